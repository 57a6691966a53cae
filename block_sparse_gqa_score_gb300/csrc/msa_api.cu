// msa_api.cu -- the extern "C" entry points declared in include/msa.h: host-side
// argument validation, per-device set-up (SM count, the device error word),
// TMA tensor-map encoding for the fp8 cache, and kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <atomic>
#include <mutex>

#include "msa.h"
#include "msa_launch.h"

// Sticky per-device error word: kernels OR MSA_ERR_* bits into it.
__device__ unsigned int msa_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 16;

struct DeviceState {
  bool ready = false;
  int sm_count = 0;
  unsigned* err = nullptr;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
// msa_set_input_overlap: whether each entry point's first kernel may start
// before the previous kernel on its stream has finished (off by default)
std::atomic<int> g_input_overlap{0};
// msa_set_union_tile: sparse decode steps of Q >= 2 over the union of each
// 4-token tile's lists (off by default; dense decode always shares pages)
std::atomic<int> g_union_tile{0};

bool input_overlap() { return g_input_overlap.load(std::memory_order_relaxed) != 0; }
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Set-up for the current device, done once: resolves the device address of the
// error word, reads the SM count and fetches the tensor-map encoder.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MSA_ECUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    void* err = nullptr;
    if (cudaGetSymbolAddress(&err, msa_error_word) != cudaSuccess) return MSA_ECUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MSA_ECUDA;
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return MSA_ECUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    st.err = static_cast<unsigned*>(err);
    st.sm_count = sms;
    st.ready = true;
  }
  *out = &st;
  return MSA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool finite_pos(float x) { return std::isfinite(x) && x > 0.f; }

// Shape checks shared by the scorer and the attend.
int check_common(const void* q, const void* kv, const int32_t* block_table,
                 const int32_t* seq_lens, int B, int Q, int Hq, int Hkv, int S,
                 int64_t num_blocks) {
  if (B < 0 || B > 65535 || Q < 1 || Q > MSA_MAX_QLEN || Hkv < 1 || Hkv > 65535 ||
      Hq != MSA_GROUP * Hkv || S < 1 || num_blocks < 1)
    return MSA_EINVAL;
  if (static_cast<int64_t>(B) * Q > INT_MAX / 4 || static_cast<int64_t>(B) * S > INT_MAX)
    return MSA_EINVAL;
  // TMA row coordinates (page * Hkv + g) * 128 must fit in int32
  if (num_blocks * Hkv * MSA_PAGE_SIZE >= (static_cast<int64_t>(1) << 31)) return MSA_EINVAL;
  if (!q || !kv || !block_table || !seq_lens) return MSA_EINVAL;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return MSA_EINVAL;
  return MSA_OK;
}

// 2-D view of the cache as [num_blocks * Hkv * 128 rows, row_bytes], read in
// 128 x 128-byte boxes (one K or V half of a page-head) with 128B swizzling.
// row_bytes is 256 for the packed K|V cache and 128 for a K-only (index-K)
// cache, whose boxes at x = 0 are then the same K tiles.  `l2_256` promotes
// L2 fills to 256 bytes (both halves of a token row, for the attend); the
// scorer reads K halves only and keeps 128-byte fills so the V halves are not
// dragged in from DRAM.
int encode_kv_map(const void* kv, int Hkv, int64_t num_blocks, CUtensorMap* map,
                  bool l2_256 = true, int row_bytes = MSA_HEAD_DIM * 2) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes),
                        static_cast<cuuint64_t>(num_blocks) * Hkv * MSA_PAGE_SIZE};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {MSA_HEAD_DIM, MSA_PAGE_SIZE};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        l2_256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                               : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MSA_OK : MSA_EINVAL;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ECUDA; }

}  // namespace

extern "C" {

int msa_version(void) { return 100; }

const char* msa_strerror(int status) {
  switch (status) {
    case MSA_OK: return "ok";
    case MSA_EINVAL: return "invalid argument (size, null or misaligned pointer)";
    case MSA_ECUDA: return "CUDA runtime error";
    case MSA_ENOSPC: return "workspace too small";
    default: return "unknown status";
  }
}

size_t msa_workspace_bytes(int B, int Q, int Hq, int num_splits) {
  if (B < 0 || Q < 1 || Hq < 1 || num_splits < 0 || num_splits > kMaxSplits) return 0;
  if (num_splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(B) * Q * Hq;
  return static_cast<size_t>(num_splits) * rows * (MSA_HEAD_DIM + 2) * sizeof(float);
}

int msa_choose_splits(int B, int Q, int Hkv, int sm_count) {
  if (B < 1 || Q < 1 || Hkv < 1 || sm_count < 1) return 1;
  if (Q >= 2 && g_union_tile.load(std::memory_order_relaxed)) {
    // the union attend: one CTA per SM per (request, 4-token tile, KV head)
    const int64_t units = static_cast<int64_t>(B) * ((Q + msa::kUnionTile - 1) / msa::kUnionTile) * Hkv;
    return msa::union_ctas_per_unit(units > INT_MAX ? INT_MAX : static_cast<int>(units), sm_count);
  }
  const int64_t units = static_cast<int64_t>(B) * Q * Hkv;  // one CTA per (token, KV head)
  const int64_t slots = 2 * static_cast<int64_t>(sm_count);  // two CTAs per SM
  if (units * 4 >= slots * 3) return 1;
  // as many splits as still fit one wave of resident CTAs
  int64_t s = slots / units;
  if (s > 8) s = 8;
  return static_cast<int>(s < 1 ? 1 : s);
}

}  // extern "C"

namespace {

// Checks and parameter block of msa_score(_kcache) and their _q8 forms:
// q_scale > 0 means q is fp8 e4m3 (value q * q_scale); k_only: kv is a K-only
// cache of 128-byte rows.  Nothing is enqueued.
int prepare_score(const void* q, float q_scale, const void* kv, const int32_t* block_table,
                  const int32_t* seq_lens, float* scores, int B, int Q, int Hq, int Hkv, int S,
                  int64_t num_blocks, float sm_scale, float k_scale, bool k_only,
                  msa::ScoreParams* p, CUtensorMap* map) {
  int st = check_common(q, kv, block_table, seq_lens, B, Q, Hq, Hkv, S, num_blocks);
  if (st != MSA_OK) return st;
  if (!scores || !aligned(scores, 4) || !finite_pos(sm_scale) || !finite_pos(k_scale) ||
      !(q_scale == 0.f || finite_pos(q_scale)))
    return MSA_EINVAL;
  if (B == 0) return MSA_OK;
  DeviceState* dev;
  if ((st = device_state(&dev)) != MSA_OK) return st;
  if ((st = encode_kv_map(kv, Hkv, num_blocks, map, /*l2_256=*/false,
                          k_only ? MSA_HEAD_DIM : 2 * MSA_HEAD_DIM)) != MSA_OK)
    return st;
  *p = msa::ScoreParams{};
  p->q = q_scale > 0.f ? nullptr : static_cast<const uint16_t*>(q);
  p->q8 = q_scale > 0.f ? static_cast<const uint8_t*>(q) : nullptr;
  p->q_scale = q_scale;
  p->block_table = block_table;
  p->seq_lens = seq_lens;
  p->scores = scores;
  p->err = dev->err;
  p->B = B;
  p->Q = Q;
  p->Hq = Hq;
  p->Hkv = Hkv;
  p->S = S;
  p->ctas = dev->sm_count;
  p->num_blocks = num_blocks;
  p->scale = sm_scale * k_scale;
  return MSA_OK;
}

int score(const void* q, float q_scale, const void* kv, const int32_t* block_table,
          const int32_t* seq_lens, float* scores, int B, int Q, int Hq, int Hkv, int S,
          int64_t num_blocks, float sm_scale, float k_scale, msa_stream_t stream,
          bool k_only = false) {
  msa::ScoreParams p;
  CUtensorMap map;
  const int st = prepare_score(q, q_scale, kv, block_table, seq_lens, scores, B, Q, Hq, Hkv, S,
                               num_blocks, sm_scale, k_scale, k_only, &p, &map);
  if (st != MSA_OK || B == 0) return st;
  return from_cuda(
      msa::launch_score(map, p, reinterpret_cast<cudaStream_t>(stream), input_overlap()));
}

}  // namespace

extern "C" {

int msa_score(const void* q, const void* kv, const int32_t* block_table, const int32_t* seq_lens,
              float* scores, int B, int Q, int Hq, int Hkv, int S, int64_t num_blocks,
              float sm_scale, float k_scale, msa_stream_t stream) {
  return score(q, 0.f, kv, block_table, seq_lens, scores, B, Q, Hq, Hkv, S, num_blocks, sm_scale,
               k_scale, stream);
}

int msa_score_q8(const void* q8, float q_scale, const void* kv, const int32_t* block_table,
                 const int32_t* seq_lens, float* scores, int B, int Q, int Hq, int Hkv, int S,
                 int64_t num_blocks, float sm_scale, float k_scale, msa_stream_t stream) {
  if (!finite_pos(q_scale)) return MSA_EINVAL;
  return score(q8, q_scale, kv, block_table, seq_lens, scores, B, Q, Hq, Hkv, S, num_blocks,
               sm_scale, k_scale, stream);
}

int msa_score_kcache(const void* q, const void* k_cache, const int32_t* block_table,
                     const int32_t* seq_lens, float* scores, int B, int Q, int Hq, int Hkv, int S,
                     int64_t num_blocks, float sm_scale, float k_scale, msa_stream_t stream) {
  return score(q, 0.f, k_cache, block_table, seq_lens, scores, B, Q, Hq, Hkv, S, num_blocks,
               sm_scale, k_scale, stream, /*k_only=*/true);
}

int msa_score_kcache_q8(const void* q8, float q_scale, const void* k_cache,
                        const int32_t* block_table, const int32_t* seq_lens, float* scores,
                        int B, int Q, int Hq, int Hkv, int S, int64_t num_blocks, float sm_scale,
                        float k_scale, msa_stream_t stream) {
  if (!finite_pos(q_scale)) return MSA_EINVAL;
  return score(q8, q_scale, k_cache, block_table, seq_lens, scores, B, Q, Hq, Hkv, S, num_blocks,
               sm_scale, k_scale, stream, /*k_only=*/true);
}

int msa_topk(const float* scores, int64_t stride_h, int64_t stride_t, int64_t stride_n,
             const int32_t* seq_lens, int32_t* topk, int B, int Q, int Hkv, int S, int k,
             msa_stream_t stream) {
  if (k != MSA_TOPK || B < 0 || Q < 1 || Q > MSA_MAX_QLEN || Hkv < 1 || S < 1) return MSA_EINVAL;
  if (static_cast<int64_t>(B) * Q * Hkv > INT_MAX / 2) return MSA_EINVAL;
  if (!scores || !seq_lens || !topk || !aligned(scores, 4) || !aligned(seq_lens, 4) ||
      !aligned(topk, 4))
    return MSA_EINVAL;
  if (B == 0) return MSA_OK;
  DeviceState* dev;
  int st = device_state(&dev);
  if (st != MSA_OK) return st;
  msa::TopkParams p{};
  p.scores = scores;
  p.stride_h = stride_h;
  p.stride_t = stride_t;
  p.stride_n = stride_n;
  p.seq_lens = seq_lens;
  p.topk = topk;
  p.err = dev->err;
  p.B = B;
  p.Q = Q;
  p.Hkv = Hkv;
  p.S = S;
  return from_cuda(msa::launch_topk(p, reinterpret_cast<cudaStream_t>(stream), input_overlap()));
}

int msa_combine(const void* workspace, void* out, int T, int Hq, int num_splits,
                msa_stream_t stream) {
  if (T < 0 || Hq < 1 || num_splits < 1 || num_splits > kMaxSplits) return MSA_EINVAL;
  if (!workspace || !out || !aligned(workspace, 16) || !aligned(out, 16)) return MSA_EINVAL;
  if (T == 0) return MSA_OK;
  const int64_t rows = static_cast<int64_t>(T) * Hq;
  const float* part_o = static_cast<const float*>(workspace);
  const float* part_ml = part_o + static_cast<int64_t>(num_splits) * rows * MSA_HEAD_DIM;
  return from_cuda(msa::launch_combine(part_o, part_ml, static_cast<uint16_t*>(out), rows,
                                       num_splits, reinterpret_cast<cudaStream_t>(stream),
                                       input_overlap()));
}

}  // extern "C"

namespace {

// Dense decode's split of a row's S blocks: up to 16 CTAs, each over a range
// of at most 128 consecutive blocks (a CTA's page list holds 128).
constexpr int kDenseMaxSpan = 128;

void dense_split(int S, int* nsplit, int* span) {
  const int groups = (S + MSA_TOPK - 1) / MSA_TOPK;  // 16-block groups
  *nsplit = groups < 1 ? 1 : (groups > kMaxSplits ? kMaxSplits : groups);
  *span = (S + *nsplit - 1) / *nsplit;
}

// An attend launch, checked and ready to enqueue.
struct AttendLaunch {
  msa::AttendParams p;
  CUtensorMap map;
  int64_t rows;  // output rows (tokens x query heads)
};

// Checks and parameter block of msa_sparse_decode, msa_sparse_decode_select and
// msa_dense_decode: `scores` null means `topk` is the input list; otherwise the
// lists are selected from the strided scores inside the attend kernel and
// written to `topk`.  dense_span > 0: no list, every visible block
// (msa_dense_decode).  cu_q non-null: a prefill-style batch of T tokens,
// request b owning tokens [cu_q[b], cu_q[b + 1]) (msa_sparse_prefill); Q is
// then unused.  Nothing is enqueued; *empty is set when there is no work.
int prepare_attend(const void* q, const void* kv, const int32_t* block_table,
                   const int32_t* seq_lens, const float* scores, int64_t stride_h,
                   int64_t stride_t, int64_t stride_n, int32_t* topk, void* workspace,
                   size_t workspace_bytes, void* out, int B, int Q, int Hq, int Hkv, int S,
                   int64_t num_blocks, float sm_scale, float k_scale, float v_scale,
                   int num_splits, int dense_span, float q_scale, const int32_t* cu_q, int T,
                   AttendLaunch* L, bool* empty) {
  *empty = true;
  if (!(q_scale == 0.f || finite_pos(q_scale))) return MSA_EINVAL;
  if (cu_q) {
    // the token count takes the place of B * Q in every size below
    if (dense_span != 0 || !aligned(cu_q, 4) || T < 0 || T > INT_MAX / 4 || (B == 0) != (T == 0))
      return MSA_EINVAL;
    if (T == 0) return B == 0 ? MSA_OK : MSA_EINVAL;
  }
  int st = check_common(q, kv, block_table, seq_lens, B, cu_q ? 1 : Q, Hq, Hkv, S, num_blocks);
  if (st != MSA_OK) return st;
  if (dense_span == 0 && (!topk || !aligned(topk, 4))) return MSA_EINVAL;
  if (!out || !aligned(out, 16) || !finite_pos(sm_scale) ||
      !finite_pos(k_scale) || !std::isfinite(v_scale) || num_splits < 0 ||
      num_splits > kMaxSplits)
    return MSA_EINVAL;
  if (scores && (!aligned(scores, 4) || stride_h < 0 || stride_t < 0 || stride_n < 0))
    return MSA_EINVAL;
  if (B == 0) return MSA_OK;
  DeviceState* dev;
  if ((st = device_state(&dev)) != MSA_OK) return st;
  // sizes over tokens: B requests of Q, or T tokens of a prefill-style batch
  const int tb = cu_q ? 1 : B, tq = cu_q ? T : Q;
  // the union attend: dense decode, or sparse decode when the union mode is on,
  // with two or more tokens per request
  const bool union_tile = !cu_q && Q >= 2 &&
                          (dense_span > 0 || g_union_tile.load(std::memory_order_relaxed) != 0);
  // prefill batches (one CTA per token): the single-token rule, msa_choose_splits(T, 1, ...)
  int splits = num_splits != 0 ? num_splits
               : cu_q ? msa_choose_splits(T, 1, Hkv, dev->sm_count)
                      : msa_choose_splits(B, Q, Hkv, dev->sm_count);
  if (union_tile && dense_span > 0) {
    // dense decode over the union.  Units that fill the SMs: one CTA each.
    // Fewer: one CTA per SM, shared out by the units' blocks (the union
    // launcher and kernel), up to the caller's split count (which sized the
    // workspace) per unit.
    const int64_t units = static_cast<int64_t>(B) * ((Q + msa::kUnionTile - 1) / msa::kUnionTile) * Hkv;
    if (units >= dev->sm_count) splits = 1;
  }
  const size_t need = msa_workspace_bytes(tb, tq, Hq, splits);
  if (splits > 1 && (!workspace || !aligned(workspace, 16) || workspace_bytes < need))
    return MSA_ENOSPC;
  if ((st = encode_kv_map(kv, Hkv, num_blocks, &L->map)) != MSA_OK) return st;
  const int64_t rows = static_cast<int64_t>(tb) * tq * Hq;
  msa::AttendParams& p = L->p;
  p = msa::AttendParams{};
  p.q = q_scale > 0.f ? nullptr : static_cast<const uint16_t*>(q);
  p.q8 = q_scale > 0.f ? static_cast<const uint8_t*>(q) : nullptr;
  p.q_scale = q_scale;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.topk = topk;
  p.scores = scores;
  p.s_stride_h = stride_h;
  p.s_stride_t = stride_t;
  p.s_stride_n = stride_n;
  p.topk_out = scores ? topk : nullptr;
  p.dense_span = dense_span;
  p.part_o = splits > 1 ? static_cast<float*>(workspace) : nullptr;
  p.part_ml = splits > 1 ? static_cast<float*>(workspace) + splits * rows * MSA_HEAD_DIM : nullptr;
  p.out = static_cast<uint16_t*>(out);
  p.err = dev->err;
  p.B = B;
  p.Q = Q;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.S = S;
  p.splits = splits;
  p.num_blocks = num_blocks;
  p.logit_scale = sm_scale * k_scale * 1.4426950408889634f;
  p.v_scale = v_scale;
  p.cu_q = cu_q;
  p.T = cu_q ? T : 0;
  p.union_tile = union_tile ? 1 : 0;
  L->rows = rows;
  *empty = false;
  return MSA_OK;
}

// Enqueues a prepared attend (+ the split merge); `pdl` for the attend kernel
// (the merge always follows it with programmatic serialization).
int enqueue_attend(const AttendLaunch& L, cudaStream_t s, bool pdl) {
  int st;
  if ((st = from_cuda(msa::launch_attend(L.map, L.p, s, pdl))) != MSA_OK) return st;
  if (L.p.splits > 1)
    return from_cuda(
        msa::launch_combine(L.p.part_o, L.p.part_ml, L.p.out, L.rows, L.p.splits, s, true));
  return MSA_OK;
}

int sparse_decode(const void* q, const void* kv, const int32_t* block_table,
                  const int32_t* seq_lens, const float* scores, int64_t stride_h,
                  int64_t stride_t, int64_t stride_n, int32_t* topk, void* workspace,
                  size_t workspace_bytes, void* out, int B, int Q, int Hq, int Hkv, int S,
                  int64_t num_blocks, float sm_scale, float k_scale, float v_scale,
                  int num_splits, msa_stream_t stream, int dense_span = 0, float q_scale = 0.f,
                  const int32_t* cu_q = nullptr, int T = 0) {
  AttendLaunch L;
  bool empty;
  const int st = prepare_attend(q, kv, block_table, seq_lens, scores, stride_h, stride_t, stride_n,
                                topk, workspace, workspace_bytes, out, B, Q, Hq, Hkv, S,
                                num_blocks, sm_scale, k_scale, v_scale, num_splits, dense_span,
                                q_scale, cu_q, T, &L, &empty);
  if (st != MSA_OK || empty) return st;
  return enqueue_attend(L, reinterpret_cast<cudaStream_t>(stream), input_overlap());
}

}  // namespace

extern "C" {

int msa_sparse_decode(const void* q, const void* kv, const int32_t* block_table,
                      const int32_t* seq_lens, const int32_t* topk, void* workspace,
                      size_t workspace_bytes, void* out, int B, int Q, int Hq, int Hkv, int S,
                      int64_t num_blocks, float sm_scale, float k_scale, float v_scale,
                      int num_splits, msa_stream_t stream) {
  return sparse_decode(q, kv, block_table, seq_lens, nullptr, 0, 0, 0, const_cast<int32_t*>(topk),
                       workspace, workspace_bytes, out, B, Q, Hq, Hkv, S, num_blocks, sm_scale,
                       k_scale, v_scale, num_splits, stream);
}

int msa_sparse_decode_select(const void* q, const void* kv, const int32_t* block_table,
                             const int32_t* seq_lens, const float* scores, int64_t stride_h,
                             int64_t stride_t, int64_t stride_n, int32_t* topk, void* workspace,
                             size_t workspace_bytes, void* out, int B, int Q, int Hq, int Hkv,
                             int S, int64_t num_blocks, float sm_scale, float k_scale,
                             float v_scale, int num_splits, msa_stream_t stream) {
  if (!scores) return MSA_EINVAL;
  return sparse_decode(q, kv, block_table, seq_lens, scores, stride_h, stride_t, stride_n, topk,
                       workspace, workspace_bytes, out, B, Q, Hq, Hkv, S, num_blocks, sm_scale,
                       k_scale, v_scale, num_splits, stream);
}

// The fp8-query variants: q8 is fp8 e4m3 [T, Hq, 128] whose value is q8 *
// q_scale; everything else as the bf16 entry points.
int msa_sparse_decode_q8(const void* q8, float q_scale, const void* kv,
                         const int32_t* block_table, const int32_t* seq_lens, const int32_t* topk,
                         void* workspace, size_t workspace_bytes, void* out, int B, int Q, int Hq,
                         int Hkv, int S, int64_t num_blocks, float sm_scale, float k_scale,
                         float v_scale, int num_splits, msa_stream_t stream) {
  if (!finite_pos(q_scale)) return MSA_EINVAL;
  return sparse_decode(q8, kv, block_table, seq_lens, nullptr, 0, 0, 0, const_cast<int32_t*>(topk),
                       workspace, workspace_bytes, out, B, Q, Hq, Hkv, S, num_blocks, sm_scale,
                       k_scale, v_scale, num_splits, stream, 0, q_scale);
}

int msa_sparse_decode_select_q8(const void* q8, float q_scale, const void* kv,
                                const int32_t* block_table, const int32_t* seq_lens,
                                const float* scores, int64_t stride_h, int64_t stride_t,
                                int64_t stride_n, int32_t* topk, void* workspace,
                                size_t workspace_bytes, void* out, int B, int Q, int Hq, int Hkv,
                                int S, int64_t num_blocks, float sm_scale, float k_scale,
                                float v_scale, int num_splits, msa_stream_t stream) {
  if (!finite_pos(q_scale) || !scores) return MSA_EINVAL;
  return sparse_decode(q8, kv, block_table, seq_lens, scores, stride_h, stride_t, stride_n, topk,
                       workspace, workspace_bytes, out, B, Q, Hq, Hkv, S, num_blocks, sm_scale,
                       k_scale, v_scale, num_splits, stream, 0, q_scale);
}

int msa_dense_splits(int S) {
  if (S < 1) return 0;
  int nsplit, span;
  dense_split(S, &nsplit, &span);
  return span > kDenseMaxSpan ? 0 : nsplit;
}

int msa_dense_decode(const void* q, const void* kv, const int32_t* block_table,
                     const int32_t* seq_lens, void* workspace, size_t workspace_bytes, void* out,
                     int B, int Q, int Hq, int Hkv, int S, int64_t num_blocks, float sm_scale,
                     float k_scale, float v_scale, msa_stream_t stream) {
  if (msa_dense_splits(S) == 0) return MSA_EINVAL;
  int nsplit, span;
  dense_split(S, &nsplit, &span);
  return sparse_decode(q, kv, block_table, seq_lens, nullptr, 0, 0, 0, nullptr, workspace,
                       workspace_bytes, out, B, Q, Hq, Hkv, S, num_blocks, sm_scale, k_scale,
                       v_scale, nsplit, stream, span);
}

int msa_dense_decode_q8(const void* q8, float q_scale, const void* kv,
                        const int32_t* block_table, const int32_t* seq_lens, void* workspace,
                        size_t workspace_bytes, void* out, int B, int Q, int Hq, int Hkv, int S,
                        int64_t num_blocks, float sm_scale, float k_scale, float v_scale,
                        msa_stream_t stream) {
  if (msa_dense_splits(S) == 0 || !finite_pos(q_scale)) return MSA_EINVAL;
  int nsplit, span;
  dense_split(S, &nsplit, &span);
  return sparse_decode(q8, kv, block_table, seq_lens, nullptr, 0, 0, 0, nullptr, workspace,
                       workspace_bytes, out, B, Q, Hq, Hkv, S, num_blocks, sm_scale, k_scale,
                       v_scale, nsplit, stream, span, q_scale);
}

// Prefill and chunked prefill: B requests, request b's query tokens being
// [cu_seqlens_q[b], cu_seqlens_q[b + 1]) of the T tokens, at the last positions
// of its seq_lens[b].  Same lists, numerics and errors as msa_sparse_decode.
int msa_sparse_prefill(const void* q, const void* kv, const int32_t* block_table,
                       const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                       const int32_t* topk, void* workspace, size_t workspace_bytes, void* out,
                       int B, int T, int Hq, int Hkv, int S, int64_t num_blocks, float sm_scale,
                       float k_scale, float v_scale, int num_splits, msa_stream_t stream) {
  if (!cu_seqlens_q) return MSA_EINVAL;
  return sparse_decode(q, kv, block_table, seq_lens, nullptr, 0, 0, 0, const_cast<int32_t*>(topk),
                       workspace, workspace_bytes, out, B, 1, Hq, Hkv, S, num_blocks, sm_scale,
                       k_scale, v_scale, num_splits, stream, 0, 0.f, cu_seqlens_q, T);
}

int msa_sparse_prefill_q8(const void* q8, float q_scale, const void* kv,
                          const int32_t* block_table, const int32_t* seq_lens,
                          const int32_t* cu_seqlens_q, const int32_t* topk, void* workspace,
                          size_t workspace_bytes, void* out, int B, int T, int Hq, int Hkv, int S,
                          int64_t num_blocks, float sm_scale, float k_scale, float v_scale,
                          int num_splits, msa_stream_t stream) {
  if (!cu_seqlens_q || !finite_pos(q_scale)) return MSA_EINVAL;
  return sparse_decode(q8, kv, block_table, seq_lens, nullptr, 0, 0, 0, const_cast<int32_t*>(topk),
                       workspace, workspace_bytes, out, B, 1, Hq, Hkv, S, num_blocks, sm_scale,
                       k_scale, v_scale, num_splits, stream, 0, q_scale, cu_seqlens_q, T);
}

int msa_sparse_prefill_select(const void* q, const void* kv, const int32_t* block_table,
                              const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                              const float* scores, int64_t stride_h, int64_t stride_t,
                              int64_t stride_n, int32_t* topk, void* workspace,
                              size_t workspace_bytes, void* out, int B, int T, int Hq, int Hkv,
                              int S, int64_t num_blocks, float sm_scale, float k_scale,
                              float v_scale, int num_splits, msa_stream_t stream) {
  if (!cu_seqlens_q || !scores) return MSA_EINVAL;
  return sparse_decode(q, kv, block_table, seq_lens, scores, stride_h, stride_t, stride_n, topk,
                       workspace, workspace_bytes, out, B, 1, Hq, Hkv, S, num_blocks, sm_scale,
                       k_scale, v_scale, num_splits, stream, 0, 0.f, cu_seqlens_q, T);
}

int msa_sparse_prefill_select_q8(const void* q8, float q_scale, const void* kv,
                                 const int32_t* block_table, const int32_t* seq_lens,
                                 const int32_t* cu_seqlens_q, const float* scores,
                                 int64_t stride_h, int64_t stride_t, int64_t stride_n,
                                 int32_t* topk, void* workspace, size_t workspace_bytes,
                                 void* out, int B, int T, int Hq, int Hkv, int S,
                                 int64_t num_blocks, float sm_scale, float k_scale, float v_scale,
                                 int num_splits, msa_stream_t stream) {
  if (!cu_seqlens_q || !scores || !finite_pos(q_scale)) return MSA_EINVAL;
  return sparse_decode(q8, kv, block_table, seq_lens, scores, stride_h, stride_t, stride_n, topk,
                       workspace, workspace_bytes, out, B, 1, Hq, Hkv, S, num_blocks, sm_scale,
                       k_scale, v_scale, num_splits, stream, 0, q_scale, cu_seqlens_q, T);
}

// One decode step: the scorer, then the selection and the attend.  Rows of at
// most kFusedMaxBlocks candidate blocks are selected inside the attend kernel
// (msa_sparse_decode_select); longer rows by the selector kernel, whose
// register paths hold up to 2048 candidates, then msa_sparse_decode.  The
// first kernel follows the input-overlap setting; the others follow a library
// kernel and may overlap it.
int msa_decode_step(const void* q, float q_scale, const void* kv, const void* index_k,
                    float index_k_scale, const int32_t* block_table, const int32_t* seq_lens,
                    float* scores, int32_t* topk, void* workspace, size_t workspace_bytes,
                    void* out, int B, int Q, int Hq, int Hkv, int S, int64_t num_blocks,
                    float sm_scale, float k_scale, float v_scale, int num_splits,
                    msa_stream_t stream) {
  constexpr int kFusedMaxBlocks = 512;
  if (!(q_scale == 0.f || finite_pos(q_scale))) return MSA_EINVAL;
  if (index_k && !finite_pos(index_k_scale)) return MSA_EINVAL;
  if (static_cast<int64_t>(B) * Q * Hkv > INT_MAX / 2) return MSA_EINVAL;
  msa::ScoreParams sp;
  CUtensorMap smap;
  int st = prepare_score(q, q_scale, index_k ? index_k : kv, block_table, seq_lens, scores, B, Q,
                         Hq, Hkv, S, num_blocks, sm_scale, index_k ? index_k_scale : k_scale,
                         index_k != nullptr, &sp, &smap);
  if (st != MSA_OK) return st;
  const bool fused = S <= kFusedMaxBlocks;
  const int64_t T = static_cast<int64_t>(B) * Q;
  AttendLaunch L;
  bool empty;
  // the scores buffer [Hkv, T, S], block dim contiguous
  st = prepare_attend(q, kv, block_table, seq_lens, fused ? scores : nullptr, T * S, S, 1, topk,
                      workspace, workspace_bytes, out, B, Q, Hq, Hkv, S, num_blocks, sm_scale,
                      k_scale, v_scale, num_splits, 0, q_scale, nullptr, 0, &L, &empty);
  if (st != MSA_OK || empty || B == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = from_cuda(msa::launch_score(smap, sp, s, input_overlap()))) != MSA_OK) return st;
  if (!fused) {
    msa::TopkParams tp{};
    tp.scores = scores;
    tp.stride_h = T * S;
    tp.stride_t = S;
    tp.stride_n = 1;
    tp.seq_lens = seq_lens;
    tp.topk = topk;
    tp.err = sp.err;
    tp.B = B;
    tp.Q = Q;
    tp.Hkv = Hkv;
    tp.S = S;
    if ((st = from_cuda(msa::launch_topk(tp, s, true))) != MSA_OK) return st;
  }
  return enqueue_attend(L, s, true);
}

int msa_test_wait_timeout(unsigned long long limit_ns, msa_stream_t stream) {
  if (limit_ns < 1000ull || limit_ns > 2000000000ull) return MSA_EINVAL;
  DeviceState* dev;
  const int st = device_state(&dev);
  if (st != MSA_OK) return st;
  return from_cuda(
      msa::launch_wait_timeout(limit_ns, dev->err, reinterpret_cast<cudaStream_t>(stream)));
}

int msa_set_union_tile(int enable) {
  return g_union_tile.exchange(enable ? 1 : 0, std::memory_order_relaxed);
}

int msa_set_input_overlap(int enable) {
  return g_input_overlap.exchange(enable ? 1 : 0, std::memory_order_relaxed);
}

int msa_get_error(unsigned int* flags, int clear) {
  DeviceState* dev;
  int st = device_state(&dev);
  if (st != MSA_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return MSA_ECUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, dev->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MSA_ECUDA;
  if (flags) *flags = v;
  if (clear) {
    const unsigned zero = 0;
    if (cudaMemcpy(dev->err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return MSA_ECUDA;
  }
  return MSA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of msa_sparse_decode.
//
// Some callers cannot allocate device memory at all: a plugin or operator
// interface that hands the library only the step's input and output buffers
// and gives it no workspace, or a runtime that forbids cudaMalloc on its hot
// path because an allocation can block on the whole device or fail under
// memory pressure.  For them the split-K partials live in one fixed scratch
// array compiled into the library.  Every GPU that loads the library holds
// this array until the process exits, so its size is kept modest.

static __device__ __align__(256) unsigned char msa_static_scratch[MSA_STATIC_SCRATCH_BYTES];

namespace {

std::mutex g_static_mutex;
void* g_static_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The array's name
// is only a host-side stand-in in host code, so the address is looked up once
// per device (with that device current) and cached.
int static_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MSA_ECUDA;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (!g_static_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, msa_static_scratch) != cudaSuccess || !ptr) return MSA_ECUDA;
    g_static_scratch_ptr[dev] = ptr;
  }
  *out = g_static_scratch_ptr[dev];
  return MSA_OK;
}

}  // namespace

extern "C" int msa_sparse_decode_static(const void* q, const void* kv,
                                        const int32_t* block_table, const int32_t* seq_lens,
                                        const int32_t* topk, void* out, int B, int Q, int Hq,
                                        int Hkv, int S, int64_t num_blocks, float sm_scale,
                                        float k_scale, float v_scale, int num_splits,
                                        msa_stream_t stream) {
  int splits = num_splits;
  if (splits == 0 && B >= 1 && Q >= 1 && Hkv >= 1) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MSA_ECUDA;
    splits = msa_choose_splits(B, Q, Hkv, sms);
  }
  const size_t need = msa_workspace_bytes(B, Q, Hq, splits);
  if (need > MSA_STATIC_SCRATCH_BYTES) return MSA_ENOSPC;
  void* scratch = nullptr;
  if (need > 0) {
    const int st = static_scratch_address(&scratch);
    if (st != MSA_OK) return st;
  }
  // Same validation and kernels as msa_sparse_decode; the partials go to the
  // static array instead of a caller-provided workspace.
  return msa_sparse_decode(q, kv, block_table, seq_lens, topk, scratch,
                           need > 0 ? static_cast<size_t>(MSA_STATIC_SCRATCH_BYTES) : 0, out, B,
                           Q, Hq, Hkv, S, num_blocks, sm_scale, k_scale, v_scale, splits, stream);
}
