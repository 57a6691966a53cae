// msa_attend.cu -- stage 3 (sparse attend) and stage 4 (split merge).
//
// Operation: minimax_m3_sparse_attn_decode / msa_cutlass_sparse_decode on the
// vLLM MiniMax-M3 pages: each query row attends only the tokens of the <= 16
// blocks its KV head's top-k list names, causally limited to pos = seq_len -
// Q + j; padding rows come out as zeros rather than NaN, and split parts are
// merged from fp32 partials (TensorRT-LLM PR #17171, flash-decoding commit).
//
// Design (sm_103a, tcgen05): one CTA per (query token, KV head, split).  The
// token's 16 query heads are the N = 16 columns of two tensor-core products
// taken transposed, so that the page's 128 keys, then its 128 value dims, fill
// the M = 128 rows of the MMA:
//   S^T = K Q^T    A = the fp8 K tile straight from the TMA stage (K-major);
//                  B = the query, scaled by a power of two and split exactly
//                  into fp8 e4m3 hi and lo parts, side by side as N = 32
//   O^T = V^T P^T  A = the fp8 V tile of the same stage, read MN-major, i.e.
//                  as stored; B = the probabilities split into e4m3 hi and lo
//                  parts, again side by side as N = 32
// both kind::f8f6f4 with fp32 accumulators in tensor memory (the softmax
// threads add the hi and lo columns), so no fp8 value is widened in
// registers and a page takes 4 + 4 MMAs.  Warp roles:
//   0    TMA producer: each selected page-head (K and V halves, 32 KiB) into a
//        3-stage ring of 128B-swizzled tiles;
//   1    issues S^T (and owns tensor memory); 2 issues O^T;
//   3-6  softmax.  A thread owns one key of the page (one TMEM lane of S^T):
//        the page's per-head maxima come from warp reductions and a
//        four-warp exchange; the reference m of a head moves only when a page
//        exceeds it by more than half a binade, so P = 2^(x - m + 8) stays
//        below 2^8.5 (the e4m3 range keeps 17 binades below it) and the
//        rescale factors are 1 on most pages; each thread keeps its share of
//        the running sums.  When a page's O^T is ready the same
//        thread owns one value dim d (one TMEM lane of O^T) and accumulates
//        O = O * alpha + O_page in registers, so O is never rescaled in place.
// The CTA's page list is the top-k list (given, or selected in the prologue
// from the block scores: select mode), or in dense decode (the TensorRT-LLM PR
// dense-decode commit: the first layers attend the whole page table) a range
// of consecutive visible blocks.  An fp8 query (value q8 * q_scale, as
// msa_cutlass_sparse_decode takes it) goes into the hi part as stored, with a
// zero lo part.  Prefill batches (one query length per request, cu_seqlens_q)
// map each token to its request by a warp-wide search and then run as decode
// tokens.  Dense decode, the fp8 query and prefill batches are template
// flags, so the bf16 list-mode decode kernel carries none of their branches.
#include "msa_device.cuh"
#include "msa_launch.h"
#include "msa_select.cuh"
#include "msa_tcgen05.cuh"

namespace msa {

namespace {

constexpr int kStages = 3;
constexpr int kWarps = 7;
constexpr int kThreads = kWarps * 32;
constexpr int kSoftmaxWarp0 = 3;              // warps 3..6; warp w reads TMEM lanes 32*(w%4)..
constexpr int kStageBytes = 2 * kHalfTile;    // K tile then V tile
constexpr int kQPart = kGroup * 128;          // one fp8 part of the query tile: 16 rows x 128 B
constexpr int kPPart = kPage * kGroup;        // one fp8 part of P^T: 128 keys x 16 heads
// P^T buffer: per block of 8 keys, the hi part's 8 x 16 B core matrix, then
// the lo part's (256 B per block, 2 * kPPart per buffer)
constexpr int kPBlock = 256;
constexpr int kTmemCols = 128;                // S^T x 2 buffers, O^T x 2 buffers, 32 columns each
constexpr uint32_t kColS = 0, kColO = 64;
constexpr float kPShift = 8.f;                // P = 2^(x - m + kPShift)
constexpr float kLazy = 0.5f;                 // m moves when a page exceeds it by more than this
// Prologue scratch in the stage ring, before its first loads (stage 0 may
// already be loading the current block's page): stage 1 holds the selector's
// keys and slots (select mode), stage 2 a copy of the request's block-table
// row (its first kTableCopy entries; later blocks are read from global memory).
constexpr int kSelectCap = 8000;              // keys cached (31.25 KiB), then the slots
constexpr int kMaxPages = 128;                // pages of one CTA (dense decode; a list has 16)
constexpr int kTableCopy = 512;               // 16 loads per lane, all in flight together

struct AttendTail {
  uint64_t full[kStages];   // TMA -> S^T issuer
  uint64_t empty[kStages];  // O^T issuer (stage's last reader) -> TMA
  uint64_t s_full[2];       // S^T ready -> softmax
  uint64_t s_empty[2];      // softmax has read S^T -> S^T issuer
  uint64_t p_full[2];       // P^T written -> O^T issuer
  uint64_t o_full[2];       // O^T ready -> softmax
  uint64_t o_empty[2];      // softmax has read O^T -> O^T issuer
  uint64_t mx_full[2];      // the four softmax warps' page maxima written
  uint64_t l_full;          // the four softmax warps' running sums written
  uint64_t finish;          // every role done and every MMA complete
  uint32_t tmem_base;
  int n_pages, pos;
  float zs;                 // logit scale (log2 units) times 2^e of the query split
  int pages[kMaxPages];
  int blocks[kMaxPages];
};

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr int kOffQ = kStages * kStageBytes;        // query hi, lo
constexpr int kOffP = kOffQ + 2 * kQPart;           // P^T [2 buffers], see kPBlock
constexpr int kOffMx = kOffP + 4 * kPPart;          // page maxima [2][4 warps][16]
constexpr int kOffL = kOffMx + 2 * 4 * kGroup * 4;  // running sums [4 warps][16]
constexpr int kOffTail = kOffL + 4 * kGroup * 4;
constexpr int kSmemBytes = kOffTail + static_cast<int>((sizeof(AttendTail) + 15) / 16 * 16) + 1024;
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "operand tiles need 1024-byte alignment");
static_assert(4 * kSelectCap + 4 * kTopK <= kStageBytes, "selector scratch fits stage 1");
static_assert(kStages >= 3, "prologue scratch uses stages 1 and 2");
static_assert(4 * kTableCopy <= kStageBytes && kTableCopy % 32 == 0, "block-table copy fits stage 2");
static_assert(kOffTail % 16 == 0, "mbarriers need 8-byte alignment");

template <int N>
__device__ __forceinline__ void fill(float (&a)[N], float v) {
#pragma unroll
  for (int k = 0; k < N; ++k) a[k] = v;
}

// Request of query token i in a variable-length batch whose request r owns
// tokens [cu_q[r], cu_q[r + 1]): b is the number of requests that end at or
// before i, found by a 32-way search across the warp (each round probes 32
// evenly spaced request ends and keeps the sub-range where the prefix of ends
// <= i stops).  Every probe reads cu_q[1..B].  Returns false, with b = 0, when
// token i lies in no request's range (cu_q not ascending, or i outside
// [cu_q[0], cu_q[B])); otherwise b, the token's offset j and the request's
// query length.  Warp-uniform arguments; all 32 lanes call it.
__device__ __forceinline__ bool varlen_token(const int32_t* __restrict__ cu_q, int B, int i,
                                             int lane, int& b, int& j, int& qlen) {
  int lo = 0, hi = B;
  while (lo < hi) {
    const int step = (hi - lo + 31) >> 5;
    const int r = lo + (lane + 1) * step - 1;
    const bool before = r < hi && cu_q[r + 1] <= i;
    const int k = __popc(__ballot_sync(0xffffffffu, before));
    lo += k * step;
    hi = min(hi, lo + step - 1);
  }
  b = 0;
  j = 0;
  qlen = 1;
  if (lo >= B) return false;
  const int start = cu_q[lo], end = cu_q[lo + 1];
  if (i < start || i >= end) return false;
  b = lo;
  j = i - start;
  qlen = end - start;
  return true;
}

// kDense: dense decode (every visible block of the CTA's range, no list);
// kFp8Q: an fp8 query (q8 * q_scale); kVarlen: prefill-style batches, one
// query length per request (cu_q), grid.x = T tokens.  Each is compiled
// separately so that the bf16 list-mode decode kernel carries none of their
// branches.
template <bool kDense, bool kFp8Q, bool kVarlen = false, bool kListsOnly = false>
__global__ void __launch_bounds__(kThreads, 2)
    attend_kernel(const __grid_constant__ CUtensorMap kv_map, const AttendParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  AttendTail* tail = reinterpret_cast<AttendTail*>(smem + kOffTail);
  uint8_t* qhi = smem + kOffQ;
  uint8_t* qlo = qhi + kQPart;
  uint8_t* pbuf = smem + kOffP;
  float* mx = reinterpret_cast<float*>(smem + kOffMx);
  float* lsum = reinterpret_cast<float*>(smem + kOffL);

  const int i = blockIdx.x;      // query token
  const int g = blockIdx.y;      // KV head
  const int split = blockIdx.z;  // split-K part
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- prologue ------------------------------------------------------------------
  if (warp == 0) {
    // the token's request b, its offset j there and the request's query length
    int b, j, qlen;
    bool tok_ok = true;
    if constexpr (kVarlen) {
      tok_ok = varlen_token(p.cu_q, p.B, i, lane, b, j, qlen);
    } else {
      b = i / p.Q;
      j = i - b * p.Q;
      qlen = p.Q;
    }
    // this CTA's page list, barriers, and the first loads.  The request's
    // block-table row goes into stage 2 while seq_lens is read: every lane
    // has all its loads in flight at once, so the row costs one round trip.
    int32_t* table_s = reinterpret_cast<int32_t*>(smem + 2 * kStageBytes);
    const int32_t* trow = p.block_table + static_cast<int64_t>(b) * p.S;
    const int ncopy = p.S < kTableCopy ? p.S : kTableCopy;
    const int L = p.seq_lens[b];
    {
      int32_t v[kTableCopy / 32];
#pragma unroll
      for (int k = 0; k < kTableCopy / 32; ++k) v[k] = 32 * k + lane < ncopy ? trow[32 * k + lane] : 0;
#pragma unroll
      for (int k = 0; k < kTableCopy / 32; ++k)
        if (32 * k + lane < ncopy) table_s[32 * k + lane] = v[k];
    }
    __syncwarp();
    // a prefill request's tokens are the last qlen of its sequence: the
    // context before them (L - qlen) cannot be negative
    const bool seq_ok = tok_ok && L >= 0 && (L == 0 || (L - 1) / kPage < p.S) &&
                        (!kVarlen || L >= qlen);
    if (!seq_ok && lane == 0) flag_error(p.err, MSA_ERR_SEQ_RANGE);
    const int pos = seq_ok ? L - qlen + j : -1;
    const int64_t list = (static_cast<int64_t>(i) * p.Hkv + g) * kTopK;
    // The current block comes first in a CTA's page order when it is listed
    // (split 0 then owns it), and it always is in select mode and in the
    // selector's lists.  Its page depends on inputs only, so it is loaded into
    // stage 0 before waiting for the previous kernel; a given list without it
    // costs one discarded load.
    const int cur = pos >= 0 ? pos / kPage : -1;
    // the CTA whose list starts with the current block: split 0 of a list,
    // the split whose block range holds it in dense decode
    const int cur_split = kDense ? (cur >= 0 ? cur / p.dense_span : -1) : 0;
    int cur_page = -1;
    if (cur >= 0 && split == cur_split) {
      const int pg = cur < ncopy ? table_s[cur] : trow[cur];
      if (pg >= 0 && static_cast<int64_t>(pg) < p.num_blocks) cur_page = pg;
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(&tail->full[s], 1);
        mbar_init(&tail->empty[s], 1);
      }
      for (int s = 0; s < 2; ++s) {
        mbar_init(&tail->s_full[s], 1);
        mbar_init(&tail->s_empty[s], 4);
        mbar_init(&tail->p_full[s], 4);
        mbar_init(&tail->o_full[s], 1);
        mbar_init(&tail->o_empty[s], 4);
        mbar_init(&tail->mx_full[s], 4);
      }
      mbar_init(&tail->l_full, 4);
      mbar_init(&tail->finish, kWarps);
      fence_barrier_init();
      prefetch_tensormap(&kv_map);
      if (cur_page >= 0) {
        const int row = (cur_page * p.Hkv + g) * kPage;
        mbar_arrive_expect_tx(&tail->full[0], kStageBytes);
        tma_load_2d(smem, &kv_map, 0, row, &tail->full[0]);
        tma_load_2d(smem + kHalfTile, &kv_map, kHeadDim, row, &tail->full[0]);
      }
    }
    int np = 0;               // this CTA's pages
    bool mine_front = false;  // its page 0 is the current block (stage 0 may hold it)
    if constexpr (kDense) {
      // dense decode: blocks [lo, hi) of the row, the current block first,
      // then ascending; nothing here comes from the previous kernel
      const int lo = split * p.dense_span;
      const int hi = min(lo + p.dense_span, cur + 1);
      if (cur >= lo && cur < hi) {
        if (cur_page >= 0) {
          if (lane == 0) {
            tail->pages[0] = cur_page;
            tail->blocks[0] = cur;
          }
          np = 1;
          mine_front = true;
        } else if (lane == 0) {
          flag_error(p.err, MSA_ERR_PAGE_RANGE);
        }
      }
      for (int base = lo; base < hi; base += 32) {
        const int n = base + lane;
        bool valid = n < hi && n != cur;
        int page = -1;
        if (valid) {
          page = n < ncopy ? table_s[n] : trow[n];
          if (page < 0 || static_cast<int64_t>(page) >= p.num_blocks) {
            flag_error(p.err, MSA_ERR_PAGE_RANGE);
            valid = false;
          }
        }
        const unsigned vm = __ballot_sync(0xffffffffu, valid);
        if (valid) {
          const int k = np + __popc(vm & ((1u << lane) - 1u));
          tail->pages[k] = page;
          tail->blocks[k] = n;
        }
        np += __popc(vm);
      }
    } else {
      pdl_wait();  // the top-k lists, or the scores they come from, are the previous kernel's
      int n;
      if (!kListsOnly && p.scores) {
        // select this row's blocks here; stage 1, not yet loaded, is the scratch
        bool nan = false;
        uint8_t* scratch = smem + kStageBytes;
        n = pos >= 0 ? select::select_row<16>(p.scores + g * p.s_stride_h + i * p.s_stride_t,
                                          p.s_stride_n, pos, lane,
                                          reinterpret_cast<uint32_t*>(scratch), kSelectCap,
                                          reinterpret_cast<int*>(scratch + 4 * kSelectCap), nan)
                     : -1;
        if (lane < kTopK) p.topk_out[list + lane] = n;
        if (__any_sync(0xffffffffu, nan) && lane == 0) flag_error(p.err, MSA_ERR_SCORE_NAN);
      } else {
        n = lane < kTopK ? p.topk[list + lane] : -1;
      }
      int page = -1;
      bool valid = false;
      if (lane < kTopK && pos >= 0) {
        if (n != -1) {
          if (n < 0 || n > pos / kPage)
            flag_error(p.err, MSA_ERR_TOPK_RANGE);
          else
            valid = true;
        }
      }
      // a block listed again at a later slot is dropped (a given list only: the
      // selector's lists hold distinct blocks)
      const unsigned same = (!kListsOnly && p.scores) ? 0u : __match_any_sync(0xffffffffu, valid ? n : -2 - lane);
      if (valid && (same & ((1u << lane) - 1u))) {
        flag_error(p.err, MSA_ERR_TOPK_DUP);
        valid = false;
      }
      if (valid) {
        page = n < ncopy ? table_s[n] : trow[n];
        if (page < 0 || static_cast<int64_t>(page) >= p.num_blocks) {
          flag_error(p.err, MSA_ERR_PAGE_RANGE);
          valid = false;
        }
      }
      // page order: the current block first when listed (in select mode it
      // always is, and may already be loading), then the others ascending; both
      // modes use this order, so they give the same bits for the same lists
      const unsigned vm = __ballot_sync(0xffffffffu, valid);
      const bool front = valid && n == cur;
      const unsigned fm = __ballot_sync(0xffffffffu, front);
      const int idx = front ? 0 : __popc(vm & ((1u << lane) - 1u)) + (fm ? 1 : 0);
      const bool mine = valid && (idx % p.splits == split);
      const unsigned mm = __ballot_sync(0xffffffffu, mine);
      mine_front = (mm & fm) != 0u;
      if (mine) {
        const int k = front ? 0 : __popc(mm & ~fm & ((1u << lane) - 1u)) + (mine_front ? 1 : 0);
        tail->pages[k] = page;
        tail->blocks[k] = n;
      }
      np = __popc(mm);
    }
    // the scratch writes in stages 1-2 come before the TMA loads into them
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tail->n_pages = np;
      tail->pos = pos;
      // stage 0 already holds (or is loading) the current block's page: it is
      // page 0 of this list when the list has it; otherwise the load lands
      // unused and stage 0's barrier starts over
      if (cur_page >= 0 && !mine_front) {
        if (!mbar_wait(&tail->full[0], 0)) flag_error(p.err, MSA_ERR_TIMEOUT);
        mbar_inval(&tail->full[0]);
        mbar_init(&tail->full[0], 1);
        fence_barrier_init();
      }
      const int t0 = (cur_page >= 0 && mine_front) ? 1 : 0;
      for (int t = t0; t < np && t < kStages; ++t) {
        uint8_t* st = smem + t * kStageBytes;
        const int row = (tail->pages[t] * p.Hkv + g) * kPage;
        mbar_arrive_expect_tx(&tail->full[t], kStageBytes);
        tma_load_2d(st, &kv_map, 0, row, &tail->full[t]);
        tma_load_2d(st + kHalfTile, &kv_map, kHeadDim, row, &tail->full[t]);
      }
    }
  } else if (warp == 1) {
    tc::tmem_alloc(&tail->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  } else if (warp == kSoftmaxWarp0) {
    const int64_t row = static_cast<int64_t>(i) * p.Hq + g * kGroup;
    if constexpr (kFp8Q) {  // fp8 query as stored; the lo rows of the product are zero
      store_query_rows_fp8(p.q8 + row * kHeadDim, 0, qhi, lane);
      zero_query_rows(0, qlo, lane);
      if (lane == 0) tail->zs = p.logit_scale * p.q_scale;
    } else {
      const int e = prepare_query_e4m3(p.q + row * kHeadDim, 0, qhi, qlo, lane);
      if (lane == 0) tail->zs = p.logit_scale * exp2i(e);
    }
    tc::fence_proxy_async_smem();  // the tiles are read by the tensor core
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const int n_pages = tail->n_pages;
  const int pos = tail->pos;
  const uint32_t tmem = tail->tmem_base;

  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------------------
    if (lane == 0) {
      int issued = n_pages < kStages ? n_pages : kStages;
      for (int t = kStages; t < n_pages; ++t) {
        const int s = t % kStages;
        if (!mbar_wait(&tail->empty[s], ((t / kStages) - 1) & 1)) {
          flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        uint8_t* st = smem + s * kStageBytes;
        const int row = (tail->pages[t] * p.Hkv + g) * kPage;
        mbar_arrive_expect_tx(&tail->full[s], kStageBytes);
        tma_load_2d(st, &kv_map, 0, row, &tail->full[s]);
        tma_load_2d(st + kHalfTile, &kv_map, kHeadDim, row, &tail->full[s]);
        issued = t + 1;
      }
      // the loads still in flight land before shared memory can be released
      for (int t = issued - kStages; t < issued; ++t)
        if (t >= 0) (void)mbar_wait(&tail->full[t % kStages], (t / kStages) & 1);
      // every load of this CTA has landed: the next kernel may start its CTAs
      pdl_trigger();
      mbar_arrive(&tail->finish);
    }
  } else if (warp == 1) {
    // ---- S^T = K Q^T ------------------------------------------------------------------------
    if (lane == 0) {
      // B: 32 rows, the hi part (rows 0-15) directly followed by the lo part
      const uint64_t a0 = tc::sw128_kmajor_desc(smem_u32(smem));
      const uint64_t bq = tc::sw128_kmajor_desc(smem_u32(qhi));
      constexpr uint32_t idesc = tc::idesc_e4m3_f32(128, 2 * kGroup);
      for (int t = 0; t < n_pages; ++t) {
        const int s = t % kStages, buf = t & 1;
        if (!mbar_wait(&tail->full[s], (t / kStages) & 1) ||
            (t >= 2 && !mbar_wait(&tail->s_empty[buf], ((t >> 1) - 1) & 1))) {
          flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        tc::fence_after_thread_sync();
        const uint64_t a = a0 + static_cast<uint64_t>(s) * (kStageBytes >> 4);
        const uint32_t d = tmem + kColS + 2 * kGroup * buf;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) tc::mma_e4m3(d, a + 2 * ks, bq + 2 * ks, idesc, ks > 0);
        tc::commit(&tail->s_full[buf]);
      }
      tc::commit(&tail->finish);  // arrives once this thread's MMAs have all completed
    }
    __syncwarp();
    // free tensor memory once every role is done with it
    (void)mbar_wait(&tail->finish, 0);
    tc::fence_after_thread_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  } else if (warp == 2) {
    // ---- O^T = V^T P^T ----------------------------------------------------------------------
    if (lane == 0) {
      const uint64_t a0 = tc::sw128_mnmajor_desc(smem_u32(smem + kHalfTile));
      // B: N = 32 (16 hi heads, then 16 lo heads 128 bytes further); core
      // matrices along K every kPBlock bytes.  Both offsets stay inside the
      // 4 KiB buffer whichever of them strides along K.
      const uint64_t b0 = tc::interleave_mnmajor_desc(smem_u32(pbuf), kPBlock, 128);
      constexpr uint32_t idesc = tc::idesc_e4m3_f32_mn(128, 2 * kGroup);
      for (int t = 0; t < n_pages; ++t) {
        const int s = t % kStages, buf = t & 1;
        if (!mbar_wait(&tail->p_full[buf], (t >> 1) & 1) ||
            (t >= 2 && !mbar_wait(&tail->o_empty[buf], ((t >> 1) - 1) & 1))) {
          flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        tc::fence_after_thread_sync();
        // k-step kk = keys 32kk .. +31: 4 KiB into the V tile, 1 KiB into P^T
        const uint64_t a = a0 + static_cast<uint64_t>(s) * (kStageBytes >> 4);
        const uint64_t bp = b0 + static_cast<uint64_t>((2 * buf * kPPart) >> 4);
        const uint32_t d = tmem + kColO + 2 * kGroup * buf;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) tc::mma_e4m3(d, a + 256 * kk, bp + 64 * kk, idesc, kk > 0);
        tc::commit(&tail->o_full[buf]);
        tc::commit(&tail->empty[s]);
      }
      tc::commit(&tail->finish);
    }
  } else {
    // ---- softmax and output ------------------------------------------------------------------
    const int quarter = warp & 3;
    const int key = 32 * quarter + lane;  // key of the page; value dim d in the O^T phase
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
    const float zs = tail->zs;
    // nref = kPShift - m, m the reference maximum of a head in log2 units
    // (+inf until the head has seen a key); l: this key slot's share of the
    // running sum; o: the running output of value dim `key`.  Both are kept
    // relative to the current m.
    float nref[kGroup], l[kGroup], o[kGroup];
    fill(nref, INFINITY);
    fill(l, 0.f);
    fill(o, 0.f);
    bool ok = true;

    // o += f * O^T of page u (hi + lo columns), once its product is complete
    auto add_page_o = [&](int u, const float (&f)[kGroup]) -> bool {
      const int ob = u & 1;
      if (!mbar_wait(&tail->o_full[ob], (u >> 1) & 1)) return false;
      tc::fence_after_thread_sync();
      uint32_t ov[32];
      tc::ld_32x32b_x32(lane_addr + kColO + 2 * kGroup * ob, ov);
      tc::wait_ld();
      tc::fence_before_thread_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->o_empty[ob]);
#pragma unroll
      for (int h = 0; h < kGroup; ++h)
        o[h] = fmaf(__uint_as_float(ov[h]) + __uint_as_float(ov[h + kGroup]), f[h], o[h]);
      return true;
    };

    for (int t = 0; t < n_pages && ok; ++t) {
      const int buf = t & 1, ph = (t >> 1) & 1;
      if (!mbar_wait(&tail->s_full[buf], ph)) {
        ok = false;
        break;
      }
      tc::fence_after_thread_sync();
      float x[kGroup], pm[kGroup];
      {
        uint32_t sv[32];
        tc::ld_32x32b_x32(lane_addr + kColS + 2 * kGroup * buf, sv);
        tc::wait_ld();
        tc::fence_before_thread_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->s_empty[buf]);
        const int lim = pos - tail->blocks[t] * kPage;  // keys <= lim are visible
        const bool vis = key <= lim;
        // raw dot products (hi + lo columns); the logit in log2 units is
        // s * zs with zs > 0, so maxima can be taken on s
#pragma unroll
        for (int h = 0; h < kGroup; ++h)
          x[h] = vis ? __uint_as_float(sv[h]) + __uint_as_float(sv[h + kGroup]) : -INFINITY;
      }
#pragma unroll
      for (int h = 0; h < kGroup; ++h) pm[h] = warp_max_f32(x[h]);
      float* mxb = mx + buf * 4 * kGroup;
      if (lane == 0) {
#pragma unroll
        for (int h4 = 0; h4 < 4; ++h4)
          *reinterpret_cast<float4*>(mxb + quarter * kGroup + 4 * h4) =
              make_float4(pm[4 * h4], pm[4 * h4 + 1], pm[4 * h4 + 2], pm[4 * h4 + 3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->mx_full[buf]);
      if (!mbar_wait(&tail->mx_full[buf], ph)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int h4 = 0; h4 < 4; ++h4) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float4 v = *reinterpret_cast<const float4*>(mxb + w * kGroup + 4 * h4);
          pm[4 * h4] = fmaxf(pm[4 * h4], v.x);
          pm[4 * h4 + 1] = fmaxf(pm[4 * h4 + 1], v.y);
          pm[4 * h4 + 2] = fmaxf(pm[4 * h4 + 2], v.z);
          pm[4 * h4 + 3] = fmaxf(pm[4 * h4 + 3], v.w);
        }
      }
      // page maximum in log2 units against m + kLazy (pm + nref > kPShift + kLazy;
      // a head without any key so far has nref = +inf and always moves)
      bool raise = false;
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
        pm[h] *= zs;
        raise |= pm[h] + nref[h] > kPShift + kLazy;
      }
      float al[kGroup];  // 2^(m_old - m_new) per head
      fill(al, 1.f);
      if (raise) {  // the same decision in every thread
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
          if (pm[h] + nref[h] > kPShift + kLazy) {
            al[h] = ex2(kPShift - nref[h] - pm[h]);  // 0 when the head had no key yet
            nref[h] = kPShift - pm[h];
          }
          o[h] *= al[h];
        }
      }
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
        x[h] = ex2(fmaf(x[h], zs, nref[h]));  // P = 2^(x - m + 8); 0 for an invisible key
        l[h] = fmaf(l[h], al[h], x[h]);
      }
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t h0, l0, h1, l1;
        split_e4m3x2(x[4 * q4], x[4 * q4 + 1], h0, l0);
        split_e4m3x2(x[4 * q4 + 2], x[4 * q4 + 3], h1, l1);
        hw[q4] = h0 | (h1 << 16);
        lw[q4] = l0 | (l1 << 16);
      }
      const int s = t % kStages;
      const int lim = pos - tail->blocks[t] * kPage;
      if (lim < kPage - 1 && key > lim) {
        // keys past the causal limit have P = 0, but their value rows may hold
        // any bytes (an fp8 NaN times 0 is NaN): zero them for the O^T product
        if (mbar_wait(&tail->full[s], (t / kStages) & 1)) {
          uint4* vrow = reinterpret_cast<uint4*>(smem + s * kStageBytes + kHalfTile + key * 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) vrow[c] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // P^T: key k's 16 hi bytes at (k/8) * kPBlock + (k%8) * 16, its lo bytes
      // 128 further (MN-major, no swizzle).  Buffer `buf` was last read by the
      // O^T product of page t-2, which add_page_o(t-2) has waited for.
      uint8_t* pk = pbuf + 2 * buf * kPPart + (key >> 3) * kPBlock + (key & 7) * 16;
      *reinterpret_cast<uint4*>(pk) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(pk + 128) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->p_full[buf]);
      // o holds pages <= t-2 relative to the new m; page t-1's product is
      // relative to the previous m, so it enters with this page's factors
      if (t >= 1 && !add_page_o(t - 1, al)) {
        ok = false;
        break;
      }
    }
    if (ok && n_pages > 0) {
      float one[kGroup];
      fill(one, 1.f);
      ok = add_page_o(n_pages - 1, one);
    }

    if (ok) {
      // running sums: this thread's share -> the whole page (128 key slots)
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
      }
      if (lane == 0) {
#pragma unroll
        for (int h4 = 0; h4 < 4; ++h4)
          *reinterpret_cast<float4*>(lsum + quarter * kGroup + 4 * h4) =
              make_float4(l[4 * h4], l[4 * h4 + 1], l[4 * h4 + 2], l[4 * h4 + 3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->l_full);
      ok = mbar_wait(&tail->l_full, 0);
    }
    if (ok) {
#pragma unroll
      for (int h4 = 0; h4 < 4; ++h4) {
        float4 t4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float4 v = *reinterpret_cast<const float4*>(lsum + w * kGroup + 4 * h4);
          t4.x += v.x;
          t4.y += v.y;
          t4.z += v.z;
          t4.w += v.w;
        }
        l[4 * h4] = t4.x;
        l[4 * h4 + 1] = t4.y;
        l[4 * h4 + 2] = t4.z;
        l[4 * h4 + 3] = t4.w;
      }
      const int d = key;
      const int64_t row0 = static_cast<int64_t>(i) * p.Hq + g * kGroup;
      // dense decode waited for no earlier kernel; the outputs (or the split
      // partials) may still be read by the previous one
      if constexpr (kDense) pdl_wait();
      if (p.splits == 1) {
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
          const float f = (l[h] > 0.f) ? p.v_scale / l[h] : 0.f;
          p.out[(row0 + h) * kHeadDim + d] = static_cast<uint16_t>(f32_to_bf16_bits(o[h] * f));
        }
      } else {
        const int64_t rows = static_cast<int64_t>(kVarlen ? p.T : p.B * p.Q) * p.Hq;
        const int64_t base = static_cast<int64_t>(split) * rows + row0;
#pragma unroll
        for (int h = 0; h < kGroup; ++h) p.part_o[(base + h) * kHeadDim + d] = o[h] * p.v_scale;
        // partial state in the combine kernel's terms: l = sum 2^(x - mref)
        if (key < kGroup) {
          float mr = -INFINITY, lr = 0.f;
#pragma unroll
          for (int h = 0; h < kGroup; ++h)
            if (h == key) {
              mr = -nref[h];  // m - kPShift; -inf for a head without keys
              lr = l[h];
            }
          p.part_ml[(base + key) * 2] = mr;
          p.part_ml[(base + key) * 2 + 1] = lr;
        }
      }
    } else if (lane == 0) {
      flag_error(p.err, MSA_ERR_TIMEOUT);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->finish);
  }
}

// Split merge: one warp per (token, query head) row, 4 d-values per lane.
// A part counts only when its l > 0 and its m is a number.
__global__ void __launch_bounds__(256)
    combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                   uint16_t* __restrict__ out, int64_t rows, int splits) {
  pdl_trigger();
  pdl_wait();  // the partials come from the attend kernel
  const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float M = -INFINITY;
  for (int s = lane; s < splits; s += 32) {
    const float m = part_ml[(s * rows + r) * 2], l = part_ml[(s * rows + r) * 2 + 1];
    if (l > 0.f && m == m) M = fmaxf(M, m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float m = part_ml[(s * rows + r) * 2], l = part_ml[(s * rows + r) * 2 + 1];
    if (!(l > 0.f) || m != m) continue;  // an empty part, or one with no valid maximum
    const float w = ex2(m - M);
    den += w * l;
    const float4 v = *reinterpret_cast<const float4*>(part_o + (s * rows + r) * kHeadDim + 4 * lane);
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  }
  const float f = den > 0.f ? 1.f / den : 0.f;
  const uint32_t lo = f32_to_bf16_bits(acc.x * f) | (f32_to_bf16_bits(acc.y * f) << 16);
  const uint32_t hi = f32_to_bf16_bits(acc.z * f) | (f32_to_bf16_bits(acc.w * f) << 16);
  *reinterpret_cast<uint2*>(out + r * kHeadDim + 4 * lane) = make_uint2(lo, hi);
}


}  // namespace

cudaError_t launch_attend(const CUtensorMap& kv_map, const AttendParams& p, cudaStream_t stream,
                          bool pdl) {
  static_assert(kSmemBytes <= 227 * 1024, "attend shared memory");
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [] {
    for (auto* k : {attend_kernel<false, false>, attend_kernel<true, false>,
                    attend_kernel<false, true>, attend_kernel<true, true>,
                    attend_kernel<false, false, true>, attend_kernel<false, true, true>,
                    attend_kernel<false, false, false, true>, attend_kernel<false, true, false, true>,
                    attend_kernel<false, false, true, true>, attend_kernel<false, true, true, true>}) {
      cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemBytes);
      if (r != cudaSuccess) return r;
      // all of the unified L1 / shared storage as shared memory: two CTAs per SM
      r = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                               static_cast<int>(cudaSharedmemCarveoutMaxShared));
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  // the union attend: one pass over the pages a 4-token tile shares
  if (p.union_tile) return launch_union_attend(kv_map, p, stream, pdl);
  const int T = p.cu_q ? p.T : p.B * p.Q;
  dim3 grid(T, p.Hkv, p.splits);
  const dim3 block(kThreads);
  if (p.cu_q) {  // prefill-style batches (no dense mode); given lists: no selector
    if (p.scores == nullptr)
      return p.q8 ? launch_pdl(attend_kernel<false, true, true, true>, grid, block, kSmemBytes,
                               stream, pdl, kv_map, p)
                  : launch_pdl(attend_kernel<false, false, true, true>, grid, block, kSmemBytes,
                               stream, pdl, kv_map, p);
    return p.q8 ? launch_pdl(attend_kernel<false, true, true>, grid, block, kSmemBytes, stream, pdl,
                             kv_map, p)
                : launch_pdl(attend_kernel<false, false, true>, grid, block, kSmemBytes, stream, pdl,
                             kv_map, p);
  }
  // decode on given lists: an instantiation without the prologue's selector
  const bool lists = p.scores == nullptr && p.dense_span == 0;
  if (p.q8)
    return p.dense_span > 0
               ? launch_pdl(attend_kernel<true, true>, grid, block, kSmemBytes, stream, pdl, kv_map, p)
           : lists ? launch_pdl(attend_kernel<false, true, false, true>, grid, block, kSmemBytes,
                                stream, pdl, kv_map, p)
                   : launch_pdl(attend_kernel<false, true>, grid, block, kSmemBytes, stream, pdl, kv_map, p);
  return p.dense_span > 0
             ? launch_pdl(attend_kernel<true, false>, grid, block, kSmemBytes, stream, pdl, kv_map, p)
         : lists ? launch_pdl(attend_kernel<false, false, false, true>, grid, block, kSmemBytes,
                              stream, pdl, kv_map, p)
                 : launch_pdl(attend_kernel<false, false>, grid, block, kSmemBytes, stream, pdl, kv_map, p);
}

cudaError_t launch_combine(const float* part_o, const float* part_ml, uint16_t* out, int64_t rows,
                           int splits, cudaStream_t stream, bool pdl) {
  const int64_t threads = rows * 32;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(grid)), dim3(block), 0, stream, pdl,
                    part_o, part_ml, out, rows, splits);
}

}  // namespace msa
