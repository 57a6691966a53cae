// msa_topk.cu -- stage 2, the block selector.
//
// For each (token, KV head) row: keep the current block cur = pos/128 and the
// 15 best earlier blocks in the order (score descending, block index
// ascending); write the kept ids ascending, -1 padded (the vLLM test file's
// _make_topk layout); all -1 for a padding row.  Scores are read through
// arbitrary element strides, as TensorRT-LLM PR #17171's selector takes the
// scorer's [head, token, block] buffer through a transposed view.
//
// Design: one warp per row.  Scores become order-preserving 32-bit keys
// (larger float -> larger key, -0 folded onto +0).  A threshold tau with at
// least 15 keys >= tau is found by a bitwise binary search: for each bit,
// count (one compare per key, one warp-wide redux add) the keys at or above
// the candidate prefix, and keep the bit when at least 15 are.  The search
// starts below the bits that the row's smallest and largest keys share (every
// key shares them, so tau does too), and stops as soon as exactly 15 keys are
// >= tau: they are then the kept set, with no tie at its boundary.  Without
// an early stop tau ends as the 15th-largest key.  Keys > tau are all kept and
// the lowest-index keys == tau fill the rest, in one ordered sweep.  Rows of up to 512 candidates live in registers (16 per
// lane), rows up to kCache in shared memory, longer rows are re-read.
#include "msa_device.cuh"
#include "msa_launch.h"

namespace msa {

namespace {

constexpr int kWarps = 4;
constexpr int kCache = 2048;  // candidates cached per warp (8 KiB)
constexpr int kRegKeys = 16;  // candidates per lane held in registers
constexpr int kSel = kTopK - 1;

__device__ __forceinline__ uint32_t order_key(float x, bool& nan) {
  uint32_t u = __float_as_uint(x);
  if (x != x) {
    nan = true;
    u = 0xFF800000u;  // rank NaN as -inf
  }
  if (u == 0x80000000u) u = 0u;  // -0 ranks equal to +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Bitwise search for the 15th-largest of a row's keys held NK per lane in
// registers (lane + 32 e); also leaves the keys in `keys` for the final sweep.
template <int NK, typename LoadKey>
__device__ __forceinline__ uint32_t tau_in_registers(LoadKey& load_key, uint32_t* keys, int cur,
                                                     int lane) {
  uint32_t kr[NK];
#pragma unroll
  for (int e = 0; e < NK; ++e) {
    const int n = lane + 32 * e;
    kr[e] = (n < cur) ? load_key(n) : 0u;  // 0 ranks below every real key
  }
  // bits above the highest one where the row's extreme keys differ are
  // common to every key (absent slots hold 0, the smallest key, and take part)
  uint32_t lo_k = 0xFFFFFFFFu, hi_k = 0u;
#pragma unroll
  for (int e = 0; e < NK; ++e) {
    if (lane + 32 * e < cur) lo_k = min(lo_k, kr[e]);
    hi_k = max(hi_k, kr[e]);
  }
  lo_k = __reduce_min_sync(0xffffffffu, lo_k);
  hi_k = __reduce_max_sync(0xffffffffu, hi_k);
  const uint32_t diff = lo_k ^ hi_k;
  const int top = diff ? 31 - __clz(diff) : -1;       // highest differing bit
  uint32_t tau = top >= 0 ? (hi_k & ~((2u << top) - 1u)) : hi_k;
  if (top == 31) tau = 0;
  for (int bit = top; bit >= 0; --bit) {
    const uint32_t cand = tau | (1u << bit);
    int cnt = 0;
#pragma unroll
    for (int e = 0; e < NK; ++e) cnt += (kr[e] >= cand) ? 1 : 0;
    const int total = __reduce_add_sync(0xffffffffu, cnt);
    if (total >= kSel) {
      tau = cand;
      if (total == kSel) break;  // exactly the 15 kept keys are >= tau
    }
  }
#pragma unroll
  for (int e = 0; e < NK; ++e)
    if (lane + 32 * e < cur) keys[lane + 32 * e] = kr[e];
  return tau;
}

__global__ void __launch_bounds__(kWarps * 32) topk_kernel(const TopkParams p) {
  __shared__ uint32_t s_keys[kWarps][kCache];
  pdl_trigger();
  pdl_wait();  // scores come from the previous kernel; topk may still be read by one
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int T = p.B * p.Q;
  if (row >= static_cast<int64_t>(T) * p.Hkv) return;
  const int i = static_cast<int>(row / p.Hkv), g = static_cast<int>(row - static_cast<int64_t>(i) * p.Hkv);
  const int b = i / p.Q, j = i - b * p.Q;
  int32_t* out = p.topk + row * kTopK;

  const int L = p.seq_lens[b];
  const bool seq_ok = L >= 0 && (L == 0 || (L - 1) / kPage < p.S);
  if (!seq_ok && lane == 0 && j == 0 && g == 0) flag_error(p.err, MSA_ERR_SEQ_RANGE);
  const int pos = seq_ok ? L - p.Q + j : -1;
  if (pos < 0) {
    if (lane < kTopK) out[lane] = -1;
    return;
  }
  const int cur = pos / kPage;
  if (cur + 1 <= kTopK) {
    if (lane < kTopK) out[lane] = (lane <= cur) ? lane : -1;
    return;
  }

  const float* srow = p.scores + g * p.stride_h + static_cast<int64_t>(i) * p.stride_t;
  uint32_t* keys = s_keys[warp];
  const bool cached = cur <= kCache;
  bool nan = false;
  auto load_key = [&](int n) -> uint32_t { return order_key(srow[n * p.stride_n], nan); };

  // tau = the largest value with at least 15 keys >= tau (the 15th-largest key)
  uint32_t tau = 0;
  if (cur <= 32 * 8) {
    tau = tau_in_registers<8>(load_key, keys, cur, lane);
  } else if (cur <= 32 * kRegKeys) {
    tau = tau_in_registers<kRegKeys>(load_key, keys, cur, lane);
  } else {
    if (cached)
      for (int n = lane; n < cur; n += 32) keys[n] = load_key(n);
    __syncwarp();
    for (int bit = 31; bit >= 0; --bit) {
      const uint32_t cand = tau | (1u << bit);
      int cnt = 0;
      for (int n = lane; n < cur; n += 32) cnt += ((cached ? keys[n] : load_key(n)) >= cand) ? 1 : 0;
      if (__reduce_add_sync(0xffffffffu, cnt) >= kSel) tau = cand;
    }
  }
  __syncwarp();
  auto key_at = [&](int n) -> uint32_t { return cached ? keys[n] : load_key(n); };
  int gt_count = 0;
  for (int n = lane; n < cur; n += 32) gt_count += (key_at(n) > tau) ? 1 : 0;
  const int need = kSel - __reduce_add_sync(0xffffffffu, gt_count);  // ties to take, >= 1

  // keys > tau all kept; keys == tau kept in ascending index order until `need`
  int written = 0, ties = 0;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = 0; base < cur; base += 32) {
    const int n = base + lane;
    const uint32_t k = (n < cur) ? key_at(n) : 0u;
    const bool gt = n < cur && k > tau;
    const bool eq = n < cur && k == tau;
    const unsigned be = __ballot_sync(0xffffffffu, eq);
    const bool take = gt || (eq && ties + __popc(be & lt) < need);
    ties += __popc(be);
    const unsigned bs = __ballot_sync(0xffffffffu, take);
    const int slot = written + __popc(bs & lt);
    if (take && slot < kTopK - 1) out[slot] = n;
    written += __popc(bs);
  }
  if (lane == 0) out[kTopK - 1] = cur;
  if (__any_sync(0xffffffffu, nan) && lane == 0) flag_error(p.err, MSA_ERR_SCORE_NAN);
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.Q * p.Hkv;
  const int64_t grid = (rows + kWarps - 1) / kWarps;
  return launch_pdl(topk_kernel, dim3(static_cast<unsigned>(grid)), dim3(kWarps * 32), 0, stream,
                    p);
}

}  // namespace msa
