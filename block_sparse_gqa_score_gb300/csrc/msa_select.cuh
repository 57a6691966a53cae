// msa_select.cuh -- the block selector of one (token, KV head) row, run by
// one warp; used by the selector kernel and by the attend kernel's fused
// select-then-attend mode.
//
// Keep the current block cur = pos/128 and the 15 best earlier blocks in the
// order (score descending, block index ascending); the kept ids come out
// ascending with cur last, -1 padded (the vLLM test file's _make_topk
// layout), as TensorRT-LLM PR #17171's selector produces them from the
// scorer's [head, token, block] buffer.
//
// Scores become order-preserving 32-bit keys (larger float -> larger key, -0
// folded onto +0, NaN ranked as -inf and reported).  A threshold tau with at
// least 15 keys >= tau is found by a bitwise binary search: for each bit,
// count (one compare per key, one warp-wide redux add) the keys at or above
// the candidate prefix, and keep the bit when at least 15 are.  The search
// starts below the bits that the row's smallest and largest keys share (every
// key shares them, so tau does too), and stops as soon as exactly 15 keys are
// >= tau: they are then the kept set, with no tie at its boundary.  Without an
// early stop tau ends as the 15th-largest key.  Keys > tau are all kept and the
// lowest-index keys == tau fill the rest, in one ordered sweep.  Rows of up to
// 2048 candidates live in registers (8 to 64 per lane) during the search,
// longer rows in the caller's shared scratch when they fit, else they are
// re-read.
#pragma once

#include "msa_device.cuh"

namespace msa {
namespace select {

constexpr int kSel = kTopK - 1;  // blocks kept besides the current one

__device__ __forceinline__ uint32_t order_key(float x, bool& nan) {
  uint32_t u = __float_as_uint(x);
  if (x != x) {
    nan = true;
    u = 0xFF800000u;  // rank NaN as -inf
  }
  if (u == 0x80000000u) u = 0u;  // -0 ranks equal to +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Start of the search from the row's smallest and largest keys: the bits
// above the highest one where they differ are common to every key.  Returns
// that prefix (lower bits 0) and the highest differing bit in `top` (-1: all
// keys equal, the prefix is the key itself).
__device__ __forceinline__ uint32_t common_prefix(uint32_t lo_k, uint32_t hi_k, int& top) {
  lo_k = __reduce_min_sync(0xffffffffu, lo_k);
  hi_k = __reduce_max_sync(0xffffffffu, hi_k);
  const uint32_t diff = lo_k ^ hi_k;
  top = diff ? 31 - __clz(diff) : -1;
  if (top == 31) return 0u;
  return top >= 0 ? (hi_k & ~((2u << top) - 1u)) : hi_k;
}

// tau for a row whose keys are held NK per lane in registers (lane + 32 e);
// also leaves the keys in `keys` for the final sweep.
template <int NK, typename LoadKey>
__device__ __forceinline__ uint32_t tau_in_registers(LoadKey& load_key, uint32_t* keys, int cur,
                                                     int lane) {
  uint32_t kr[NK];
#pragma unroll
  for (int e = 0; e < NK; ++e) {
    const int n = lane + 32 * e;
    kr[e] = (n < cur) ? load_key(n) : 0u;  // 0 ranks below every real key
  }
  uint32_t lo_k = 0xFFFFFFFFu, hi_k = 0u;
#pragma unroll
  for (int e = 0; e < NK; ++e) {
    if (lane + 32 * e < cur) lo_k = min(lo_k, kr[e]);
    hi_k = max(hi_k, kr[e]);
  }
  int top;
  uint32_t tau = common_prefix(lo_k, hi_k, top);
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

// tau for a longer row, keys read through key_at (shared scratch or global).
template <typename KeyAt>
__device__ __forceinline__ uint32_t tau_in_memory(KeyAt& key_at, int cur, int lane) {
  uint32_t lo_k = 0xFFFFFFFFu, hi_k = 0u;
  for (int n = lane; n < cur; n += 32) {
    const uint32_t k = key_at(n);
    lo_k = min(lo_k, k);
    hi_k = max(hi_k, k);
  }
  int top;
  uint32_t tau = common_prefix(lo_k, hi_k, top);
  for (int bit = top; bit >= 0; --bit) {
    const uint32_t cand = tau | (1u << bit);
    int cnt = 0;
    for (int n = lane; n < cur; n += 32) cnt += (key_at(n) >= cand) ? 1 : 0;
    const int total = __reduce_add_sync(0xffffffffu, cnt);
    if (total >= kSel) {
      tau = cand;
      if (total == kSel) break;
    }
  }
  return tau;
}

// The kept blocks of a row whose token sits at causal position pos >= 0:
// returns the k-th kept block (ascending, cur last, -1 padded) in lane k < 16,
// -1 in lanes 16-31.  kMaxRegKeys (16, 32 or 64) bounds the keys a lane holds
// in registers, i.e. the register pressure the caller can afford.
// srow[n * stride_n] is the score of block n.  `keys` is
// shared scratch for `cap` >= 512 keys, `slots` shared scratch for 16 ints
// (both used only by this warp).  `nan` is set when a score is NaN.
template <int kMaxRegKeys>
__device__ __forceinline__ int select_row(const float* __restrict__ srow, int64_t stride_n, int pos,
                                          int lane, uint32_t* keys, int cap, int* slots,
                                          bool& nan) {
  const int cur = pos / kPage;
  if (cur + 1 <= kTopK) return (lane < kTopK && lane <= cur) ? lane : -1;
  auto load_key = [&](int n) -> uint32_t { return order_key(srow[n * stride_n], nan); };
  const bool cached = cur <= cap;
  uint32_t tau;
  if (cur <= 32 * 8) {
    tau = tau_in_registers<8>(load_key, keys, cur, lane);
  } else if (cur <= 32 * 16) {
    tau = tau_in_registers<16>(load_key, keys, cur, lane);
  } else if (kMaxRegKeys >= 32 && cur <= 32 * 32 && cap >= 32 * 32) {
    tau = tau_in_registers<(kMaxRegKeys >= 32 ? 32 : 16)>(load_key, keys, cur, lane);
  } else if (kMaxRegKeys >= 64 && cur <= 32 * 64 && cap >= 32 * 64) {
    tau = tau_in_registers<(kMaxRegKeys >= 64 ? 64 : 16)>(load_key, keys, cur, lane);
  } else {
    if (cached)
      for (int n = lane; n < cur; n += 32) keys[n] = load_key(n);
    __syncwarp();
    auto mem_key = [&](int n) -> uint32_t { return cached ? keys[n] : load_key(n); };
    tau = tau_in_memory(mem_key, cur, lane);
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
    if (take && slot < kSel) slots[slot] = n;
    written += __popc(bs);
  }
  if (lane == 0) slots[kSel] = cur;
  __syncwarp();
  const int v = lane < kTopK ? slots[lane] : -1;
  __syncwarp();  // slots may be reused once every lane has read it
  return v;
}

}  // namespace select
}  // namespace msa
