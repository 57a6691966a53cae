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
// (larger float -> larger key, -0 folded onto +0).  A most-significant-digit
// radix select (8 passes of 4 bits, shared-memory histograms) finds the exact
// 15th-largest key tau and how many keys equal to tau are still needed; a
// final ordered sweep keeps every key > tau and the lowest-index keys == tau.
// Rows of up to kCache candidates are staged once in shared memory.
#include "msa_device.cuh"
#include "msa_launch.h"

namespace msa {

namespace {

constexpr int kWarps = 4;
constexpr int kCache = 2048;  // candidates cached per warp (8 KiB)

__device__ __forceinline__ uint32_t order_key(float x, bool& nan) {
  uint32_t u = __float_as_uint(x);
  if (x != x) {
    nan = true;
    u = 0xFF800000u;  // rank NaN as -inf
  }
  if (u == 0x80000000u) u = 0u;  // -0 ranks equal to +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kWarps * 32) topk_kernel(const TopkParams p) {
  __shared__ uint32_t s_keys[kWarps][kCache];
  __shared__ int s_hist[kWarps][16];
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
  const bool cached = cur <= kCache;
  uint32_t* keys = s_keys[warp];
  bool nan = false;
  auto key_at = [&](int n) -> uint32_t {
    return cached ? keys[n] : order_key(srow[n * p.stride_n], nan);
  };
  if (cached) {
    for (int n = lane; n < cur; n += 32) keys[n] = order_key(srow[n * p.stride_n], nan);
    __syncwarp();
  }

  int need = kTopK - 1;  // keys still to take among those matching the prefix
  uint32_t prefix = 0, pmask = 0;
  for (int shift = 28; shift >= 0; shift -= 4) {
    if (lane < 16) s_hist[warp][lane] = 0;
    __syncwarp();
    for (int n = lane; n < cur; n += 32) {
      const uint32_t k = key_at(n);
      if ((k & pmask) == prefix) atomicAdd(&s_hist[warp][(k >> shift) & 15], 1);
    }
    __syncwarp();
    // suffix[d] = number of matching keys whose digit is >= d
    int suf = (lane < 16) ? s_hist[warp][lane] : 0;
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) {
      const int v = __shfl_down_sync(0xffffffffu, suf, off);
      if (lane + off < 16) suf += v;
    }
    const unsigned ok = __ballot_sync(0xffffffffu, lane < 16 && suf >= need);
    const int D = ok ? 31 - __clz(ok) : 0;          // largest digit reaching `need`
    const int above = __shfl_sync(0xffffffffu, suf, (D + 1) & 31);
    need -= (D < 15) ? above : 0;
    prefix |= static_cast<uint32_t>(D) << shift;
    pmask |= 15u << shift;
    __syncwarp();
  }
  const uint32_t tau = prefix;

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
  topk_kernel<<<static_cast<unsigned>(grid), kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace msa
