// msa_topk.cu -- stage 2, the block selector.
//
// For each (token, KV head) row: keep the current block cur = pos/128 and the
// 15 best earlier blocks in the order (score descending, block index
// ascending); write the kept ids ascending, -1 padded (the vLLM test file's
// _make_topk layout); all -1 for a padding row.  Scores are read through
// arbitrary element strides, as TensorRT-LLM PR #17171's selector takes the
// scorer's [head, token, block] buffer through a transposed view.  One warp
// per row; the per-row algorithm is in msa_select.cuh.
#include "msa_device.cuh"
#include "msa_launch.h"
#include "msa_select.cuh"

namespace msa {

namespace {

constexpr int kWarps = 4;
constexpr int kCache = 2048;  // candidates cached per warp (8 KiB)

__global__ void __launch_bounds__(kWarps * 32) topk_kernel(const TopkParams p) {
  __shared__ uint32_t s_keys[kWarps][kCache];
  __shared__ int s_slots[kWarps][kTopK];
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
  const float* srow = p.scores + g * p.stride_h + static_cast<int64_t>(i) * p.stride_t;
  bool nan = false;
  const int v = select::select_row<64>(srow, p.stride_n, pos, lane, s_keys[warp], kCache,
                                   s_slots[warp], nan);
  if (lane < kTopK) out[lane] = v;
  if (__any_sync(0xffffffffu, nan) && lane == 0) flag_error(p.err, MSA_ERR_SCORE_NAN);
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream, bool pdl) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.Q * p.Hkv;
  const int64_t grid = (rows + kWarps - 1) / kWarps;
  return launch_pdl(topk_kernel, dim3(static_cast<unsigned>(grid)), dim3(kWarps * 32), 0, stream, pdl,
                    p);
}

}  // namespace msa
