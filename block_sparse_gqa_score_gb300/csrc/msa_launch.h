// msa_launch.h -- parameter blocks and host launchers of the sm_103a kernels
// (internal to the library; the public interface is include/msa.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace msa {

struct ScoreParams {
  const uint16_t* q;           // bf16 bits [T, Hq, 128] (when q8 is null)
  const int32_t* block_table;  // [B, S]
  const int32_t* seq_lens;     // [B]
  float* scores;               // [Hkv, T, S]
  unsigned* err;               // device error word
  int B, Q, Hq, Hkv, S;
  int ctas;                    // SM count (the scorer runs one or two CTAs per SM)
  int64_t num_blocks;
  float scale;                 // sm_scale * k_scale
  const uint8_t* q8;           // fp8 e4m3 [T, Hq, 128], value q8 * q_scale; or nullptr
  float q_scale;
};

struct TopkParams {
  const float* scores;
  int64_t stride_h, stride_t, stride_n;  // element strides of scores[g, i, n]
  const int32_t* seq_lens;
  int32_t* topk;                         // [T, Hkv, 16]
  unsigned* err;
  int B, Q, Hkv, S;
};

struct AttendParams {
  const uint16_t* q;           // bf16 bits [T, Hq, 128] (when q8 is null)
  const int32_t* block_table;  // [B, S]
  const int32_t* seq_lens;     // [B]
  const int32_t* topk;         // [T, Hkv, 16]; unused when `scores` is given
  // select-then-attend: each row's top-k list is selected inside the kernel
  // from scores[g * s_stride_h + i * s_stride_t + n * s_stride_n] and written
  // to topk_out [T, Hkv, 16]; nullptr: `topk` is the input list
  const float* scores;
  int64_t s_stride_h, s_stride_t, s_stride_n;
  int32_t* topk_out;
  // dense decode: > 0 means no list at all; CTA z attends blocks
  // [z * dense_span, (z + 1) * dense_span) that its token may see
  int dense_span;
  float* part_o;               // [splits, T, Hq, 128]     (splits > 1)
  float* part_ml;              // [splits, T, Hq, 2]       (splits > 1)
  uint16_t* out;               // bf16 bits [T, Hq, 128]   (splits == 1)
  unsigned* err;
  int B, Q, Hq, Hkv, S, splits;
  int64_t num_blocks;
  float logit_scale;           // sm_scale * k_scale * log2(e)
  float v_scale;
  const uint8_t* q8;           // fp8 e4m3 [T, Hq, 128], value q8 * q_scale; or nullptr
  float q_scale;
  // prefill-style batches: request r owns tokens [cu_q[r], cu_q[r + 1]) of the
  // T tokens (then Q is unused); nullptr: every request has Q tokens
  const int32_t* cu_q;
  int T;
  // 1: the union attend (msa_union.cu) over 4-token tiles of each request;
  // 0: one CTA per (token, KV head)
  int union_tile;
};

// Runs `set_up` once per device (e.g. raising a kernel's dynamic shared-memory
// limit), so that later launches, including ones inside a CUDA-graph capture,
// make no attribute calls.
template <typename F>
inline cudaError_t once_per_device(std::atomic<unsigned long long>& done, F&& set_up) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = set_up();
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launch with programmatic stream serialization when `pdl` is set: the kernel
// may then start while the previous kernel on the stream finishes (its CTAs
// call pdl_wait before touching that kernel's results, but may read the
// caller's inputs before it).  Without `pdl` it is an ordinary launch that
// starts after all earlier work on the stream has completed (pdl_wait then
// returns at once).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Each launcher's `pdl`: whether its kernel may overlap the previous kernel on
// the stream (see launch_pdl).  The first kernel of a public entry point
// passes the library-wide input-overlap setting; a kernel that follows
// another library kernel inside one call passes true.
cudaError_t launch_score(const CUtensorMap& kv_map, const ScoreParams& p, cudaStream_t stream,
                         bool pdl);
cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_attend(const CUtensorMap& kv_map, const AttendParams& p, cudaStream_t stream,
                          bool pdl);
// The union attend (msa_union.cu): decode steps of Q >= 2 tokens per request,
// one CTA per (request, tile of 4 tokens, KV head, split) over the union of the
// tile's lists; grid (B * ceil(Q / 4) * Hkv, splits).
cudaError_t launch_union_attend(const CUtensorMap& kv_map, const AttendParams& p,
                                cudaStream_t stream, bool pdl);
// Its split count for `units` (request, tile, KV head) units: as many CTAs per
// unit as fit one CTA per SM (at most 8), 1 when the units fill the SMs.
int union_ctas_per_unit(int units, int sm_count);
constexpr int kUnionTile = 4;   // query tokens per union tile

// The bounded-wait exit exercised on purpose (msa_waittest.cu).
cudaError_t launch_wait_timeout(unsigned long long limit_ns, unsigned* err, cudaStream_t stream);

cudaError_t launch_combine(const float* part_o, const float* part_ml, uint16_t* out, int64_t rows,
                           int splits, cudaStream_t stream, bool pdl);

}  // namespace msa
