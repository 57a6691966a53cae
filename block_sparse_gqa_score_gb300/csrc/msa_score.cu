// msa_score.cu -- stage 1, the block scorer.
//
// Operation (TensorRT-LLM PR #17171, scorer commit): for each KV head g, query
// token i and logical block n, the causal max of sm_scale * k_scale * q.k over
// the query heads of g's group and the block's keys the token may see; -inf
// past the token's current block and for padding rows.  Output [Hkv, T, S].
//
// Design (sm_103a): one CTA per (chunk of logical blocks, KV head, request),
// i.e. a grid sized to the batch rather than a 128-row query tile per token.
// A producer warp streams the K halves (16 KiB per page-head) of the chunk's
// pages with TMA into 128B-swizzled stages; four compute warps each take 32
// keys of a page and run the request's Q tokens x 16 heads against them with
// fp16 tensor-core MMAs, widening fp8 keys in registers.  Query fragments are
// prepared once per CTA in shared memory.
#include "msa_device.cuh"
#include "msa_launch.h"

namespace msa {

namespace {

constexpr int kComputeWarps = 4;
constexpr int kThreads = (kComputeWarps + 1) * 32;
constexpr int kScoreStages = 4;
constexpr int kMaxChunk = 32;
constexpr int kTokensPerPass = 4;   // query tokens whose fragments a warp holds at once

struct ScoreSmemTail {
  uint64_t full[kScoreStages];
  uint64_t empty[kScoreStages];
  uint64_t drained;
  int abort;
  int n_pages;
  int pages[kMaxChunk];
  int loc[kMaxChunk];  // block offset inside the chunk
};

__host__ __device__ constexpr int score_qfrag_bytes(int Q) { return Q * 8 * 32 * 16; }

__host__ __device__ inline int score_smem_bytes(int Q, int chunk) {
  return kScoreStages * kHalfTile + score_qfrag_bytes(Q) + Q * kGroup * 4 +
         chunk * kComputeWarps * Q * 4 + static_cast<int>(sizeof(ScoreSmemTail)) + 1024;
}

template <bool kHoist>
__global__ void __launch_bounds__(kThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap kv_map, const ScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int Q = p.Q, chunk = p.chunk;
  uint8_t* stages = smem;
  uint4* qfrag = reinterpret_cast<uint4*>(stages + kScoreStages * kHalfTile);  // [Q][8][32]
  float* qmul = reinterpret_cast<float*>(stages + kScoreStages * kHalfTile + score_qfrag_bytes(Q));
  float* red = qmul + Q * kGroup;                                  // [chunk][4][Q]
  ScoreSmemTail* tail = reinterpret_cast<ScoreSmemTail*>(red + chunk * kComputeWarps * Q);

  const int n0 = blockIdx.x * chunk;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.B * Q;

  int L = p.seq_lens[b];
  const bool seq_ok = L >= 0 && (L == 0 || (L - 1) / kPage < p.S);
  if (!seq_ok) L = 0;

  for (int idx = threadIdx.x; idx < chunk * kComputeWarps * Q; idx += kThreads) red[idx] = -INFINITY;

  if (warp == kComputeWarps) {
    if (!seq_ok && lane == 0 && blockIdx.x == 0) flag_error(p.err, MSA_ERR_SEQ_RANGE);
    const int n_hi = min(min(n0 + chunk, p.S), (L >= 1) ? (L - 1) / kPage + 1 : 0);
    const int n = n0 + lane;
    bool valid = false;
    int page = -1;
    if (lane < chunk && n < n_hi) {
      page = p.block_table[static_cast<int64_t>(b) * p.S + n];
      if (page < 0 || static_cast<int64_t>(page) >= p.num_blocks)
        flag_error(p.err, MSA_ERR_PAGE_RANGE);
      else
        valid = true;
    }
    const unsigned vm = __ballot_sync(0xffffffffu, valid);
    if (valid) {
      const int k = __popc(vm & ((1u << lane) - 1u));
      tail->pages[k] = page;
      tail->loc[k] = lane;
    }
    if (lane == 0) {
      tail->n_pages = __popc(vm);
      tail->abort = 0;
      for (int s = 0; s < kScoreStages; ++s) {
        mbar_init(&tail->full[s], 1);
        mbar_init(&tail->empty[s], kComputeWarps);
      }
      mbar_init(&tail->drained, kComputeWarps);
      fence_barrier_init();
    }
  }
  __syncthreads();
  const int n_pages = tail->n_pages;

  if (warp == kComputeWarps) {
    if (lane == 0) {
      prefetch_tensormap(&kv_map);
      for (int t = 0; t < n_pages; ++t) {
        const int s = t % kScoreStages;
        if (t >= kScoreStages && !mbar_wait(&tail->empty[s], ((t / kScoreStages) - 1) & 1)) {
          flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&tail->full[s], kHalfTile);
        tma_load_2d(stages + s * kHalfTile, &kv_map, 0, (tail->pages[t] * p.Hkv + g) * kPage,
                    &tail->full[s]);
      }
    }
    return;
  }

  // ---- query fragments of every token of the request, once per CTA ----------
  const int gr = lane >> 2, c = lane & 3;
  for (int jq = warp; jq < Q; jq += kComputeWarps) {
    uint32_t a[8][4];
    float mul0, mul1;
    load_query_fragments(p.q + ((static_cast<int64_t>(b) * Q + jq) * p.Hq + g * kGroup) * kHeadDim,
                         lane, p.scale, a, mul0, mul1);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      qfrag[(jq * 8 + ks) * 32 + lane] = make_uint4(a[ks][0], a[ks][1], a[ks][2], a[ks][3]);
    if (c == 0) {
      qmul[jq * kGroup + gr] = mul0;
      qmul[jq * kGroup + gr + 8] = mul1;
    }
  }
  named_barrier(1, kComputeWarps * 32);

  const int key0 = warp * 32;
  const int n_passes = (Q + kTokensPerPass - 1) / kTokensPerPass;
  uint32_t a[kTokensPerPass][8][4];
  float mul[kTokensPerPass][2];
  auto load_pass = [&](int pass) {
#pragma unroll
    for (int jj = 0; jj < kTokensPerPass; ++jj) {
      const int jq = min(pass * kTokensPerPass + jj, Q - 1);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint4 v = qfrag[(jq * 8 + ks) * 32 + lane];
        a[jj][ks][0] = v.x;
        a[jj][ks][1] = v.y;
        a[jj][ks][2] = v.z;
        a[jj][ks][3] = v.w;
      }
      mul[jj][0] = qmul[jq * kGroup + gr];
      mul[jj][1] = qmul[jq * kGroup + gr + 8];
    }
  };
  if (kHoist) load_pass(0);

  bool timed_out = false;
  int consumed = 0;
  for (int t = 0; t < n_pages; ++t) {
    const int s = t % kScoreStages;
    if (!mbar_wait(&tail->full[s], (t / kScoreStages) & 1)) {
      if (lane == 0) flag_error(p.err, MSA_ERR_TIMEOUT);
      timed_out = true;
      break;
    }
    consumed = t + 1;
    const uint8_t* kt = stages + s * kHalfTile;
    const int nl = tail->loc[t];
    const int n = n0 + nl;
    for (int pass = 0; pass < n_passes; ++pass) {
      // tokens of this pass that see at least one key of block n
      const int lim_base = L - Q - n * kPage;  // lim of token j is lim_base + j
      const int j_first = pass * kTokensPerPass;
      if (lim_base + min(j_first + kTokensPerPass, Q) - 1 < 0) continue;
      if (!kHoist) load_pass(pass);
      float runmax[kTokensPerPass][2];
#pragma unroll
      for (int jj = 0; jj < kTokensPerPass; ++jj) runmax[jj][0] = runmax[jj][1] = -INFINITY;
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        const int row = key0 + 8 * tt + gr;
        uint32_t bk[8][2];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(kt + sw128(row, ks) + 4 * c);
          bk[ks][0] = e4m3x2_to_f16x2(w & 0xFFFF);
          bk[ks][1] = e4m3x2_to_f16x2(w >> 16);
        }
        const int key = key0 + 8 * tt + 2 * c;
#pragma unroll
        for (int jj = 0; jj < kTokensPerPass; ++jj) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) mma_f16(acc, a[jj][ks], bk[ks][0], bk[ks][1]);
          const int lim = lim_base + j_first + jj;
          if (key <= lim) {
            runmax[jj][0] = fmaxf(runmax[jj][0], acc[0]);
            runmax[jj][1] = fmaxf(runmax[jj][1], acc[2]);
          }
          if (key + 1 <= lim) {
            runmax[jj][0] = fmaxf(runmax[jj][0], acc[1]);
            runmax[jj][1] = fmaxf(runmax[jj][1], acc[3]);
          }
        }
      }
#pragma unroll
      for (int jj = 0; jj < kTokensPerPass; ++jj) {
        const int jq = j_first + jj;
        float v = fmaxf(runmax[jj][0] * mul[jj][0], runmax[jj][1] * mul[jj][1]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
        if (lane == 0 && jq < Q) red[(nl * kComputeWarps + warp) * Q + jq] = v;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->empty[s]);
  }

  if (timed_out) {
    if (lane == 0) {
      *reinterpret_cast<volatile int*>(&tail->abort) = 1;
      __threadfence_block();
      mbar_arrive(&tail->drained);
    }
    for (int t = consumed; t < n_pages && t < consumed + kScoreStages; ++t)
      (void)mbar_wait(&tail->full[t % kScoreStages], (t / kScoreStages) & 1);
    return;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&tail->drained);
  if (!mbar_wait(&tail->drained, 0)) {
    if (lane == 0) flag_error(p.err, MSA_ERR_TIMEOUT);
    return;
  }
  if (*reinterpret_cast<volatile int*>(&tail->abort)) return;

  // ---- write the chunk's scores for every token (blocks not computed: -inf) --
  const int tid = threadIdx.x;
  for (int idx = tid; idx < chunk * Q; idx += kComputeWarps * 32) {
    const int jq = idx / chunk, nl = idx - jq * chunk;
    const int n = n0 + nl;
    if (n >= p.S) continue;
    float v = -INFINITY;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) v = fmaxf(v, red[(nl * kComputeWarps + w) * Q + jq]);
    p.scores[(static_cast<int64_t>(g) * T + static_cast<int64_t>(b) * Q + jq) * p.S + n] = v;
  }
}

}  // namespace

cudaError_t launch_score(const CUtensorMap& kv_map, const ScoreParams& p, cudaStream_t stream) {
  if (p.chunk < 1 || p.chunk > kMaxChunk) return cudaErrorInvalidValue;
  const int smem = score_smem_bytes(p.Q, p.chunk);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  const bool hoist = p.Q <= kTokensPerPass;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [] {
    constexpr int kMax = 227 * 1024;
    cudaError_t r = cudaFuncSetAttribute(score_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kMax);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(score_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kMax);
  });
  if (e != cudaSuccess) return e;
  dim3 grid((p.S + p.chunk - 1) / p.chunk, p.Hkv, p.B);
  if (hoist)
    score_kernel<true><<<grid, kThreads, smem, stream>>>(kv_map, p);
  else
    score_kernel<false><<<grid, kThreads, smem, stream>>>(kv_map, p);
  return cudaGetLastError();
}

}  // namespace msa
