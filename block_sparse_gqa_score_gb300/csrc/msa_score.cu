// msa_score.cu -- stage 1, the block scorer.
//
// Operation (TensorRT-LLM PR #17171, scorer commit): for each KV head g, query
// token i and logical block n, the causal max of sm_scale * k_scale * q.k over
// the query heads of g's group and the block's keys the token may see; -inf
// past the token's current block and for padding rows.  Output [Hkv, T, S].
//
// Design (sm_103a, tcgen05): one CTA per (chunk of logical blocks, KV head,
// request) -- a grid sized to the batch, not a 128-row query tile per token.
//  * warp 0 streams the K halves (16 KiB per page-head) of the chunk's pages
//    with TMA into 128B-swizzled stages;
//  * warp 1 issues, from one thread, kind::f8f6f4 MMAs with the fp8 K tile
//    straight from the TMA stage as operand A (M = 128 keys, K-major) and the
//    request's Q x 16 query rows as operand B (N = 16 Q), accumulating fp32
//    in tensor memory;
//  * warps 2-5 read the accumulator from tensor memory (one key per lane),
//    take the max over each token's 16 heads, apply the causal limit, and
//    reduce over the 128 keys.
// The bf16 query is represented exactly as the sum of two fp8 e4m3 parts
// (q' = hi + lo after a per-token power-of-two scale; bf16's 8 significant
// bits are 4 + 4), and both parts accumulate into the same tensor-memory
// columns, so the fp8 keys need no widening at all.
#include "msa_device.cuh"
#include "msa_launch.h"
#include "msa_tcgen05.cuh"

namespace msa {

namespace {

constexpr int kStages = 4;
constexpr int kThreads = 192;      // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2-5 epilogue
constexpr int kEpiWarp0 = 2;
constexpr int kMaxChunk = 32;
constexpr int kSmemPerSM = 233472;  // shared memory of one SM available to CTAs

struct ScoreTail {
  uint64_t full[kStages];   // TMA -> MMA
  uint64_t empty[kStages];  // MMA -> TMA
  uint64_t dfull[2];        // MMA -> epilogue (accumulator buffer ready)
  uint64_t dempty[2];       // epilogue -> MMA (accumulator buffer drained)
  uint64_t epi_done;        // epilogue warps finished their pages
  uint64_t finish;          // every role finished (TMEM may be freed)
  uint32_t tmem_base;
  int n_pages;
  int pages[kMaxChunk];
  int loc[kMaxChunk];
};

static_assert(alignof(ScoreTail) <= 16, "tail alignment");

struct ScoreGeometry {
  int Q, chunk, nh, Qu, ncols;
  int qtile_bytes;  // one of the hi / lo query tiles: 16 Q rows x 128 B
  // byte offsets from the 1024-aligned base; every region starts 16-byte aligned
  int off_qhi, off_qlo, off_qmul, off_red, off_tail;
  int smem_needed, smem_request;
};

__host__ __device__ constexpr int align16(int x) { return (x + 15) & ~15; }

__host__ __device__ inline ScoreGeometry score_geometry(int Q, int chunk) {
  ScoreGeometry G{};
  G.Q = Q;
  G.chunk = chunk;
  G.nh = (16 * Q > 256) ? 2 : 1;        // MMA N is at most 256: split the tokens in two
  G.Qu = (Q + G.nh - 1) / G.nh;         // tokens per accumulator unit
  int cols = 2 * 16 * G.Qu;             // two accumulator buffers
  int nc = 32;
  while (nc < cols) nc <<= 1;
  G.ncols = nc;
  G.qtile_bytes = 16 * Q * 128;
  G.off_qhi = kStages * kHalfTile;
  G.off_qlo = G.off_qhi + G.qtile_bytes;
  G.off_qmul = G.off_qlo + G.qtile_bytes;
  G.off_red = G.off_qmul + align16(Q * 4);
  G.off_tail = G.off_red + align16(chunk * 4 * Q * 4);
  G.smem_needed = G.off_tail + align16(static_cast<int>(sizeof(ScoreTail))) + 1024;
  // ask for enough shared memory that no more CTAs share an SM than its
  // tensor memory (512 columns) can hold at once
  const int kmax = 512 / nc;
  const int floor_bytes = kSmemPerSM / (kmax + 1) - 1024 + 16;
  G.smem_request = G.smem_needed > floor_bytes ? G.smem_needed : floor_bytes;
  return G;
}

__device__ __forceinline__ int order_int(float x) {
  const int i = __float_as_int(x);
  return i >= 0 ? i : i ^ 0x7FFFFFFF;
}

__device__ __forceinline__ float order_float(int i) {
  return __int_as_float(i >= 0 ? i : i ^ 0x7FFFFFFF);
}

__global__ void __launch_bounds__(kThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap kv_map, const ScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int Q = p.Q;
  const ScoreGeometry G = score_geometry(Q, p.chunk);
  uint8_t* stages = smem;                                         // [kStages][128][128 B]
  uint8_t* qhi = smem + G.off_qhi;                                // [16Q][128 B] swizzled
  uint8_t* qlo = smem + G.off_qlo;
  float* qmul = reinterpret_cast<float*>(smem + G.off_qmul);      // [Q]
  float* red = reinterpret_cast<float*>(smem + G.off_red);        // [chunk][4][Q]
  ScoreTail* tail = reinterpret_cast<ScoreTail*>(smem + G.off_tail);

  const int chunk = p.chunk;
  const int n0 = blockIdx.x * chunk;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.B * Q;

  int L = p.seq_lens[b];
  const bool seq_ok = L >= 0 && (L == 0 || (L - 1) / kPage < p.S);
  if (!seq_ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(p.err, MSA_ERR_SEQ_RANGE);
    L = 0;
  }
  const int n_hi = min(min(n0 + chunk, p.S), (L >= 1) ? (L - 1) / kPage + 1 : 0);
  const int n_end = min(n0 + chunk, p.S);

  if (n0 >= n_hi) {
    // nothing visible in this chunk: every score is -inf
    for (int idx = threadIdx.x; idx < (n_end - n0) * Q; idx += kThreads) {
      const int jq = idx / (n_end - n0), nl = idx - jq * (n_end - n0);
      p.scores[(static_cast<int64_t>(g) * T + static_cast<int64_t>(b) * Q + jq) * p.S + n0 + nl] =
          -INFINITY;
    }
    return;
  }

  for (int idx = threadIdx.x; idx < chunk * 4 * Q; idx += kThreads) red[idx] = -INFINITY;

  if (warp == 0) {
    // page list of the chunk
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
      for (int s = 0; s < kStages; ++s) {
        mbar_init(&tail->full[s], 1);
        mbar_init(&tail->empty[s], 1);
      }
      for (int s = 0; s < 2; ++s) {
        mbar_init(&tail->dfull[s], 1);
        mbar_init(&tail->dempty[s], 4);
      }
      mbar_init(&tail->epi_done, 4);
      mbar_init(&tail->finish, 6);
      fence_barrier_init();
    }
  } else if (warp == 1) {
    tc::tmem_alloc(&tail->tmem_base, G.ncols);
    tc::tmem_relinquish();
  }

  // ---- query tiles: per token, q' = q * 2^-e split into fp8 hi + lo -------------
  // Token j's 16 heads are rows 16j..16j+15 of both tiles; lane = (head, half of d).
  for (int jq = warp; jq < Q; jq += kThreads / 32) {
    const int r = lane >> 1, half = lane & 1;
    const uint16_t* src =
        p.q + ((static_cast<int64_t>(b) * Q + jq) * p.Hq + g * kGroup + r) * kHeadDim + 64 * half;
    uint4 raw[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) raw[k] = __ldg(reinterpret_cast<const uint4*>(src) + k);
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w[e] & 0xFFFF)));
        amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w[e] >> 16)));
      }
    }
    amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
    const int biased = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);
    int e = (biased == 0 || biased == 0xFF) ? 0 : biased - 127 - 7;  // amax*2^-e in [2^7, 2^8)
    e = e < -100 ? -100 : (e > 100 ? 100 : e);
    const float sd = exp2i(-e);
    const int R = jq * kGroup + r;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        // elements 16*c4 + 4*wi .. +3 of this lane's 64
        const int el = 16 * c4 + 4 * wi;
        const uint4 v = raw[el >> 3];
        const uint32_t pair0 = ((el & 7) == 0) ? v.x : v.z;
        const uint32_t pair1 = ((el & 7) == 0) ? v.y : v.w;
        float x[4] = {bf16_bits_to_f32(pair0 & 0xFFFF) * sd, bf16_bits_to_f32(pair0 >> 16) * sd,
                      bf16_bits_to_f32(pair1 & 0xFFFF) * sd, bf16_bits_to_f32(pair1 >> 16) * sd};
        const uint32_t h01 = f32x2_to_e4m3x2(x[0], x[1]), h23 = f32x2_to_e4m3x2(x[2], x[3]);
        uint32_t w01 = e4m3x2_to_f16x2(h01), w23 = e4m3x2_to_f16x2(h23);
        const __half2 f01 = *reinterpret_cast<const __half2*>(&w01);
        const __half2 f23 = *reinterpret_cast<const __half2*>(&w23);
        const uint32_t l01 = f32x2_to_e4m3x2(x[0] - __low2float(f01), x[1] - __high2float(f01));
        const uint32_t l23 = f32x2_to_e4m3x2(x[2] - __low2float(f23), x[3] - __high2float(f23));
        hw[wi] = h01 | (h23 << 16);
        lw[wi] = l01 | (l23 << 16);
      }
      const int off = sw128(R, 4 * half + c4);
      *reinterpret_cast<uint4*>(qhi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(qlo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    if (lane == 0) qmul[jq] = p.scale * exp2i(e);
  }
  tc::fence_proxy_async_smem();   // query tiles are read by the tensor core
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const int n_pages = tail->n_pages;
  const uint32_t tmem = tail->tmem_base;

  if (warp == 0) {
    // ---- TMA producer ----------------------------------------------------------
    if (lane == 0) {
      prefetch_tensormap(&kv_map);
      int issued = 0;
      for (int t = 0; t < n_pages; ++t) {
        const int s = t % kStages;
        if (t >= kStages && !mbar_wait(&tail->empty[s], ((t / kStages) - 1) & 1)) {
          flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&tail->full[s], kHalfTile);
        tma_load_2d(stages + s * kHalfTile, &kv_map, 0, (tail->pages[t] * p.Hkv + g) * kPage,
                    &tail->full[s]);
        ++issued;
      }
      // the last loads in flight land before shared memory can be released
      for (int t = issued - kStages; t < issued; ++t)
        if (t >= 0) (void)mbar_wait(&tail->full[t % kStages], (t / kStages) & 1);
      mbar_arrive(&tail->finish);
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----------------------------------------------------------------
    if (lane == 0) {
      const uint32_t stage_addr = smem_u32(stages);
      const uint32_t qhi_addr = smem_u32(qhi), qlo_addr = smem_u32(qlo);
      bool ok = true;
      for (int t = 0; t < n_pages && ok; ++t) {
        const int s = t % kStages;
        if (!mbar_wait(&tail->full[s], (t / kStages) & 1)) {
          flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        tc::fence_after_thread_sync();
        const uint32_t a_base = stage_addr + s * kHalfTile;
        for (int h = 0; h < G.nh; ++h) {
          const int u = t * G.nh + h, buf = u & 1, use = u >> 1;
          if (use >= 1) {
            if (!mbar_wait(&tail->dempty[buf], (use - 1) & 1)) {
              flag_error(p.err, MSA_ERR_TIMEOUT);
              ok = false;
              break;
            }
            tc::fence_after_thread_sync();
          }
          const int tok0 = h * G.Qu, ntok = min(G.Qu, Q - tok0);
          const uint32_t idesc = tc::idesc_e4m3_f32(128, 16 * ntok);
          const uint32_t d = tmem + buf * 16 * G.Qu;
          const uint32_t b_off = tok0 * kGroup * 128;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc::mma_e4m3(d, tc::sw128_kmajor_desc(a_base + 32 * ks),
                         tc::sw128_kmajor_desc(qhi_addr + b_off + 32 * ks), idesc, ks > 0);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc::mma_e4m3(d, tc::sw128_kmajor_desc(a_base + 32 * ks),
                         tc::sw128_kmajor_desc(qlo_addr + b_off + 32 * ks), idesc, 1);
          tc::commit(&tail->dfull[buf]);
        }
        tc::commit(&tail->empty[s]);
      }
      mbar_arrive(&tail->finish);
    }
    __syncwarp();
    // free tensor memory once every role is done with it
    (void)mbar_wait(&tail->finish, 0);
    tc::fence_after_thread_sync();
    tc::tmem_dealloc(tmem, G.ncols);
  } else {
    // ---- epilogue: accumulator -> per-token block maxima ----------------------------
    const int quarter = warp & 3;                // TMEM lanes 32*quarter .. +31
    const int key = 32 * quarter + lane;         // key (row of the page) of this thread
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
    bool ok = true;
    for (int t = 0; t < n_pages && ok; ++t) {
      const int nl = tail->loc[t];
      const int lim_base = L - Q - (n0 + nl) * kPage;   // token j sees keys <= lim_base + j
      for (int h = 0; h < G.nh; ++h) {
        const int u = t * G.nh + h, buf = u & 1, use = u >> 1;
        if (!mbar_wait(&tail->dfull[buf], use & 1)) {
          if (lane == 0) flag_error(p.err, MSA_ERR_TIMEOUT);
          ok = false;
          break;
        }
        tc::fence_after_thread_sync();
        const int tok0 = h * G.Qu, ntok = min(G.Qu, Q - tok0);
        for (int jj = 0; jj < ntok; ++jj) {
          const int jq = tok0 + jj;
          const int lim = lim_base + jq;
          if (lim < 0) continue;                 // warp-uniform: token sees nothing here
          uint32_t v[16];
          tc::ld_32x32b_x16(lane_addr + buf * 16 * G.Qu + jj * 16, v);
          tc::wait_ld();
          float m = __uint_as_float(v[0]);
#pragma unroll
          for (int e = 1; e < 16; ++e) m = fmaxf(m, __uint_as_float(v[e]));
          if (key > lim) m = -INFINITY;
          const float wmax = order_float(__reduce_max_sync(0xffffffffu, order_int(m)));
          if (lane == 0) red[(nl * 4 + quarter) * Q + jq] = wmax;
        }
        tc::fence_before_thread_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->dempty[buf]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->epi_done);
    const bool all_done = mbar_wait(&tail->epi_done, 0);
    if (all_done && ok) {
      // write the chunk's scores for every token (blocks not computed: -inf)
      const int et = threadIdx.x - kEpiWarp0 * 32;
      for (int idx = et; idx < (n_end - n0) * Q; idx += 128) {
        const int jq = idx / (n_end - n0), nl = idx - jq * (n_end - n0);
        float v = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) v = fmaxf(v, red[(nl * 4 + w) * Q + jq]);
        if (v != -INFINITY) v *= qmul[jq];
        p.scores[(static_cast<int64_t>(g) * T + static_cast<int64_t>(b) * Q + jq) * p.S + n0 + nl] =
            v;
      }
    } else if (!all_done && lane == 0) {
      flag_error(p.err, MSA_ERR_TIMEOUT);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->finish);
  }
}

}  // namespace

cudaError_t launch_score(const CUtensorMap& kv_map, const ScoreParams& p, cudaStream_t stream) {
  if (p.chunk < 1 || p.chunk > kMaxChunk) return cudaErrorInvalidValue;
  const ScoreGeometry G = score_geometry(p.Q, p.chunk);
  if (G.smem_request > 227 * 1024) return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                227 * 1024);
  });
  if (e != cudaSuccess) return e;
  dim3 grid((p.S + p.chunk - 1) / p.chunk, p.Hkv, p.B);
  score_kernel<<<grid, kThreads, G.smem_request, stream>>>(kv_map, p);
  return cudaGetLastError();
}

}  // namespace msa
