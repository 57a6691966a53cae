// msa_attend.cu -- stage 3 (sparse attend) and stage 4 (split merge).
//
// Operation: minimax_m3_sparse_attn_decode / msa_cutlass_sparse_decode on the
// vLLM MiniMax-M3 pages: each query row attends only the tokens of the <= 16
// blocks its KV head's top-k list names, causally limited to pos = seq_len -
// Q + j; padding rows give zero (TensorRT-LLM PR #17171, flash-decoding
// commit: "zeroed (not NaN) output for graph padding rows", fp32 split-K
// partials).
//
// Design (sm_103a):
//  * One CTA per (query token, KV head, split).  The token's 16 query heads of
//    the group form exactly one m16 tile of the MMA, so no rows are wasted and
//    pages are fetched per token; pages shared by the Q tokens of a request
//    are deduplicated by L2, since the tokens' CTAs run side by side.
//  * A producer warp streams each selected page-head (K half and V half, 16 KiB
//    each) with two TMA tile loads into a ring of 128B-swizzled shared-memory
//    stages; four compute warps each take 32 of the page's 128 keys.
//  * fp8 K/V bytes are widened to fp16 in registers (cvt.rn.f16x2.e4m3x2) while
//    building the MMA B fragments, so shared memory holds only the raw page.
//  * Each warp keeps its own online-softmax state (m, l, O) over its keys; the
//    four states are merged through shared memory at the end.
#include "msa_device.cuh"
#include "msa_launch.h"

namespace msa {

namespace {

constexpr int kComputeWarps = 4;
constexpr int kThreads = (kComputeWarps + 1) * 32;
constexpr int kStageBytes = 2 * kHalfTile;  // K tile then V tile

struct AttendSmemTail {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t drained;  // the compute warps are done with the stage ring
  uint64_t merged;   // the compute warps have written their softmax states
  int abort;         // set by a warp whose wait timed out
  int pages[kTopK];
  int blocks[kTopK];
  int n_pages;
  int pos;
};

// fp16 query fragments shared by the compute warps: [k-step][lane] uint4
constexpr int kQfragBytes = 8 * 32 * 16;
constexpr int kTailBytes = static_cast<int>((sizeof(AttendSmemTail) + 15) / 16 * 16);

template <int NST>
constexpr int attend_smem_bytes() {
  return NST * kStageBytes + kTailBytes + kQfragBytes + 1024;
}

// Returns the PRMT selector that gathers byte r of x and byte r of y into the
// low two bytes of the result.
__device__ __forceinline__ uint32_t pair_bytes(uint32_t x, uint32_t y, int r) {
  return __byte_perm(x, y, static_cast<uint32_t>(r | ((r + 4) << 4)));
}

template <int NST>
__global__ void __launch_bounds__(kThreads, 2)
    attend_kernel(const __grid_constant__ CUtensorMap kv_map, const AttendParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  AttendSmemTail* tail = reinterpret_cast<AttendSmemTail*>(smem + NST * kStageBytes);
  uint4* qfrag = reinterpret_cast<uint4*>(smem + NST * kStageBytes + kTailBytes);  // [8][32]

  const int i = blockIdx.x;      // query token
  const int g = blockIdx.y;      // KV head
  const int split = blockIdx.z;  // split-K part
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = i / p.Q, j = i - b * p.Q;

  // ---- prologue: the producer warp resolves this CTA's page list ----------
  if (warp == kComputeWarps) {
    const int L = p.seq_lens[b];
    const bool seq_ok = L >= 0 && (L == 0 || (L - 1) / kPage < p.S);
    if (!seq_ok && lane == 0) flag_error(p.err, MSA_ERR_SEQ_RANGE);
    const int pos = seq_ok ? L - p.Q + j : -1;
    int n = -1, page = -1;
    bool valid = false;
    if (lane < kTopK && pos >= 0) {
      n = p.topk[(static_cast<int64_t>(i) * p.Hkv + g) * kTopK + lane];
      if (n != -1) {
        if (n < 0 || n > pos / kPage)
          flag_error(p.err, MSA_ERR_TOPK_RANGE);
        else
          valid = true;
      }
    }
    // a block listed again at a later slot is dropped
    const unsigned same = __match_any_sync(0xffffffffu, valid ? n : -2 - lane);
    if (valid && (same & ((1u << lane) - 1u))) {
      flag_error(p.err, MSA_ERR_TOPK_DUP);
      valid = false;
    }
    if (valid) {
      page = p.block_table[static_cast<int64_t>(b) * p.S + n];
      if (page < 0 || static_cast<int64_t>(page) >= p.num_blocks) {
        flag_error(p.err, MSA_ERR_PAGE_RANGE);
        valid = false;
      }
    }
    const unsigned vm = __ballot_sync(0xffffffffu, valid);
    const int idx = __popc(vm & ((1u << lane) - 1u));
    const bool mine = valid && (idx % p.splits == split);
    const unsigned mm = __ballot_sync(0xffffffffu, mine);
    if (mine) {
      const int k = __popc(mm & ((1u << lane) - 1u));
      tail->pages[k] = page;
      tail->blocks[k] = n;
    }
    if (lane == 0) {
      tail->n_pages = __popc(mm);
      tail->pos = pos;
      for (int s = 0; s < NST; ++s) {
        mbar_init(&tail->full[s], 1);
        mbar_init(&tail->empty[s], kComputeWarps);
      }
      mbar_init(&tail->drained, kComputeWarps);
      mbar_init(&tail->merged, kComputeWarps);
      tail->abort = 0;
      fence_barrier_init();
    }
  }
  __syncthreads();
  const int n_pages = tail->n_pages;
  const int pos = tail->pos;

  if (warp == kComputeWarps) {
    // ---- producer: stream the selected page-heads through the stage ring ----
    if (lane == 0) {
      prefetch_tensormap(&kv_map);
      int issued = 0;
      for (int t = 0; t < n_pages; ++t) {
        const int s = t % NST;
        if (t >= NST && !mbar_wait(&tail->empty[s], ((t / NST) - 1) & 1)) {
          flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        uint8_t* st = smem + s * kStageBytes;
        const int row = (tail->pages[t] * p.Hkv + g) * kPage;
        mbar_arrive_expect_tx(&tail->full[s], kStageBytes);
        tma_load_2d(st, &kv_map, 0, row, &tail->full[s]);
        tma_load_2d(st + kHalfTile, &kv_map, kHeadDim, row, &tail->full[s]);
        ++issued;
      }
      (void)issued;
    }
    return;
  }

  // ---- compute warps ---------------------------------------------------------
  const int gr = lane >> 2, c = lane & 3;
  const int key0 = warp * 32;
  float zs0, zs1;  // logit scales (log2 units) of rows gr / gr+8, times their power-of-two factors
  {
    // every warp prepares the fp16 query fragments; warp w stores k-steps 2w, 2w+1
    uint32_t qa[8][4];
    load_query_fragments(p.q + (static_cast<int64_t>(i) * p.Hq + g * kGroup) * kHeadDim, lane,
                         p.logit_scale, qa, zs0, zs1);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      if ((ks >> 1) == warp)
        qfrag[ks * 32 + lane] = make_uint4(qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
  }
  named_barrier(1, kComputeWarps * 32);  // no wait precedes it: every compute warp arrives

  // m0/m1: the reference maximum used for rows gr / gr+8 (lazily raised: it
  // only moves when a page's maximum exceeds it by more than kLazy, so the
  // probabilities stay <= 2^kLazy, well inside fp16).
  constexpr float kLazy = 8.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[16][4];
#pragma unroll
  for (int dt = 0; dt < 16; ++dt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[dt][e] = 0.f;

  bool timed_out = false;
  int consumed = 0;
  for (int t = 0; t < n_pages; ++t) {
    const int s = t % NST;
    if (!mbar_wait(&tail->full[s], (t / NST) & 1)) {
      if (lane == 0) flag_error(p.err, MSA_ERR_TIMEOUT);
      timed_out = true;
      break;
    }
    consumed = t + 1;
    const uint8_t* kt = smem + s * kStageBytes;
    const uint8_t* vt = kt + kHalfTile;
    const int lim = pos - tail->blocks[t] * kPage;  // keys <= lim are visible
    const bool whole = lim >= kPage - 1;            // same for the whole CTA

    // S = Q K^T (fp16 MMA; fp8 keys widened in registers)
    float acc[4][4];
#pragma unroll
    for (int tt = 0; tt < 4; ++tt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[tt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint4 qv = qfrag[ks * 32 + lane];
      const uint32_t qa[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        const int row = key0 + 8 * tt + gr;
        const uint32_t w = *reinterpret_cast<const uint32_t*>(kt + sw128(row, ks) + 4 * c);
        mma_f16(acc[tt], qa, e4m3x2_to_f16x2(w & 0xFFFF), e4m3x2_to_f16x2(w >> 16));
      }
    }
    if (!whole) {
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        const int key = key0 + 8 * tt + 2 * c;
        if (key > lim) acc[tt][0] = acc[tt][2] = -INFINITY;
        if (key + 1 > lim) acc[tt][1] = acc[tt][3] = -INFINITY;
      }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      mx0 = fmaxf(mx0, fmaxf(acc[tt][0], acc[tt][1]));
      mx1 = fmaxf(mx1, fmaxf(acc[tt][2], acc[tt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mz0 = mx0 * zs0, mz1 = mx1 * zs1;   // page maxima in log2 units
    const bool r0 = mz0 > m0 + kLazy, r1 = mz1 > m1 + kLazy;
    if (__any_sync(0xffffffffu, r0 || r1)) {
      const float al0 = r0 ? ex2(m0 - mz0) : 1.f;  // ex2(-inf) = 0 on the first raise
      const float al1 = r1 ? ex2(m1 - mz1) : 1.f;
      if (r0) m0 = mz0;
      if (r1) m1 = mz1;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int dt = 0; dt < 16; ++dt) {
        o[dt][0] *= al0;
        o[dt][1] *= al0;
        o[dt][2] *= al1;
        o[dt][3] *= al1;
      }
    }
    // p = 2^(acc*zs - m); a row with no visible key yet has m = -inf and only
    // -inf logits, which give 0
    const float nm0 = (m0 == -INFINITY) ? 0.f : -m0;
    const float nm1 = (m1 == -INFINITY) ? 0.f : -m1;
    uint32_t pa[2][4];
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      const float p0 = ex2(fmaf(acc[tt][0], zs0, nm0)), p1 = ex2(fmaf(acc[tt][1], zs0, nm0));
      const float p2 = ex2(fmaf(acc[tt][2], zs1, nm1)), p3 = ex2(fmaf(acc[tt][3], zs1, nm1));
      l0 += p0 + p1;
      l1 += p2 + p3;
      // C fragments of key tiles (2k, 2k+1) form the A fragment of PV k-step k
      pa[tt >> 1][(tt & 1) * 2 + 0] = pack_f16x2(p0, p1);
      pa[tt >> 1][(tt & 1) * 2 + 1] = pack_f16x2(p2, p3);
    }

    // O += P V (fp16 MMA).  Logical d-column n of d-tile 4*q4 + r is physical
    // d = 4*(n + 8*q4) + r, so each lane's 4-byte load of one V row covers
    // four d-tiles; rows 2c, 2c+1, 2c+8, 2c+9 of the k-step give the B pairs.
    // On the current block's page, rows past the causal limit are zeroed so
    // that whatever bytes they hold cannot reach the output.
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int rb = key0 + 16 * kk + 2 * c;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int chunk = (gr >> 2) + 2 * q4;
        const int word = 4 * (gr & 3);
        uint32_t w0 = *reinterpret_cast<const uint32_t*>(vt + sw128(rb, chunk) + word);
        uint32_t w1 = *reinterpret_cast<const uint32_t*>(vt + sw128(rb + 1, chunk) + word);
        uint32_t w2 = *reinterpret_cast<const uint32_t*>(vt + sw128(rb + 8, chunk) + word);
        uint32_t w3 = *reinterpret_cast<const uint32_t*>(vt + sw128(rb + 9, chunk) + word);
        if (!whole) {
          if (rb > lim) w0 = 0u;
          if (rb + 1 > lim) w1 = 0u;
          if (rb + 8 > lim) w2 = 0u;
          if (rb + 9 > lim) w3 = 0u;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const uint32_t b0 = e4m3x2_to_f16x2(pair_bytes(w0, w1, r));
          const uint32_t b1 = e4m3x2_to_f16x2(pair_bytes(w2, w3, r));
          mma_f16(o[4 * q4 + r], pa[kk], b0, b1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->empty[s]);
  }

  if (timed_out) {
    // Tell the other warps to stop, release them from the two merge barriers,
    // and let copies already in flight land before the CTA's shared memory
    // goes away.
    if (lane == 0) {
      *reinterpret_cast<volatile int*>(&tail->abort) = 1;
      __threadfence_block();
      mbar_arrive(&tail->drained);
      mbar_arrive(&tail->merged);
    }
    for (int t = consumed; t < n_pages && t < consumed + NST; ++t)
      (void)mbar_wait(&tail->full[t % NST], (t / NST) & 1);
    return;
  }

  // ---- merge the four warps' states ------------------------------------------
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  // every warp must be done reading the stages before they are reused
  __syncwarp();
  if (lane == 0) mbar_arrive(&tail->drained);
  if (!mbar_wait(&tail->drained, 0)) {
    if (lane == 0) flag_error(p.err, MSA_ERR_TIMEOUT);
    return;
  }
  if (*reinterpret_cast<volatile int*>(&tail->abort)) return;
  float* s_o = reinterpret_cast<float*>(smem);                   // [4][16][128]
  float* s_m = s_o + kComputeWarps * kGroup * kHeadDim;          // [4][16]
  float* s_l = s_m + kComputeWarps * kGroup;                     // [4][16]
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    float4 lo0, hi0, lo1, hi1;  // rows gr and gr+8, d = 32q4 + 8c + (0..3 | 4..7)
    lo0 = make_float4(o[4 * q4 + 0][0], o[4 * q4 + 1][0], o[4 * q4 + 2][0], o[4 * q4 + 3][0]);
    hi0 = make_float4(o[4 * q4 + 0][1], o[4 * q4 + 1][1], o[4 * q4 + 2][1], o[4 * q4 + 3][1]);
    lo1 = make_float4(o[4 * q4 + 0][2], o[4 * q4 + 1][2], o[4 * q4 + 2][2], o[4 * q4 + 3][2]);
    hi1 = make_float4(o[4 * q4 + 0][3], o[4 * q4 + 1][3], o[4 * q4 + 2][3], o[4 * q4 + 3][3]);
    float* d0 = s_o + (warp * kGroup + gr) * kHeadDim + 32 * q4 + 8 * c;
    float* d1 = d0 + 8 * kHeadDim;
    *reinterpret_cast<float4*>(d0) = lo0;
    *reinterpret_cast<float4*>(d0 + 4) = hi0;
    *reinterpret_cast<float4*>(d1) = lo1;
    *reinterpret_cast<float4*>(d1 + 4) = hi1;
  }
  if (c == 0) {
    s_m[warp * kGroup + gr] = m0;
    s_m[warp * kGroup + gr + 8] = m1;
    s_l[warp * kGroup + gr] = l0;
    s_l[warp * kGroup + gr + 8] = l1;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&tail->merged);
  if (!mbar_wait(&tail->merged, 0)) {
    if (lane == 0) flag_error(p.err, MSA_ERR_TIMEOUT);
    return;
  }
  if (*reinterpret_cast<volatile int*>(&tail->abort)) return;

  // 128 threads: row r = tid / 8, 16 consecutive d per thread
  const int tid = threadIdx.x;
  const int r = tid >> 3, d0 = (tid & 7) * 16;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, s_m[w * kGroup + r]);
  float wt[kComputeWarps];
  float Lsum = 0.f;
#pragma unroll
  for (int w = 0; w < kComputeWarps; ++w) {
    const float mw = s_m[w * kGroup + r];
    wt[w] = (mw == -INFINITY) ? 0.f : ex2(mw - M);
    Lsum += wt[w] * s_l[w * kGroup + r];
  }
  float acc_o[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc_o[e] = 0.f;
#pragma unroll
  for (int w = 0; w < kComputeWarps; ++w) {
    const float* src = s_o + (w * kGroup + r) * kHeadDim + d0;
#pragma unroll
    for (int e = 0; e < 16; e += 4) {
      const float4 v = *reinterpret_cast<const float4*>(src + e);
      acc_o[e] += wt[w] * v.x;
      acc_o[e + 1] += wt[w] * v.y;
      acc_o[e + 2] += wt[w] * v.z;
      acc_o[e + 3] += wt[w] * v.w;
    }
  }
  const int h = g * kGroup + r;
  const int64_t row_idx = static_cast<int64_t>(i) * p.Hq + h;
  if (p.splits == 1) {
    const float f = (Lsum > 0.f) ? p.v_scale / Lsum : 0.f;
    uint32_t packed[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      packed[e] = f32_to_bf16_bits(acc_o[2 * e] * f) | (f32_to_bf16_bits(acc_o[2 * e + 1] * f) << 16);
    uint4* dst = reinterpret_cast<uint4*>(p.out + row_idx * kHeadDim + d0);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  } else {
    const int64_t rows = static_cast<int64_t>(p.B) * p.Q * p.Hq;
    float* dst = p.part_o + (static_cast<int64_t>(split) * rows + row_idx) * kHeadDim + d0;
#pragma unroll
    for (int e = 0; e < 16; e += 4)
      *reinterpret_cast<float4*>(dst + e) =
          make_float4(acc_o[e] * p.v_scale, acc_o[e + 1] * p.v_scale, acc_o[e + 2] * p.v_scale,
                      acc_o[e + 3] * p.v_scale);
    if ((tid & 7) == 0) {
      float* ml = p.part_ml + (static_cast<int64_t>(split) * rows + row_idx) * 2;
      ml[0] = M;
      ml[1] = Lsum;
    }
  }
}

// Split merge: one warp per (token, query head) row, 4 d-values per lane.
__global__ void __launch_bounds__(256)
    combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                   uint16_t* __restrict__ out, int64_t rows, int splits) {
  const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float M = -INFINITY;
  for (int s = lane; s < splits; s += 32) {
    const float m = part_ml[(s * rows + r) * 2], l = part_ml[(s * rows + r) * 2 + 1];
    if (l > 0.f) M = fmaxf(M, m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float m = part_ml[(s * rows + r) * 2], l = part_ml[(s * rows + r) * 2 + 1];
    if (!(l > 0.f)) continue;
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

constexpr int kAttendStages = 3;

}  // namespace

cudaError_t launch_attend(const CUtensorMap& kv_map, const AttendParams& p, cudaStream_t stream) {
  constexpr int smem = attend_smem_bytes<kAttendStages>();
  static_assert(smem <= 227 * 1024, "attend shared memory");
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [] {
    cudaError_t r = cudaFuncSetAttribute(attend_kernel<kAttendStages>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(attend_kernel<kAttendStages>,
                                cudaFuncAttributePreferredSharedMemoryCarveout,
                                static_cast<int>(cudaSharedmemCarveoutMaxShared));
  });
  if (e != cudaSuccess) return e;
  const int T = p.B * p.Q;
  dim3 grid(T, p.Hkv, p.splits);
  attend_kernel<kAttendStages><<<grid, kThreads, smem, stream>>>(kv_map, p);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* part_o, const float* part_ml, uint16_t* out, int64_t rows,
                           int splits, cudaStream_t stream) {
  const int64_t threads = rows * 32;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  combine_kernel<<<static_cast<unsigned>(grid), block, 0, stream>>>(part_o, part_ml, out, rows,
                                                                   splits);
  return cudaGetLastError();
}

}  // namespace msa
