// msa_device.cuh -- device helpers of the sm_103a sparse-decode kernels:
// inline PTX for mbarriers, TMA tile loads, the m16n8k16 fp16 tensor-core MMA,
// fp8 -> fp16 widening, and the fp16 query-row preparation.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "msa.h"

namespace msa {

constexpr int kHeadDim = 128;
constexpr int kPage = 128;
constexpr int kRowBytes = 256;    // one cached token: K (128 B) then V (128 B)
constexpr int kHalfTile = kPage * 128;  // bytes of one K or V half-page tile
constexpr int kTopK = 16;
constexpr int kGroup = 16;        // query heads per KV head
constexpr int kMaxQ = 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s bound on any wait

// ----------------------------------------------------------------------------
// error word

__device__ __forceinline__ void flag_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

// ----------------------------------------------------------------------------
// shared-memory addressing, timers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may be suspended (it issues nothing) for up
// to `hint_ns` while the phase is incomplete; it resumes when the phase
// completes or the hint expires.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, unsigned parity,
                                                    unsigned hint_ns) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, for at most kWaitLimitNs.
// Waiting warps sleep inside try_wait instead of spinning, so they leave the
// issue slots to the warps doing work.  Returns false on timeout (the caller
// flags MSA_ERR_TIMEOUT and bails out).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  constexpr unsigned kHintNs = 1000000u;  // re-check the time limit every 1 ms at most
  if (mbar_try_wait_sleep(bar, parity, kHintNs)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kHintNs)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ----------------------------------------------------------------------------
// TMA: 2-D tiled load global -> shared, completion counted on an mbarrier

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Byte offset of (row, 16-byte chunk) inside a [rows x 128 B] tile written by
// TMA with 128-byte swizzling (tile base 1024-byte aligned): the chunk index
// is XORed with the row index modulo 8.
__device__ __forceinline__ int sw128(int row, int chunk) {
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

// ----------------------------------------------------------------------------
// numerics

// Two fp8 e4m3 values (low byte first) -> two fp16 (low half first); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(two_bytes));
  return r;
}

// Two fp32 -> two fp8 e4m3 (round to nearest even, saturating), `lo` in the
// low byte of the result.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float x) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

// Power-of-two exponent e for a query row with largest magnitude `amax`, such
// that amax * 2^-e lies in [2^14, 2^15): the row then rounds to fp16 with every
// element >= amax * 2^-28 exact (bf16 has 8 significant bits).
__device__ __forceinline__ int row_exponent(float amax) {
  const int biased = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);
  if (biased == 0 || biased == 0xFF) return 0;  // zero/subnormal or non-finite row
  int e = biased - 127 - 14;
  return e < -100 ? -100 : (e > 100 ? 100 : e);
}

__device__ __forceinline__ float exp2i(int e) {  // 2^e for |e| <= 126
  return __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
}

// m16n8k16 tensor-core MMA, fp16 inputs, fp32 accumulate (in place).
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// m16n8k32 tensor-core MMA, fp8 e4m3 inputs, fp32 accumulate (in place).
// A (16 x 32, row): a0/a2 = row lane/4, k 4(lane%4)..+3 and 16 + that; a1/a3
// the same for row lane/4 + 8.  B (32 x 8, col): b0/b1 = k 4(lane%4)..+3 and
// 16 + that, column lane/4.
__device__ __forceinline__ void mma_e4m3_k32(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four floats -> four e4m3 bytes (x0 in the low byte).
__device__ __forceinline__ uint32_t f32x4_to_e4m3x4(float x0, float x1, float x2, float x3) {
  return f32x2_to_e4m3x2(x0, x1) | (f32x2_to_e4m3x2(x2, x3) << 16);
}

// Exact split of four floats (each with at most 8 significant bits and a
// magnitude below 2^8) into fp8 e4m3 hi + lo words with hi + lo == x for
// every element whose magnitude is at least 2^-2.
__device__ __forceinline__ void split_e4m3x4(const float (&x)[4], uint32_t& hi, uint32_t& lo) {
  const uint32_t h01 = f32x2_to_e4m3x2(x[0], x[1]), h23 = f32x2_to_e4m3x2(x[2], x[3]);
  uint32_t w01 = e4m3x2_to_f16x2(h01), w23 = e4m3x2_to_f16x2(h23);
  const __half2 f01 = *reinterpret_cast<const __half2*>(&w01);
  const __half2 f23 = *reinterpret_cast<const __half2*>(&w23);
  hi = h01 | (h23 << 16);
  lo = f32x4_to_e4m3x4(x[0] - __low2float(f01), x[1] - __high2float(f01),
                       x[2] - __low2float(f23), x[3] - __high2float(f23));
}

// Query fragments for the fp8 QK^T MMA (m16n8k32): the 16 query heads of one
// (token, KV head), scaled by a per-token power of two 2^-e so that the
// largest element lies in [2^7, 2^8), then split exactly into e4m3 hi + lo.
// Lane (gr = lane/4, c = lane%4) gets, for k-step ks (d = 32ks .. 32ks+31):
//   hi/lo[0] = row gr,   d 32ks + 4c .. +3      hi/lo[2] = row gr,   d +16
//   hi/lo[1] = row gr+8, d 32ks + 4c .. +3      hi/lo[3] = row gr+8, d +16
// Only k-step `ks_only` (0..3) is split and returned; the exponent e always
// comes from the whole token.  `mul` receives scale * 2^e.
__device__ __forceinline__ void load_query_fragments_e4m3(const uint16_t* __restrict__ q_rows,
                                                          int lane, float scale, int ks_only,
                                                          uint32_t (&hi)[4], uint32_t (&lo)[4],
                                                          float& mul) {
  const int gr = lane >> 2, c = lane & 3;
  uint2 raw[4][4];  // [ks][fragment register]
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
    for (int f = 0; f < 4; ++f) {
      const int row = gr + 8 * (f & 1), d = 32 * ks + 16 * (f >> 1) + 4 * c;
      raw[ks][f] = __ldg(reinterpret_cast<const uint2*>(q_rows + row * kHeadDim + d));
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int ks = 0; ks < 4; ++ks)
#pragma unroll
    for (int f = 0; f < 4; ++f) {
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(raw[ks][f].x & 0xFFFF)));
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(raw[ks][f].x >> 16)));
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(raw[ks][f].y & 0xFFFF)));
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(raw[ks][f].y >> 16)));
    }
  amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
  const int biased = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);
  int e = (biased == 0 || biased == 0xFF) ? 0 : biased - 127 - 7;
  e = e < -100 ? -100 : (e > 100 ? 100 : e);
  const float sd = exp2i(-e);
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    if (ks != ks_only) continue;
#pragma unroll
    for (int f = 0; f < 4; ++f) {
      const float x[4] = {bf16_bits_to_f32(raw[ks][f].x & 0xFFFF) * sd,
                          bf16_bits_to_f32(raw[ks][f].x >> 16) * sd,
                          bf16_bits_to_f32(raw[ks][f].y & 0xFFFF) * sd,
                          bf16_bits_to_f32(raw[ks][f].y >> 16) * sd};
      split_e4m3x4(x, hi[f], lo[f]);
    }
  }
  mul = scale * exp2i(e);
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ----------------------------------------------------------------------------
// Query fragments.
//
// The 128-wide head dimension is permuted inside every 16-wide k-step of the
// MMA so that each lane's four k values are four consecutive bytes of a cached
// fp8 key row: logical k (2c, 2c+1, 2c+8, 2c+9) of k-step ks <-> physical d
// (16ks + 4c .. 16ks + 4c + 3).  The same permutation is applied to q, so the
// dot products are unchanged.  Lane (gr = lane/4, c = lane%4) of a warp holds,
// for the 16 query heads of one (token, KV head), A-fragment registers
//   a[ks][0] = q[gr  ][16ks+4c .. +1]   a[ks][2] = q[gr  ][16ks+4c+2 .. +3]
//   a[ks][1] = q[gr+8][16ks+4c .. +1]   a[ks][3] = q[gr+8][16ks+4c+2 .. +3]
// as fp16 after scaling row r by 2^-e_r.  `mul0/mul1` receive
// `scale * 2^e_r` for rows gr and gr+8.
__device__ __forceinline__ void load_query_fragments(const uint16_t* __restrict__ q_rows,
                                                     int lane, float scale, uint32_t (&a)[8][4],
                                                     float& mul0, float& mul1) {
  const int gr = lane >> 2, c = lane & 3;
  const uint16_t* r0 = q_rows + gr * kHeadDim + 4 * c;
  const uint16_t* r1 = r0 + 8 * kHeadDim;
  uint2 raw0[8], raw1[8];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    raw0[ks] = __ldg(reinterpret_cast<const uint2*>(r0 + 16 * ks));
    raw1[ks] = __ldg(reinterpret_cast<const uint2*>(r1 + 16 * ks));
  }
  float amax0 = 0.f, amax1 = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    amax0 = fmaxf(amax0, fabsf(bf16_bits_to_f32(raw0[ks].x & 0xFFFF)));
    amax0 = fmaxf(amax0, fabsf(bf16_bits_to_f32(raw0[ks].x >> 16)));
    amax0 = fmaxf(amax0, fabsf(bf16_bits_to_f32(raw0[ks].y & 0xFFFF)));
    amax0 = fmaxf(amax0, fabsf(bf16_bits_to_f32(raw0[ks].y >> 16)));
    amax1 = fmaxf(amax1, fabsf(bf16_bits_to_f32(raw1[ks].x & 0xFFFF)));
    amax1 = fmaxf(amax1, fabsf(bf16_bits_to_f32(raw1[ks].x >> 16)));
    amax1 = fmaxf(amax1, fabsf(bf16_bits_to_f32(raw1[ks].y & 0xFFFF)));
    amax1 = fmaxf(amax1, fabsf(bf16_bits_to_f32(raw1[ks].y >> 16)));
  }
  amax0 = fmaxf(amax0, __shfl_xor_sync(0xffffffffu, amax0, 1));
  amax0 = fmaxf(amax0, __shfl_xor_sync(0xffffffffu, amax0, 2));
  amax1 = fmaxf(amax1, __shfl_xor_sync(0xffffffffu, amax1, 1));
  amax1 = fmaxf(amax1, __shfl_xor_sync(0xffffffffu, amax1, 2));
  const int e0 = row_exponent(amax0), e1 = row_exponent(amax1);
  const float s0 = exp2i(-e0), s1 = exp2i(-e1);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    a[ks][0] = pack_f16x2(bf16_bits_to_f32(raw0[ks].x & 0xFFFF) * s0,
                          bf16_bits_to_f32(raw0[ks].x >> 16) * s0);
    a[ks][2] = pack_f16x2(bf16_bits_to_f32(raw0[ks].y & 0xFFFF) * s0,
                          bf16_bits_to_f32(raw0[ks].y >> 16) * s0);
    a[ks][1] = pack_f16x2(bf16_bits_to_f32(raw1[ks].x & 0xFFFF) * s1,
                          bf16_bits_to_f32(raw1[ks].x >> 16) * s1);
    a[ks][3] = pack_f16x2(bf16_bits_to_f32(raw1[ks].y & 0xFFFF) * s1,
                          bf16_bits_to_f32(raw1[ks].y >> 16) * s1);
  }
  mul0 = scale * exp2i(e0);
  mul1 = scale * exp2i(e1);
}

// S = Q K^T for one warp: the 16 query heads of `a` against 32 keys
// (rows key0 .. key0+31) of a swizzled K half-page tile.  acc[tile][0..1] are
// row gr, keys key0 + 8*tile + 2c + {0,1}; acc[tile][2..3] row gr+8.
__device__ __forceinline__ void qk_32keys(const uint8_t* __restrict__ ktile, int key0, int lane,
                                          const uint32_t (&a)[8][4], float (&acc)[4][4]) {
  const int gr = lane >> 2, c = lane & 3;
#pragma unroll
  for (int t = 0; t < 4; ++t)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int row = key0 + 8 * t + gr;
      const uint32_t w = *reinterpret_cast<const uint32_t*>(ktile + sw128(row, ks) + 4 * c);
      mma_f16(acc[t], a[ks], e4m3x2_to_f16x2(w & 0xFFFF), e4m3x2_to_f16x2(w >> 16));
    }
  }
}

}  // namespace msa
