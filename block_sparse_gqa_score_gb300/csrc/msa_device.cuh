// msa_device.cuh -- device helpers of the sm_103a sparse-decode kernels:
// inline PTX for mbarriers and TMA tile loads, fp8 conversions, warp
// reductions, and the preparation of fp8 query tiles for the tensor core.
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
// programmatic dependent launch
//
// pdl_trigger: this CTA lets the next kernel on the stream (launched with the
// programmatic stream serialization attribute) schedule its CTAs once every
// CTA of this grid has triggered or exited, so that their prologue overlaps
// this kernel's tail (the streaming kernels trigger after their last load).  pdl_wait: the calling thread
// waits until the previous kernel on the stream has completed and its memory
// writes are visible (at once when this launch overlapped no kernel).  Each
// kernel calls pdl_wait before its first read of a previous kernel's output
// and before its first write of anything a previous kernel may still read.

__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ----------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Invalidate an mbarrier that has no pending arrivals or waiters, so that it
// can be initialised again.
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// `count` arrivals at once (count >= 1).
__device__ __forceinline__ void mbar_arrive_count(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
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

// Whether phase `parity` of `bar` has completed, without waiting (try_wait may
// suspend the thread for a while before it reports an incomplete phase; a
// thread polling several barriers uses this instead).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
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

// Wait for phase `parity` of `bar` to complete, for at most limit_ns
// (mbar_wait: kWaitLimitNs).
// The first two tries carry no suspend-time hint: on the kernels' per-page
// hand-offs (TMA -> MMA -> softmax -> MMA) they return sooner after the phase
// completes than a hinted try does (the batch-16, qlen-4 step 69.3 vs 70.3 us,
// its attend alone 24.5 vs 25.1 us).  Longer waits then sleep inside try_wait
// with a 1 ms hint, leaving the issue slots to the warps doing work (polling
// with test_wait instead cost 17 us per step).  Returns false on timeout (the
// caller flags MSA_ERR_TIMEOUT and bails out).
__device__ __forceinline__ bool mbar_wait_limit(uint64_t* bar, unsigned parity,
                                                unsigned long long limit_ns) {
  constexpr unsigned kHintNs = 1000000u;  // re-check the time limit every 1 ms at most
  if (mbar_try_wait(bar, parity) || mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  const unsigned hint = limit_ns < kHintNs ? static_cast<unsigned>(limit_ns) : kHintNs;
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, hint)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  return mbar_wait_limit(bar, parity, kWaitLimitNs);
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

// Untiled bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global into shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, unsigned bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(smem_dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
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

__device__ __forceinline__ float exp2i(int e) {  // 2^e for |e| <= 126
  return __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
}

// Four floats -> four e4m3 bytes (x0 in the low byte).
__device__ __forceinline__ uint32_t f32x4_to_e4m3x4(float x0, float x1, float x2, float x3) {
  return f32x2_to_e4m3x2(x0, x1) | (f32x2_to_e4m3x2(x2, x3) << 16);
}

// Split of four floats (magnitude at most 448) into fp8 e4m3 hi + lo words:
// hi = x rounded to e4m3, lo = (x - hi) rounded to e4m3, so hi + lo carries
// about 8 significant bits of x, and is exact for a value with at most 8
// significant bits and magnitude in [2^-2, 2^8).
__device__ __forceinline__ void split_e4m3x4(const float (&x)[4], uint32_t& hi, uint32_t& lo) {
  const uint32_t h01 = f32x2_to_e4m3x2(x[0], x[1]), h23 = f32x2_to_e4m3x2(x[2], x[3]);
  uint32_t w01 = e4m3x2_to_f16x2(h01), w23 = e4m3x2_to_f16x2(h23);
  const __half2 f01 = *reinterpret_cast<const __half2*>(&w01);
  const __half2 f23 = *reinterpret_cast<const __half2*>(&w23);
  hi = h01 | (h23 << 16);
  lo = f32x4_to_e4m3x4(x[0] - __low2float(f01), x[1] - __high2float(f01),
                       x[2] - __low2float(f23), x[3] - __high2float(f23));
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Two non-negative floats (at most 448) -> fp8 e4m3 hi and lo pairs (x0 in
// the low byte): hi = x rounded to e4m3 (through fp16), lo = the remainder
// rounded to e4m3; hi + lo carries about 8 significant bits of x.
__device__ __forceinline__ void split_e4m3x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  uint16_t h8, l8;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(h8) : "r"(*reinterpret_cast<const uint32_t*>(&h)));
  const uint32_t hb = e4m3x2_to_f16x2(h8);
  const __half2 r = __hsub2(h, *reinterpret_cast<const __half2*>(&hb));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(l8) : "r"(*reinterpret_cast<const uint32_t*>(&r)));
  hi = h8;
  lo = l8;
}

// Largest of a float across the warp (every lane gets it); NaN inputs are
// ignored unless every lane holds one.
__device__ __forceinline__ float warp_max_f32(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}

// ----------------------------------------------------------------------------
// Query tiles for the fp8 tensor-core products.
//
// The 16 query rows of one (token, KV head) (bf16, 16 x 128, row stride 128)
// are scaled by a power of two 2^-e, e chosen so that the largest magnitude
// of the 16 rows lies in [2^7, 2^8), and split into fp8 e4m3 hi + lo parts
// (bf16's 8 significant bits are 4 + 4, so hi + lo equals the scaled value for
// every element of magnitude >= 2^-2, i.e. all but those 2^9 times smaller
// than the largest).  The parts are written as rows row0 .. row0+15 of two
// K-major tiles with 128-byte rows and 128-byte swizzling.  One warp (lane:
// row lane/2, d 64*(lane&1) .. +63).

// The lane's 64 bf16 values (global loads only; nothing waits on them yet).
__device__ __forceinline__ void load_query_rows(const uint16_t* __restrict__ rows, int lane,
                                                uint4 (&raw)[8]) {
  const uint4* src = reinterpret_cast<const uint4*>(rows + (lane >> 1) * kHeadDim + 64 * (lane & 1));
#pragma unroll
  for (int k = 0; k < 8; ++k) raw[k] = __ldg(src + k);
}

// Scale, split and store the values load_query_rows fetched; returns e (the
// same in every lane).
__device__ __forceinline__ int store_query_e4m3(const uint4 (&raw)[8], int row0, uint8_t* hi,
                                                uint8_t* lo, int lane) {
  const int r = lane >> 1, half = lane & 1;
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
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      const int el = 16 * c4 + 4 * wi;  // elements el .. el+3 of this lane's 64
      const uint4 v = raw[el >> 3];
      const uint32_t pair0 = ((el & 7) == 0) ? v.x : v.z;
      const uint32_t pair1 = ((el & 7) == 0) ? v.y : v.w;
      const float x[4] = {bf16_bits_to_f32(pair0 & 0xFFFF) * sd, bf16_bits_to_f32(pair0 >> 16) * sd,
                          bf16_bits_to_f32(pair1 & 0xFFFF) * sd, bf16_bits_to_f32(pair1 >> 16) * sd};
      split_e4m3x4(x, hw[wi], lw[wi]);
    }
    const int off = sw128(row0 + r, 4 * half + c4);
    *reinterpret_cast<uint4*>(hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  return e;
}

// max(a, b, c) in one instruction (the three-input fp32 max of sm_100 and
// later); exact, and like fmaxf it returns the other operands' max when one is
// NaN.
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// The largest of 16 fp32 values held as raw bits (8 three-input maxima).
__device__ __forceinline__ float max16(const uint32_t (&v)[16]) {
  float a[5];
#pragma unroll
  for (int k = 0; k < 5; ++k)
    a[k] = fmax3f(__uint_as_float(v[3 * k]), __uint_as_float(v[3 * k + 1]),
                  __uint_as_float(v[3 * k + 2]));
  return fmaxf(fmax3f(a[0], a[1], a[2]), fmax3f(a[3], a[4], __uint_as_float(v[15])));
}

// An fp8 e4m3 query token's 16 rows (16 heads x 128 B, contiguous) copied as
// stored into rows row0 .. row0 + 15 of a 128B-swizzled K-major tile; lane l
// moves 64 bytes of row l / 2.
__device__ __forceinline__ void store_query_rows_fp8(const uint8_t* __restrict__ rows, int row0,
                                                     uint8_t* tile, int lane) {
  const int r = lane >> 1, half = lane & 1;
  const uint4* src = reinterpret_cast<const uint4*>(rows + r * 128 + 64 * half);
  uint4 v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = __ldg(src + k);
#pragma unroll
  for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4*>(tile + sw128(row0 + r, 4 * half + k)) = v[k];
}

// Rows row0 .. row0 + 15 of a 128B-swizzled tile set to zero (lane l: 64
// bytes of row l / 2).
__device__ __forceinline__ void zero_query_rows(int row0, uint8_t* tile, int lane) {
  const int r = lane >> 1, half = lane & 1;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *reinterpret_cast<uint4*>(tile + sw128(row0 + r, 4 * half + k)) = make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ int prepare_query_e4m3(const uint16_t* __restrict__ rows, int row0,
                                                  uint8_t* hi, uint8_t* lo, int lane) {
  uint4 raw[8];
  load_query_rows(rows, lane, raw);
  return store_query_e4m3(raw, row0, hi, lo, lane);
}

}  // namespace msa
