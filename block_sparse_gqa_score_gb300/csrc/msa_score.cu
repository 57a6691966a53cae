// msa_score.cu -- stage 1, the block scorer.
//
// Operation (TensorRT-LLM PR #17171, scorer commit): for each KV head g, query
// token i and logical block n, the causal max of sm_scale * k_scale * q.k over
// the query heads of g's group and the block's keys the token may see; -inf
// past the token's current block and for padding rows.  Output [Hkv, T, S].
//
// Design (sm_103a, tcgen05, persistent): one or two CTAs per SM (two whenever
// tensor and shared memory hold two pipelines).  The visible pages of
// the batch, in (request, KV head, block) order, are split into equal
// contiguous ranges, one per CTA; every CTA derives the same split from
// seq_lens with a block-wide prefix sum, so no scratch memory or atomics are
// needed and the grid stays fixed for a given shape.  Inside a CTA:
//  * warp 0 streams the K halves (16 KiB per page-head) of its range with TMA
//    into a ring of 128B-swizzled stages, from the first microseconds on;
//  * warp 1 issues, from one thread, kind::f8f6f4 MMAs with the fp8 K tile
//    straight from the TMA stage as operand A (M = 128 keys, K-major) and the
//    request's Q x 16 query rows as operand B (N = 16 Q), accumulating fp32 in
//    two or four tensor-memory accumulator buffers;
//  * warp 2 prepares the query tile of each (request, KV head) unit of the
//    range (the first one together with warps 3-6, a token each): the bf16
//    query, scaled per token by a power of two 2^-e, is represented exactly
//    as the sum of two fp8 e4m3 parts (bf16's 8 significant bits are 4 + 4)
//    that accumulate into the same columns (up to qlen 2: side by side as one
//    B operand of N = 32 Q, summed by the epilogue), so the fp8 keys need no
//    widening (an fp8 query, value q8 * q_scale, is the hi part as stored and
//    only its MMAs are issued: half the tensor work); it also writes the -inf
//    tails;
//  * warps 3-6 read the accumulator (one key per lane), take each token's max
//    over its 16 heads and visible keys, and publish their four quarter-page
//    maxima through shared memory and a per-slot mbarrier; with one CTA per
//    SM (qlen >= 8, where this epilogue costs as much as the MMAs) warps 8-19
//    form three more sets on the same lane quarters, the four sets taking
//    groups of two tokens in turn (20 warps: registers capped near 96);
//  * warp 7 combines the quarters and writes the scores.
#include "msa_device.cuh"
#include "msa_launch.h"
#include "msa_tcgen05.cuh"

namespace msa {

namespace {

// 8 warps, see above; 20 with the extra epilogue warp sets (ScoreGeometry::threads)
constexpr int kMaxWarps = 20;
constexpr int kWideSub = 4;      // epilogue warp sets when one CTA runs per SM
constexpr int kMaxAcc = 4;          // tensor-memory accumulator buffers
constexpr int kMaxStages = 8;
constexpr int kRedSlots = 8;        // pages in flight between the epilogue warps
// A second unit that starts within this many pages of a CTA's range gets its
// query tile in the prologue (bf16 query, two CTAs per SM), from the warps
// that build the first one: built by the query warp alone (about a microsecond per token) it
// came late, and the CTAs whose range crosses a unit boundary in its first
// pages ran up to 6 us behind the rest (a page every 1.2-1.3 us, not 1.02).
constexpr int kNearUnit = 8;
constexpr int kQmulRing = 16;       // units whose scale factors are kept (> nqb + nacc + kRedSlots)
constexpr int kSmemLimit = 227 * 1024;
constexpr int kSmemPerSM = 233472;  // shared memory of one SM available to CTAs
static_assert(kMaxStages <= 32 && kMaxAcc <= 32 && kRedSlots <= 32 && kQmulRing <= 32,
              "one lane initialises each barrier of a ring");

struct ScoreTail {
  uint64_t full[kMaxStages];   // TMA -> MMA
  uint64_t empty[kMaxStages];  // MMA -> TMA
  uint64_t dfull[kMaxAcc];     // MMA -> epilogue (accumulator buffer ready)
  uint64_t dempty[kMaxAcc];    // epilogue -> MMA (accumulator buffer drained)
  uint64_t red_full[kRedSlots];   // epilogue -> combiner (four quarter maxima written)
  uint64_t red_empty[kRedSlots];  // combiner -> epilogue (slot read)
  uint64_t qfull[2];           // query prep -> MMA (query tile ready)
  uint64_t qempty[2];          // MMA -> query prep (query tile no longer read)
  uint64_t qmul_ready[kQmulRing];  // query prep -> epilogue (unit scale factors)
  uint64_t qstage;             // query prep -> TMA: the last stage, the first tile's staging, is free
  uint64_t finish;             // every role finished (TMEM may be freed)
  uint32_t tmem_base;
  int start_b, start_rem, count;   // this CTA's page range
  int any_invalid;                 // some page of the range has a bad block-table entry
  int64_t warp_sums[kMaxWarps];
};

struct ScoreGeometry {
  int Q, nh, Qu, nacc, ncols, nqb, stages, per_sm;
  int fuse;     // a bf16 query's hi and lo parts in one MMA (N = 32 Qu), summed by the epilogue
  int ucols;    // accumulator columns of one unit: 16 Qu, or 32 Qu when fused
  int nsub;     // epilogue warps per TMEM lane quarter (2 with one CTA per SM)
  int threads;  // 32 * (8 + 4 * (nsub - 1))
  int qtile_bytes;  // hi + lo query tiles of one unit: 2 x 16Q rows x 128 B
  int off_q, off_qmul, off_red, off_tail, smem;
};

__host__ __device__ constexpr int align16(int x) { return (x + 15) & ~15; }

__host__ __device__ inline ScoreGeometry score_geometry(int Q, bool fp8) {
  ScoreGeometry G{};
  G.Q = Q;
  G.nh = (16 * Q > 256) ? 2 : 1;        // MMA N is at most 256: split the tokens in two
  G.Qu = (Q + G.nh - 1) / G.nh;         // tokens per accumulator unit
  // Up to qlen 2 the hi and lo query tiles, adjacent in shared memory, form
  // one B operand of N = 32 Qu <= 64: the K tile is read once per k-step
  // instead of twice, and the two parts land in separate columns (batch 128,
  // qlen 1: scorer 232 -> 215 us).  At qlen 4 the wider accumulators would
  // leave room for two buffers instead of four, which measured slower
  // (43.3 vs 40.9 us at batch 16).
  G.fuse = (!fp8 && kMaxAcc * 32 * G.Qu <= 256) ? 1 : 0;
  G.ucols = (G.fuse ? 32 : 16) * G.Qu;
  G.nacc = (kMaxAcc * G.ucols <= 256) ? kMaxAcc : 2;   // accumulator buffers
  int cols = G.nacc * G.ucols;
  int nc = 32;
  while (nc < cols) nc <<= 1;
  G.ncols = nc;
  G.qtile_bytes = 2 * 16 * Q * 128;
  // two CTAs per SM (two independent pipelines) when tensor memory and shared
  // memory hold two; each then gets half an SM's shared memory
  const int two_budget = kSmemPerSM / 2 - 1024;
  // Small query tiles are double-buffered: the next unit's tile is built
  // while the current one is in use.  (A single buffer, which leaves room for
  // one more K stage at qlen 2-8, measured slower at qlen 4: 43.1 vs 40.3 us,
  // the tile hand-over at a unit boundary stalling the CTAs that cross one.)
  G.nqb = (2 * G.qtile_bytes <= 64 * 1024) ? 2 : 1;
  auto fixed_for = [&](int nqb) {
    return nqb * G.qtile_bytes + align16(kQmulRing * Q * 4) + align16(kRedSlots * 4 * Q * 4) +
           align16(static_cast<int>(sizeof(ScoreTail))) + 1024;
  };
  const int fixed1 = fixed_for(G.nqb);
  G.per_sm = (nc <= 256 && (two_budget - fixed1) / kHalfTile >= 3) ? 2 : 1;
  // one CTA per SM has the registers for a second set of epilogue warps
  G.nsub = G.per_sm == 1 ? kWideSub : 1;
  G.threads = 32 * (8 + 4 * (G.nsub - 1));
  const int red_bytes = align16(kRedSlots * 4 * G.nsub * Q * 4);
  const int fixed = fixed1 - align16(kRedSlots * 4 * Q * 4) + red_bytes;
  const int budget = G.per_sm == 2 ? two_budget : kSmemLimit;
  int st = (budget - fixed) / kHalfTile;
  G.stages = st > kMaxStages ? kMaxStages : st;
  G.off_q = G.stages * kHalfTile;
  G.off_qmul = G.off_q + G.nqb * G.qtile_bytes;
  G.off_red = G.off_qmul + align16(kQmulRing * Q * 4);
  G.off_tail = G.off_red + red_bytes;
  G.smem = G.off_tail + align16(static_cast<int>(sizeof(ScoreTail))) + 1024;
  return G;
}

// Whether the first query tile is staged through the last K stage: one
// query buffer, and the tile's raw rows (Q tokens x 16 rows) fit in a stage.
__host__ __device__ inline bool stage_staging(const ScoreGeometry& G, bool fp8) {
  return G.nqb == 1 && G.Q * kGroup * (fp8 ? 128 : 256) <= kHalfTile;
}

// Where the first unit's raw query rows are staged: the second tile buffer
// (free until the second tile is built) or, with one buffer, the last K
// stage (which the producer loads only once the first tile is built).
__device__ __forceinline__ uint8_t* first_tile_staging(const ScoreGeometry& G, bool fp8,
                                                       uint8_t* stages, uint8_t* qtiles) {
  return G.nqb == 2 ? qtiles + G.qtile_bytes
         : stage_staging(G, fp8) ? stages + (G.stages - 1) * kHalfTile : nullptr;
}

__device__ __forceinline__ int order_int(float x) {
  const int i = __float_as_int(x);
  return i >= 0 ? i : i ^ 0x7FFFFFFF;
}

__device__ __forceinline__ float order_float(int i) {
  return __int_as_float(i >= 0 ? i : i ^ 0x7FFFFFFF);
}

// Visible blocks of request b: ceil(seq_len / 128), or 0 for an empty or
// inconsistent request (seq_len < 0 or more blocks than the table holds).
__device__ __forceinline__ int visible_blocks(const ScoreParams& p, int b) {
  const int L = p.seq_lens[b];
  if (L <= 0 || (L - 1) / kPage >= p.S) return 0;
  return (L - 1) / kPage + 1;
}

// Sequential walk over this CTA's pages in (request, KV head, block) order.
struct PageWalk {
  int b, g, n, nhi, L;
  __device__ void load(const ScoreParams& p) {
    L = p.seq_lens[b];
    nhi = visible_blocks(p, b);
  }
  __device__ void begin(const ScoreParams& p, int b0, int rem) {
    b = b0;
    load(p);
    g = rem / nhi;
    n = rem - g * nhi;
  }
  // Move k pages forward (k >= 0), crossing requests as needed.
  __device__ void advance(const ScoreParams& p, int64_t k) {
    while (k > 0 && b < p.B) {
      const int64_t here = static_cast<int64_t>(g) * nhi + n;
      const int64_t left = static_cast<int64_t>(p.Hkv) * nhi - here;  // incl. the current page
      if (k < left) {
        const int64_t rem = here + k;
        g = static_cast<int>(rem / nhi);
        n = static_cast<int>(rem - static_cast<int64_t>(g) * nhi);
        return;
      }
      k -= left;
      g = 0;
      n = 0;
      do {
        ++b;
        if (b >= p.B) return;
        load(p);
      } while (nhi == 0);
    }
  }
  __device__ void next(const ScoreParams& p) {
    if (++n < nhi) return;
    n = 0;
    if (++g < p.Hkv) return;
    g = 0;
    do {
      ++b;
      if (b >= p.B) return;
      load(p);
    } while (nhi == 0);
  }
};

// Whether the range's second unit (if any) starts within kNearUnit pages, so
// that the prologue builds its tile too (two tile buffers only).
__device__ __forceinline__ bool second_tile_early(const ScoreGeometry& G, const PageWalk& w0,
                                                  int count) {
  const int first_len = w0.nhi - w0.n;   // pages of the first unit in the range
  return G.nqb == 2 && first_len < count && first_len <= kNearUnit;
}

__device__ __forceinline__ bool page_valid(const ScoreParams& p, const PageWalk& w, int& page) {
  page = p.block_table[static_cast<int64_t>(w.b) * p.S + w.n];
  return page >= 0 && static_cast<int64_t>(page) < p.num_blocks;
}

// Query tile of unit (b, g) into hi / lo (16 Q rows x 128 B each, 128B
// swizzled, K-major), per-token factors into qmul[0..Q): a bf16 query scaled
// by 2^-e and split exactly into hi + lo (factor scale * 2^e), or an fp8 query
// as stored in hi (lo unused; factor scale * q_scale).  The calling warp
// builds tokens j0, j0 + jstep, ... (each token's scale is its own).  With
// `staging` (Q * 4 KiB of shared memory nothing else uses meanwhile), those
// tokens' rows are first copied there with asynchronous copies, all in flight
// at once, so that the tile costs one memory round trip instead of one per
// token.
template <bool kFp8Q, bool kShared = false>
__device__ void prepare_query_tile(const ScoreParams& p, int b, int g, uint8_t* qhi, uint8_t* qlo,
                                   float* qmul, int lane, uint8_t* staging, int j0_ = 0,
                                   int jstep_ = 1) {
  // kShared: several warps build the tile, this one tokens j0, j0 + jstep, ...;
  // otherwise all tokens, in a plain loop
  const int j0 = kShared ? j0_ : 0, jstep = kShared ? jstep_ : 1;
  constexpr int kRowBytes = kFp8Q ? 128 : 256;   // one query head's row
  constexpr int kTokBytes = kGroup * kRowBytes;  // one token's 16 rows, contiguous
  if (staging) {
    for (int jq = j0; jq < p.Q; jq += jstep) {
      const int64_t row = (static_cast<int64_t>(b) * p.Q + jq) * p.Hq + g * kGroup;
      const uint8_t* src = kFp8Q ? p.q8 + row * kHeadDim
                                 : reinterpret_cast<const uint8_t*>(p.q + row * kHeadDim);
      for (int c = lane; c < kTokBytes / 16; c += 32)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(
                         smem_u32(staging + jq * kTokBytes + 16 * c)),
                     "l"(src + 16 * c)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    __syncwarp();
  }
  for (int jq = j0; jq < p.Q; jq += jstep) {
    const int64_t row = (static_cast<int64_t>(b) * p.Q + jq) * p.Hq + g * kGroup;
    if constexpr (kFp8Q) {
      if (staging) {
        // lane l: 64 bytes of row l / 2, copied as stored into the swizzled tile
        const int r = lane >> 1, half = lane & 1;
        const uint4* src = reinterpret_cast<const uint4*>(staging + jq * kTokBytes + r * 128 + 64 * half);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4*>(qhi + sw128(jq * kGroup + r, 4 * half + k)) = src[k];
      } else
        store_query_rows_fp8(p.q8 + row * kHeadDim, jq * kGroup, qhi, lane);
      if (lane == 0) qmul[jq] = p.scale * p.q_scale;
    } else {
      uint4 raw[8];
      if (staging) {
        const uint4* src = reinterpret_cast<const uint4*>(staging + jq * kTokBytes +
                                                          (lane >> 1) * kRowBytes + 128 * (lane & 1));
#pragma unroll
        for (int k = 0; k < 8; ++k) raw[k] = src[k];
      } else {
        load_query_rows(p.q + row * kHeadDim, lane, raw);
      }
      const int e = store_query_e4m3(raw, jq * kGroup, qhi, qlo, lane);
      if (lane == 0) qmul[jq] = p.scale * exp2i(e);
    }
  }
}

// At most 128 registers: registers are allocated per SM sub-partition (16K
// each), so two 7-warp CTAs per SM need <= 128 per thread.  kFp8Q: the query
// is fp8 (q8 * q_scale), compiled separately so that the bf16 kernel carries
// none of its branches.  kWide: the extra sets of epilogue warps (one CTA
// per SM, 640 threads), likewise a separate instantiation; the launch bounds
// keep 128 registers for the two-CTA kernel.  kFuse: a bf16 query's hi and lo
// parts in one product (qlen <= 2, ScoreGeometry::fuse), its own
// instantiation too, so that the qlen 3-8 kernel carries none of it.  kQ:
// the query length as a compile-time constant (0: read from the arguments).
// With it the whole geometry (stages, accumulator and tile buffers, token
// groups) is constant, and the ring indices of the per-page loops divide by
// constants instead of by runtime values: the qlen-4 scorer went from 39.9
// to 31.6 us.  The common lengths are instantiated (see launch_score).
template <bool kFp8Q, bool kWide, bool kFuse = false, int kQ = 0>
__global__ void __launch_bounds__(kWide ? 640 : 256, kWide ? 1 : 2)
    score_kernel(const __grid_constant__ CUtensorMap kv_map, const ScoreParams p) {
  constexpr int kSub = kWide ? kWideSub : 1;              // epilogue warps per TMEM lane quarter
  constexpr int kGrp = kWide ? 2 : 4;              // tokens per epilogue group
  constexpr int kNumThreads = 32 * (8 + 4 * (kSub - 1));
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int Q = kQ > 0 ? kQ : p.Q;   // kQ: the query length compiled in (0: the argument's)
  const ScoreGeometry G = score_geometry(Q, kFp8Q);
  // Ring indices of the per-page loops: with the length compiled in the
  // divisors are constants; otherwise the stage count (2-8) divides through
  // a multiply-high by ceil(2^32 / stages) (exact for indices below 2^29),
  // and the accumulator and tile buffer counts (powers of two) by shifts
  // (generic qlen 9-24 scorers 9-15 % faster).  The fused qlen 1-2 kernel
  // keeps plain divisions: like this, or with qlen 1 compiled in, batch 128 /
  // qlen 1 ran 269 and 263 instead of 257 us.
  constexpr bool kPlainDiv = kQ > 0 || kFuse;
  const uint32_t st_magic = kPlainDiv ? 0u : static_cast<uint32_t>(0xFFFFFFFFull / G.stages + 1);
  const int acc_sh = G.nacc == 4 ? 2 : 1, qb_sh = G.nqb == 2 ? 1 : 0;
  auto st_div = [&](int x) -> int {
    if constexpr (kPlainDiv) return x / G.stages;
    else return static_cast<int>(__umulhi(static_cast<uint32_t>(x), st_magic));
  };
  auto st_mod = [&](int x) -> int {
    if constexpr (kPlainDiv) return x % G.stages;
    else return x - st_div(x) * G.stages;
  };
  auto acc_div = [&](int x) -> int {
    if constexpr (kPlainDiv) return x / G.nacc;
    else return x >> acc_sh;
  };
  auto acc_mod = [&](int x) -> int {
    if constexpr (kPlainDiv) return x % G.nacc;
    else return x & (G.nacc - 1);
  };
  auto qb_div = [&](int x) -> int {
    if constexpr (kPlainDiv) return x / G.nqb;
    else return x >> qb_sh;
  };
  auto qb_mod = [&](int x) -> int {
    if constexpr (kPlainDiv) return x % G.nqb;
    else return x & (G.nqb - 1);
  };
  uint8_t* stages = smem;                                              // [stages][128][128 B]
  uint8_t* qtiles = smem + G.off_q;                                    // [nqb][hi, lo][16Q][128 B]
  float* qmul_ring = reinterpret_cast<float*>(smem + G.off_qmul);      // [kQmulRing][Q]
  float* red = reinterpret_cast<float*>(smem + G.off_red);             // [kRedSlots][4][nsub][Q]
  ScoreTail* tail = reinterpret_cast<ScoreTail*>(smem + G.off_tail);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int T = p.B * Q;
  const int qtile_half = G.qtile_bytes / 2;

  // Tensor memory first when two CTAs share an SM: the hardware places the
  // second CTA only once the first has relinquished its allocation permit
  // (allocating after the prefix sum below started the second CTA of every SM
  // 2 us after the first).  With one CTA per SM it is allocated after the
  // prefix sum, which keeps the wide instantiation free of spills (allocated
  // first, its qlen-32 scorer spilled and took 1735 instead of 1591 us).
  if (!kWide && warp == 1) {
    tc::tmem_alloc(&tail->tmem_base, G.ncols);
    tc::tmem_relinquish();
  } else if (warp == 0) {
    // the pipeline's barriers, spread over the lanes
    if (lane < G.stages) {
      mbar_init(&tail->full[lane], 1);
      mbar_init(&tail->empty[lane], 1);
    }
    if (lane < kMaxAcc) {
      mbar_init(&tail->dfull[lane], 1);
      mbar_init(&tail->dempty[lane], 4 * kSub);
    }
    if (lane < 2) {
      mbar_init(&tail->qfull[lane], 1);
      mbar_init(&tail->qempty[lane], 1);
    }
    if (lane < kRedSlots) {
      mbar_init(&tail->red_full[lane], 4 * kSub);
      mbar_init(&tail->red_empty[lane], 1);
    }
    if (lane < kQmulRing) mbar_init(&tail->qmul_ready[lane], 1);
    if (lane == 0) {
      mbar_init(&tail->qstage, 1);
      mbar_init(&tail->finish, kNumThreads / 32);
      tail->any_invalid = 0;
    }
    fence_barrier_init();
  }

  // ---- this CTA's page range: block-wide prefix sum over the requests -----------
  {
    const int per = (p.B + kNumThreads - 1) / kNumThreads;
    const int b_lo = min(p.B, tid * per), b_hi = min(p.B, b_lo + per);
    int64_t local = 0;
    for (int b = b_lo; b < b_hi; ++b) {
      const int L = p.seq_lens[b];
      if (blockIdx.x == 0 && (L < 0 || (L > 0 && (L - 1) / kPage >= p.S)))
        flag_error(p.err, MSA_ERR_SEQ_RANGE);
      local += static_cast<int64_t>(p.Hkv) * visible_blocks(p, b);
    }
    int64_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) tail->warp_sums[warp] = incl;
    __syncthreads();
    int64_t before = 0, total = 0;
    for (int w = 0; w < kNumThreads / 32; ++w) {
      if (w < warp) before += tail->warp_sums[w];
      total += tail->warp_sums[w];
    }
    const int64_t excl = before + incl - local;
    const int64_t w0 = total * blockIdx.x / gridDim.x, w1 = total * (blockIdx.x + 1) / gridDim.x;
    if (tid == 0) tail->count = static_cast<int>(w1 - w0);
    if (w0 < w1 && excl <= w0 && w0 < excl + local) {
      int64_t acc = excl;
      for (int b = b_lo; b < b_hi; ++b) {
        const int64_t pb = static_cast<int64_t>(p.Hkv) * visible_blocks(p, b);
        if (w0 < acc + pb) {
          tail->start_b = b;
          tail->start_rem = static_cast<int>(w0 - acc);
          break;
        }
        acc += pb;
      }
    }
  }
  if (kWide && warp == 1) {
    tc::tmem_alloc(&tail->tmem_base, G.ncols);
    tc::tmem_relinquish();
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const int count = tail->count;
  const uint32_t tmem = tail->tmem_base;

  // The first query tile, which the first products wait for, is built by
  // warps 2-6 together, a token each in turn (converting one token's 16 rows
  // to e4m3 hi + lo takes one warp about a microsecond); warp 2 publishes it.
  const int nq0 = Q < 5 ? Q : 5;
  if (count > 0 && warp >= 2 && warp < 2 + nq0) {
    PageWalk w0;
    w0.begin(p, tail->start_b, tail->start_rem);
    if (!kFp8Q && !kWide && warp == 2 && second_tile_early(G, w0, count)) {
      // the second unit's query rows into L2 for its tile (built below)
      PageWalk w1 = w0;
      w1.advance(p, w1.nhi - w1.n);
      for (int jq = 0; jq < Q; ++jq) {
        const int64_t row = (static_cast<int64_t>(w1.b) * Q + jq) * p.Hq + w1.g * kGroup;
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q + row * kHeadDim);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(src + 128 * lane));
      }
    }
    prepare_query_tile<kFp8Q, true>(p, w0.b, w0.g, qtiles, qtiles + qtile_half, qmul_ring, lane,
                                    first_tile_staging(G, kFp8Q, stages, qtiles), warp - 2, nq0);
    tc::fence_proxy_async_smem();   // read by the tensor core (and the staging rewritten by TMA)
    named_barrier(3, 32 * nq0);
    if (warp == 2 && lane == 0) {
      mbar_arrive(&tail->qfull[0]);
      mbar_arrive(&tail->qmul_ready[0]);
      mbar_arrive(&tail->qstage);
    }
  }

  // Warps 1 and 3-7 check every block-table entry of the range once, in
  // parallel, while warp 0 starts streaming and warp 2 prepares the first
  // query tile; when all are valid (the normal case) the MMA and epilogue
  // roles need no per-page table reads on their critical path.
  bool all_valid = true;
  if (warp != 0 && warp != 2) {
    const int nthr = kNumThreads - 64, t_id = tid - (warp == 1 ? 32 : 64);
    const int t0 = static_cast<int>(static_cast<int64_t>(count) * t_id / nthr);
    const int t1 = static_cast<int>(static_cast<int64_t>(count) * (t_id + 1) / nthr);
    if (t0 < t1) {
      PageWalk w;
      w.begin(p, tail->start_b, tail->start_rem);
      w.advance(p, t0);
      bool bad = false;
      for (int t = t0; t < t1; ++t, w.next(p)) {
        int page;
        bad |= !page_valid(p, w, page);
      }
      if (bad) atomicOr(&tail->any_invalid, 1);
    }
    named_barrier(2, kNumThreads - 64);  // no wait precedes it: warps 1 and 3+ all arrive
    all_valid = *reinterpret_cast<volatile int*>(&tail->any_invalid) == 0;
  }

  // A second unit near the start of the range: its tile by the query warp and
  // the combiner warp (idle until the first page's maxima), after the check
  // above, into the second buffer (the first tile's staging there has been
  // read), rows read directly.  An fp8 query's tile is a plain copy, quick
  // for the query warp alone.
  if (!kFp8Q && !kWide && count > 0 && (warp == 2 || warp == 7)) {
    PageWalk w1;
    w1.begin(p, tail->start_b, tail->start_rem);
    if (second_tile_early(G, w1, count)) {
      w1.advance(p, w1.nhi - w1.n);
      prepare_query_tile<kFp8Q, true>(p, w1.b, w1.g, qtiles + G.qtile_bytes,
                                      qtiles + G.qtile_bytes + qtile_half, qmul_ring + Q, lane,
                                      nullptr, warp == 2 ? 0 : 1, 2);
      tc::fence_proxy_async_smem();
      named_barrier(1, 64);
      if (warp == 2 && lane == 0) {
        mbar_arrive(&tail->qfull[1]);
        mbar_arrive(&tail->qmul_ready[1]);
      }
    }
  }

  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------------
    if (lane == 0) {
      prefetch_tensormap(&kv_map);
      PageWalk w;
      if (count > 0) w.begin(p, tail->start_b, tail->start_rem);
      int vp = 0;
      for (int t = 0; t < count; ++t, w.next(p)) {
        int page;
        if (!page_valid(p, w, page)) {
          if (p.err) flag_error(p.err, MSA_ERR_PAGE_RANGE);
          continue;
        }
        const int s = st_mod(vp);
        if (vp >= G.stages && !mbar_wait(&tail->empty[s], (st_div(vp) - 1) & 1)) {
          flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        // with one query buffer the last stage first stages the first query tile
        if (stage_staging(G, kFp8Q) && vp == G.stages - 1 && !mbar_wait(&tail->qstage, 0)) {
          flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&tail->full[s], kHalfTile);
        tma_load_2d(stages + s * kHalfTile, &kv_map, 0, (page * p.Hkv + w.g) * kPage,
                    &tail->full[s]);
        ++vp;
      }
      // the last loads in flight land before shared memory can be released
      for (int t = vp - G.stages; t < vp; ++t)
        if (t >= 0) (void)mbar_wait(&tail->full[st_mod(t)], st_div(t) & 1);
      // every load of this CTA has landed: the next kernel may start its CTAs
      pdl_trigger();
      mbar_arrive(&tail->finish);
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----------------------------------------------------------------
    if (lane == 0) {
      // descriptors are built once and advanced by constants: the start
      // address field counts 16-byte units (stage = 1024, k-step = 2)
      const uint64_t adesc0 = tc::sw128_kmajor_desc(smem_u32(stages));
      const uint64_t bdesc0 = tc::sw128_kmajor_desc(smem_u32(qtiles));
      const uint64_t lo_step = static_cast<uint64_t>(qtile_half >> 4);
      uint32_t idesc[2];
      for (int h = 0; h < 2; ++h)
        idesc[h] = tc::idesc_e4m3_f32(128, ((kWide ? G.fuse != 0 : kFuse) ? 32 : 16) *
                                               max(1, min(G.Qu, Q - h * G.Qu)));
      PageWalk w;
      if (count > 0) w.begin(p, tail->start_b, tail->start_rem);
      int k = -1, pb = -1, pg = -1, vp = 0;
      bool q_ready = false, ok = true;
      for (int t = 0; t < count && ok; ++t, w.next(p)) {
        if (w.b != pb || w.g != pg) {
          if (k >= 0) tc::commit(&tail->qempty[qb_mod(k)]);  // old tile free once its MMAs end
          ++k;
          pb = w.b;
          pg = w.g;
          q_ready = false;
        }
        int page;
        if (!all_valid && !page_valid(p, w, page)) continue;
        if (!q_ready) {
          if (!mbar_wait(&tail->qfull[qb_mod(k)], qb_div(k) & 1)) {
            flag_error(p.err, MSA_ERR_TIMEOUT);
            break;
          }
          tc::fence_after_thread_sync();
          q_ready = true;
        }
        const int s = st_mod(vp);
        if (!mbar_wait(&tail->full[s], st_div(vp) & 1)) {
          flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        tc::fence_after_thread_sync();
        const uint64_t a = adesc0 + static_cast<uint64_t>(s) * (kHalfTile >> 4);
        const uint64_t bq = bdesc0 + static_cast<uint64_t>(qb_mod(k) * (G.qtile_bytes >> 4));
        for (int h = 0; h < G.nh; ++h) {
          const int u = vp * G.nh + h, buf = acc_mod(u), use = acc_div(u);
          if (use >= 1) {
            if (!mbar_wait(&tail->dempty[buf], (use - 1) & 1)) {
              flag_error(p.err, MSA_ERR_TIMEOUT);
              ok = false;
              break;
            }
            tc::fence_after_thread_sync();
          }
          const uint32_t d = tmem + buf * G.ucols;
          const uint64_t bh = bq + static_cast<uint64_t>((h * G.Qu * kGroup * 128) >> 4);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) tc::mma_e4m3(d, a + 2 * ks, bh + 2 * ks, idesc[h], ks > 0);
          if (!kFp8Q && (kWide ? !G.fuse : !kFuse)) {  // the lo part of a bf16 query adds into the same columns
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc::mma_e4m3(d, a + 2 * ks, bh + lo_step + 2 * ks, idesc[h], 1);
          }
          tc::commit(&tail->dfull[buf]);
        }
        tc::commit(&tail->empty[s]);
        ++vp;
      }
      mbar_arrive(&tail->finish);
    }
    __syncwarp();
    // free tensor memory once every role is done with it
    (void)mbar_wait(&tail->finish, 0);
    tc::fence_after_thread_sync();
    tc::tmem_dealloc(tmem, G.ncols);
  } else if (warp == 2) {
    // ---- query tiles, then the -inf tails ----------------------------------------------
    PageWalk w;
    if (count > 0) w.begin(p, tail->start_b, tail->start_rem);
    const bool pre1 = !kFp8Q && !kWide && count > 0 && second_tile_early(G, w, count);   // tile 1 built above
    int t = 0, k = 0;
    bool ok = true;
    while (t < count && ok) {
      if (k > 0 && !(k == 1 && pre1)) {   // the first tile is built above
        const int qb = qb_mod(k);
        if (k >= G.nqb && !mbar_wait(&tail->qempty[qb], (qb_div(k) - 1) & 1)) {
          if (lane == 0) flag_error(p.err, MSA_ERR_TIMEOUT);
          ok = false;
          break;
        }
        uint8_t* qhi = qtiles + qb * G.qtile_bytes;
        prepare_query_tile<kFp8Q>(p, w.b, w.g, qhi, qhi + qtile_half,
                                  qmul_ring + (k % kQmulRing) * Q, lane, nullptr);
        tc::fence_proxy_async_smem();   // the tile is read by the tensor core
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&tail->qfull[qb]);
          mbar_arrive(&tail->qmul_ready[k % kQmulRing]);
        }
      }
      // skip to the first page of the next unit
      const int in_unit = w.nhi - w.n;
      for (int s = 0; s < in_unit && t < count; ++s, ++t) w.next(p);
      // its query rows into L2 now, so that its tile is quick to build
      if (t < count) {
        constexpr int kTokBytes = kGroup * (kFp8Q ? 128 : 256);
        for (int jq = 0; jq < Q; ++jq) {
          const int64_t row = (static_cast<int64_t>(w.b) * Q + jq) * p.Hq + w.g * kGroup;
          const uint8_t* src = kFp8Q ? p.q8 + row * kHeadDim
                                     : reinterpret_cast<const uint8_t*>(p.q + row * kHeadDim);
          for (int c = lane; c < kTokBytes / 128; c += 32)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(src + 128 * c));
        }
      }
      ++k;
    }
    // -inf for blocks past each request's last visible block (units dealt
    // round-robin over the CTAs; disjoint from every page written above);
    // the previous kernel on the stream may still be reading scores
    pdl_wait();
    for (int64_t u = blockIdx.x; u < static_cast<int64_t>(p.B) * p.Hkv; u += gridDim.x) {
      const int b = static_cast<int>(u / p.Hkv), g = static_cast<int>(u - static_cast<int64_t>(b) * p.Hkv);
      const int nhi = visible_blocks(p, b);
      const int width = p.S - nhi;
      for (int idx = lane; idx < width * Q; idx += 32) {
        const int jq = idx / width, n = nhi + (idx - jq * width);
        p.scores[(static_cast<int64_t>(g) * T + static_cast<int64_t>(b) * Q + jq) * p.S + n] =
            -INFINITY;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->finish);
  } else if (warp != 7) {
    // ---- epilogue: accumulator -> per-token block maxima ----------------------------
    const int quarter = warp & 3;                // TMEM lanes 32*quarter .. +31
    const int sub = kWide ? (warp >= 8 ? (warp - 4) / 4 : 0) : 0;  // epilogue set
    const int key = 32 * quarter + lane;         // key (row of the page) of this thread
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
    PageWalk w;
    if (count > 0) w.begin(p, tail->start_b, tail->start_rem);
    int vp = 0;
    bool ok = true;
    for (int t = 0; t < count && ok; ++t, w.next(p)) {
      int page;
      if (!all_valid && !page_valid(p, w, page)) continue;
      const int lim_base = w.L - Q - w.n * kPage;   // token j sees keys <= lim_base + j
      float myv = -INFINITY;                        // lane jq: this quarter's max of token jq
      for (int h = 0; h < G.nh && ok; ++h) {
        const int u = vp * G.nh + h, buf = acc_mod(u), use = acc_div(u);
        if (!mbar_wait(&tail->dfull[buf], use & 1)) {
          if (lane == 0) flag_error(p.err, MSA_ERR_TIMEOUT);
          ok = false;
          break;
        }
        tc::fence_after_thread_sync();
        const int tok0 = h * G.Qu, ntok = min(G.Qu, Q - tok0);
        const uint32_t acc = lane_addr + buf * G.ucols;
        if (kFuse) {   // (fused only at qlen <= 2: two CTAs per SM)
          // token by token: its hi columns (16 j) and lo columns (16 Qu + 16 j),
          // summed head by head before the maximum
          for (int j = sub; j < ntok; j += kSub) {
            const int lim = lim_base + tok0 + j;
            if (lim < 0) continue;                 // warp-uniform: nothing visible
            uint32_t vh[16], vl[16];
            tc::ld_32x32b_x16(acc + j * 16, vh);
            tc::ld_32x32b_x16(acc + 16 * G.Qu + j * 16, vl);
            tc::wait_ld();
#pragma unroll
            for (int c = 0; c < 16; ++c)
              vh[c] = __float_as_uint(__uint_as_float(vh[c]) + __uint_as_float(vl[c]));
            const int ord = __reduce_max_sync(0xffffffffu,
                                              order_int(key <= lim ? max16(vh) : -INFINITY));
            if (lane == tok0 + j) myv = order_float(ord);
          }
        } else
        // groups of four tokens: four TMEM loads in flight under one wait, then
        // four independent tree maxima and four back-to-back warp reductions
        for (int j0 = kGrp * sub; j0 < ntok; j0 += kGrp * kSub) {
          const int nj = min(kGrp, ntok - j0);
          if (lim_base + tok0 + j0 + nj - 1 < 0) continue;   // warp-uniform: nothing visible
          uint32_t v[kGrp][16];
#pragma unroll
          for (int jj = 0; jj < kGrp; ++jj)
            if (jj < nj) tc::ld_32x32b_x16(acc + (j0 + jj) * 16, v[jj]);
          tc::wait_ld();
          int ord[kGrp];
#pragma unroll
          for (int jj = 0; jj < kGrp; ++jj) {
            const float m = max16(v[jj]);
            const int lim = lim_base + tok0 + j0 + jj;
            ord[jj] = order_int((jj < nj && key <= lim) ? m : -INFINITY);
          }
#pragma unroll
          for (int jj = 0; jj < kGrp; ++jj) ord[jj] = __reduce_max_sync(0xffffffffu, ord[jj]);
#pragma unroll
          for (int jj = 0; jj < kGrp; ++jj)
            if (jj < nj && lane == tok0 + j0 + jj) myv = order_float(ord[jj]);
        }
        tc::fence_before_thread_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->dempty[buf]);
      }
      if (!ok) break;
      // publish this quarter's maxima to the combiner
      const int slot = vp % kRedSlots;
      if (vp >= kRedSlots && !mbar_wait(&tail->red_empty[slot], ((vp / kRedSlots) - 1) & 1)) {
        if (lane == 0) flag_error(p.err, MSA_ERR_TIMEOUT);
        break;
      }
      // this set's row of the quarter (-inf for the tokens the other set takes)
      if (lane < Q) red[((slot * 4 + quarter) * kSub + sub) * Q + lane] = myv;
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->red_full[slot]);
      ++vp;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->finish);
  } else {
    // ---- combiner: four quarters -> scores ---------------------------------------------
    pdl_wait();  // the first write of scores
    PageWalk w;
    if (count > 0) w.begin(p, tail->start_b, tail->start_rem);
    int k = -1, pb = -1, pg = -1, vp = 0;
    float qm = 0.f;                              // scale of token `lane` of the current unit
    bool have_qm = false;
    for (int t = 0; t < count; ++t, w.next(p)) {
      if (w.b != pb || w.g != pg) {
        ++k;
        pb = w.b;
        pg = w.g;
        have_qm = false;
      }
      const int64_t row0 = (static_cast<int64_t>(w.g) * T + static_cast<int64_t>(w.b) * Q) * p.S + w.n;
      int page;
      if (!all_valid && !page_valid(p, w, page)) {
        if (lane < Q) p.scores[row0 + static_cast<int64_t>(lane) * p.S] = -INFINITY;
        continue;
      }
      if (!have_qm) {
        if (!mbar_wait(&tail->qmul_ready[k % kQmulRing], (k / kQmulRing) & 1)) {
          if (lane == 0) flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        qm = lane < Q ? qmul_ring[(k % kQmulRing) * Q + lane] : 0.f;
        have_qm = true;
      }
      const int slot = vp % kRedSlots;
      if (!mbar_wait(&tail->red_full[slot], (vp / kRedSlots) & 1)) {
        if (lane == 0) flag_error(p.err, MSA_ERR_TIMEOUT);
        break;
      }
      if (lane < Q) {
        float v = -INFINITY;
#pragma unroll
        for (int r = 0; r < 4 * kSub; ++r) v = fmaxf(v, red[(slot * 4 * kSub + r) * Q + lane]);
        p.scores[row0 + static_cast<int64_t>(lane) * p.S] = (v == -INFINITY) ? v : v * qm;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->red_empty[slot]);
      ++vp;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->finish);
  }
}

}  // namespace

// The instantiations with the query length compiled in: bf16 qlen 3-7 and
// fp8 qlen 1-7 (two CTAs per SM), bf16 and fp8 qlen 8, 16 and 32 (one CTA per
// SM).  Measured at batch 16 over 8k-32k tokens, generic -> compiled in: bf16
// qlen 4 39.9 -> 31.6 us, 5 52.1 -> 40.8, 8 87.5 -> 67.7, 16 116.3 -> 95.7,
// 32 1574 -> 1362 (the qlen-32 workload); fp8 qlen 4 34.1 -> 31.7, 5 47.2 ->
// 35.0, 8 67.6 -> 52.8, 16 88.9 -> 69.6.  The other lengths read it from the
// arguments, and so does the fused bf16 qlen 1-2 path (with qlen 1 compiled
// in, batch 128 / qlen 1 ran 263.2 instead of 256.7 us).
#define MSA_SCORE_KERNELS(X)                                                                    \
  X(false, false, true, 0) X(false, false, false, 3) X(false, false, false, 4)                  \
  X(false, false, false, 5) X(false, false, false, 6) X(false, false, false, 7)                 \
  X(false, false, false, 0) X(true, false, false, 1) X(true, false, false, 2)                   \
  X(true, false, false, 3) X(true, false, false, 4) X(true, false, false, 5)                    \
  X(true, false, false, 6) X(true, false, false, 7) X(true, false, false, 0)                    \
  X(false, true, false, 8) X(false, true, false, 16) X(false, true, false, 32)                  \
  X(false, true, false, 0) X(true, true, false, 8) X(true, true, false, 16)                   \
  X(true, true, false, 32) X(true, true, false, 0)

cudaError_t launch_score(const CUtensorMap& kv_map, const ScoreParams& p, cudaStream_t stream,
                         bool pdl) {
  if (p.ctas < 1) return cudaErrorInvalidValue;
  const ScoreGeometry G = score_geometry(p.Q, p.q8 != nullptr);
  if (G.stages < 2 || G.smem > kSmemLimit) return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [] {
#define MSA_SET_ATTR(F8, W, FU, QQ)                                                              \
    {                                                                                          \
      auto* k = score_kernel<F8, W, FU, QQ>;                                                   \
      cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,     \
                                           kSmemLimit);                                        \
      if (r != cudaSuccess) return r;                                                          \
      r = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,              \
                               static_cast<int>(cudaSharedmemCarveoutMaxShared));              \
      if (r != cudaSuccess) return r;                                                          \
    }
    // all of the unified L1 / shared storage as shared memory, so that two
    // CTAs of ~100 KB can be resident on one SM
    MSA_SCORE_KERNELS(MSA_SET_ATTR)
#undef MSA_SET_ATTR
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const dim3 grid(p.ctas * G.per_sm), block(G.threads);
  const bool f8 = p.q8 != nullptr, wide = G.nsub > 1, fuse = G.fuse != 0;
#define MSA_LAUNCH_IF(F8, W, FU, QQ)                                                             \
  if (f8 == F8 && wide == W && fuse == FU && (QQ == 0 || p.Q == QQ))                            \
    return launch_pdl(score_kernel<F8, W, FU, QQ>, grid, block, G.smem, stream, pdl, kv_map, p);
  // the instantiations with the length compiled in come before the generic ones
  MSA_SCORE_KERNELS(MSA_LAUNCH_IF)
#undef MSA_LAUNCH_IF
  return cudaErrorInvalidValue;   // unreachable: every (fp8, wide, fused) has a generic kernel
}

}  // namespace msa
