// msa_union.cu -- stage 3 (sparse attend) for decode steps of two or more
// query tokens per request: one CTA per (request, tile of up to four query
// tokens, KV head, split) over the UNION of the tile's top-k lists.
//
// Operation: as attend_kernel (minimax_m3_sparse_attn_decode /
// msa_cutlass_sparse_decode on the vLLM MiniMax-M3 pages): each query row
// attends only the tokens of the blocks its own list names, causally limited
// to pos = seq_len - Q + j; padding rows give zeros; split parts are merged
// from fp32 partials (TensorRT-LLM PR #17171, flash-decoding commit).  The
// CUTLASS decode plan on the vLLM page sizes its work by the request's query
// length (qo_lens) with kv_block_num = topk: a request's decode tokens share
// one pass over the KV pages.  Here the tokens of a tile share each page:
//
//  * the tile's lists (given, or selected in the prologue from the block
//    scores, one warp per token) are merged into their ascending union, each
//    union page carrying a mask of the tokens that listed it; a request's
//    tokens select mostly the same recent blocks, so the union is smaller
//    than the sum of the lists, and each union page is loaded once;
//  * the union is cut into `splits` equal contiguous ranges, one per CTA (the
//    current block, the union's largest, first in the last range: its page is
//    loaded before the lists are known);
//  * each token then runs its own softmax over the pages it listed, in its
//    own four warps (one key per thread, attend_kernel's online softmax), with
//    its own tensor-core products: S^T = K Q^T with N = 32 (the query's exact
//    fp8 hi and lo parts, three buffers), O^T += V^T P^T with N = 32 (P's hi
//    and lo parts), both transposed so that the page's 128 keys, then its 128
//    value dims, fill the MMA's M.  A token's O^T accumulates in tensor memory
//    across its pages and is rescaled there on the rare pages where its
//    softmax reference maximum moves.  The tokens share only the loaded
//    pages: a token is never held up by a page it did not list, and a stage
//    is refilled once every token that listed its page is done with it.
//
// Dense decode (the TensorRT-LLM PR #17171 dense-decode commit: the first
// layers attend the whole page table) is the same kernel with every block a
// token may see as its list: the tile's union is the blocks up to its last
// token's current block, each token listing a prefix of it, so every page is
// loaded once for the whole tile.  With fewer units than SMs the launch has
// one CTA per SM and each unit takes CTAs in proportion to its blocks (the
// requests' lengths differ), so that no CTA holds much more than its share;
// a page's tokens then share one S^T and one O^T product and three commits.
//
// Warp roles (20 warps, one CTA per SM):
//   0      union, page list, TMA producer (5-stage ring of 32 KiB K|V pages)
//   1      walks the pages in order: issues S^T for each token that listed
//          the page (when that token's S^T buffer is free), releases the page
//          for the tokens that did not; owns tensor memory
//   2      issues each token's O^T as soon as its P^T is written
//   3      copies the request's block-table row
//   4..19  token j = (warp - 4) / 4: softmax; warp 4+4j selects or reads the
//          token's list, warp 5+4j prepares its query rows
#include "msa_device.cuh"
#include "msa_launch.h"
#include "msa_select.cuh"
#include "msa_tcgen05.cuh"

namespace msa {

namespace {

constexpr int kQt = kUnionTile;               // query tokens per tile
constexpr int kStages = 5;
constexpr int kWarps = 4 + 4 * kQt;
constexpr int kThreads = kWarps * 32;
constexpr int kSoftWarp0 = 4;
constexpr int kN = 32 * kQt;                  // query tile rows: hi | lo per token
constexpr int kStageBytes = 2 * kHalfTile;    // K tile then V tile
constexpr int kQTile = kN * 128;              // query tile: kN rows x 128 B
// P^T, two buffers: per block of 8 keys, for each token j its hi 8 x 16 B core
// matrix at 256 j and its lo one at 256 j + 128 (MN-major, no swizzle), so the
// columns of consecutive tokens are contiguous
constexpr int kPBlock = 8 * kN;               // 1 KiB
constexpr int kPBuf = kPage * kN;             // 16 KiB
constexpr int kMaxUnion = kTopK * kQt;        // 64
// tensor memory: S^T buffer b of token j at columns kN b + 32 j (three
// buffers), token j's O^T accumulator at kColAcc + 32 j; the columns of
// consecutive tokens are contiguous, so one product can cover several
constexpr int kSBufs = 3;
constexpr uint32_t kColAcc = kSBufs * kN;
constexpr int kTmemCols = 512;
constexpr int kMaxDenseBlocks = 2048;         // dense decode: blocks of one CTA's range
// dense decode with fewer (request, tile, KV head) units than SMs and split
// parts: one CTA per SM, shared out in the kernel among up to this many
// (request, tile) units in proportion to their blocks
constexpr int kBalancedTiles = 256;
constexpr float kPShift = 8.f;                // P = 2^(x - m + kPShift)
constexpr float kLazy = 0.5f;                 // m moves when a page exceeds it by more than this
constexpr int kTableCopy = 512;               // block-table entries copied to shared memory
constexpr int kSelectCap = (kStageBytes - 4 * kTopK) / 4;  // selector keys per scratch stage

struct UnionTail {
  uint64_t full[kStages];   // TMA -> the S^T walker (and the V-row fix)
  uint64_t empty[kStages];  // one release per token and use (walker for non-listing tokens, O^T commits)
  uint64_t s_full[kQt][kSBufs];  // token j's S^T ready -> its softmax
  uint64_t s_free[kQt][kSBufs];  // token j's four warps have read an S^T buffer -> walker
  uint64_t p_full[kQt][2];  // token j's four warps' P^T written -> O^T issuer
  uint64_t o_done[kQt][2];  // token j's O^T of a page complete (its P^T buffer free again)
  uint64_t mx_full[kQt][2]; // token j's four warps' page maxima written
  uint64_t l_full[kQt];     // token j's four warps' running sums written
  uint64_t vfix;            // value rows past the request's last token zeroed (4 warps)
  uint64_t finish;          // every role done and every MMA complete
  uint32_t tmem_base;
  int n_pages;
  int fix_slot;             // slot of the request's last block (-1: none here)
  int last_rows;            // rows of that block holding tokens
  int pos[kQt];             // token positions (-1: padding row or no token)
  float zs[kQt];            // logit scale (log2 units) times 2^e of each token's query split
  int lists[kQt][kTopK];    // each token's checked list (-1: unused slot)
  uint32_t sorted[kMaxUnion];
  int pages[kMaxUnion];
  int blocks[kMaxUnion];
  uint32_t masks[kMaxUnion];
  int n_tok[kQt];           // pages each token listed among this CTA's
  int tok_slots[kQt][kMaxUnion];  // their slots, in page order
  int dense_lo;             // dense decode: this CTA's pages are blocks dense_lo + slot
  uint32_t dense_bad[kMaxDenseBlocks / 32];  // dense decode: slots whose block-table entry is bad
};

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr int kOffQ = kStages * kStageBytes;
constexpr int kOffP = kOffQ + kQTile;                   // P^T [kQt tokens][2 buffers]
constexpr int kOffMx = kOffP + 2 * kPBuf;               // page maxima [kQt][2][4 warps][16]
constexpr int kOffL = kOffMx + kQt * 2 * 4 * kGroup * 4;  // running sums [kQt][4 warps][16]
constexpr int kOffTail = kOffL + kQt * 4 * kGroup * 4;
constexpr int kSmemBytes = kOffTail + static_cast<int>((sizeof(UnionTail) + 15) / 16 * 16) + 1024;
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "operand tiles need 1024-byte alignment");
static_assert(kSmemBytes <= 227 * 1024, "union attend shared memory");
static_assert(kStages >= 1 + kQt, "the selectors' scratch uses stages 1..kQt");
static_assert(4 * kTableCopy <= 2 * kPBuf, "block-table copy fits the P^T buffers");
static_assert(kColAcc + kN <= kTmemCols, "tensor memory layout");
static_assert(kOffTail % 16 == 0, "mbarriers need 8-byte alignment");

template <int N>
__device__ __forceinline__ void fill(float (&a)[N], float v) {
#pragma unroll
  for (int k = 0; k < N; ++k) a[k] = v;
}

// Ascending sort of 64 keys held two per lane (element e = 32 r + lane in
// v[r]) by a bitonic network across the warp.
__device__ __forceinline__ void warp_sort64(uint32_t (&v)[2], int lane) {
#pragma unroll
  for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j == 32) {  // partners in the same lane: element lane vs lane + 32
        const uint32_t a = v[0], b = v[1];
        // k == 64: one ascending run, the lower element keeps the minimum
        v[0] = min(a, b);
        v[1] = max(a, b);
      } else {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int e = 32 * r + lane;
          const uint32_t other = __shfl_xor_sync(0xffffffffu, v[r], j);
          const bool asc = (e & k) == 0;
          const bool lower = (e & j) == 0;
          v[r] = (asc == lower) ? min(v[r], other) : max(v[r], other);
        }
      }
    }
  }
}

// Blocks a dense-decode unit (request, tile) attends: up to its last token's
// current block (0 for a padding request or a tile of padding rows).
__device__ __forceinline__ int dense_tile_blocks(const AttendParams& p, int tu, int ntiles) {
  const int b = tu / ntiles, tile = tu - b * ntiles;
  const int L = p.seq_lens[b];
  const bool seq_ok = L >= 0 && (L == 0 || (L - 1) / kPage < p.S);
  const int tok = min(kQt * tile + kQt - 1, p.Q - 1);
  const int pos = seq_ok ? L - p.Q + tok : -1;
  return pos >= 0 ? pos / kPage + 1 : 0;
}

struct DenseSlot {
  int unit;    // (request, tile, KV head) unit, in blockIdx.x order of the plain grid; -1: none
  int part;    // which of its equal block ranges
  int nparts;  // how many ranges the unit is cut into
};

// Dense decode's work for this CTA.  With a grid of one CTA per unit and split
// that is (blockIdx.x, blockIdx.y, gridDim.y).  With more CTAs than units (one
// per SM, launch_union_attend) the units share them out by their blocks: unit u (n_u blocks)
// takes z_u = min(ceil(n_u / T), splits) CTAs (at least one) for the smallest
// T at which every unit's CTAs fit the grid, so that no CTA holds much more
// than its share of the batch's pages; the CTAs go to the units in order, a
// unit's KV heads in turn, each head's ranges in turn.  Every CTA computes the
// same assignment from seq_lens (one warp, every lane the same result); CTAs
// past the last unit's get none.
__device__ DenseSlot dense_slot(const AttendParams& p, int ntiles, int lane) {
  const int NT = p.B * ntiles, H = p.Hkv, Z = p.splits, C = static_cast<int>(gridDim.x);
  if (C <= NT * H)
    return DenseSlot{static_cast<int>(blockIdx.x), static_cast<int>(blockIdx.y),
                     static_cast<int>(gridDim.y)};
  constexpr int kPer = kBalancedTiles / 32;
  int n[kPer];
  int maxn = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int tu = 32 * k + lane;
    n[k] = tu < NT ? dense_tile_blocks(p, tu, ntiles) : 0;
    maxn = max(maxn, n[k]);
  }
  maxn = __reduce_max_sync(0xffffffffu, maxn);
  auto parts = [&](int k, int T) { return min(max((n[k] + T - 1) / T, 1), Z); };
  auto ctas = [&](int T) {
    int s = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (32 * k + lane < NT) s += parts(k, T);
    return static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(s))) * H;
  };
  // at T = max(n) every unit takes one CTA per head, NT * H <= C (the host's rule)
  int lo = 1, hi = max(maxn, 1);
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (ctas(mid) <= C) hi = mid;
    else lo = mid + 1;
  }
  const int c = static_cast<int>(blockIdx.x);
  int run = 0;   // CTAs of the units before this group of 32
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int tu = 32 * k + lane;
    const int zc = tu < NT ? parts(k, lo) : 0;
    int incl = zc * H;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    const int start = run + incl - zc * H;
    const unsigned hit = __ballot_sync(0xffffffffu, zc > 0 && c >= start && c < start + zc * H);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const int st = __shfl_sync(0xffffffffu, start, src);
      const int z = __shfl_sync(0xffffffffu, zc, src);
      const int rel = c - st;
      return DenseSlot{(32 * k + src) * H + rel / z, rel % z, z};
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  return DenseSlot{-1, 0, 1};
}

// kFp8Q: an fp8 query (q8 * q_scale); kDense: dense decode (no lists);
// each compiled separately.
template <bool kFp8Q, bool kDense>
__global__ void __launch_bounds__(kThreads, 1)
    union_attend_kernel(const __grid_constant__ CUtensorMap kv_map, const AttendParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  UnionTail* tail = reinterpret_cast<UnionTail*>(smem + kOffTail);
  uint8_t* qtile = smem + kOffQ;
  uint8_t* pbuf = smem + kOffP;
  float* mx_all = reinterpret_cast<float*>(smem + kOffMx);
  float* lsum_all = reinterpret_cast<float*>(smem + kOffL);
  int32_t* table_s = reinterpret_cast<int32_t*>(pbuf);   // prologue only

  const int ntiles = (p.Q + kQt - 1) / kQt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int unit = static_cast<int>(blockIdx.x), split = static_cast<int>(blockIdx.y);
  int nsplit = static_cast<int>(gridDim.y);
  if constexpr (kDense) {
    const DenseSlot ds = dense_slot(p, ntiles, lane);
    if (ds.unit < 0) return;   // the whole CTA: no unit left for it
    unit = ds.unit;
    split = ds.part;
    nsplit = ds.nparts;
  }
  const int g = unit % p.Hkv;
  const int tile = (unit / p.Hkv) % ntiles;
  const int b = unit / (p.Hkv * ntiles);
  const int32_t* trow = p.block_table + static_cast<int64_t>(b) * p.S;
  const int ncopy = p.S < kTableCopy ? p.S : kTableCopy;

  // ---- prologue, part 1: positions, barriers, the current block's page, the
  // ---- block-table row, the lists and the query tile -------------------------------
  const int L = p.seq_lens[b];
  const bool seq_ok = L >= 0 && (L == 0 || (L - 1) / kPage < p.S);
  if (warp == 0) {
    if (!seq_ok && lane == 0 && tile == 0 && g == 0 && split == 0)
      flag_error(p.err, MSA_ERR_SEQ_RANGE);
    int cur_max = -1;
#pragma unroll
    for (int j = 0; j < kQt; ++j) {
      const int tok = kQt * tile + j;
      const int pos = (seq_ok && tok < p.Q) ? L - p.Q + tok : -1;
      if (lane == 0) tail->pos[j] = pos;
      if (pos >= 0) cur_max = pos / kPage;
    }
    // the union's largest block is the last token's current block when listed
    // (always in select mode); the last split owns it and loads it now, before
    // the lists are known (it depends on inputs only)
    int cur_page = -1;
    if (!kDense && cur_max >= 0 && split == nsplit - 1) {
      const int pg = trow[cur_max];
      if (pg >= 0 && static_cast<int64_t>(pg) < p.num_blocks) cur_page = pg;
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(&tail->full[s], 1);
        // one release per token and use; dense decode: one per page (its
        // tokens' joint O^T product)
        mbar_init(&tail->empty[s], kDense ? 1 : kQt);
      }
      for (int j = 0; j < kQt; ++j) {
        for (int s = 0; s < kSBufs; ++s) {
          mbar_init(&tail->s_full[j][s], 1);
          mbar_init(&tail->s_free[j][s], 4);
        }
        for (int s = 0; s < 2; ++s) {
          mbar_init(&tail->p_full[j][s], 4);
          mbar_init(&tail->o_done[j][s], 1);
          mbar_init(&tail->mx_full[j][s], 4);
        }
        mbar_init(&tail->l_full[j], 4);
      }
      mbar_init(&tail->vfix, 4);
      // the producer, the 16 softmax warps, and the two MMA issuers' last products
      mbar_init(&tail->finish, 1 + 4 * kQt + 2);
      fence_barrier_init();
      prefetch_tensormap(&kv_map);
      tail->pages[0] = cur_page;   // read back after the union is built
      tail->last_rows = (seq_ok && L > 0) ? L - ((L - 1) / kPage) * kPage : 0;
      if (cur_page >= 0) {
        const int row = (cur_page * p.Hkv + g) * kPage;
        mbar_arrive_expect_tx(&tail->full[0], kStageBytes);
        tma_load_2d(smem, &kv_map, 0, row, &tail->full[0]);
        tma_load_2d(smem + kHalfTile, &kv_map, kHeadDim, row, &tail->full[0]);
      }
    }
  } else if (warp == 1) {
    tc::tmem_alloc(&tail->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  } else if (warp == 3) {
    // the request's block-table row (its first kTableCopy entries), all loads in flight
    int32_t v[kTableCopy / 32];
#pragma unroll
    for (int k = 0; k < kTableCopy / 32; ++k) v[k] = 32 * k + lane < ncopy ? trow[32 * k + lane] : 0;
#pragma unroll
    for (int k = 0; k < kTableCopy / 32; ++k)
      if (32 * k + lane < ncopy) table_s[32 * k + lane] = v[k];
  } else if (warp >= kSoftWarp0 && (warp & 3) == 0) {
    // token j's list: selected from the block scores, or read
    const int j = (warp - kSoftWarp0) >> 2;
    const int tok = kQt * tile + j;
    const int pos = (seq_ok && tok < p.Q) ? L - p.Q + tok : -1;
    const int64_t i = static_cast<int64_t>(b) * p.Q + tok;
    pdl_wait();  // the lists, the scores they come from, or the outputs, are the previous kernel's
    int n = -1;
    if (kDense) {
      // no lists: every block the token sees
    } else if (p.scores) {
      // stage 1 + j, not loaded before the union is built, is this warp's scratch
      uint8_t* scratch = smem + (1 + j) * kStageBytes;
      bool nan = false;
      if (pos >= 0)
        n = select::select_row<16>(p.scores + g * p.s_stride_h + i * p.s_stride_t, p.s_stride_n,
                                   pos, lane, reinterpret_cast<uint32_t*>(scratch), kSelectCap,
                                   reinterpret_cast<int*>(scratch + 4 * kSelectCap), nan);
      if (lane < kTopK && tok < p.Q && split == 0)
        p.topk_out[(i * p.Hkv + g) * kTopK + lane] = n;
      if (__any_sync(0xffffffffu, nan) && lane == 0) flag_error(p.err, MSA_ERR_SCORE_NAN);
      tc::fence_proxy_async_smem();   // scratch writes before the TMA loads into it
    } else if (lane < kTopK && tok < p.Q) {
      n = p.topk[(i * p.Hkv + g) * kTopK + lane];
    }
    if (lane < kTopK && pos >= 0 && n != -1 && (n < 0 || n > pos / kPage)) {
      if (split == 0) flag_error(p.err, MSA_ERR_TOPK_RANGE);
      n = -1;
    }
    if (pos < 0) n = -1;
    if (lane < kTopK) tail->lists[j][lane] = n;
  } else if (warp >= kSoftWarp0 && (warp & 3) == 1) {
    // token j's query rows: hi at tile rows 32 j .. +15, lo at 32 j + 16 .. +31
    const int j = (warp - kSoftWarp0) >> 2;
    const int tok = kQt * tile + j;
    if (tok < p.Q) {
      const int64_t row = (static_cast<int64_t>(b) * p.Q + tok) * p.Hq + g * kGroup;
      if constexpr (kFp8Q) {
        store_query_rows_fp8(p.q8 + row * kHeadDim, 32 * j, qtile, lane);
        zero_query_rows(32 * j + 16, qtile, lane);
        if (lane == 0) tail->zs[j] = p.logit_scale * p.q_scale;
      } else {
        const int e = prepare_query_e4m3(p.q + row * kHeadDim, 32 * j, qtile,
                                         qtile + 16 * 128, lane);
        if (lane == 0) tail->zs[j] = p.logit_scale * exp2i(e);
      }
    } else {
      zero_query_rows(32 * j, qtile, lane);
      zero_query_rows(32 * j + 16, qtile, lane);
      if (lane == 0) tail->zs[j] = 0.f;
    }
    tc::fence_proxy_async_smem();  // the tile is read by the tensor core
  }
  // Warp 0 builds the union once the lists and the block-table row are in
  // shared memory: a barrier over warps 0 and 3 and the list warps only, so
  // that the query tiles are prepared meanwhile.
  constexpr int kListBarrier = 1, kListThreads = 32 * (2 + kQt);
  if (warp == 0 || warp == 3 || (warp >= kSoftWarp0 && (warp & 3) == 0))
    named_barrier(kListBarrier, kListThreads);

  // ---- prologue, part 2 (warp 0): the union and this CTA's pages --------------------
  if (kDense && warp == 0) {
    // the tile's blocks 0 .. cur_max cut into equal ranges; token j lists the
    // prefix of this CTA's range up to its own current block
    int cur_max = -1;
#pragma unroll
    for (int j = 0; j < kQt; ++j)
      if (tail->pos[j] >= 0) cur_max = tail->pos[j] / kPage;
    const int nblk = cur_max + 1;
    const int lo = static_cast<int>(static_cast<int64_t>(nblk) * split / nsplit);
    const int hi = static_cast<int>(static_cast<int64_t>(nblk) * (split + 1) / nsplit);
    const int np = hi - lo;
    // bad block-table entries: flagged, and attended by no token (their slot
    // loads page 0 instead, so that the stage holds finite bytes)
    for (int base = 0; base < np; base += 32) {
      const int t = base + lane;
      bool bad = false;
      if (t < np) {
        const int pg = lo + t < ncopy ? table_s[lo + t] : trow[lo + t];
        bad = pg < 0 || static_cast<int64_t>(pg) >= p.num_blocks;
      }
      const unsigned bb = __ballot_sync(0xffffffffu, bad);
      if (lane == 0 && base / 32 < kMaxDenseBlocks / 32) tail->dense_bad[base / 32] = bb;
      if (bb && lane == 0) flag_error(p.err, MSA_ERR_PAGE_RANGE);
    }
    if (lane == 0) {
      const int last_block = (seq_ok && L > 0) ? (L - 1) / kPage : -1;
      tail->fix_slot = (last_block >= lo && last_block < hi) ? last_block - lo : -1;
      tail->dense_lo = lo;
      tail->n_pages = np;
      for (int j = 0; j < kQt; ++j) {
        const int cur = tail->pos[j] >= 0 ? tail->pos[j] / kPage : -1;
        const int nj = cur + 1 - lo;
        tail->n_tok[j] = nj < 0 ? 0 : (nj > np ? np : nj);
      }
      for (int t = 0; t < np && t < kStages; ++t) {
        int pg = lo + t < ncopy ? table_s[lo + t] : trow[lo + t];
        if (pg < 0 || static_cast<int64_t>(pg) >= p.num_blocks) pg = 0;
        const int row = (pg * p.Hkv + g) * kPage;
        uint8_t* st = smem + t * kStageBytes;
        mbar_arrive_expect_tx(&tail->full[t], kStageBytes);
        tma_load_2d(st, &kv_map, 0, row, &tail->full[t]);
        tma_load_2d(st + kHalfTile, &kv_map, kHeadDim, row, &tail->full[t]);
      }
    }
  } else if (warp == 0) {
    // keys (block << 2 | token), invalid slots last; lane holds slots lane and lane + 32
    uint32_t v[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int e = 32 * r + lane, j = e >> 4;
      const int n = tail->lists[j][e & 15];
      v[r] = n >= 0 ? (static_cast<uint32_t>(n) << 2) | static_cast<uint32_t>(j) : 0xFFFFFFFFu;
    }
    warp_sort64(v, lane);
    // neighbours in sorted order by shuffles: the previous key, and the next
    // four (a block's run is at most one key per token in a valid list)
    uint32_t prev[2], nxt[2][4];
    {
      const uint32_t up0 = __shfl_up_sync(0xffffffffu, v[0], 1);
      const uint32_t up1 = __shfl_up_sync(0xffffffffu, v[1], 1);
      const uint32_t last0 = __shfl_sync(0xffffffffu, v[0], 31);
      prev[0] = lane == 0 ? 0xFFFFFFFFu : up0;
      prev[1] = lane == 0 ? last0 : up1;
#pragma unroll
      for (int d = 1; d <= 4; ++d) {
        const uint32_t dn0 = __shfl_down_sync(0xffffffffu, v[0], d);
        const uint32_t dn1 = __shfl_down_sync(0xffffffffu, v[1], d);
        const uint32_t wrap = __shfl_sync(0xffffffffu, v[1], (lane + d) & 31);
        nxt[0][d - 1] = lane + d < 32 ? dn0 : wrap;
        nxt[1][d - 1] = lane + d < 32 ? dn1 : 0xFFFFFFFFu;
      }
    }
    // per distinct block: first occurrence, the tokens listing it, its page
    bool keep[2];
    uint32_t mk[2];
    int pg[2];
    bool long_run = false;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint32_t k = v[r];
      const bool valid = k != 0xFFFFFFFFu;
      if (valid && prev[r] == k && split == 0)  // the same block twice in one token's list
        flag_error(p.err, MSA_ERR_TOPK_DUP);
      const bool first = valid && (prev[r] == 0xFFFFFFFFu || (prev[r] >> 2) != (k >> 2));
      uint32_t m = 0;
      if (first) {
        m = 1u << (k & 3);
        bool same = true;
#pragma unroll
        for (int d = 0; d < 4; ++d) {
          const uint32_t kf = nxt[r][d];
          same = same && kf != 0xFFFFFFFFu && (kf >> 2) == (k >> 2);
          if (same && d < 3) m |= 1u << (kf & 3);
          if (same && d == 3) long_run = true;   // five or more keys: duplicates
        }
      }
      int page = -1;
      bool ok = first;
      if (first) {
        const int n = static_cast<int>(k >> 2);
        page = n < ncopy ? table_s[n] : trow[n];
        if (page < 0 || static_cast<int64_t>(page) >= p.num_blocks) {
          if (split == 0) flag_error(p.err, MSA_ERR_PAGE_RANGE);
          ok = false;
        }
      }
      keep[r] = ok;
      mk[r] = m;
      pg[r] = page;
    }
    if (__any_sync(0xffffffffu, long_run)) {
      // a list with duplicates: each run's tokens from the whole sorted sequence
      tail->sorted[lane] = v[0];
      tail->sorted[32 + lane] = v[1];
      __syncwarp();
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (!keep[r]) continue;
        const uint32_t k = v[r];
        uint32_t m = 0;
        for (int f = 32 * r + lane; f < kMaxUnion; ++f) {
          const uint32_t kf = tail->sorted[f];
          if (kf == 0xFFFFFFFFu || (kf >> 2) != (k >> 2)) break;
          m |= 1u << (kf & 3);
        }
        mk[r] = m;
      }
      __syncwarp();
    }
    const unsigned b0 = __ballot_sync(0xffffffffu, keep[0]);
    const unsigned b1 = __ballot_sync(0xffffffffu, keep[1]);
    const int U = __popc(b0) + __popc(b1);
    // this CTA's range of the union, [lo, hi); the last range holds the union's
    // largest block, which goes first (its page may already be in stage 0)
    const int lo = static_cast<int>(static_cast<int64_t>(U) * split / nsplit);
    const int hi = static_cast<int>(static_cast<int64_t>(U) * (split + 1) / nsplit);
    const int np = hi - lo;
    const bool last_first = np > 0 && hi == U;
    const unsigned lt = (1u << lane) - 1u;
    const int pre_page = tail->pages[0];   // stage 0's page (or -1)
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (!keep[r]) continue;
      const int rank = (r == 0 ? 0 : __popc(b0)) + __popc((r == 0 ? b0 : b1) & lt);
      if (rank < lo || rank >= hi) continue;
      int slot = rank - lo;
      if (last_first) slot = (rank == U - 1) ? 0 : slot + 1;
      tail->pages[slot] = pg[r];
      tail->blocks[slot] = static_cast<int>(v[r] >> 2);
      tail->masks[slot] = mk[r];
    }
    __syncwarp();
    // each token's slots in page order, and the slot of the request's last block
    const int last_block = (seq_ok && L > 0) ? (L - 1) / kPage : -1;
    int fix = -1;
    for (int base = 0; base < np; base += 32) {
      const int t = base + lane;
      const uint32_t m = t < np ? tail->masks[t] : 0u;
      if (t < np && tail->blocks[t] == last_block) fix = t;
#pragma unroll
      for (int j = 0; j < kQt; ++j) {
        const unsigned bj = __ballot_sync(0xffffffffu, (m >> j) & 1u);
        const int before = base == 0 ? 0 : tail->n_tok[j];
        if ((m >> j) & 1u) tail->tok_slots[j][before + __popc(bj & lt)] = t;
        __syncwarp();
        if (lane == 0) tail->n_tok[j] = before + __popc(bj);
        __syncwarp();
      }
    }
    fix = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(fix + 1)) - 1;
    if (lane == 0) {
      if (np == 0)
        for (int j = 0; j < kQt; ++j) tail->n_tok[j] = 0;
      tail->fix_slot = fix;
      tail->n_pages = np;
      // stage 0 holds (or is loading) pre_page: it is page 0 of this list when
      // that is the union's largest block; otherwise the load lands unused and
      // stage 0's barrier starts over
      const bool stage0_used = pre_page >= 0 && last_first && tail->pages[0] == pre_page;
      if (pre_page >= 0 && !stage0_used) {
        if (!mbar_wait(&tail->full[0], 0)) flag_error(p.err, MSA_ERR_TIMEOUT);
        mbar_inval(&tail->full[0]);
        mbar_init(&tail->full[0], 1);
        fence_barrier_init();
      }
      for (int t = 0; t < np && t < kStages; ++t) {
        if (t > 0 || !stage0_used) {
          uint8_t* st = smem + t * kStageBytes;
          const int row = (tail->pages[t] * p.Hkv + g) * kPage;
          mbar_arrive_expect_tx(&tail->full[t], kStageBytes);
          tma_load_2d(st, &kv_map, 0, row, &tail->full[t]);
          tma_load_2d(st + kHalfTile, &kv_map, kHeadDim, row, &tail->full[t]);
        }
      }
    }
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const int n_pages = tail->n_pages;
  const uint32_t tmem = tail->tmem_base;
  const int dense_lo = kDense ? tail->dense_lo : 0;
  // slot t's tokens (mask), physical page and block; token j's k-th slot
  auto slot_mask = [&](int t) -> uint32_t {
    if constexpr (kDense) {
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < kQt; ++j)
        if (t < tail->n_tok[j]) m |= 1u << j;
      return m;
    } else {
      return tail->masks[t];
    }
  };
  auto slot_page = [&](int t) -> int {
    if constexpr (kDense) {
      const int pg = trow[dense_lo + t];
      return (pg < 0 || static_cast<int64_t>(pg) >= p.num_blocks) ? 0 : pg;
    } else {
      return tail->pages[t];
    }
  };
  auto slot_block = [&](int t) -> int { return kDense ? dense_lo + t : tail->blocks[t]; };
  auto slot_bad = [&](int t) -> bool {
    return kDense && t < kMaxDenseBlocks && ((tail->dense_bad[t >> 5] >> (t & 31)) & 1u);
  };
  auto tok_slot = [&](int j, int k) -> int { return kDense ? k : tail->tok_slots[j][k]; };

  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------------------
    if (lane == 0) {
      int issued = n_pages < kStages ? n_pages : kStages;
      for (int t = kStages; t < n_pages; ++t) {
        const int s = t % kStages;
        if (!mbar_wait(&tail->empty[s], ((t / kStages) - 1) & 1)) {
          flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        uint8_t* st = smem + s * kStageBytes;
        const int row = (slot_page(t) * p.Hkv + g) * kPage;
        mbar_arrive_expect_tx(&tail->full[s], kStageBytes);
        tma_load_2d(st, &kv_map, 0, row, &tail->full[s]);
        tma_load_2d(st + kHalfTile, &kv_map, kHeadDim, row, &tail->full[s]);
        issued = t + 1;
      }
      // the loads still in flight land before shared memory can be released
      for (int t = issued - kStages; t < issued; ++t)
        if (t >= 0) (void)mbar_wait(&tail->full[t % kStages], (t / kStages) & 1);
      pdl_trigger();   // every load of this CTA has landed
      mbar_arrive(&tail->finish);
    }
  } else if (warp == 1) {
    // ---- S^T walker: the pages in order -------------------------------------------------
    // Each page, once landed, is released at once for the tokens that did not
    // list it, and each listing token's S^T = K Q^T (its 32 query rows: hi,
    // then lo) goes into its next buffer as soon as that buffer has been read.
    if (lane == 0) {
      const uint64_t ak0 = tc::sw128_kmajor_desc(smem_u32(smem));
      const uint64_t bq0 = tc::sw128_kmajor_desc(smem_u32(qtile));
      constexpr uint32_t idesc = tc::idesc_e4m3_f32(128, 32);
      int cnt[kQt] = {0, 0, 0, 0};   // pages issued per token
      bool ok = true;
      for (int t = 0; t < n_pages && ok; ++t) {
        const int s = t % kStages;
        if (!mbar_wait(&tail->full[s], (t / kStages) & 1)) {
          flag_error(p.err, MSA_ERR_TIMEOUT);
          break;
        }
        tc::fence_after_thread_sync();
        const uint32_t mask = slot_mask(t);
        const int others = kQt - __popc(mask);
        if (!kDense && others > 0) mbar_arrive_count(&tail->empty[s], static_cast<unsigned>(others));
        const uint64_t a = ak0 + static_cast<uint64_t>(s) * (kStageBytes >> 4);
        // dense decode: the listing tokens are consecutive and all at their
        // t-th page (their lists are prefixes of the range), so one product
        // covers them, with one commit (to the last token's barrier, which
        // lists every page of the range and on which they all wait);
        // otherwise one product per listing token
        const int j0 = __ffs(mask) - 1, j1 = 31 - __clz(mask);
        const bool joint = kDense && mask == ((2u << j1) - (1u << j0));
        if (joint) {
          const int b = t % kSBufs;
          for (int j = j0; j <= j1 && ok; ++j) {
            if (t >= kSBufs && !mbar_wait(&tail->s_free[j][b], ((t / kSBufs) - 1) & 1)) {
              flag_error(p.err, MSA_ERR_TIMEOUT);
              ok = false;
            }
            cnt[j] = t + 1;
          }
          if (!ok) break;
          tc::fence_after_thread_sync();
          const uint64_t bj = bq0 + static_cast<uint64_t>((32 * j0 * 128) >> 4);
          const uint32_t d = tmem + kN * b + 32 * j0;
          const uint32_t idesc_m = tc::idesc_e4m3_f32(128, 32 * (j1 - j0 + 1));
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) tc::mma_e4m3(d, a + 2 * ks, bj + 2 * ks, idesc_m, ks > 0);
          tc::commit(&tail->s_full[j1][b]);
          continue;
        }
#pragma unroll
        for (int j = 0; j < kQt; ++j) {
          if (!(mask & (1u << j))) continue;
          const int k = cnt[j]++, b = k % kSBufs;
          if (k >= kSBufs && !mbar_wait(&tail->s_free[j][b], ((k / kSBufs) - 1) & 1)) {
            flag_error(p.err, MSA_ERR_TIMEOUT);
            ok = false;
            break;
          }
          tc::fence_after_thread_sync();
          const uint64_t bj = bq0 + static_cast<uint64_t>((32 * j * 128) >> 4);
          const uint32_t d = tmem + kN * b + 32 * j;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) tc::mma_e4m3(d, a + 2 * ks, bj + 2 * ks, idesc, ks > 0);
          tc::commit(&tail->s_full[j][b]);
        }
      }
      tc::commit(&tail->finish);  // arrives once this thread's MMAs have all completed
    }
    __syncwarp();
    (void)mbar_wait(&tail->finish, 0);
    tc::fence_after_thread_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  } else if (warp == 2) {
    // ---- O^T issuer: each token's next page once its P^T is written --------------------
    if (lane == 0) {
      const uint64_t av0 = tc::sw128_mnmajor_desc(smem_u32(smem + kHalfTile));
      // B: consecutive tokens' P^T columns (each token's hi, lo core matrices;
      // 128 bytes apart), 8-key blocks kPBlock apart
      const uint64_t bp0 = tc::interleave_mnmajor_desc(smem_u32(pbuf), kPBlock, 128);
      constexpr uint32_t idesc = tc::idesc_e4m3_f32_mn(128, 32);
      const int fix_slot = tail->fix_slot;
      if constexpr (kDense) {
        // pages in order; each page's listing tokens (consecutive, all at their
        // t-th page) share one product once all their P^T is written
        for (int t = 0; t < n_pages; ++t) {
          const uint32_t mask = slot_mask(t);
          const int j0 = __ffs(mask) - 1, j1 = 31 - __clz(mask), buf = t & 1, s = t % kStages;
          bool ok = mask != 0u;
          for (int j = j0; j <= j1 && ok; ++j)
            ok = mbar_wait(&tail->p_full[j][buf], (t >> 1) & 1);
          if (ok && t == fix_slot) ok = mbar_wait(&tail->vfix, 0);
          if (!ok) {
            flag_error(p.err, MSA_ERR_TIMEOUT);
            break;
          }
          tc::fence_after_thread_sync();
          const uint64_t a = av0 + static_cast<uint64_t>(s) * (kStageBytes >> 4);
          const uint64_t bp = bp0 + static_cast<uint64_t>((buf * kPBuf + 256 * j0) >> 4);
          const uint32_t d = tmem + kColAcc + 32 * j0;
          const uint32_t idesc_m = tc::idesc_e4m3_f32_mn(128, 32 * (j1 - j0 + 1));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_e4m3(d, a + 256 * kk, bp + ((4 * kPBlock) >> 4) * kk, idesc_m,
                         (t > 0 || kk > 0) ? 1u : 0u);
          // one commit for the tokens (the last token's barrier, on which
          // they all wait) and one for the stage
          tc::commit(&tail->o_done[j1][buf]);
          tc::commit(&tail->empty[s]);
        }
      } else {
        int k[kQt], n[kQt];
        int left = 0;
#pragma unroll
        for (int j = 0; j < kQt; ++j) {
          k[j] = 0;
          n[j] = tail->n_tok[j];
          left += n[j];
        }
        const unsigned long long t0 = global_ns();
        while (left > 0) {
          bool progress = false;
#pragma unroll
          for (int j = 0; j < kQt; ++j) {
            if (k[j] >= n[j]) continue;
            const int kj = k[j], buf = kj & 1;
            if (!mbar_test_wait(&tail->p_full[j][buf], (kj >> 1) & 1)) continue;
            const int t = tok_slot(j, kj), s = t % kStages;
            // on the request's last block the value rows past its last token are zeroed first
            if (t == fix_slot && !mbar_wait(&tail->vfix, 0)) {
              flag_error(p.err, MSA_ERR_TIMEOUT);
              left = 0;
              break;
            }
            tc::fence_after_thread_sync();
            const uint64_t a = av0 + static_cast<uint64_t>(s) * (kStageBytes >> 4);
            const uint64_t bp = bp0 + static_cast<uint64_t>((buf * kPBuf + 256 * j) >> 4);
            const uint32_t d = tmem + kColAcc + 32 * j;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_e4m3(d, a + 256 * kk, bp + ((4 * kPBlock) >> 4) * kk, idesc,
                           (kj > 0 || kk > 0) ? 1u : 0u);
            tc::commit(&tail->o_done[j][buf]);
            tc::commit(&tail->empty[s]);    // this token is done with the page
            k[j] = kj + 1;
            --left;
            progress = true;
          }
          if (!progress && global_ns() - t0 > kWaitLimitNs) {
            flag_error(p.err, MSA_ERR_TIMEOUT);
            break;
          }
        }
      }
      tc::commit(&tail->finish);
    }
  } else if (warp >= kSoftWarp0) {
    // ---- token j: softmax and output ------------------------------------------------------
    const int j = (warp - kSoftWarp0) >> 2;
    const int quarter = warp & 3;
    const int key = 32 * quarter + lane;  // key of the page; value dim d at the end
    // this thread's lane of token j's columns: S^T buffer b at + kN b, O^T hi | lo at + kColAcc
    const uint32_t lane_addr = tmem + 32 * j + (static_cast<uint32_t>(32 * quarter) << 16);
    const uint32_t acc_addr = lane_addr + kColAcc;
    const float zs = tail->zs[j];
    const int pos = tail->pos[j];
    const int n_j = tail->n_tok[j];
    const int fix_slot = tail->fix_slot;
    // the value rows past the request's last token are zeroed by the lowest
    // token that listed that page
    const int fix_tok = fix_slot >= 0 ? __ffs(slot_mask(fix_slot)) - 1 : -1;
    uint8_t* pj = pbuf + 256 * j;      // token j's P^T columns
    // the barriers token j waits on for its products: its own, or in dense
    // decode the last listing token's (it lists every page of the range, and
    // the products it commits are the tokens' joint ones; the others' pages
    // are a prefix of its, so no barrier runs two phases ahead of a wait)
    const int jw = kDense ? max(0, 31 - __clz(slot_mask(0))) : j;
    float* mxj = mx_all + j * 2 * 4 * kGroup;
    float* lsum = lsum_all + j * 4 * kGroup;
    bool ok = true;

    // Lane h < 16 of every warp keeps head h's nref = kPShift - m, m the
    // reference maximum in log2 units (+inf until the head has seen a key);
    // the other lanes read it by shuffle.  l: this key slot's share of each
    // head's running sum relative to m.  The output accumulates in tensor
    // memory, relative to m.
    float nref_h = INFINITY;
    float l[kGroup];
    fill(l, 0.f);
    uint32_t sv[32];   // page k's S^T row (hi | lo columns)
    for (int k = 0; k < n_j && ok; ++k) {
      const int t = tok_slot(j, k), buf = k & 1, sb = k % kSBufs;
      const int s = t % kStages;
      if (!mbar_wait(&tail->s_full[jw][sb], (k / kSBufs) & 1)) {
        ok = false;
        break;
      }
      tc::fence_after_thread_sync();
      tc::ld_32x32b_x32(lane_addr + kN * sb, sv);
      // keys <= lim are visible to this token (none on a dense slot with a bad entry)
      const int lim = slot_bad(t) ? -1 : pos - slot_block(t) * kPage;
      float x[kGroup];
      {
        tc::wait_ld();
        tc::fence_before_thread_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->s_free[j][sb]);
        const bool vis = key <= lim;
#pragma unroll
        for (int h = 0; h < kGroup; ++h)
          x[h] = vis ? __uint_as_float(sv[h]) + __uint_as_float(sv[h + kGroup]) : -INFINITY;
      }
      // this warp's 32 keys' maximum of each head, lane h keeping head h's
      float wm = -INFINITY;
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
        const float r = warp_max_f32(x[h]);
        if (lane == h) wm = r;
      }
      float* mxb = mxj + buf * 4 * kGroup;
      if (lane < kGroup) mxb[quarter * kGroup + lane] = wm;
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->mx_full[j][buf]);
      if (!mbar_wait(&tail->mx_full[j][buf], (k >> 1) & 1)) {
        ok = false;
        break;
      }
      // page maximum against m + kLazy, per head in lane h (a head without any
      // key so far has nref = +inf and always moves)
      float al_h = 1.f;   // 2^(m_old - m_new): 1 when m stays, 0 when the head had no key
      bool raise_h = false;
      if (lane < kGroup) {
        const float pm = fmaxf(fmaxf(mxb[lane], mxb[kGroup + lane]),
                               fmaxf(mxb[2 * kGroup + lane], mxb[3 * kGroup + lane])) * zs;
        raise_h = pm + nref_h > kPShift + kLazy;
        if (raise_h) {
          al_h = ex2(kPShift - nref_h - pm);
          nref_h = kPShift - pm;
        }
      }
      if (__any_sync(0xffffffffu, raise_h)) {  // the same decision in all four warps
#pragma unroll
        for (int h = 0; h < kGroup; ++h) l[h] *= __shfl_sync(0xffffffffu, al_h, h);
        if (k > 0) {
          // the accumulator holds the earlier pages relative to the old m: once
          // their products are complete (page k - 1's, and with it the earlier
          // ones), rescale it; page k's product waits for this page's P^T
          if (!mbar_wait(&tail->o_done[jw][(k - 1) & 1], ((k - 1) >> 1) & 1)) {
            ok = false;
            break;
          }
          tc::fence_after_thread_sync();
#pragma unroll
          for (int part = 0; part < 2; ++part) {   // the hi columns, then the lo ones
            uint32_t av[kGroup];
            tc::ld_32x32b_x16(acc_addr + kGroup * part, av);
            tc::wait_ld();
#pragma unroll
            for (int h = 0; h < kGroup; ++h)
              av[h] = __float_as_uint(__uint_as_float(av[h]) * __shfl_sync(0xffffffffu, al_h, h));
            tc::st_32x32b_x16(acc_addr + kGroup * part, av);
          }
          tc::wait_st();
        }
      }
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
        // P = 2^(x - m + 8); 0 for an invisible key
        x[h] = ex2(fmaf(x[h], zs, __shfl_sync(0xffffffffu, nref_h, h)));
        l[h] += x[h];
      }
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t h0, l0, h1, l1;
        split_e4m3x2(x[4 * q4], x[4 * q4 + 1], h0, l0);
        split_e4m3x2(x[4 * q4 + 2], x[4 * q4 + 3], h1, l1);
        hw[q4] = h0 | (h1 << 16);
        lw[q4] = l0 | (l1 << 16);
      }
      if (t == fix_slot && j == fix_tok) {
        // rows past the request's last token hold no key: P is 0 there for
        // every token, but the bytes may be anything (an fp8 NaN times 0 is
        // NaN), so they are zeroed before any O^T product reads them
        if (key >= tail->last_rows) {
          uint4* vrow = reinterpret_cast<uint4*>(smem + s * kStageBytes + kHalfTile + key * 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) vrow[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->vfix);
      }
      // P^T buffer `buf` was last read by page k - 2's product
      if (k >= 2 && !mbar_wait(&tail->o_done[jw][buf], ((k >> 1) - 1) & 1)) {
        ok = false;
        break;
      }
      // key k's 16 hi bytes at (key / 8) * kPBlock + 256 j + (key % 8) * 16, its lo bytes 128 further
      uint8_t* pk = pj + buf * kPBuf + (key >> 3) * kPBlock + (key & 7) * 16;
      *reinterpret_cast<uint4*>(pk) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(pk + 128) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      tc::fence_proxy_async_smem();
      tc::fence_before_thread_sync();   // the accumulator's rescale, if any, before O^T
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->p_full[j][buf]);
    }
    // no load is in flight here; with this wait the batch-16 dense decode
    // measured 149 instead of 152 us (code placement)
    tc::wait_ld();

    // the output: every O^T product complete, this thread's value dim of each head
    float o[kGroup];
    fill(o, 0.f);
    if (ok && n_j > 0) {
      ok = mbar_wait(&tail->o_done[jw][(n_j - 1) & 1], ((n_j - 1) >> 1) & 1);
      if (ok) {
        tc::fence_after_thread_sync();
        uint32_t av[32];
        tc::ld_32x32b_x32(acc_addr, av);
        tc::wait_ld();
#pragma unroll
        for (int h = 0; h < kGroup; ++h) o[h] = __uint_as_float(av[h]) + __uint_as_float(av[h + kGroup]);
      }
      tc::fence_before_thread_sync();
    }
    if (ok) {
      // running sums: this thread's share -> the whole page (128 key slots)
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
      }
      if (lane == 0) {
#pragma unroll
        for (int h4 = 0; h4 < 4; ++h4)
          *reinterpret_cast<float4*>(lsum + quarter * kGroup + 4 * h4) =
              make_float4(l[4 * h4], l[4 * h4 + 1], l[4 * h4 + 2], l[4 * h4 + 3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->l_full[j]);
      ok = mbar_wait(&tail->l_full[j], 0);
    }
    const int tok = kQt * tile + j;
    if (ok && tok < p.Q) {
#pragma unroll
      for (int h4 = 0; h4 < 4; ++h4) {
        float4 t4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float4 v = *reinterpret_cast<const float4*>(lsum + w * kGroup + 4 * h4);
          t4.x += v.x;
          t4.y += v.y;
          t4.z += v.z;
          t4.w += v.w;
        }
        l[4 * h4] = t4.x;
        l[4 * h4 + 1] = t4.y;
        l[4 * h4 + 2] = t4.z;
        l[4 * h4 + 3] = t4.w;
      }
      const int d = key;
      const int64_t row0 = (static_cast<int64_t>(b) * p.Q + tok) * p.Hq + g * kGroup;
      if (p.splits == 1) {
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
          const float f = (l[h] > 0.f) ? p.v_scale / l[h] : 0.f;
          p.out[(row0 + h) * kHeadDim + d] = static_cast<uint16_t>(f32_to_bf16_bits(o[h] * f));
        }
      } else {
        const int64_t rows = static_cast<int64_t>(p.B) * p.Q * p.Hq;
        const int64_t base = static_cast<int64_t>(split) * rows + row0;
#pragma unroll
        for (int h = 0; h < kGroup; ++h) p.part_o[(base + h) * kHeadDim + d] = o[h] * p.v_scale;
        // partial state in the merge kernel's terms: l = sum 2^(x - mref)
        if (key < kGroup) {
          float lr = 0.f;
#pragma unroll
          for (int h = 0; h < kGroup; ++h)
            if (h == key) lr = l[h];
          p.part_ml[(base + key) * 2] = -nref_h;  // m - kPShift; -inf for a head without keys
          p.part_ml[(base + key) * 2 + 1] = lr;
          // dense decode: a unit cut into fewer ranges than the workspace's
          // parts; its first range marks the rest empty for the merge
          if (kDense && split == 0)
            for (int s2 = nsplit; s2 < p.splits; ++s2) {
              p.part_ml[(static_cast<int64_t>(s2) * rows + row0 + key) * 2] = -INFINITY;
              p.part_ml[(static_cast<int64_t>(s2) * rows + row0 + key) * 2 + 1] = 0.f;
            }
        }
      }
    } else if (!ok && lane == 0) {
      flag_error(p.err, MSA_ERR_TIMEOUT);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->finish);
  }
}

}  // namespace

int union_ctas_per_unit(int units, int sm_count) {
  if (units >= sm_count) return 1;
  const int z = sm_count / units;
  return z > 8 ? 8 : z;
}

cudaError_t launch_union_attend(const CUtensorMap& kv_map, const AttendParams& p,
                                cudaStream_t stream, bool pdl) {
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [] {
    for (auto* k : {union_attend_kernel<false, false>, union_attend_kernel<true, false>,
                    union_attend_kernel<false, true>, union_attend_kernel<true, true>}) {
      cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemBytes);
      if (r != cudaSuccess) return r;
      r = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                               static_cast<int>(cudaSharedmemCarveoutMaxShared));
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const int ntiles = (p.Q + kQt - 1) / kQt;
  dim3 grid(p.B * ntiles * p.Hkv, p.splits);
  if (p.dense_span > 0 && p.splits > 1 && p.B * ntiles <= kBalancedTiles) {
    // dense decode on fewer units than SMs: one CTA per SM, shared out by the
    // units' blocks in the kernel (dense_slot), up to `splits` parts per unit
    int dev = 0, sms = 0;
    cudaError_t r = cudaGetDevice(&dev);
    if (r == cudaSuccess) r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (r != cudaSuccess) return r;
    if (p.B * ntiles * p.Hkv < sms) grid = dim3(sms, 1);
  }
  const dim3 block(kThreads);
  if (p.dense_span > 0)
    return p.q8 ? launch_pdl(union_attend_kernel<true, true>, grid, block, kSmemBytes, stream,
                             pdl, kv_map, p)
                : launch_pdl(union_attend_kernel<false, true>, grid, block, kSmemBytes, stream,
                             pdl, kv_map, p);
  return p.q8 ? launch_pdl(union_attend_kernel<true, false>, grid, block, kSmemBytes, stream, pdl,
                           kv_map, p)
              : launch_pdl(union_attend_kernel<false, false>, grid, block, kSmemBytes, stream, pdl,
                           kv_map, p);
}

}  // namespace msa
