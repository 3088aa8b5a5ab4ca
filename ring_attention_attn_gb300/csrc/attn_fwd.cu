// Blockwise ring-attention forward for sm_103a (GB300): TMA -> tcgen05 MMA
// into tensor memory -> online softmax in registers -> tcgen05 MMA -> epilogue.
//
// What it computes (k8ai "Sequence and Context Parallel", "How context
// parallel works"; "day 83" blog, "Context parallelism: splitting the
// sequence"): rank r's queries attend to the key/value blocks (r - s) mod P of
// its ring steps s, one 128-key tile at a time, folding every tile into a
// running row max m, row sum l and output O with the online softmax
//     m' = max(m, max_j s_j),  O = e^(m - m') O + sum_j e^(s_j - m') v_j,
//     l = e^(m - m') l + sum_j e^(s_j - m'),
// and finally writes O / l and LSE = m + ln l.  Scores are q.k / sqrt(d),
// masked by global token position (key <= query) for the zigzag causal split.
//
// CTA structure (384 threads, one CTA per SM, ~225 KB shared memory).  A
// unit is one query-tile pair with its steps; a CTA runs one unit, or, for
// short units, walks units blockIdx.x + k * gridDim.x (persistent), every
// role counting barrier phases across units:
//   warp 0       TMA producer: per unit the Q tile pair (once the previous
//                pair's last QK^T is done), then K_j, V_j tiles through a
//                ring of shared-memory slots (mbarrier full/empty pairs).
//   warp 1       allocates 512 TMEM columns and issues every tcgen05.mma and
//                tcgen05.commit: the whole warp runs the issue loop (so its
//                operands stay warp-uniform) and one elected lane executes
//                each tcgen05 instruction.
//   warps 4..7   softmax for query tile 0 (one thread per query row),
//   warps 8..11  softmax for query tile 1; the two tiles ping-pong so the
//                tensor core computes one tile's PV / next QK^T while the
//                other tile's softmax runs.
//   The producer/MMA warpgroup hands registers to the softmax warpgroups
//   (setmaxnreg).
// Tensor memory: S0 cols [0,128), S1 [128,256), O0 [256,256+d), O1 [384,384+d).
// P (bf16 probabilities) overwrites the first 64 columns of its tile's S (one
// bf16 pair per 32-bit column) and is the A operand of the PV MMA straight
// from tensor memory; QK^T takes both operands from shared memory.  Because
// P_i lives in S_i's columns, S_i of the next tile is issued after PV_i of
// this one; the MMAs of one thread execute in issue order.
//
// The O rescale is lazy: a row's reference max only moves when the new max
// exceeds it by more than 2^8 (in exp2 units), so P entries stay <= 256 and
// the O accumulator in TMEM is touched only on such rare jumps.
//
// Compile-time variants (ring_attn_kernel<D, OUT_F32, PK, CAUSAL, REM>): the
// head dimension; fp32 per-step partials or normalised bf16 output; the tile
// layout PK (0 row tiles, 1 packed short problems, 2 packed with 16 or 32
// rows per problem so each softmax warp owns one 32-column chunk); the
// causal mask; and REM, launches whose ranks' short last tiles are stacked
// into one query tile (rem_pack).  Code a variant does not use is not
// compiled into it, which keeps the softmax warpgroups' registers for the
// work that is there.
#include <math.h>

#include "ra_device.cuh"
#include "ra_internal.h"
#include "attn_common.cuh"

namespace ra {
namespace {

constexpr int kThreads = 384;
constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per tile
constexpr float kRescaleThreshold = 8.0f;
constexpr int kPersistMaxTiles = 32;  // key tiles per unit up to which CTAs persist
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;         // 128-byte swizzle atoms along d
  static constexpr int kChunkBytes = 128 * 128;  // one atom column of a 128-row tile
  static constexpr int kQTile = kBM * D * 2;
  static constexpr int kKVTile = kBN * D * 2;
  static constexpr int kSlots = (D == 128) ? 5 : 12;
  static constexpr int kOffQ0 = 0;
  static constexpr int kOffQ1 = kQTile;
  static constexpr int kOffKV = 2 * kQTile;
  static constexpr int kOffBar = kOffKV + kSlots * kKVTile;
  static constexpr int kBarBytes = 512;
  static_assert(8 * (9 + 2 * kSlots + 6) <= 496, "barriers overlap the TMEM slot");
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;  // + alignment slack
};

// Barrier indices (8 bytes each) in the barrier block.
enum : int {
  kBarQFull = 0,
  kBarSFull = 1,   // +wg
  kBarPFull = 3,   // +wg
  kBarODone = 5,   // +wg
  kBarDrain = 7,
  kBarQEmpty = 8,  // the Q pair's last QK^T has completed
  kBarKVFull = 9,  // +slot; kv_empty follows the kv_full block
};
// Split units (PK 3) use two more barriers after the K/V block: the softmax
// warpgroups' (m, l) exchange and "both O accumulators read" (256 arrivals
// each).
template <int D>
__device__ __forceinline__ int bar_xchg() { return kBarKVFull + 2 * Cfg<D>::kSlots; }
template <int D>
__device__ __forceinline__ int bar_ofree() { return kBarKVFull + 2 * Cfg<D>::kSlots + 1; }
// Split units at d = 64 keep three S tiles in tensor memory, and S_full and
// P_full belong to the S buffer instead of the warpgroup (a warpgroup may
// finish its next tile before the MMA warp has seen this one's P): the third
// buffer's S_full and P_full, and per warpgroup "its last PV has completed"
// (for the rare O rescale, which may no longer assume it).
template <int D>
__device__ __forceinline__ int bar_sfull2() { return kBarKVFull + 2 * Cfg<D>::kSlots + 2; }
template <int D>
__device__ __forceinline__ int bar_pvdone(int wg) { return kBarKVFull + 2 * Cfg<D>::kSlots + 3 + wg; }
template <int D>
__device__ __forceinline__ int bar_pfull2() { return kBarKVFull + 2 * Cfg<D>::kSlots + 5; }
constexpr int kTmemSlotOff = 496;
constexpr int kAbortOff = 500;
constexpr uint32_t kTmemCols = 512;
// TMEM columns of S_i and O_i.
__device__ __forceinline__ uint32_t col_s(int i) { return static_cast<uint32_t>(i) * 128u; }
__device__ __forceinline__ uint32_t col_o(int i) { return 256u + static_cast<uint32_t>(i) * 128u; }
// With three S tiles (split units, d = 64): S_0..S_2 at [0,384), O_0 at
// [384,448), O_1 at [448,512).
template <bool S3>
__device__ __forceinline__ uint32_t col_o_v(int i) {
  return S3 ? 384u + static_cast<uint32_t>(i) * 64u : col_o(i);
}

struct Unit {
  int bh, g, rank, s_lo, s_hi, pair, part;
  int64_t q_row0;  // first row of the rank's query chunk in the Q tensor
  bool rem;        // every rank's last rows in one tile (rem_pack)
};

// When a rank's last query-tile pair holds a single tile (L mod 256 <= 128),
// its units cost about half of the others; they are numbered last so that
// the block scheduler, which hands out CTAs in index order, packs them into
// the final, partial wave (longest units first).
template <bool REM, bool SPLIT, bool CAUSAL>
__device__ __forceinline__ Unit decode_unit(const AttnParams &p, int u) {
  Unit w;
  w.rem = false;
  if (SPLIT && CAUSAL) {
    // Causal split units (one query tile each) are numbered longest first:
    // the rank chunks' last query tiles of every head before their first
    // ones (in both zigzag halves a tile's visible key tiles grow with its
    // row), so that the block scheduler starts the longest in the first wave.
    const int nbg = p.BH * p.G;
    const int bhg = u % nbg;
    u /= nbg;
    w.part = u % p.n_stepgroups;
    u /= p.n_stepgroups;
    const int ri = u % p.n_ranks;
    w.pair = p.n_pairs - 1 - u / p.n_ranks;
    w.g = bhg % p.G;
    w.bh = bhg / p.G;
    w.rank = p.rank_begin + (p.pack_ranks ? 2 * ri : ri);
    w.s_lo = p.step_begin + w.part * p.steps_per_group;
    w.s_hi = w.s_lo + p.steps_per_group;
    w.q_row0 = static_cast<int64_t>(w.bh) * p.q_rows_bh + static_cast<int64_t>(w.g) * p.q_rows_g +
               static_cast<int64_t>(ri) * (p.q_rank_stride ? p.q_rank_stride : p.L);
    return w;
  }
  int np = p.n_pairs, pair_base = 0;
  // (Non-causal split units hold one query tile each: all cost alike.)
  if (!SPLIT && p.n_pairs > 1 && p.L - static_cast<int64_t>(p.n_pairs - 1) * 2 * kBM <= kBM) {
    const int heavy = (p.n_pairs - 1) * p.n_stepgroups * p.n_ranks * p.G * p.BH;
    if (u < heavy) {
      np = p.n_pairs - 1;
    } else {
      u -= heavy;
      np = 1;
      pair_base = p.n_pairs - 1;
      if (REM && p.rem_pack > 0) {
        // One unit per (head, problem, step group) for all ranks' last rows.
        w.rem = true;
        w.pair = pair_base;
        w.part = u % p.n_stepgroups;
        u /= p.n_stepgroups;
        w.g = u % p.G;
        w.bh = u / p.G;
        w.rank = p.rank_begin;
        w.s_lo = p.step_begin + w.part * p.steps_per_group;
        w.s_hi = w.s_lo + p.steps_per_group;
        w.q_row0 =
            static_cast<int64_t>(w.bh) * p.q_rows_bh + static_cast<int64_t>(w.g) * p.q_rows_g;
        return w;
      }
    }
  }
  w.pair = pair_base + u % np;
  u /= np;
  w.part = u % p.n_stepgroups;
  u /= p.n_stepgroups;
  const int ri = u % p.n_ranks;
  u /= p.n_ranks;
  w.g = u % p.G;
  w.bh = u / p.G;
  w.rank = p.rank_begin + (p.pack_ranks ? 2 * ri : ri);
  w.s_lo = p.step_begin + w.part * p.steps_per_group;
  w.s_hi = w.s_lo + p.steps_per_group;
  w.q_row0 = static_cast<int64_t>(w.bh) * p.q_rows_bh + static_cast<int64_t>(w.g) * p.q_rows_g +
             static_cast<int64_t>(ri) * (p.q_rank_stride ? p.q_rank_stride : p.L);
  return w;
}

// Walks the key tiles of a unit in ring order: steps s_lo..s_hi-1, block
// (rank - s) mod P, tiles of 128 keys; with the causal mask, tiles that no
// query of the pair may see are skipped.
struct TileIter {
  int s, t;
  int src;
  __device__ __forceinline__ void init(const AttnParams &p, const Unit &w) {
    s = w.s_lo;
    t = 0;
    src = ((w.rank - s) % p.P + p.P) % p.P;
  }
  template <bool CAUSAL>
  __device__ __forceinline__ void settle(const AttnParams &p, const Unit &w, int n_t,
                                         int64_t gq_max) {
    while (s < w.s_hi) {
      if (t >= n_t) {
        t = 0;
        ++s;
        src = (src == 0) ? p.P - 1 : src - 1;  // next block in ring order
        continue;
      }
      if (CAUSAL) {
        const int64_t gk_min = zz_pos(src, static_cast<int64_t>(t) * kBN, p.L >> 1, p.P);
        if (gk_min > gq_max) {
          ++t;
          continue;
        }
      }
      return;
    }
  }
  __device__ __forceinline__ bool valid(const Unit &w) const { return s < w.s_hi; }
};

// Geometry of one unit: its query-tile pair, whether the second tile holds
// rows, and (causal) the last global query position of the pair.
struct UnitGeo {
  Unit w;
  int64_t pair_row0, gq_max;
  bool has_q1;
};

template <bool CAUSAL, bool REM, bool SPLIT = false>
__device__ __forceinline__ UnitGeo unit_geo(const AttnParams &p, int u) {
  UnitGeo g;
  g.w = decode_unit<REM, SPLIT, CAUSAL>(p, u);
  // Split units: "pair" counts single query tiles and there is no tile 1.
  constexpr int kRows = SPLIT ? kBM : 2 * kBM;
  g.pair_row0 = static_cast<int64_t>(g.w.pair) * kRows;
  // Packed mode pairs rank chunks: tile 1 is the next rank's chunk.
  g.has_q1 = SPLIT    ? false
             : p.pack ? (p.pack_ranks > 0 && g.w.rank + 1 < p.rank_begin + p.pack_ranks)
                      : g.pair_row0 + kBM < p.L;
  g.gq_max = CAUSAL ? zz_pos(g.w.rank, min64(g.pair_row0 + kRows - 1, p.L - 1), p.L >> 1, p.P)
                      : 0;
  return g;
}

template <int D, bool OUT_F32, int PK, bool CAUSAL, bool REM>
__global__ void __launch_bounds__(kThreads, 1)
    ring_attn_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_qr, const AttnParams p, int n_units) {
  using C = Cfg<D>;
  // PK: 0 = row tiles, 1 = packed short problems, 2 = packed with 16 or 32
  // rows per problem (warp-packed softmax).
  // PK 3 = split units: one query tile per unit whose key tiles alternate
  // between the two softmax warpgroups (each with its own m, l and O), merged
  // in the epilogue; for launches with fewer units than SMs.
  constexpr bool kPack = PK == 1 || PK == 2;
  constexpr bool kSplit = PK == 3;
  static_assert(!kSplit || (!OUT_F32 && !REM), "split units: bf16 output, no stacked rows");
  // Non-causal split units at d = 64 ring three S tiles: S of tile t + 3 is
  // issued after PV of tile t, so a warpgroup's next S is usually complete
  // when its softmax of this tile ends (with two, each warpgroup waits a
  // PV + QK^T round trip per tile).  Tile t uses S buffer (T + t) mod 3, T
  // the tiles of the CTA's earlier units.  (Causal rows rescale O more
  // often, and each rescale must then wait for the warpgroup's last PV:
  // measured slower there.)
  constexpr bool kS3 = kSplit && D == 64 && !CAUSAL;
  // REM: launches with packed remainders (rem_pack > 0), non-causal row
  // tiles only.
  static_assert(!REM || (PK == 0 && !CAUSAL), "packed remainders: non-causal row tiles");
  constexpr bool kRem = REM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kOffBar;
  const uint32_t kv_full0 = bar0 + 8 * kBarKVFull;
  const uint32_t kv_empty0 = kv_full0 + 8 * C::kSlots;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffBar + kAbortOff);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffBar + kTmemSlotOff);
  const Watchdog wd{p.wd.status, p.wd.limit_ns};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_t = static_cast<int>((p.L + kBN - 1) / kBN);

  if (threadIdx.x == 0) {
    mbar_init(bar0 + 8 * kBarQFull, 1);
    mbar_init(bar0 + 8 * kBarQEmpty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar0 + 8 * (kBarSFull + i), 1);
      mbar_init(bar0 + 8 * (kBarPFull + i), 128);
      mbar_init(bar0 + 8 * (kBarODone + i), 1);
    }
    mbar_init(bar0 + 8 * kBarDrain, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(kv_full0 + 8 * s, 1);
      mbar_init(kv_empty0 + 8 * s, 1);
    }
    if (kSplit) {
      mbar_init(bar0 + 8 * bar_xchg<D>(), 256);
      mbar_init(bar0 + 8 * bar_ofree<D>(), 256);
    }
    if (kS3) {
      mbar_init(bar0 + 8 * bar_sfull2<D>(), 1);
      mbar_init(bar0 + 8 * bar_pfull2<D>(), 128);
      for (int i = 0; i < 2; ++i) mbar_init(bar0 + 8 * bar_pvdone<D>(i), 1);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (kPack) {
    // Rows past pack * pLrow of the Q tiles and of every K/V slot are never
    // written by TMA: zero them once so that masked keys meet finite values
    // (P = 0 times V must stay 0).
    const int r0 = p.pack * p.pLrow;
    const int per_chunk = (kBM - r0) * 8;  // 16-byte units
    const int regions = (C::kSlots + 2) * C::kChunks;
    for (int idx = threadIdx.x; idx < regions * per_chunk; idx += kThreads) {
      const int reg = idx / per_chunk, u = idx - reg * per_chunk;
      const int slot = reg / C::kChunks, c = reg - slot * C::kChunks;
      const uint32_t base = (slot < C::kSlots    ? sbase + C::kOffKV + slot * C::kKVTile
                             : slot == C::kSlots ? sbase + C::kOffQ0
                                                 : sbase + C::kOffQ1) +
                            c * C::kChunkBytes;
      st_shared_v4(base + r0 * 128 + u * 16, 0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Every role walks the same units (blockIdx.x, + gridDim.x, ...) and skips
  // the same empty ones (no visible key tile), so the barrier phases they
  // count stay in step across units.

  // Registers: the producer / MMA warpgroup gives most of its share to the
  // two softmax warpgroups (128*104 + 256*184 <= 384*168, the launch total).
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 104;\n" ::: "memory");
  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      const uint32_t qfull = bar0 + 8 * kBarQFull;
      const uint32_t pack_bytes = static_cast<uint32_t>(p.pack * p.pLrow) * 128u * C::kChunks;
      const uint64_t keep = l2_policy_evict_last();
      int it = 0;        // K/V slot sequence over all units
      int n_loaded = 0;  // Q pairs loaded
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const UnitGeo g = unit_geo<CAUSAL, kRem, kSplit>(p, u);
        const Unit &w = g.w;
        TileIter ti;
        ti.init(p, w);
        ti.settle<CAUSAL>(p, w, n_t, g.gq_max);
        if (!ti.valid(w)) continue;
        // The previous pair's last QK^T must have read the Q buffers.
        if (n_loaded > 0 &&
            !mbar_wait(bar0 + 8 * kBarQEmpty, (n_loaded - 1) & 1, wd, abort_flag))
          break;
        // Packed mode: box {64 d, Lf frames, pack positions, 1 head} of the
        // [head][frame][position][d] tensor, starting at the rank's first
        // frame and the unit's first position.
        int32_t pn = w.g * p.pack;
        int32_t pbh = w.bh;
        if (kPack) {
          int32_t f0 = w.rank * p.Lf, f1 = (w.rank + 1) * p.Lf;
          if (!RA_IN_BOUNDS(pn >= 0 && pn < p.pN && pbh >= 0 && pbh < p.BH && f0 >= 0 &&
                                f0 < p.pT && (!g.has_q1 || f1 < p.pT),
                            wd.status))
            pn = pbh = f0 = f1 = 0;
          mbar_arrive_expect_tx(qfull, g.has_q1 ? 2 * pack_bytes : pack_bytes);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c) {
            tma_load_4d(sbase + C::kOffQ0 + c * C::kChunkBytes, &tm_q, c * 64, f0, pn, pbh, qfull);
            if (g.has_q1)
              tma_load_4d(sbase + C::kOffQ1 + c * C::kChunkBytes, &tm_q, c * 64, f1, pn, pbh,
                          qfull);
          }
        } else if (kRem && w.rem) {
          // rem_pack rows of each rank, stacked in the first query tile
          // (rem_pack % 8 == 0 keeps the 128-byte swizzle phase).
          const int rr = p.rem_pack;
          const int64_t rstride = p.q_rank_stride ? p.q_rank_stride : p.L;
          mbar_arrive_expect_tx(qfull, static_cast<uint32_t>(p.n_ranks * rr * 128 * C::kChunks));
          for (int r = 0; r < p.n_ranks; ++r) {
            int32_t qy = static_cast<int32_t>(w.q_row0 + r * rstride + g.pair_row0);
            if (!RA_IN_BOUNDS(qy >= 0 && static_cast<int64_t>(qy) + rr <= p.chk_q_rows,
                              wd.status))
              qy = 0;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_2d(sbase + C::kOffQ0 + c * C::kChunkBytes + r * rr * 128, &tm_qr, c * 64, qy,
                          qfull);
          }
        } else {
          int32_t qy = static_cast<int32_t>(w.q_row0 + g.pair_row0);
          if (!RA_IN_BOUNDS(qy >= 0 && qy < p.chk_q_rows &&
                                (!g.has_q1 || static_cast<int64_t>(qy) + kBM < p.chk_q_rows),
                            wd.status))
            qy = 0;
          // Split units read one query tile (the Q1 buffer holds the
          // warpgroups' (m, l) exchange instead).
          mbar_arrive_expect_tx(qfull, kSplit ? C::kQTile : 2 * C::kQTile);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c) {
            tma_load_2d(sbase + C::kOffQ0 + c * C::kChunkBytes, &tm_q, c * 64, qy, qfull);
            if (!kSplit)
              tma_load_2d(sbase + C::kOffQ1 + c * C::kChunkBytes, &tm_q, c * 64, qy + kBM,
                          qfull);
          }
        }
        ++n_loaded;
        const int64_t kv_base =
            static_cast<int64_t>(w.bh) * p.kv_rows_bh + static_cast<int64_t>(w.g) * p.kv_rows_g;
        while (ok && ti.valid(w)) {
          const int64_t blk = p.kv_own ? static_cast<int64_t>(w.rank) * p.kv_rank_stride +
                                             static_cast<int64_t>(w.bh) * p.kv_rows_bh
                                       : kv_base + static_cast<int64_t>(ti.src) * p.L;
          int32_t ky = static_cast<int32_t>(blk + static_cast<int64_t>(ti.t) * kBN);
          int32_t kf = ti.src * p.Lf;
          if (!RA_IN_BOUNDS(kPack ? (kf >= 0 && kf < p.pT) : (ky >= 0 && ky < p.chk_kv_rows),
                            wd.status))
            ky = kf = 0;
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            const int slot = it % C::kSlots;
            const uint32_t ph = (it / C::kSlots) & 1;
            if (!mbar_wait(kv_empty0 + 8 * slot, ph ^ 1, wd, abort_flag)) {
              ok = false;
              break;
            }
            const CUtensorMap *map = which ? &tm_v : &tm_k;
            if (kPack) {
              mbar_arrive_expect_tx(kv_full0 + 8 * slot, pack_bytes);
#pragma unroll
              for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sbase + C::kOffKV + slot * C::kKVTile + c * C::kChunkBytes, map,
                            c * 64, kf, pn, pbh, kv_full0 + 8 * slot);
            } else {
              mbar_arrive_expect_tx(kv_full0 + 8 * slot, C::kKVTile);
#pragma unroll
              for (int c = 0; c < C::kChunks; ++c)
                tma_load_2d_hint(sbase + C::kOffKV + slot * C::kKVTile + c * C::kChunkBytes, map,
                                 c * 64, ky, kv_full0 + 8 * slot, keep);
            }
            ++it;
          }
          ++ti.t;
          ti.settle<CAUSAL>(p, w, n_t, g.gq_max);
        }
      }
      // Drain: every copy issued must land before the CTA may exit.
      if (n_loaded > 0) mbar_wait_drain(qfull, (n_loaded - 1) & 1, p.wd.limit_ns);
      for (int i = max(0, it - C::kSlots); i < it; ++i)
        mbar_wait_drain(kv_full0 + 8 * (i % C::kSlots), (i / C::kSlots) & 1, p.wd.limit_ns);
    }
  } else if (warp == 2 || warp == 3) {
    // ----------------------------------------------- in-launch ring exchange --
    // (Overlapped ring without a comm stream: this launch copies the blocks
    // the next step reads while its other warps compute.  A device copy would
    // need SMs that the launch holds.)
    if (p.x_on) {
      // Work items of up to 64 KB of one row, grid-strided over the CTAs; the
      // 64 threads keep eight 16-byte loads each in flight.
      constexpr int kU = 8;
      constexpr int64_t kChunk = 4096;  // 16-byte pieces per work item
      const int tid = static_cast<int>(threadIdx.x) - 64;
      const int64_t per_row = p.x_row_bytes >> 4;
      const int64_t chunks = (per_row + kChunk - 1) / kChunk;
      const int64_t rows = static_cast<int64_t>(p.x_ranks) * p.x_bh;
      const int64_t n_items = 2 * rows * chunks;
      for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int64_t row2 = item / chunks, c = item - row2 * chunks;
        const int tsel = row2 >= rows;
        const int64_t row = row2 - (tsel ? rows : 0);
        const int r = static_cast<int>(row / p.x_bh);
        const int64_t h = row - static_cast<int64_t>(r) * p.x_bh;
        const int from = (r + p.x_ranks - 1) % p.x_ranks;
        const int64_t so = from * p.x_src_rank + h * p.x_src_head;
        const int64_t dof = r * p.x_dst_rank + h * p.x_dst_head;
        const int64_t p0 = c * kChunk, p1 = min64(per_row, p0 + kChunk);
        if (!RA_IN_BOUNDS(so >= 0 && so + p1 * 16 <= p.x_src_span && dof >= 0 &&
                              dof + p1 * 16 <= p.x_dst_span,
                          wd.status))
          continue;
        const uint4 *src = reinterpret_cast<const uint4 *>((tsel ? p.xv_src : p.xk_src) + so);
        uint4 *dst = reinterpret_cast<uint4 *>((tsel ? p.xv_dst : p.xk_dst) + dof);
        for (int64_t pc = p0 + tid; pc < p1; pc += 64 * kU) {
          uint4 val[kU];
#pragma unroll
          for (int u = 0; u < kU; ++u)
            if (pc + u * 64 < p1) val[u] = src[pc + u * 64];
#pragma unroll
          for (int u = 0; u < kU; ++u)
            if (pc + u * 64 < p1) dst[pc + u * 64] = val[u];
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issue --
    {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, 0, 1);
      bool issued = false;
      const uint64_t dq[2] = {smem_desc_sw128(sbase + C::kOffQ0, 16, 1024),
                              smem_desc_sw128(sbase + C::kOffQ1, 16, 1024)};
      const uint64_t dk0 = smem_desc_sw128(sbase + C::kOffKV, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(sbase + C::kOffKV, C::kChunkBytes, 1024);
      auto issue_s = [&](int i, int slot) {
        issue_qk<D>(tmem + col_s(i), dq[i], dk0 + static_cast<uint64_t>(slot * (C::kKVTile >> 4)),
                    idesc_s);
      };
      auto issue_o = [&](int i, int slot, bool acc) {
        issue_pv(tmem + col_o(i), tmem + col_s(i),
                 dv0 + static_cast<uint64_t>(slot * (C::kKVTile >> 4)), idesc_o, acc);
      };
      // S_full barrier of S buffer b.
      auto sfull = [&](int b) -> uint32_t {
        return bar0 + 8 * (b < 2 ? kBarSFull + b : bar_sfull2<D>());
      };
      int it = 0;          // K/V slot sequence: K_j at 2j, V_j at 2j+1 of each unit
      int n_loaded = 0;    // Q pairs consumed
      int jt[2] = {0, 0};  // tiles handed to each softmax warpgroup so far
      bool ok = true;
      if constexpr (kSplit) {
        // Split units: visible key tile t of the unit goes to warpgroup t % 2;
        // both S_i read the one query tile.  S of tile t + 2 is issued right
        // after PV of tile t (it overwrites the same TMEM columns); with three
        // S buffers (d = 64), S of tile t + 3.
        int n_units_done = 0;  // units with at least one tile (O_done / O_free phases)
        int t_base = 0;        // tiles of earlier units (S buffer rotation, three buffers)
        for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
          const UnitGeo g = unit_geo<CAUSAL, kRem, kSplit>(p, u);
          const Unit &w = g.w;
          TileIter ts;  // next tile whose S is to be issued
          ts.init(p, w);
          ts.settle<CAUSAL>(p, w, n_t, g.gq_max);
          if (!ts.valid(w)) continue;
          if (!(ok = mbar_wait(bar0 + 8 * kBarQFull, n_loaded & 1, wd, abort_flag))) break;
          ++n_loaded;
          tc_fence_after();
          const int base = it;
          int ns = 0;  // tiles whose S has been issued
          auto issue_next_s = [&](int i) -> bool {
            const int seq = base + 2 * ns;
            if (!mbar_wait(kv_full0 + 8 * (seq % C::kSlots), (seq / C::kSlots) & 1, wd,
                           abort_flag))
              return false;
            tc_fence_after();
            if (kS3) i = (t_base + ns) % 3;
            issue_qk<D>(tmem + col_s(i), dq[0],
                        dk0 + static_cast<uint64_t>((seq % C::kSlots) * (C::kKVTile >> 4)),
                        idesc_s);
            mma_commit_e(sfull(i));
            mma_commit_e(kv_empty0 + 8 * (seq % C::kSlots));
            ++ns;
            ++ts.t;
            ts.settle<CAUSAL>(p, w, n_t, g.gq_max);
            // The unit's last QK^T has been issued: the Q buffer is free once
            // it completes.
            if (!ts.valid(w)) mma_commit_e(bar0 + 8 * kBarQEmpty);
            return true;
          };
          ok = issue_next_s(0) && (!ts.valid(w) || issue_next_s(1)) &&
               (!kS3 || !ts.valid(w) || issue_next_s(2));
          issued = true;
          for (int t = 0; ok && t < ns; ++t) {
            const int i = t & 1;
            const int seq_v = base + 2 * t + 1;
            if (!(ok = mbar_wait(kv_full0 + 8 * (seq_v % C::kSlots), (seq_v / C::kSlots) & 1, wd,
                                 abort_flag)))
              break;
            {
              uint32_t p_bar = bar0 + 8 * (kBarPFull + i), p_par = (jt[i] + (t >> 1)) & 1;
              if (kS3) {
                const int gt = t_base + t, b = gt % 3;
                p_bar = bar0 + 8 * (b < 2 ? kBarPFull + b : bar_pfull2<D>());
                p_par = (gt / 3) & 1;
              }
              if (!(ok = mbar_wait(p_bar, p_par, wd, abort_flag))) break;
            }
            // The first PV of a unit overwrites O_i: both warpgroups must
            // have read the previous unit's accumulators.
            if (t < 2 && n_units_done > 0 &&
                !(ok = mbar_wait(bar0 + 8 * bar_ofree<D>(), (n_units_done - 1) & 1, wd,
                                 abort_flag)))
              break;
            tc_fence_after();
            if (kS3) {
              // P_t sits in S buffer (t_base + t) mod 3; S of tile t + 3
              // takes that buffer after this PV.
              issue_pv(tmem + col_o_v<kS3>(i), tmem + col_s((t_base + t) % 3),
                       dv0 + static_cast<uint64_t>((seq_v % C::kSlots) * (C::kKVTile >> 4)),
                       idesc_o, t >= 2);
              mma_commit_e(bar0 + 8 * bar_pvdone<D>(i));
            } else {
              issue_o(i, seq_v % C::kSlots, t >= 2);
            }
            mma_commit_e(kv_empty0 + 8 * (seq_v % C::kSlots));
            if (ts.valid(w) && !(ok = issue_next_s(i))) break;
          }
          if (!ok) break;
          it = base + 2 * ns;
          t_base += ns;
          for (int i = 0; i < 2; ++i) mma_commit_e(bar0 + 8 * (kBarODone + i));
          jt[0] += (ns + 1) >> 1;
          jt[1] += ns >> 1;
          ++n_units_done;
        }
      } else
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const UnitGeo g = unit_geo<CAUSAL, kRem, kSplit>(p, u);
        const Unit &w = g.w;
        const bool has_q1 = g.has_q1;
        const int nq = has_q1 ? 2 : 1;
        TileIter ti;
        ti.init(p, w);
        ti.settle<CAUSAL>(p, w, n_t, g.gq_max);
        if (!ti.valid(w)) continue;
        if (!(ok = mbar_wait(bar0 + 8 * kBarQFull, n_loaded & 1, wd, abort_flag))) break;
        ++n_loaded;
        tc_fence_after();
        if (!(ok = mbar_wait(kv_full0 + 8 * (it % C::kSlots), (it / C::kSlots) & 1, wd,
                             abort_flag)))
          break;
        tc_fence_after();
        for (int i = 0; i < nq; ++i) {
          issue_s(i, it % C::kSlots);
          mma_commit_e(bar0 + 8 * (kBarSFull + i));
        }
        mma_commit_e(kv_empty0 + 8 * (it % C::kSlots));
        issued = true;
        ++it;
        int j = 0;
        for (;; ++j) {
          const int v_it = it;
          ++ti.t;
          ti.settle<CAUSAL>(p, w, n_t, g.gq_max);
          const bool more = ti.valid(w);
          // The pair's last QK^T has been issued: the Q buffers are free once
          // it completes.
          if (!more) mma_commit_e(bar0 + 8 * kBarQEmpty);
          if (!(ok = mbar_wait(kv_full0 + 8 * (v_it % C::kSlots), (v_it / C::kSlots) & 1, wd,
                               abort_flag)))
            break;
          if (!(ok = mbar_wait(bar0 + 8 * kBarPFull, (jt[0] + j) & 1, wd, abort_flag))) break;
          tc_fence_after();
          issue_o(0, v_it % C::kSlots, j > 0);
          const int k_it = v_it + 1;
          if (more) {
            if (!(ok = mbar_wait(kv_full0 + 8 * (k_it % C::kSlots), (k_it / C::kSlots) & 1, wd,
                                 abort_flag)))
              break;
            tc_fence_after();
            issue_s(0, k_it % C::kSlots);
            mma_commit_e(bar0 + 8 * kBarSFull);
          }
          if (has_q1) {
            if (!(ok = mbar_wait(bar0 + 8 * (kBarPFull + 1), (jt[1] + j) & 1, wd, abort_flag)))
              break;
            tc_fence_after();
            issue_o(1, v_it % C::kSlots, j > 0);
          }
          mma_commit_e(kv_empty0 + 8 * (v_it % C::kSlots));
          if (!more) break;
          if (has_q1) {
            issue_s(1, k_it % C::kSlots);
            mma_commit_e(bar0 + 8 * (kBarSFull + 1));
          }
          mma_commit_e(kv_empty0 + 8 * (k_it % C::kSlots));
          it = k_it + 1;
        }
        if (!ok) break;
        it = it + 1;  // the last tile's V slot
        for (int i = 0; i < nq; ++i) mma_commit_e(bar0 + 8 * (kBarODone + i));
        jt[0] += j + 1;
        if (has_q1) jt[1] += j + 1;
      }
      if (issued) {
        // Nothing may still be running on the tensor core when TMEM is freed.
        mma_commit_e(bar0 + 8 * kBarDrain);
        mbar_wait_drain(bar0 + 8 * kBarDrain, 0, p.wd.limit_ns);
      }
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;\n" ::: "memory");
    // ------------------------------------------------------------- softmax --
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t tS = tmem + lane_bits + col_s(wg);  // per tile with three S buffers
    const uint32_t tO = tmem + lane_bits + col_o_v<kS3>(wg);
    // This thread's TMEM lanes and columns: its S tiles and O accumulator.
    (void)RA_IN_BOUNDS(wg < 2 && row < kBM && col_s(kS3 ? 2 : 1) + kBN <= col_o_v<kS3>(0) &&
                           col_o_v<kS3>(wg) + D <= kTmemCols &&
                           (col_o_v<kS3>(1) >= col_o_v<kS3>(0) + D),
                       wd.status);
    const float sl2 = p.scale_log2;
    // Rows start 32-byte aligned when the output and its part stride are
    // (the entry points only promise 16): then 32-byte stores are used.
    const bool out_v8 = ((reinterpret_cast<uintptr_t>(p.out) |
                          static_cast<uintptr_t>(p.out_part_stride * (OUT_F32 ? 4 : 2))) &
                         31u) == 0;
    int jt = 0;      // tiles of this warpgroup so far (S_full / P_full phases)
    int n_done = 0;  // units whose O this warpgroup has read (O_done phases)
    int t_base = 0;  // tiles of earlier units (three S buffers)
    // The next unit's geometry is decoded while the last PV of the current
    // one runs, off the path from this unit's epilogue to the next S.
    UnitGeo g_next = unit_geo<CAUSAL, kRem, kSplit>(p, blockIdx.x);
    // Packed tiles: this thread's row is frame row_fr of problem row_pr in
    // every unit.
    const int row_pr = kPack ? row / p.pLrow : 0;
    const int row_fr = kPack ? row - row_pr * p.pLrow : 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const UnitGeo g = g_next;
      const int u_next = u + static_cast<int>(gridDim.x);
      const Unit &w = g.w;
      if (!kSplit && !(wg == 0 || g.has_q1)) {
        if (u_next < n_units) g_next = unit_geo<CAUSAL, kRem, kSplit>(p, u_next);
        continue;
      }
      // Row within the rank's chunk; in packed mode within the tile, whose
      // rank is w.rank + wg; split units: both warpgroups hold the same rows.
      const int64_t qi = kPack ? row : g.pair_row0 + (kSplit ? 0 : wg * kBM) + row;
      // Packed mode: row qi is frame qi % pLrow of the chunk of problem
      // g * pack + qi / pLrow (pLrow >= Lf rows per problem; rows past Lf
      // hold the next frames and are not written) and sees only the first Lf
      // keys of that problem (columns [lo, lo + Lf) of a tile).
      const int pr = row_pr;
      bool row_valid =
          qi < p.L && (!kPack || (static_cast<int64_t>(w.g) * p.pack + pr < p.pN &&
                                   row_fr < p.Lf));
      // Packed remainders: tile row r * rem_pack + i is row i of rank r's
      // last rows (offset from the first rank's chunk).
      int64_t rem_off = qi;
      if (kRem && w.rem) {
        const int rr = p.rem_pack;
        row_valid = row < p.n_ranks * rr;
        rem_off = static_cast<int64_t>(row / rr) * (p.q_rank_stride ? p.q_rank_stride : p.L) +
                  g.pair_row0 + row % rr;
      }
      const int64_t gq = CAUSAL ? zz_pos(w.rank, min64(qi, p.L - 1), p.L >> 1, p.P) : 0;

      // l sums the probabilities as computed (it gives the LSE); packed tiles
      // also sum them as rounded to bf16 (lr), the weights the PV MMA
      // actually applies, and normalise O by that: rows of a few dozen keys,
      // often dominated by one, would otherwise carry the rounding of the
      // dominant probability (up to 2^-9 relative) straight into O.
      float m_ref = -INFINITY, l = 0.f, lr = 0.f;
      int j = 0;
      int tv = 0;  // visible tiles of the unit walked (split units take every other)
      TileIter ti;
      ti.init(p, w);
      ti.settle<CAUSAL>(p, w, n_t, g.gq_max);
      while (ti.valid(w)) {
        if (kSplit && (tv & 1) != wg) {
          ++tv;
          ++ti.t;
          ti.settle<CAUSAL>(p, w, n_t, g.gq_max);
          continue;
        }
        uint32_t s_bar = bar0 + 8 * (kBarSFull + wg), s_par = (jt + j) & 1;
        uint32_t p_bar = bar0 + 8 * (kBarPFull + wg);
        if (kS3) {
          // Tile tv's S buffer b = (t_base + tv) mod 3, used (t_base + tv) / 3
          // times before.
          const int gt = t_base + tv, b = gt % 3;
          tS = tmem + lane_bits + col_s(b);
          s_bar = bar0 + 8 * (b < 2 ? kBarSFull + b : bar_sfull2<D>());
          s_par = (gt / 3) & 1;
          p_bar = bar0 + 8 * (b < 2 ? kBarPFull + b : bar_pfull2<D>());
        }
        const bool ok = __all_sync(0xffffffffu, mbar_wait(s_bar, s_par, wd, abort_flag));
        if (!ok) break;
        tc_fence_after();
        if constexpr (PK == 2) {
          float alpha = 1.f;
          bool rescale = false;
          float2 rs[4], rq[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) rs[x] = rq[x] = make_float2(0.f, 0.f);
          // Warp-packed temporal tiles: problems of pLrow = 16 or 32 rows sit
          // at the same offsets in the query and the key tile, so the keys
          // of this warp's 32 rows are exactly its own 32-column chunk: only
          // that chunk is loaded and exponentiated, and the other chunks of
          // P are zero.  A row sees the first Lf columns of its problem.
          float s[32];
          tmem_ld32(tS + 32 * quarter, s);
          tmem_wait_ld();
          const int lo = p.pLrow == 16 ? (lane & 16) : 0;
          const int hi = lo + p.Lf;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c < lo || c >= hi) s[c] = -INFINITY;
          float mx[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) mx[x] = fmaxf(s[2 * x], s[2 * x + 1]);
#pragma unroll
          for (int c = 8; c < 32; c += 8)
#pragma unroll
            for (int x = 0; x < 4; ++x) mx[x] = fmax3(mx[x], s[c + 2 * x], s[c + 2 * x + 1]);
          const float mxs = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sl2;
          if (mxs > m_ref + kRescaleThreshold) {
            if (m_ref != -INFINITY) {
              alpha = ex2(m_ref - mxs);
              rescale = true;
            }
            m_ref = mxs;
          }
          const float shift = (m_ref == -INFINITY) ? 0.f : m_ref;
          const float2 sl2v = make_float2(sl2, sl2);
          const float2 nshift = make_float2(-shift, -shift);
          uint32_t pk[16], zero[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const float2 a = ffma2(make_float2(s[2 * x], s[2 * x + 1]), sl2v, nshift);
            const float2 e = make_float2(ex2(a.x), ex2(a.y));
            rs[x & 3] = fadd2(rs[x & 3], e);
            pk[x] = pack_bf16x2(e.x, e.y);
            rq[x & 3] = fadd2(rq[x & 3], unpack_bf16x2(pk[x]));
            zero[x] = 0u;
          }
#pragma unroll
          for (int c = 0; c < kBN / 32; ++c) tmem_st16(tS + c * 16, c == quarter ? pk : zero);
          const float2 r01 = fadd2(rs[0], rs[1]), r23 = fadd2(rs[2], rs[3]);
          const float2 r = fadd2(r01, r23);
          const float rsum = r.x + r.y;
          l = l * alpha + rsum;
          const float2 q01 = fadd2(rq[0], rq[1]), q23 = fadd2(rq[2], rq[3]);
          const float2 rqs = fadd2(q01, q23);
          lr = lr * alpha + (rqs.x + rqs.y);
          if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              float o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int x = 0; x < 32; ++x) o[x] *= alpha;
              tmem_st32(tO + c * 32, o);
            }
          }
        } else {
          float s[kBN];
#pragma unroll
          for (int c = 0; c < kBN / 32; ++c)
            tmem_ld32(tS + c * 32, *reinterpret_cast<float(*)[32]>(&s[c * 32]));
          tmem_wait_ld();

          const int64_t k0 = static_cast<int64_t>(ti.t) * kBN;
          int nvis = static_cast<int>(min64(kBN, p.L - k0));
          if (CAUSAL) nvis = causal_visible(ti.src, k0, gq, p.L, p.P);
          int lo = 0;
          if (kPack) {
            lo = pr * p.pLrow;
            nvis = min(nvis, lo + p.Lf);
          }
          if (lo > 0 || nvis < kBN) {
#pragma unroll
            for (int c = 0; c < kBN; ++c)
              if (c < lo || c >= nvis) s[c] = -INFINITY;
          }
          // Row max with 3-input max (two new scores per instruction), 4 chains.
          float mx[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) mx[x] = fmaxf(s[2 * x], s[2 * x + 1]);
#pragma unroll
          for (int c = 8; c < kBN; c += 8)
#pragma unroll
            for (int x = 0; x < 4; ++x) mx[x] = fmax3(mx[x], s[c + 2 * x], s[c + 2 * x + 1]);
          const float mxs = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sl2;
          float alpha = 1.f;
          bool rescale = false;
          if (mxs > m_ref + kRescaleThreshold) {
            if (m_ref != -INFINITY) {
              alpha = ex2(m_ref - mxs);
              rescale = true;
            }
            m_ref = mxs;
          }
          const float shift = (m_ref == -INFINITY) ? 0.f : m_ref;
          const float2 sl2v = make_float2(sl2, sl2);
          const float2 nshift = make_float2(-shift, -shift);
          float2 rs[4], rq[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) rs[x] = rq[x] = make_float2(0.f, 0.f);
          // P overwrites the first 64 columns of this tile's S (already in
          // registers): bf16 pairs, lower key in the low half.  Scale/shift and
          // the row sum use packed f32x2 arithmetic (two scores per instruction).
#pragma unroll
          for (int c = 0; c < kBN / 32; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) {
              const float2 a = ffma2(make_float2(s[32 * c + 2 * x], s[32 * c + 2 * x + 1]), sl2v, nshift);
              const float2 e = make_float2(ex2(a.x), ex2(a.y));
              rs[x & 3] = fadd2(rs[x & 3], e);
              pk[x] = pack_bf16x2(e.x, e.y);
              if constexpr (kPack) rq[x & 3] = fadd2(rq[x & 3], unpack_bf16x2(pk[x]));
            }
            tmem_st16(tS + c * 16, pk);
          }
          const float2 r01 = fadd2(rs[0], rs[1]), r23 = fadd2(rs[2], rs[3]);
          const float2 r = fadd2(r01, r23);
          const float rsum = r.x + r.y;
          l = l * alpha + rsum;
          if constexpr (kPack) {
            const float2 q01 = fadd2(rq[0], rq[1]), q23 = fadd2(rq[2], rq[3]);
            const float2 rqs = fadd2(q01, q23);
            lr = lr * alpha + (rqs.x + rqs.y);
          }
          if (__any_sync(0xffffffffu, rescale)) {
            // Three S buffers: this warpgroup's previous PV (tile tv - 2) may
            // still be accumulating into O.
            if (kS3 && !__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * bar_pvdone<D>(wg),
                                                           (jt + j - 1) & 1, wd, abort_flag)))
              break;
            if (kS3) tc_fence_after();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              float o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int x = 0; x < 32; ++x) o[x] *= alpha;
              tmem_st32(tO + c * 32, o);
            }
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_bar);
        ++j;
        ++tv;
        ++ti.t;
        ti.settle<CAUSAL>(p, w, n_t, g.gq_max);
      }
      __syncwarp();
      const bool aborted = __shfl_sync(0xffffffffu, *abort_flag, 0) != 0;
      if (aborted) break;
      if (u_next < n_units) g_next = unit_geo<CAUSAL, kRem, kSplit>(p, u_next);
      if constexpr (kSplit) {
        // Merge the two warpgroups' partial softmax states of each row:
        //   M = max(m0, m1),  a_i = 2^(m_i - M),  l = a0 l0 + a1 l1,
        //   O = (a0 O0 + a1 O1) / l,  LSE = (M + log2 l) ln 2,
        // the (m, l) pairs exchanged through shared memory (double-buffered
        // by unit), O0 and O1 read from tensor memory; warpgroup i writes
        // columns [i D/2, (i+1) D/2) of the row.
        jt += j;
        t_base += tv;
        if (tv == 0) continue;  // no visible key tile: the MMA warp skipped the unit too
        float *xb = reinterpret_cast<float *>(smem + C::kOffQ1) + (n_done & 1) * (4 * kBM);
        xb[(wg * kBM + row) * 2] = m_ref;
        xb[(wg * kBM + row) * 2 + 1] = l;
        mbar_arrive(bar0 + 8 * bar_xchg<D>());
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bar0 + 8 * bar_xchg<D>(), n_done & 1, wd, abort_flag)))
          break;
        const float m_o = xb[((1 - wg) * kBM + row) * 2];
        const float l_o = xb[((1 - wg) * kBM + row) * 2 + 1];
        const float M = fmaxf(m_ref, m_o);
        const float a_s = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - M);
        const float a_o = (m_o == -INFINITY) ? 0.f : ex2(m_o - M);
        const float lt = a_s * l + a_o * l_o;
        const float inv = (lt > 0.f) ? 1.f / lt : 0.f;
        const float c0 = (wg == 0 ? a_s : a_o) * inv, c1 = (wg == 0 ? a_o : a_s) * inv;
        const bool have1 = tv >= 2;  // warpgroup 1 met a tile: O1 holds this unit's sum
        const bool done = __all_sync(
            0xffffffffu, mbar_wait(bar0 + 8 * kBarODone, n_done & 1, wd, abort_flag) &&
                             mbar_wait(bar0 + 8 * (kBarODone + 1), n_done & 1, wd, abort_flag));
        ++n_done;
        if (!done) break;
        tc_fence_after();
        const int64_t orow = w.q_row0 + qi;
        if (row_valid && !RA_IN_BOUNDS(orow >= 0 && orow < p.chk_out_rows, wd.status))
          row_valid = false;
        __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(p.out) + orow * D;
        const uint32_t tO0 = tmem + lane_bits + col_o_v<kS3>(0);
        const uint32_t tO1 = tmem + lane_bits + col_o_v<kS3>(1);
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          const int c = wg * (D / 64) + cc;
          float o0[32], o1[32];
          tmem_ld32(tO0 + c * 32, o0);
          if (have1) tmem_ld32(tO1 + c * 32, o1);
          tmem_wait_ld();
          if (!have1) {
#pragma unroll
            for (int x = 0; x < 32; ++x) o1[x] = 0.f;
          }
          if (row_valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(out + c * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              uint32_t v4[4];
#pragma unroll
              for (int y = 0; y < 4; ++y) {
                const int e = 8 * x + 2 * y;
                v4[y] = pack_bf16x2(fmaf(c0, o0[e], c1 * o1[e]),
                                    fmaf(c0, o0[e + 1], c1 * o1[e + 1]));
              }
              dst[x] = make_uint4(v4[0], v4[1], v4[2], v4[3]);
            }
          }
        }
        // Both accumulators have been read: the next unit's PVs may start.
        tc_fence_before();
        mbar_arrive(bar0 + 8 * bar_ofree<D>());
        if (row_valid && wg == 0) p.lse[orow] = (lt > 0.f) ? (M + lg2(lt)) * kLn2 : -INFINITY;
        continue;
      }
      bool have_o = false;
      if (j > 0) {
        have_o = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (kBarODone + wg), n_done & 1, wd,
                                                   abort_flag));
        ++n_done;
        if (!have_o) break;
        tc_fence_after();
      }
      jt += j;
      const float l_o = kPack ? lr : l;  // the normaliser of O
      const float inv_l = (l_o > 0.f) ? 1.f / l_o : 0.f;
      const float lse_val = (l > 0.f) ? (m_ref + lg2(l)) * kLn2 : -INFINITY;
      const int part = p.part_by_block ? ((w.rank - w.s_lo) % p.P + p.P) % p.P : w.part;
      // Packed mode: frame f = (w.rank + wg) * Lf + qi % pLrow of position
      // n = g * pack + qi / pLrow.
      const int64_t pf = static_cast<int64_t>(w.rank + wg) * p.Lf + row_fr;
      const int64_t pn = static_cast<int64_t>(w.g) * p.pack + pr;
      const int64_t orow =
          !kPack                 ? w.q_row0 + rem_off
          : p.pack_frame_major ? (static_cast<int64_t>(w.bh) * p.pT + pf) * p.pN + pn
                               : (static_cast<int64_t>(w.bh) * p.pN + pn) * p.pT + pf;
      if (row_valid && !RA_IN_BOUNDS(orow >= 0 && orow < p.chk_out_rows && part >= 0 &&
                                         part < p.chk_parts,
                                     wd.status))
        row_valid = false;
      if (OUT_F32) {
        float *out = reinterpret_cast<float *>(p.out) + part * p.out_part_stride + orow * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          if (have_o) {
            tmem_ld32(tO + c * 32, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = 0.f;
          }
          if (row_valid && out_v8) {
            // 32-byte stores: every lane writes whole L2 sectors of its row.
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              uint32_t v8[8];
#pragma unroll
              for (int y = 0; y < 8; ++y) v8[y] = __float_as_uint(o[8 * x + y] * inv_l);
              st_global_v8(out + c * 32 + 8 * x, v8);
            }
          } else if (row_valid) {
            float4 *dst = reinterpret_cast<float4 *>(out + c * 32);
#pragma unroll
            for (int x = 0; x < 8; ++x)
              dst[x] = make_float4(o[4 * x] * inv_l, o[4 * x + 1] * inv_l, o[4 * x + 2] * inv_l,
                                   o[4 * x + 3] * inv_l);
          }
        }
      } else {
        __nv_bfloat16 *out =
            reinterpret_cast<__nv_bfloat16 *>(p.out) + part * p.out_part_stride + orow * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          if (have_o) {
            tmem_ld32(tO + c * 32, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = 0.f;
          }
          if (row_valid && out_v8) {
            // 32-byte stores: every lane writes whole L2 sectors of its row.
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              uint32_t v8[8];
#pragma unroll
              for (int y = 0; y < 8; ++y)
                v8[y] = pack_bf16x2(o[16 * x + 2 * y] * inv_l, o[16 * x + 2 * y + 1] * inv_l);
              st_global_v8(out + c * 32 + 16 * x, v8);
            }
          } else if (row_valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(out + c * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x)
              dst[x] = make_uint4(pack_bf16x2(o[8 * x] * inv_l, o[8 * x + 1] * inv_l),
                                  pack_bf16x2(o[8 * x + 2] * inv_l, o[8 * x + 3] * inv_l),
                                  pack_bf16x2(o[8 * x + 4] * inv_l, o[8 * x + 5] * inv_l),
                                  pack_bf16x2(o[8 * x + 6] * inv_l, o[8 * x + 7] * inv_l));
          }
        }
      }
      if (row_valid) p.lse[part * p.lse_part_stride + orow] = lse_val;
      // O of this unit has been read into registers: the next unit's first
      // PV (accumulate off) may overwrite it once this warpgroup's next
      // P_full arrival, which follows these loads, has been seen.
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}


// A kernel whose only wait can never complete (nothing arrives on the
// barrier): exercises the bounded-wait path.
__global__ void watchdog_selftest_kernel(WatchdogParams wdp) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const Watchdog wd{wdp.status, wdp.limit_ns};
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, wd, &abort_flag);
  __syncthreads();
}

// Checks one index against a bound it exceeds, touching no memory through
// it: the RA_CHECKS build records RA_ERR_BOUNDS, the default build nothing.
__global__ void checks_selftest_kernel(int *status, int index, int bound) {
  (void)RA_IN_BOUNDS(index < bound, status);
}

// --------------------------------------------------------------- host side --
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

// 2-D bf16 row matrix [rows, d], box = 128 rows x 64 elements (128 bytes),
// 128-byte swizzle; rows past the end read as zero.
cudaError_t make_row_map(CUtensorMap *map, const void *base, int64_t rows, int d,
                         int box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Packed temporal problems read in place: the bf16 tensor [BH][T][N][d]
// (frame-major video tokens) seen as 4-D with dims (d, frame, position,
// head) and strides (2 B, N·d·2, d·2, T·N·d·2), box = 64 elements x Lrow
// frames x pack positions x 1 head, so a box lands in shared memory
// position-major (pack problems of Lrow rows each).  128-byte swizzle;
// coordinates past the end read as zero.
cudaError_t make_pack_map(CUtensorMap *map, const void *base, int64_t BH, int T, int64_t N, int Lrow,
                          int pack, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t row = static_cast<cuuint64_t>(d) * 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[3] = {row * static_cast<cuuint64_t>(N), row,
                           row * static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(T)};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(Lrow), static_cast<cuuint32_t>(pack), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, bool OUT_F32, int PK, bool CAUSAL, bool REM>
cudaError_t launch_kernel(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                          const CUtensorMap &mqr, const AttnParams &p, int64_t n_units,
                          int64_t grid, int dev, cudaStream_t stream) {
  using C = Cfg<D>;
  static bool configured[64] = {};
  if (!configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(ring_attn_kernel<D, OUT_F32, PK, CAUSAL, REM>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  ring_attn_kernel<D, OUT_F32, PK, CAUSAL, REM>
      <<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(
          mq, mk, mv, mqr, p, static_cast<int>(n_units));
  return cudaGetLastError();
}

// Multiprocessors of device `dev` (cached; 0 on failure).
int sm_count(int dev) {
  static int sms[64] = {};
  if (dev < 0 || dev >= 64) return 0;
  if (sms[dev] == 0 &&
      cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms[dev] = 0;
  return sms[dev];
}

template <int D, bool OUT_F32, int PK, bool CAUSAL>
cudaError_t launch_variant(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                           const CUtensorMap &mqr, const AttnParams &p, int64_t n_units,
                           cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  // Short units (a few key tiles each: 900-token frames, packed temporal
  // problems) run persistently, one CTA per SM walking units blockIdx.x,
  // + gridDim.x, ..., so that a CTA's next query pair and key tiles load
  // while its current pair finishes.  Long units get one CTA each and the
  // block scheduler balances them (static striding costs ~1% there).
  const int sms = sm_count(dev);
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int64_t tiles_per_unit = ((p.L + kBN - 1) / kBN) * p.steps_per_group;
  const int64_t grid =
      (tiles_per_unit <= kPersistMaxTiles && n_units > sms) ? sms : n_units;
  if constexpr (PK == 0 && !OUT_F32) {
    // A launch of fewer pair units than SMs runs as split units (one query
    // tile each, its key tiles shared by the two softmax warpgroups): twice
    // the units, half the work on the longest one.  One unit per CTA.
    if (p.rem_pack == 0 && n_units < sms) {
      AttnParams ps = p;
      ps.n_pairs = static_cast<int>((p.L + kBM - 1) / kBM);
      const int64_t nu = static_cast<int64_t>(ps.BH) * ps.G * ps.n_stepgroups * ps.n_ranks *
                         ps.n_pairs;
      return launch_kernel<D, false, 3, CAUSAL, false>(mq, mk, mv, mqr, ps, nu, nu, dev, stream);
    }
  }
  if constexpr (PK == 0 && !CAUSAL) {
    if (p.rem_pack > 0)
      return launch_kernel<D, OUT_F32, PK, CAUSAL, true>(mq, mk, mv, mqr, p, n_units, grid, dev,
                                                         stream);
  }
  return launch_kernel<D, OUT_F32, PK, CAUSAL, false>(mq, mk, mv, mqr, p, n_units, grid, dev,
                                                      stream);
}

}  // namespace

cudaError_t launch_ring_attn(const void *q, int64_t q_total_rows, const void *k, const void *v,
                             int64_t kv_total_rows, int d, bool out_f32,
                             const AttnParams &params, cudaStream_t stream) {
  const int64_t per_pair = static_cast<int64_t>(params.BH) * params.G * params.n_stepgroups;
  // With rem_pack every rank's single last tile shares one unit.
  const int64_t n_units =
      params.rem_pack > 0 ? per_pair * ((params.n_pairs - 1) * params.n_ranks + 1)
                          : per_pair * params.n_ranks * params.n_pairs;
  if (n_units <= 0) return cudaSuccess;
  if (n_units > 0x7fffffff) return cudaErrorInvalidConfiguration;
  // Extents the RA_CHECKS build checks indices against: outputs have as many
  // rows per part as the Q row matrix, one part per step group (or per block).
  AttnParams pc = params;
  pc.chk_q_rows = q_total_rows;
  pc.chk_kv_rows = kv_total_rows;
  pc.chk_out_rows = q_total_rows;
  pc.chk_parts = pc.part_by_block ? pc.P : pc.n_stepgroups;
  const AttnParams &p = pc;
  CUtensorMap mq, mk, mv, mqr;
  cudaError_t e;
  if (p.pack) {
    if (out_f32 || p.causal || p.pLrow < p.Lf || p.pack * p.pLrow > kBM)
      return cudaErrorInvalidValue;
    if ((e = make_pack_map(&mq, q, p.BH, p.pT, p.pN, p.pLrow, p.pack, d)) != cudaSuccess) return e;
    if ((e = make_pack_map(&mk, k, p.BH, p.pT, p.pN, p.pLrow, p.pack, d)) != cudaSuccess) return e;
    if ((e = make_pack_map(&mv, v, p.BH, p.pT, p.pN, p.pLrow, p.pack, d)) != cudaSuccess) return e;
    mqr = mq;
    // Problems of 16 or 32 rows: every warp's rows and keys share one
    // 32-column chunk (the warp-packed softmax).
    const bool wp = p.pLrow == 16 || p.pLrow == 32;
    if (d == 128)
      return wp ? launch_variant<128, false, 2, false>(mq, mk, mv, mqr, p, n_units, stream)
                : launch_variant<128, false, 1, false>(mq, mk, mv, mqr, p, n_units, stream);
    return wp ? launch_variant<64, false, 2, false>(mq, mk, mv, mqr, p, n_units, stream)
              : launch_variant<64, false, 1, false>(mq, mk, mv, mqr, p, n_units, stream);
  } else {
    if ((e = make_row_map(&mq, q, q_total_rows, d)) != cudaSuccess) return e;
    if ((e = make_row_map(&mk, k, kv_total_rows, d)) != cudaSuccess) return e;
    if ((e = make_row_map(&mv, v, kv_total_rows, d)) != cudaSuccess) return e;
  }
  if (p.rem_pack > 0) {
    if (p.pack || p.causal || p.rem_pack % 8 != 0 || p.n_ranks * p.rem_pack > kBM)
      return cudaErrorInvalidValue;
    if ((e = make_row_map(&mqr, q, q_total_rows, d, p.rem_pack)) != cudaSuccess) return e;
  } else {
    mqr = mq;
  }
  // Row tiles: the causal mask and the tile skipping it allows are compiled
  // only into the causal instantiations.
  if (d == 128) {
    if (p.causal)
      return out_f32 ? launch_variant<128, true, 0, true>(mq, mk, mv, mqr, p, n_units, stream)
                     : launch_variant<128, false, 0, true>(mq, mk, mv, mqr, p, n_units, stream);
    return out_f32 ? launch_variant<128, true, 0, false>(mq, mk, mv, mqr, p, n_units, stream)
                   : launch_variant<128, false, 0, false>(mq, mk, mv, mqr, p, n_units, stream);
  }
  if (p.causal)
    return out_f32 ? launch_variant<64, true, 0, true>(mq, mk, mv, mqr, p, n_units, stream)
                   : launch_variant<64, false, 0, true>(mq, mk, mv, mqr, p, n_units, stream);
  return out_f32 ? launch_variant<64, true, 0, false>(mq, mk, mv, mqr, p, n_units, stream)
                 : launch_variant<64, false, 0, false>(mq, mk, mv, mqr, p, n_units, stream);
}

cudaError_t launch_checks_selftest(int *status, cudaStream_t stream) {
  if (status == nullptr) return cudaErrorInvalidValue;
  checks_selftest_kernel<<<1, 1, 0, stream>>>(status, 1, 1);
  return cudaGetLastError();
}

cudaError_t launch_watchdog_selftest(const WatchdogParams &wd, cudaStream_t stream) {
  watchdog_selftest_kernel<<<1, 32, 0, stream>>>(wd);
  return cudaGetLastError();
}

}  // namespace ra
