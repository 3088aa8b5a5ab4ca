// Ring-attention backward for sm_103a: gradients dQ, dK, dV of the forward
// in attn_fwd.cu (the ring's exchanges recur in the backward pass of every
// attention layer: k8ai "Sequence and Context Parallel", "Communication
// profile").  With s_ij = scale q_i.k_j, P_ij = exp(s_ij - LSE_i) (LSE from
// the forward) and D_i = dO_i . O_i:
//     dP_ij = dO_i . v_j,   dS_ij = P_ij (dP_ij - D_i),
//     dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,
//     dQ_i = scale sum_j dS_ij k_j.
// The ring order is kept: rank r's dQ visits K/V blocks (r - s) mod P at
// step s, as in the forward; block b's dK/dV gather the query chunks of the
// ranks the block passes through, r = (b + s) mod P at step s.
//
// Two launches:
//   bwd_prep_kernel   D_i = dO_i . O_i (fp32), one warp per row.
//   bwd_kernel        one CTA per unit of either kind (dK/dV units first, so
//                     the shorter dQ units fill the launch's last wave):
//     dQ unit         one 128-row query tile, whose Q and dO the compute
//                     warpgroups first copy into TMEM.  Per K/V tile, in two
//                     halves of 64 keys: S_h = Q K_h^T and dP_h = dO V_h^T
//                     (Q, dO from TMEM, K, V from SMEM) into TMEM; compute
//                     warpgroup h writes dS_h (bf16) over S_h; dQ += dS_h K_h
//                     takes it from TMEM.
//     dK/dV unit      one 128-key tile.  Per query tile, in two halves of 64
//                     queries: S^T_h = K Q_h^T and dP^T_h = V dO_h^T; compute
//                     warpgroup h writes P^T_h over S^T_h and dS^T_h over
//                     dP^T_h (bf16); dV += P^T_h dO_h and dK += dS^T_h Q_h
//                     take them from TMEM.
//   Non-causal chunks whose last tile is short stack every chunk's last rows
//   (queries for dQ, keys for dK/dV) into one tile per head (REM variants):
//   one unit instead of P nearly empty ones.
// Roles (384 threads): warp 0 TMA producer, warp 1 TMEM allocation and
// elected MMA issue, warps 4..7 / 8..11 compute warpgroups 0 / 1, one thread
// per row of the tile and half h of its columns.  The halves pipeline: while
// warpgroup h works on half h of tile j, the tensor core runs the other
// half's products and half h's MMAs of tile j+1 wait only for it.
#include <math.h>

#include "attn_common.cuh"
#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kThreadsB = 384;
constexpr float kLog2eB = 1.44269504088896340736f;

constexpr int kBKVFirst = 11;

template <int D>
struct BCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = 128 * 128;
  static constexpr int kTile = 128 * D * 2;
  // as many streamed-tile slots as fit next to the two fixed tiles
  static constexpr int kSlots = (232448 - 1024 - 512 - 2048 - 2 * kTile) / kTile;
  static constexpr int kOffA = 0;           // Q (dQ kernel) or K (dK/dV kernel)
  static constexpr int kOffB = kTile;       // dO (dQ kernel) or V (dK/dV kernel)
  static constexpr int kOffKV = 2 * kTile;  // ring of streamed tiles
  static constexpr int kOffBar = kOffKV + kSlots * kTile;
  static constexpr int kBarBytes = 512;
  static constexpr int kOffLD = kOffBar + kBarBytes;  // [half][buffer](-LSE[64], -D[64]) fp32
  static constexpr int kLDBytes = 2048;
  static constexpr int kSmemBytes = kOffLD + kLDBytes + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(8 * (kBKVFirst + 2 * kSlots) <= 496, "barriers overlap the TMEM slot");
};

// Barriers: fixed tiles loaded, half h of S/dP ready (+h), half h computed
// (+h, 128 arrivals), accumulators done, drain, the dK/dV kernel's LSE/D
// staging (+2h + buffer, 128 arrivals), then full/empty per ring slot.
enum : int { kBA = 0, kBH = 1, kBC = 3, kBO = 5, kBDrain = 6, kBLd = 7, kBKV = kBKVFirst };
constexpr int kBTmemSlot = 496;
constexpr int kBAbort = 500;
constexpr uint32_t kColS = 0, kColP = 128, kColAcc0 = 256, kColAcc1 = 384;
// dQ units: Q at kColQT and dO at kColQT + D/2 (bf16 pairs), the A operands
// of S and dP straight from tensor memory; kBQT (256 arrivals) = both copied.
constexpr uint32_t kColQT = 384;
constexpr int kBQT = 7;

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// D[tmem] = A[tmem] B[smem]^T over d: A (128 rows x d, bf16 pairs, 8 columns
// per 16 elements) from tensor memory, B K-major with the 128-byte swizzle.
template <int D>
__device__ __forceinline__ void issue_qk_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t db,
                                            uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
    mma_ts_e(d_tmem, a_tmem + kk * 8, db + off, idesc, kk > 0 ? 1u : 0u);
  }
}

__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16 *__restrict__ out,
                                                       const __nv_bfloat16 *__restrict__ dout,
                                                       float *__restrict__ Dv, int64_t rows, int d) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (row >= rows) return;
  float acc = 0.f;
  for (int c = lane * 2; c < d; c += 64) {
    const __nv_bfloat162 o = *reinterpret_cast<const __nv_bfloat162 *>(out + row * d + c);
    const __nv_bfloat162 g = *reinterpret_cast<const __nv_bfloat162 *>(dout + row * d + c);
    acc = fmaf(__low2float(o), __low2float(g), acc);
    acc = fmaf(__high2float(o), __high2float(g), acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) Dv[row] = acc;
}

// K/V blocks for rank r (dQ) or query chunks for block b (dK/dV), in ring
// order, in 128-row tiles; causal tiles with nothing visible are skipped.
template <bool CAUSAL>
struct BIter {
  int s, t, blk;
  int P, n_t, dir;  // dir -1: blk = (r - s) mod P; +1: blk = (b + s) mod P
  int64_t C, limit;         // causal: dQ skips tiles with min position > limit,
                            //         dK/dV skips tiles with max position < limit
  int64_t L;
  __device__ __forceinline__ void settle() {
    while (s < P) {
      if (t >= n_t) {
        t = 0;
        ++s;
        blk = dir < 0 ? (blk == 0 ? P - 1 : blk - 1) : (blk == P - 1 ? 0 : blk + 1);
        continue;
      }
      if (CAUSAL) {
        const int64_t t0 = static_cast<int64_t>(t) * 128;
        const bool skip = dir < 0 ? zz_pos(blk, t0, C, P) > limit
                                  : zz_pos(blk, min64(t0 + 127, L - 1), C, P) < limit;
        if (skip) {
          ++t;
          continue;
        }
      }
      return;
    }
  }
  __device__ __forceinline__ bool valid() const { return s < P; }
};

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16 *dst, const float (&o)[32], float mul) {
  uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int x = 0; x < 4; ++x)
    d4[x] = make_uint4(pack_bf16x2(o[8 * x] * mul, o[8 * x + 1] * mul),
                       pack_bf16x2(o[8 * x + 2] * mul, o[8 * x + 3] * mul),
                       pack_bf16x2(o[8 * x + 4] * mul, o[8 * x + 5] * mul),
                       pack_bf16x2(o[8 * x + 6] * mul, o[8 * x + 7] * mul));
}

// One barrier-block layout for both kernels.
struct BBars {
  uint32_t bar0, kv_full0, kv_empty0;
  __device__ __forceinline__ uint32_t b(int i) const { return bar0 + 8 * i; }
};

template <int D>
__device__ __forceinline__ BBars init_bars(uint32_t sbase) {
  using C = BCfg<D>;
  BBars r;
  r.bar0 = sbase + C::kOffBar;
  r.kv_full0 = r.bar0 + 8 * kBKV;
  r.kv_empty0 = r.kv_full0 + 8 * C::kSlots;
  return r;
}

// Half-tile MMA issue: an accumulation over 64 rows of the streamed tile
// (K = 64: four MMAs of 16) with A (bf16 pairs) from TMEM and B MN-major.
__device__ __forceinline__ void issue_acc_k64(uint32_t d_tmem, uint32_t a_tmem, uint64_t db,
                                              uint32_t idesc, bool acc) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_ts_e(d_tmem, a_tmem + kk * 8, db + static_cast<uint64_t>(kk * (2048 >> 4)), idesc,
             (acc || kk > 0) ? 1u : 0u);
}

// Descriptor offset of row 64 of a 128-row, 128-byte-swizzled tile.
constexpr uint64_t kHalfRows = (64 * 128) >> 4;

// ------------------------------------------------------------------ dQ ----
template <int D, bool CAUSAL, bool REM>
__device__ __forceinline__ void bwd_dq_body(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                            const CUtensorMap &tm_v, const CUtensorMap &tm_do,
                                            const CUtensorMap &tm_qr, const CUtensorMap &tm_dor,
                                            const BwdParams &p, int unit) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const BBars bb = init_bars<D>(sbase);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffBar + kBAbort);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffBar + kBTmemSlot);
  const Watchdog wd{p.wd.status, p.wd.limit_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // With REM, units past BH * P * (n_t - 1) stack every rank's last rows.
  int u = unit;
  const int nt_full = REM ? p.n_t - 1 : p.n_t;
  const bool stacked = REM && u >= p.BH * p.P * nt_full;
  int qt, r, bh;
  if (stacked) {
    qt = p.n_t - 1;
    r = 0;
    bh = u - p.BH * p.P * nt_full;
  } else {
    qt = u % nt_full;
    u /= nt_full;
    r = u % p.P;
    bh = u / p.P;
  }
  const int64_t C2 = p.L >> 1;
  const int64_t n_rows = static_cast<int64_t>(p.BH) * p.S;  // rows of every [BH, S] tensor
  const int64_t q0 = static_cast<int64_t>(qt) * 128;
  const int64_t nq = stacked ? static_cast<int64_t>(p.P) * p.rem : min64(128, p.L - q0);
  const int64_t q_row0 = static_cast<int64_t>(bh) * p.S + static_cast<int64_t>(r) * p.L + q0;
  const int64_t gq_max = CAUSAL ? zz_pos(r, q0 + nq - 1, C2, p.P) : 0;
  auto make_iter = [&]() {
    BIter<CAUSAL> it{0, 0, r, p.P, p.n_t, -1, C2, gq_max, p.L};
    it.settle();
    return it;
  };

  if (threadIdx.x == 0) {
    mbar_init(bb.b(kBA), 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(bb.b(kBH + h), 1);
      mbar_init(bb.b(kBC + h), 128);
    }
    mbar_init(bb.b(kBO), 1);
    mbar_init(bb.b(kBDrain), 1);
    mbar_init(bb.b(kBQT), 256);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bb.kv_full0 + 8 * s, 1);
      mbar_init(bb.kv_empty0 + 8 * s, 1);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      if (stacked) {
        // Each rank's rem last rows of Q and dO, stacked (rem % 8 == 0 keeps
        // the 128-byte swizzle phase).
        mbar_arrive_expect_tx(bb.b(kBA), static_cast<uint32_t>(2 * p.P * p.rem * 128 * C::kChunks));
        for (int rr = 0; rr < p.P; ++rr) {
          int32_t y = static_cast<int32_t>(q_row0 + static_cast<int64_t>(rr) * p.L);
          if (!RA_IN_BOUNDS(y >= 0 && static_cast<int64_t>(y) + p.rem <= n_rows, wd.status)) y = 0;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c) {
            tma_load_2d(sbase + C::kOffA + c * C::kChunkBytes + rr * p.rem * 128, &tm_qr, c * 64, y,
                        bb.b(kBA));
            tma_load_2d(sbase + C::kOffB + c * C::kChunkBytes + rr * p.rem * 128, &tm_dor, c * 64,
                        y, bb.b(kBA));
          }
        }
      } else {
        int32_t y = static_cast<int32_t>(q_row0);
        if (!RA_IN_BOUNDS(q_row0 >= 0 && q_row0 < n_rows, wd.status)) y = 0;
        mbar_arrive_expect_tx(bb.b(kBA), 2 * C::kTile);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_2d(sbase + C::kOffA + c * C::kChunkBytes, &tm_q, c * 64, y, bb.b(kBA));
          tma_load_2d(sbase + C::kOffB + c * C::kChunkBytes, &tm_do, c * 64, y, bb.b(kBA));
        }
      }
      int it = 0;
      bool ok = true;
      for (auto ti = make_iter(); ok && ti.valid(); ++ti.t, ti.settle()) {
        int32_t ky = static_cast<int32_t>(static_cast<int64_t>(bh) * p.S +
                                          static_cast<int64_t>(ti.blk) * p.L +
                                          static_cast<int64_t>(ti.t) * 128);
        if (!RA_IN_BOUNDS(ky >= 0 && ky < n_rows, wd.status)) ky = 0;
        for (int which = 0; which < 2 && ok; ++which, ++it) {
          const int slot = it % C::kSlots;
          if (!(ok = mbar_wait(bb.kv_empty0 + 8 * slot, ((it / C::kSlots) & 1) ^ 1, wd, abort_flag)))
            break;
          mbar_arrive_expect_tx(bb.kv_full0 + 8 * slot, C::kTile);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_2d(sbase + C::kOffKV + slot * C::kTile + c * C::kChunkBytes,
                        which ? &tm_v : &tm_k, c * 64, ky, bb.kv_full0 + 8 * slot);
        }
      }
      mbar_wait_drain(bb.b(kBA), 0, p.wd.limit_ns);
      for (int i = max(0, it - C::kSlots); i < it; ++i)
        mbar_wait_drain(bb.kv_full0 + 8 * (i % C::kSlots), (i / C::kSlots) & 1, p.wd.limit_ns);
    }
  } else if (warp == 1) {
    constexpr uint32_t idesc_h = idesc_bf16_f32(128, 64, 0, 0);
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);
    constexpr uint32_t kSlotDesc = C::kTile >> 4;
    const uint64_t dKV = smem_desc_sw128(sbase + C::kOffKV, 16, 1024);
    const uint64_t dKVmn = smem_desc_sw128(sbase + C::kOffKV, C::kChunkBytes, 1024);
    // S_h = Q K_h^T and dP_h = dO V_h^T for the 64 keys of half h of the
    // K/V tiles in slots ks, vs.
    auto issue_s = [&](int h, int ks, int vs) {
      issue_qk_ts<D>(tmem + kColS + 64 * h, tmem + kColQT,
                     dKV + static_cast<uint64_t>(ks * kSlotDesc) + h * kHalfRows, idesc_h);
      issue_qk_ts<D>(tmem + kColP + 64 * h, tmem + kColQT + D / 2,
                     dKV + static_cast<uint64_t>(vs * kSlotDesc) + h * kHalfRows, idesc_h);
      mma_commit_e(bb.b(kBH + h));
    };
    bool issued = false, ok = true;
    auto ti = make_iter();
    // Q and dO reach tensor memory through the compute warpgroups.
    if (ti.valid() && mbar_wait(bb.b(kBQT), 0, wd, abort_flag)) {
      tc_fence_after();
      int it = 0;  // K_j in slot it, V_j in it + 1
      ok = mbar_wait(bb.kv_full0 + 8 * (it % C::kSlots), (it / C::kSlots) & 1, wd, abort_flag) &&
           mbar_wait(bb.kv_full0 + 8 * ((it + 1) % C::kSlots), ((it + 1) / C::kSlots) & 1, wd,
                     abort_flag);
      if (ok) {
        tc_fence_after();
        issue_s(0, it % C::kSlots, (it + 1) % C::kSlots);
        issue_s(1, it % C::kSlots, (it + 1) % C::kSlots);
        mma_commit_e(bb.kv_empty0 + 8 * ((it + 1) % C::kSlots));  // V_0: last use issued
        issued = true;
      }
      for (int j = 0; ok; ++j) {
        const int ks = it % C::kSlots;
        const int nk = it + 2;
        ++ti.t;
        ti.settle();
        const bool more = ti.valid();
        for (int h = 0; h < 2 && ok; ++h) {
          if (!(ok = mbar_wait(bb.b(kBC + h), j & 1, wd, abort_flag))) break;
          tc_fence_after();
          // dQ += dS_h K_h: dS_h over S_h's columns, K MN-major (d contiguous).
          issue_acc_k64(tmem + kColAcc0, tmem + kColS + 64 * h,
                        dKVmn + static_cast<uint64_t>(ks * kSlotDesc) + h * kHalfRows, idesc_o,
                        j > 0 || h > 0);
          if (h == 1) mma_commit_e(bb.kv_empty0 + 8 * ks);  // K_j: last use issued
          if (more) {
            if (h == 0) {
              ok = mbar_wait(bb.kv_full0 + 8 * (nk % C::kSlots), (nk / C::kSlots) & 1, wd,
                             abort_flag) &&
                   mbar_wait(bb.kv_full0 + 8 * ((nk + 1) % C::kSlots), ((nk + 1) / C::kSlots) & 1,
                             wd, abort_flag);
              if (!ok) break;
              tc_fence_after();
            }
            issue_s(h, nk % C::kSlots, (nk + 1) % C::kSlots);
            if (h == 1) mma_commit_e(bb.kv_empty0 + 8 * ((nk + 1) % C::kSlots));  // V_{j+1}
          }
        }
        if (!ok || !more) break;
        it = nk;
      }
      if (ok) mma_commit_e(bb.b(kBO));
    }
    if (issued) {
      mma_commit_e(bb.b(kBDrain));
      mbar_wait_drain(bb.b(kBDrain), 0, p.wd.limit_ns);
    }
  } else if (warp >= 4) {
    const int h = (warp - 4) >> 2;  // half of the key tile this warpgroup handles
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_bits + kColS + 64 * h, tP = tmem + lane_bits + kColP + 64 * h;
    const int64_t grow =
        stacked ? q_row0 + static_cast<int64_t>(row / p.rem) * p.L + row % p.rem : q_row0 + row;
    const bool valid =
        row < nq && RA_IN_BOUNDS(grow >= 0 && grow < n_rows && (D / 2) * h + D / 2 <= D &&
                                     kColQT + (D / 2) * (h + 1) <= 512,
                                 wd.status);
    const float lse2 = valid ? p.lse[grow] * kLog2eB : 0.f;
    const float Drow = valid ? p.Dv[grow] : 0.f;
    const int64_t gq = CAUSAL ? zz_pos(r, min64(q0 + row, p.L - 1), C2, p.P) : 0;
    const float sl2 = p.scale_log2;
    const float2 sl2v = make_float2(sl2, sl2), nlse2 = make_float2(-lse2, -lse2),
                 nD2 = make_float2(-Drow, -Drow);
    // Warpgroup 0 copies this row of Q, warpgroup 1 of dO, from the swizzled
    // shared-memory tile (16-byte piece c of a 128-byte row segment sits at
    // piece c ^ (row % 8)) into tensor memory as bf16 pairs.
    if (__all_sync(0xffffffffu, mbar_wait(bb.b(kBA), 0, wd, abort_flag))) {
      const uint32_t src = sbase + (h == 0 ? C::kOffA : C::kOffB) + row * 128;
      const uint32_t dst = tmem + lane_bits + kColQT + (D / 2) * h;
#pragma unroll
      for (int k = 0; k < D / 64; ++k) {
        uint32_t u0[16], u1[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 a = ld_shared_v4(src + k * C::kChunkBytes + ((c ^ (row & 7)) << 4));
          const uint4 b = ld_shared_v4(src + k * C::kChunkBytes + (((c + 4) ^ (row & 7)) << 4));
          u0[4 * c] = a.x; u0[4 * c + 1] = a.y; u0[4 * c + 2] = a.z; u0[4 * c + 3] = a.w;
          u1[4 * c] = b.x; u1[4 * c + 1] = b.y; u1[4 * c + 2] = b.z; u1[4 * c + 3] = b.w;
        }
        tmem_st16(dst + k * 32, u0);
        tmem_st16(dst + k * 32 + 16, u1);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bb.b(kBQT));
    }
    int j = 0;
    for (auto ti = make_iter(); ti.valid(); ++j, ++ti.t, ti.settle()) {
      if (!__all_sync(0xffffffffu, mbar_wait(bb.b(kBH + h), j & 1, wd, abort_flag))) break;
      tc_fence_after();
      const int64_t k0 = static_cast<int64_t>(ti.t) * 128;
      int nvis = static_cast<int>(min64(128, p.L - k0));
      if (CAUSAL) nvis = causal_visible(ti.blk, k0, gq, p.L, p.P);
      // Keys [0, nvis) of the tile are visible; when every row of the warp
      // sees all of this half, no column needs a mask.
      const bool full = __all_sync(0xffffffffu, nvis >= 64 * h + 64);
      // Four 16-column chunks, software-pipelined: chunk c + 1's TMEM loads
      // are in flight while chunk c is computed (two chunks of S and dP live).
      float sv[2][16], pv[2][16];
      tmem_ld16(tS, sv[0]);
      tmem_ld16(tP, pv[0]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int b = c & 1;
        if (c < 3) {
          tmem_ld16(tS + (c + 1) * 16, sv[b ^ 1]);
          tmem_ld16(tP + (c + 1) * 16, pv[b ^ 1]);
        }
        uint32_t pk[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const float2 a = ffma2(make_float2(sv[b][2 * x], sv[b][2 * x + 1]), sl2v, nlse2);
          float2 e = make_float2(ex2(a.x), ex2(a.y));
          if (!full) {
            const int cc = 64 * h + c * 16 + 2 * x;
            e.x = cc < nvis ? e.x : 0.f;
            e.y = cc + 1 < nvis ? e.y : 0.f;
          }
          const float2 ds = fmul2(e, fadd2(make_float2(pv[b][2 * x], pv[b][2 * x + 1]), nD2));
          pk[x] = pack_bf16x2(ds.x, ds.y);
        }
        // dS of columns [16c, 16c + 16) over S columns [8c, 8c + 8): already read.
        tmem_st8(tS + c * 8, pk);
        if (c < 3) tmem_wait_ld();
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bb.b(kBC + h));
    }
    __syncwarp();
    const bool aborted = __shfl_sync(0xffffffffu, *abort_flag, 0) != 0;
    if (!aborted) {
      const bool have = j > 0 && __all_sync(0xffffffffu, mbar_wait(bb.b(kBO), 0, wd, abort_flag));
      tc_fence_after();
      // Warpgroup h writes columns [h D/2, (h+1) D/2) of its dQ rows.
      const uint32_t tQ = tmem + lane_bits + kColAcc0 + (D / 2) * h;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        float o[32];
        if (have) {
          tmem_ld32(tQ + c * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0.f;
        }
        if (valid) store_row_bf16(p.dq + grow * D + (D / 2) * h + c * 32, o, p.scale);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- dK/dV ----
template <int D, bool CAUSAL, bool REM>
__device__ __forceinline__ void bwd_dkv_body(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                             const CUtensorMap &tm_v, const CUtensorMap &tm_do,
                                             const CUtensorMap &tm_kr, const CUtensorMap &tm_vr,
                                             const BwdParams &p, int unit) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const BBars bb = init_bars<D>(sbase);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffBar + kBAbort);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffBar + kBTmemSlot);
  float *sm_ld = reinterpret_cast<float *>(smem + C::kOffLD);  // [half][buffer](-LSE 64 | -D 64)
  const Watchdog wd{p.wd.status, p.wd.limit_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // With REM, units past BH * P * (n_t - 1) stack every block's last keys.
  int u = unit;
  const int nt_full = REM ? p.n_t - 1 : p.n_t;
  const bool stacked = REM && u >= p.BH * p.P * nt_full;
  int kt, b, bh;
  if (stacked) {
    kt = p.n_t - 1;
    b = 0;
    bh = u - p.BH * p.P * nt_full;
  } else {
    kt = u % nt_full;
    u /= nt_full;
    b = u % p.P;
    bh = u / p.P;
  }
  const int64_t C2 = p.L >> 1;
  const int64_t n_rows = static_cast<int64_t>(p.BH) * p.S;  // rows of every [BH, S] tensor
  const int64_t k0 = static_cast<int64_t>(kt) * 128;
  const int64_t nk = stacked ? static_cast<int64_t>(p.P) * p.rem : min64(128, p.L - k0);
  const int64_t k_row0 = static_cast<int64_t>(bh) * p.S + static_cast<int64_t>(b) * p.L + k0;
  const int64_t gk_min = CAUSAL ? zz_pos(b, k0, C2, p.P) : 0;
  auto make_iter = [&]() {
    BIter<CAUSAL> it{0, 0, b, p.P, p.n_t, +1, C2, gk_min, p.L};
    it.settle();
    return it;
  };

  if (threadIdx.x == 0) {
    mbar_init(bb.b(kBA), 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(bb.b(kBH + h), 1);
      mbar_init(bb.b(kBC + h), 128);
      mbar_init(bb.b(kBLd + 2 * h), 128);
      mbar_init(bb.b(kBLd + 2 * h + 1), 128);
    }
    mbar_init(bb.b(kBO), 1);
    mbar_init(bb.b(kBDrain), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bb.kv_full0 + 8 * s, 1);
      mbar_init(bb.kv_empty0 + 8 * s, 1);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      if (stacked) {
        mbar_arrive_expect_tx(bb.b(kBA), static_cast<uint32_t>(2 * p.P * p.rem * 128 * C::kChunks));
        for (int rr = 0; rr < p.P; ++rr) {
          int32_t y = static_cast<int32_t>(k_row0 + static_cast<int64_t>(rr) * p.L);
          if (!RA_IN_BOUNDS(y >= 0 && static_cast<int64_t>(y) + p.rem <= n_rows, wd.status)) y = 0;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c) {
            tma_load_2d(sbase + C::kOffA + c * C::kChunkBytes + rr * p.rem * 128, &tm_kr, c * 64, y,
                        bb.b(kBA));
            tma_load_2d(sbase + C::kOffB + c * C::kChunkBytes + rr * p.rem * 128, &tm_vr, c * 64, y,
                        bb.b(kBA));
          }
        }
      } else {
        int32_t y = static_cast<int32_t>(k_row0);
        if (!RA_IN_BOUNDS(k_row0 >= 0 && k_row0 < n_rows, wd.status)) y = 0;
        mbar_arrive_expect_tx(bb.b(kBA), 2 * C::kTile);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_2d(sbase + C::kOffA + c * C::kChunkBytes, &tm_k, c * 64, y, bb.b(kBA));
          tma_load_2d(sbase + C::kOffB + c * C::kChunkBytes, &tm_v, c * 64, y, bb.b(kBA));
        }
      }
      int it = 0;
      bool ok = true;
      for (auto ti = make_iter(); ok && ti.valid(); ++ti.t, ti.settle()) {
        int32_t qy = static_cast<int32_t>(static_cast<int64_t>(bh) * p.S +
                                          static_cast<int64_t>(ti.blk) * p.L +
                                          static_cast<int64_t>(ti.t) * 128);
        if (!RA_IN_BOUNDS(qy >= 0 && qy < n_rows, wd.status)) qy = 0;
        for (int which = 0; which < 2 && ok; ++which, ++it) {
          const int slot = it % C::kSlots;
          if (!(ok = mbar_wait(bb.kv_empty0 + 8 * slot, ((it / C::kSlots) & 1) ^ 1, wd, abort_flag)))
            break;
          mbar_arrive_expect_tx(bb.kv_full0 + 8 * slot, C::kTile);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_2d(sbase + C::kOffKV + slot * C::kTile + c * C::kChunkBytes,
                        which ? &tm_do : &tm_q, c * 64, qy, bb.kv_full0 + 8 * slot);
        }
      }
      mbar_wait_drain(bb.b(kBA), 0, p.wd.limit_ns);
      for (int i = max(0, it - C::kSlots); i < it; ++i)
        mbar_wait_drain(bb.kv_full0 + 8 * (i % C::kSlots), (i / C::kSlots) & 1, p.wd.limit_ns);
    }
  } else if (warp == 1) {
    constexpr uint32_t idesc_h = idesc_bf16_f32(128, 64, 0, 0);
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);
    constexpr uint32_t kSlotDesc = C::kTile >> 4;
    const uint64_t dKd = smem_desc_sw128(sbase + C::kOffA, 16, 1024);
    const uint64_t dVd = smem_desc_sw128(sbase + C::kOffB, 16, 1024);
    const uint64_t dRing = smem_desc_sw128(sbase + C::kOffKV, 16, 1024);
    const uint64_t dRingMn = smem_desc_sw128(sbase + C::kOffKV, C::kChunkBytes, 1024);
    // S^T_h = K Q_h^T and dP^T_h = V dO_h^T (rows = keys, 64 query columns)
    // for half h of the Q / dO tiles in slots qs, gs.
    auto issue_s = [&](int h, int qs, int gs) {
      issue_qk<D>(tmem + kColS + 64 * h, dKd,
                  dRing + static_cast<uint64_t>(qs * kSlotDesc) + h * kHalfRows, idesc_h);
      issue_qk<D>(tmem + kColP + 64 * h, dVd,
                  dRing + static_cast<uint64_t>(gs * kSlotDesc) + h * kHalfRows, idesc_h);
      mma_commit_e(bb.b(kBH + h));
    };
    bool issued = false, ok = true;
    auto ti = make_iter();
    if (ti.valid() && mbar_wait(bb.b(kBA), 0, wd, abort_flag)) {
      tc_fence_after();
      int it = 0;  // Q_j in slot it, dO_j in it + 1
      ok = mbar_wait(bb.kv_full0 + 8 * (it % C::kSlots), (it / C::kSlots) & 1, wd, abort_flag) &&
           mbar_wait(bb.kv_full0 + 8 * ((it + 1) % C::kSlots), ((it + 1) / C::kSlots) & 1, wd,
                     abort_flag);
      if (ok) {
        tc_fence_after();
        issue_s(0, it % C::kSlots, (it + 1) % C::kSlots);
        issue_s(1, it % C::kSlots, (it + 1) % C::kSlots);
        issued = true;
      }
      for (int j = 0; ok; ++j) {
        const int qs = it % C::kSlots, gs = (it + 1) % C::kSlots;
        const int nx = it + 2;
        ++ti.t;
        ti.settle();
        const bool more = ti.valid();
        for (int h = 0; h < 2 && ok; ++h) {
          if (!(ok = mbar_wait(bb.b(kBC + h), j & 1, wd, abort_flag))) break;
          tc_fence_after();
          // dV += P^T_h dO_h and dK += dS^T_h Q_h (dO, Q MN-major).
          issue_acc_k64(tmem + kColAcc0, tmem + kColS + 64 * h,
                        dRingMn + static_cast<uint64_t>(gs * kSlotDesc) + h * kHalfRows, idesc_o,
                        j > 0 || h > 0);
          issue_acc_k64(tmem + kColAcc1, tmem + kColP + 64 * h,
                        dRingMn + static_cast<uint64_t>(qs * kSlotDesc) + h * kHalfRows, idesc_o,
                        j > 0 || h > 0);
          if (h == 1) {
            mma_commit_e(bb.kv_empty0 + 8 * qs);  // Q_j and dO_j: last uses issued
            mma_commit_e(bb.kv_empty0 + 8 * gs);
          }
          if (more) {
            if (h == 0) {
              ok = mbar_wait(bb.kv_full0 + 8 * (nx % C::kSlots), (nx / C::kSlots) & 1, wd,
                             abort_flag) &&
                   mbar_wait(bb.kv_full0 + 8 * ((nx + 1) % C::kSlots), ((nx + 1) / C::kSlots) & 1,
                             wd, abort_flag);
              if (!ok) break;
              tc_fence_after();
            }
            issue_s(h, nx % C::kSlots, (nx + 1) % C::kSlots);
          }
        }
        if (!ok || !more) break;
        it = nx;
      }
      if (ok) mma_commit_e(bb.b(kBO));
    }
    if (issued) {
      mma_commit_e(bb.b(kBDrain));
      mbar_wait_drain(bb.b(kBDrain), 0, p.wd.limit_ns);
    }
  } else if (warp >= 4) {
    const int h = (warp - 4) >> 2;  // half of the query tile this warpgroup handles
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key row of the tile; thread index in the warpgroup
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_bits + kColS + 64 * h, tP = tmem + lane_bits + kColP + 64 * h;
    const bool kvalid = row < nk;
    const int64_t gk = CAUSAL ? zz_pos(b, min64(k0 + row, p.L - 1), C2, p.P) : 0;
    const float sl2 = p.scale_log2;
    // -LSE (log2 units) and -D of this half's 64 queries are staged in SMEM,
    // double-buffered: thread t < 64 holds query t's, thread 64 + t its -D,
    // read from global memory one tile ahead.
    const int qi = row & 63;
    auto staged = [&](const BIter<CAUSAL> &t) -> float {
      const int64_t tq0 = static_cast<int64_t>(t.t) * 128;
      if (64 * h + qi >= min64(128, p.L - tq0)) return 0.f;
      const int64_t qrow = static_cast<int64_t>(bh) * p.S + static_cast<int64_t>(t.blk) * p.L +
                           tq0 + 64 * h + qi;
      if (!RA_IN_BOUNDS(qrow >= 0 && qrow < n_rows, wd.status)) return 0.f;
      return row < 64 ? -(p.lse[qrow] * kLog2eB) : -p.Dv[qrow];
    };
    int j = 0;
    auto ti = make_iter();
    float val = ti.valid() ? staged(ti) : 0.f;
    for (; ti.valid(); ++j) {
      BIter<CAUSAL> tn = ti;
      ++tn.t;
      tn.settle();
      float *ld = sm_ld + (2 * h + (j & 1)) * 128;
      const int64_t q0 = static_cast<int64_t>(ti.t) * 128;
      const int64_t nq = min64(128, p.L - q0);
      // Buffer (h, j&1) was last read two tiles ago; no thread of this
      // warpgroup can still be there, since half h of this tile's S^T needs
      // every one of its arrivals for the previous tile.
      ld[row < 64 ? qi : 64 + qi] = val;
      val = tn.valid() ? staged(tn) : 0.f;         // next tile's value, in flight
      mbar_arrive(bb.b(kBLd + 2 * h + (j & 1)));  // release: the value above
      if (!__all_sync(0xffffffffu,
                      mbar_wait(bb.b(kBLd + 2 * h + (j & 1)), (j >> 1) & 1, wd, abort_flag)))
        break;
      // Visible queries of this key: positions >= its own (a suffix of the tile).
      int first = 0, last = static_cast<int>(nq);
      if (!kvalid) first = last;
      else if (CAUSAL) first = causal_visible(ti.blk, q0, gk - 1, p.L, p.P);
      if (!__all_sync(0xffffffffu, mbar_wait(bb.b(kBH + h), j & 1, wd, abort_flag))) break;
      tc_fence_after();
      // When every key row of the warp sees every query of this half, no
      // column needs a mask.
      const bool full = __all_sync(0xffffffffu, first <= 64 * h && last >= 64 * h + 64);
      const float2 sl2v = make_float2(sl2, sl2);
      // Four 16-column chunks, software-pipelined: chunk c + 1's TMEM loads
      // are in flight while chunk c is computed (two chunks of S^T and dP^T
      // live).
      float sv[2][16], pv[2][16];
      tmem_ld16(tS, sv[0]);
      tmem_ld16(tP, pv[0]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int b = c & 1;
        if (c < 3) {
          tmem_ld16(tS + (c + 1) * 16, sv[b ^ 1]);
          tmem_ld16(tP + (c + 1) * 16, pv[b ^ 1]);
        }
        uint32_t pkp[8], pks[8];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const float4 nl = *reinterpret_cast<const float4 *>(ld + c * 16 + 4 * y);
          const float4 nd = *reinterpret_cast<const float4 *>(ld + 64 + c * 16 + 4 * y);
#pragma unroll
          for (int z = 0; z < 2; ++z) {
            const int x = 2 * y + z;
            const float2 a = ffma2(make_float2(sv[b][2 * x], sv[b][2 * x + 1]), sl2v,
                                   z ? make_float2(nl.z, nl.w) : make_float2(nl.x, nl.y));
            float2 e = make_float2(ex2(a.x), ex2(a.y));
            if (!full) {
              const int cc = 64 * h + c * 16 + 2 * x;  // column within the tile
              e.x = cc >= first && cc < last ? e.x : 0.f;
              e.y = cc + 1 >= first && cc + 1 < last ? e.y : 0.f;
            }
            const float2 ds = fmul2(e, fadd2(make_float2(pv[b][2 * x], pv[b][2 * x + 1]),
                                             z ? make_float2(nd.z, nd.w) : make_float2(nd.x, nd.y)));
            pkp[x] = pack_bf16x2(e.x, e.y);
            pks[x] = pack_bf16x2(ds.x, ds.y);
          }
        }
        // P^T and dS^T of columns [16c, 16c + 16) over columns [8c, 8c + 8)
        // of S^T and dP^T: already read.
        tmem_st8(tS + c * 8, pkp);
        tmem_st8(tP + c * 8, pks);
        if (c < 3) tmem_wait_ld();
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bb.b(kBC + h));
      ti = tn;
    }
    __syncwarp();
    const bool aborted = __shfl_sync(0xffffffffu, *abort_flag, 0) != 0;
    if (!aborted) {
      const bool have = j > 0 && __all_sync(0xffffffffu, mbar_wait(bb.b(kBO), 0, wd, abort_flag));
      tc_fence_after();
      // Warpgroup 0 writes the dV row, warpgroup 1 the dK row.
      const int64_t grow =
          stacked ? k_row0 + static_cast<int64_t>(row / p.rem) * p.L + row % p.rem : k_row0 + row;
      const bool store = kvalid && RA_IN_BOUNDS(grow >= 0 && grow < n_rows, wd.status);
      const uint32_t tA = tmem + lane_bits + (h == 0 ? kColAcc0 : kColAcc1);
      __nv_bfloat16 *dst = (h == 0 ? p.dv : p.dk) + grow * D;
      const float mul = h == 0 ? 1.f : p.scale;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        if (have) {
          tmem_ld32(tA + c * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0.f;
        }
        if (store) store_row_bf16(dst + c * 32, o, mul);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host ----
// One launch for both gradients: the first n_dkv CTAs run dK/dV units (the
// longer ones), the rest dQ units, so the dQ units fill the dK/dV tail.
template <int D, bool CAUSAL, bool REM>
__global__ void __launch_bounds__(kThreadsB, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_qr, const __grid_constant__ CUtensorMap tm_kr,
               const __grid_constant__ CUtensorMap tm_vr, const __grid_constant__ CUtensorMap tm_dor,
               const BwdParams p, int n_dkv) {
  static_assert(!(REM && CAUSAL), "stacked last tiles: non-causal only");
  const int b = static_cast<int>(blockIdx.x);
  if (b < n_dkv)
    bwd_dkv_body<D, CAUSAL, REM>(tm_q, tm_k, tm_v, tm_do, tm_kr, tm_vr, p, b);
  else
    bwd_dq_body<D, CAUSAL, REM>(tm_q, tm_k, tm_v, tm_do, tm_qr, tm_dor, p, b - n_dkv);
}

typedef CUresult (*EncodeTiledFnB)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnB encode_fn_b() {
  static EncodeTiledFnB fn = [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<EncodeTiledFnB>(ptr);
  }();
  return fn;
}

cudaError_t row_map_b(CUtensorMap *map, const void *base, int64_t rows, int d,
                      int box_rows = 128) {
  EncodeTiledFnB fn = encode_fn_b();
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

template <int D, bool CAUSAL, bool REM>
cudaError_t launch_bwd_variant(const CUtensorMap *maps, const BwdParams &p, int64_t units,
                               cudaStream_t stream) {
  using C = BCfg<D>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    if ((e = cudaFuncSetAttribute(bwd_kernel<D, CAUSAL, REM>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes)) !=
        cudaSuccess)
      return e;
    configured[dev] = true;
  }
  const unsigned grid = static_cast<unsigned>(2 * units);
  bwd_kernel<D, CAUSAL, REM><<<grid, kThreadsB, C::kSmemBytes, stream>>>(
      maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], p,
      static_cast<int>(units));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(const void *q, const void *k, const void *v, const void *out,
                            const void *dout, int d, const BwdParams &params,
                            cudaStream_t stream) {
  BwdParams p = params;
  const int64_t rows = static_cast<int64_t>(p.BH) * p.S;
  if (rows == 0) return cudaSuccess;
  // Non-causal chunks ending in a short tile: every chunk's last rows share
  // one tile per head (and kind of unit) when they fit.
  const int64_t rem = p.L - static_cast<int64_t>(p.n_t - 1) * 128;
  p.rem = (!p.causal && p.n_t > 1 && p.P > 1 && rem < 128 && rem % 8 == 0 && p.P * rem <= 128)
              ? static_cast<int>(rem)
              : 0;
  const int64_t units = p.rem ? static_cast<int64_t>(p.BH) * (p.P * (p.n_t - 1) + 1)
                              : static_cast<int64_t>(p.BH) * p.P * p.n_t;
  if (2 * units > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const int64_t prep_blocks = (rows + 7) / 8;
  bwd_prep_kernel<<<static_cast<unsigned>(prep_blocks), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16 *>(out), static_cast<const __nv_bfloat16 *>(dout), p.Dv, rows,
      d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // q, k, v, dO with 128-row boxes, then with rem-row boxes (stacked tiles).
  CUtensorMap maps[8];
  const void *src[4] = {q, k, v, dout};
  for (int i = 0; i < 4; ++i) {
    if ((e = row_map_b(&maps[i], src[i], rows, d)) != cudaSuccess) return e;
    if (p.rem) {
      if ((e = row_map_b(&maps[4 + i], src[i], rows, d, p.rem)) != cudaSuccess) return e;
    } else {
      maps[4 + i] = maps[i];
    }
  }
  // Kernel parameter order: q, k, v, dO, then the stacked maps q, k, v, dO.
  // The causal mask and tile skipping are compiled only into the causal
  // instantiations, the stacked last tiles only into the REM ones.
  if (d == 128) {
    if (p.causal) return launch_bwd_variant<128, true, false>(maps, p, units, stream);
    return p.rem ? launch_bwd_variant<128, false, true>(maps, p, units, stream)
                 : launch_bwd_variant<128, false, false>(maps, p, units, stream);
  }
  if (p.causal) return launch_bwd_variant<64, true, false>(maps, p, units, stream);
  return p.rem ? launch_bwd_variant<64, false, true>(maps, p, units, stream)
               : launch_bwd_variant<64, false, false>(maps, p, units, stream);
}

}  // namespace ra
