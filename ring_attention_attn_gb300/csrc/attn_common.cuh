// Helpers shared by the forward and backward attention kernels: zigzag
// token positions, causal prefix counts and the tcgen05 MMA issue loops of a
// 128-row tile.  Internal to the library.
#pragma once

#include <stdint.h>

#include "ra_device.cuh"

namespace ra {
namespace {

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Global token position of local row i of rank `rank`'s chunk (zigzag: the
// chunk is global chunks rank and 2P-1-rank, each C = L/2 rows).
__device__ __forceinline__ int64_t zz_pos(int rank, int64_t i, int64_t C, int P) {
  return i < C ? static_cast<int64_t>(rank) * C + i
               : static_cast<int64_t>(2 * P - 1 - rank) * C + (i - C);
}

// Number of keys of tile [k0, k0+128) of block `src` that query position gq
// may see.  Global key positions increase with the local index, so the
// visible keys are a prefix of the tile.
__device__ __forceinline__ int causal_visible(int src, int64_t k0, int64_t gq, int64_t L, int P) {
  const int64_t C = L >> 1;
  const int64_t n = min64(128, L - k0);
  const int64_t endA = min64(k0 + n, C);
  const int64_t lenA = max64(0, endA - k0);
  const int64_t cntA = min64(lenA, max64(0, gq - (static_cast<int64_t>(src) * C + k0) + 1));
  const int64_t startB = max64(k0, C);
  const int64_t lenB = max64(0, k0 + n - startB);
  const int64_t gB0 = static_cast<int64_t>(2 * P - 1 - src) * C + (startB - C);
  const int64_t cntB = min64(lenB, max64(0, gq - gB0 + 1));
  return static_cast<int>(cntA + cntB);
}


// S_i = Q_i K^T over d: 16 columns of d per MMA; dq / dk are the tiles'
// base descriptors, the k-step offset is added to the address field.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t dq, uint64_t dk, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
    mma_ss_e(d_tmem, dq + off, dk + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O_i (+)= P_i V over 128 keys: P (bf16 pairs) from TMEM, 8 columns per
// 16 keys; V MN-major, 16 keys = 2048 bytes per MMA.
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t dv,
                                         uint32_t idesc, bool acc) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts_e(d_tmem, p_tmem + kk * 8, dv + static_cast<uint64_t>(kk * (2048 >> 4)), idesc,
             (acc || kk > 0) ? 1u : 0u);
}


}  // namespace
}  // namespace ra
