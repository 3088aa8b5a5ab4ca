// Row permutations of [BH, S, row] tensors: sequence sharding for context
// parallelism and the frame transpose of factored video attention.
//
// Sharding ("day 83" blog, "Context parallelism: splitting the sequence";
// k8ai "How context parallel works", balanced causal split read as zigzag):
// sharded row j = r*L + i of rank r holds global token
//   contiguous: r*L + i
//   zigzag:     r*C + i (i < C), (2P-1-r)*C + (i - C) (i >= C),  C = S/(2P).
// Frame transpose ("day 83" blog, "The spatial-temporal twist"): token t*N + n
// of [T, N] order is row n*T + t of [N, T] order.
//
// Each thread moves 16-byte pieces (or 4-byte elements for fp32 rows) with
// plain vector loads/stores; consecutive threads take consecutive pieces of a
// row, so both sides are fully coalesced 128-byte lines.
#include <stdint.h>

#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {
namespace {

struct PermuteArgs {
  int64_t S;
  int mode;       // 0 shard, 1 unshard, 2 [T,N]->[N,T], 3 [N,T]->[T,N],
                  // 4 Ulysses sequence-split -> head-split, 5 back,
                  // 6 per-rank [P][B][H][L] -> rank-major [B][H][P*L], 7 back
  int64_t a, b;   // modes 0/1: a = P; modes 2/3: a = T, b = N; modes 4-7: a = P, b = H
  int layout;     // modes 0/1: 0 contiguous, 1 zigzag; modes 4-7: B
};

// Ulysses all-to-all (k8ai "An alternative: all-to-all on heads"), over the
// whole tensor.  Sequence-split per-rank layout [P][B][H][L][d]: rank r's
// chunk of every head.  Head-split per-rank layout [P][B][H/P][S][d]: rank
// r's heads r*H/P .. (r+1)*H/P - 1, every token (contiguous split: token
// r*L + i is row i of rank r).  Modes 6/7 gather per-rank buffers into the
// rank-major order [B][H][P*L] and scatter back.  Returns the source row of
// output row o.  Row counts are below 2^31, so 32-bit arithmetic is exact.
__device__ __forceinline__ uint32_t global_source_row(const PermuteArgs &p, uint32_t o) {
  const uint32_t P = static_cast<uint32_t>(p.a), H = static_cast<uint32_t>(p.b);
  const uint32_t B = static_cast<uint32_t>(p.layout), S = static_cast<uint32_t>(p.S);
  const uint32_t L = S / P, Hp = H / P;
  if (p.mode == 6) {  // rank-major [B][H][S] <- per-rank [P][B][H][L] (all-gather)
    const uint32_t bh = o / S, t = o - bh * S;
    const uint32_t r = t / L, i = t - r * L;
    return (r * B * H + bh) * L + i;
  }
  if (p.mode == 7) {  // per-rank <- rank-major (scatter)
    const uint32_t r = o / (B * H * L), r1 = o - r * (B * H * L);
    const uint32_t bh = r1 / L, i = r1 - bh * L;
    return bh * S + r * L + i;
  }
  if (p.mode == 4) {  // head-split <- sequence-split
    const uint32_t R = o / (B * Hp * S), r1 = o - R * (B * Hp * S);
    const uint32_t b = r1 / (Hp * S), r2 = r1 - b * (Hp * S);
    const uint32_t hh = r2 / S, t = r2 - hh * S;
    const uint32_t r = t / L, i = t - r * L;
    return ((r * B + b) * H + R * Hp + hh) * L + i;
  }
  // sequence-split <- head-split
  const uint32_t r = o / (B * H * L), r1 = o - r * (B * H * L);
  const uint32_t b = r1 / (H * L), r2 = r1 - b * (H * L);
  const uint32_t h = r2 / L, i = r2 - h * L;
  const uint32_t R = h / Hp;
  return ((R * B + b) * Hp + (h - R * Hp)) * S + r * L + i;
}

// Source row (within one (b,h) slice) of output row o; 32-bit arithmetic
// (rows are below 2^31).
__device__ __forceinline__ uint32_t source_row(const PermuteArgs &p, uint32_t o) {
  const uint32_t S = static_cast<uint32_t>(p.S);
  switch (p.mode) {
    case 0: {  // y[j] = x[s2g(j)]
      if (p.layout == 0) return o;
      const uint32_t P = static_cast<uint32_t>(p.a), L = S / P, C = L >> 1;
      const uint32_t r = o / L, i = o - r * L;
      return i < C ? r * C + i : (2 * P - 1 - r) * C + (i - C);
    }
    case 1: {  // y[g] = x[g2s(g)]
      if (p.layout == 0) return o;
      const uint32_t P = static_cast<uint32_t>(p.a), L = S / P, C = L >> 1;
      const uint32_t chunk = o / C, off = o - chunk * C;
      return chunk < P ? chunk * L + off : (2 * P - 1 - chunk) * L + C + off;
    }
    case 2: {  // output [N, T]: row n*T + t <- input row t*N + n
      const uint32_t T = static_cast<uint32_t>(p.a), N = static_cast<uint32_t>(p.b);
      const uint32_t n = o / T, t = o - n * T;
      return t * N + n;
    }
    default: {  // output [T, N]: row t*N + n <- input row n*T + t
      const uint32_t T = static_cast<uint32_t>(p.a), N = static_cast<uint32_t>(p.b);
      const uint32_t t = o / N, n = o - t * N;
      return n * T + t;
    }
  }
}

template <typename Vec, int PIECES>
__global__ void __launch_bounds__(256) row_permute_kernel(const Vec *__restrict__ x,
                                                          Vec *__restrict__ y, int64_t total_rows,
                                                          PermuteArgs p, int *status) {
  constexpr int kUnroll = 4;
  const int64_t total = total_rows * PIECES;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; idx < total; idx += kUnroll * stride) {
    Vec v[kUnroll];
    int64_t dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t e = idx + u * stride;
      dst[u] = -1;
      if (e < total) {
        const int64_t row = e / PIECES;
        const int piece = static_cast<int>(e - row * PIECES);
        int64_t src;
        if (p.mode >= 4) {
          src = global_source_row(p, static_cast<uint32_t>(row));
        } else {
          const uint32_t S = static_cast<uint32_t>(p.S), r32 = static_cast<uint32_t>(row);
          const uint32_t bh = r32 / S, o = r32 - bh * S;
          src = static_cast<int64_t>(bh * S + source_row(p, o));
        }
        if (!RA_IN_BOUNDS(src >= 0 && src < total_rows, status)) continue;
        v[u] = x[src * PIECES + piece];
        dst[u] = e;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (dst[u] >= 0) y[dst[u]] = v[u];
  }
}

// One block per 256 x kUnroll pieces: every thread moves its pieces once
// and exits (a grid capped at the resident blocks, striding over the rest,
// reached only 80-85% of the copy bandwidth against 97-98% this way).
int grid_for(int64_t work, int threads) {
  const int64_t want = (work + threads - 1) / threads;
  const int64_t cap = 0x7fffffff;
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_row_permute(const void *x, void *y, int64_t BH, int64_t S, int row_bytes,
                               int mode, int64_t a, int64_t b, int layout, int *status,
                               cudaStream_t stream) {
  const int64_t rows = BH * S;
  if (rows == 0) return cudaSuccess;
  if (status == nullptr) return cudaErrorInvalidValue;
  PermuteArgs p{S, mode, a, b, layout};
  if (row_bytes % 16 == 0) {
    const int pieces = row_bytes / 16;
    const int grid = grid_for(rows * pieces / 4, 256);
    if (pieces == 16)
      row_permute_kernel<uint4, 16><<<grid, 256, 0, stream>>>(
          static_cast<const uint4 *>(x), static_cast<uint4 *>(y), rows, p, status);
    else if (pieces == 8)
      row_permute_kernel<uint4, 8><<<grid, 256, 0, stream>>>(
          static_cast<const uint4 *>(x), static_cast<uint4 *>(y), rows, p, status);
    else
      return cudaErrorInvalidValue;
  } else if (row_bytes == 4) {
    const int grid = grid_for(rows / 4, 256);
    row_permute_kernel<uint32_t, 1><<<grid, 256, 0, stream>>>(
        static_cast<const uint32_t *>(x), static_cast<uint32_t *>(y), rows, p, status);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ra
