// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ra {

struct WatchdogParams {
  int *status;       // device status word
  int64_t limit_ns;  // bound on every barrier wait
};

// One launch of the blockwise ring-attention kernel.
//
// A "problem" is one (bh, g) pair: G independent attention problems per
// (batch, head), e.g. the frames of spatial attention (G = 1 for the ring).
// Each problem's keys form P ring blocks of L rows; a query chunk of rank r
// (L rows) visits blocks (r - s) mod P for its steps s.  Work unit =
// (bh, g, rank, step group, pair of 128-row query tiles); units are numbered
// with the query-tile pair fastest, then step group, rank, g, bh.
struct AttnParams {
  int BH, G, n_ranks, n_stepgroups, n_pairs;
  int64_t q_rows_bh, q_rows_g;    // Q / out / lse row strides (rows)
  int64_t q_rank_stride;          // rows between consecutive ranks' query chunks (0: L)
  int64_t kv_rows_bh, kv_rows_g;  // K / V row strides (rows)
  int64_t L;                      // rows per ring block (and per rank chunk)
  int P, rank_begin, step_begin, steps_per_group;
  int causal;                     // zigzag positions + key <= query mask
  float scale_log2;               // log2(e) / sqrt(d)
  void *out;                      // bf16 or fp32
  float *lse;
  int64_t out_part_stride;        // elements between step groups' outputs
  int64_t lse_part_stride;
  // Packed short problems (temporal factored attention): when pack > 0 the
  // Q/K/V tensors are frame-major video tokens [BH][pT frames][pN positions]
  // [d] read in place, each position a problem of pT rows; one tile holds
  // the rank's chunk (Lf frames) of `pack` consecutive positions:
  // L = pack * Lf, G = ceil(pN / pack), and a query only sees keys of its
  // own position.  Outputs are written position-major [BH][pN][pT], or,
  // with pack_frame_major, frame-major [BH][pT][pN] like the inputs.
  int pack, Lf, pT;
  int pLrow;  // tile rows per problem, >= Lf (16 or 32 for the warp-packed softmax)
  int pack_frame_major;
  int64_t pN;
  // Packed mode only: when pack_ranks > 0 a unit holds the chunks of two
  // consecutive ranks (2 * unit index and the next, below pack_ranks) as its
  // two query tiles; n_ranks then counts rank pairs.  Both tiles meet the
  // same key/value tiles, in the first rank's ring order.
  int pack_ranks;
  // Per-rank K/V buffers (overlapped ring): when kv_own != 0, rank r's
  // current block for head bh is rows [r * kv_rank_stride + bh * kv_rows_bh,
  // + L) of the K/V tensors, whatever block of the ring it holds.
  int kv_own;
  int64_t kv_rank_stride;
  // Per-step partials indexed by the K/V block that produced them
  // ((rank - step) mod P) instead of by step (reduce-scatter form).
  int part_by_block;
  // Row tiles, non-causal, every rank's chunk ending in a short single tile:
  // when rem_pack > 0 one unit per (head, problem, step group) holds the
  // last rem_pack rows of each of the n_ranks chunks in one query tile
  // (rank r at tile rows [r * rem_pack, (r + 1) * rem_pack)), meeting the
  // key tiles in the first rank's ring order.
  int rem_pack;
  // Overlapped ring, exchange inside the launch: when x_on != 0 the CTAs'
  // otherwise idle warps 2 and 3 copy, for both K and V, every rank r's
  // next block: x_ranks x x_bh rows of x_row_bytes from
  // src + ((r - 1) mod x_ranks) * x_src_rank + h * x_src_head to
  // dst + r * x_dst_rank + h * x_dst_head.  x_src_span / x_dst_span bound
  // the byte offsets (bounds-checked build).
  int x_on, x_ranks, x_bh;
  const uint8_t *xk_src, *xv_src;
  uint8_t *xk_dst, *xv_dst;
  int64_t x_src_rank, x_src_head, x_dst_rank, x_dst_head, x_row_bytes, x_src_span, x_dst_span;
  WatchdogParams wd;
  // Extents for the RA_CHECKS build's bounds checks (set by launch_ring_attn):
  // rows of the Q and K/V row matrices, output rows per part, output parts.
  int64_t chk_q_rows, chk_kv_rows, chk_out_rows;
  int chk_parts;
};

// Backward pass (attn_bwd.cu).  All tensors [BH, S, d] in sharded order.
struct BwdParams {
  int BH, P, n_t;  // n_t = ceil(L / 128) tiles per rank chunk / ring block
  int64_t S, L;
  int causal;
  float scale_log2, scale;
  const float *lse;  // forward LSE [BH, S]
  float *Dv;         // D_i = dO_i . O_i [BH, S] (scratch, written by the prep kernel)
  __nv_bfloat16 *dq, *dk, *dv;
  // Non-causal chunks whose last tile holds rem < 128 rows (rem % 8 == 0,
  // P * rem <= 128): one unit per head of each kind stacks every chunk's
  // last rows in one tile (chunk r at tile rows [r * rem, (r + 1) * rem)).
  // Set by launch_attn_bwd; 0 = off.
  int rem;
  WatchdogParams wd;
};

cudaError_t launch_attn_bwd(const void *q, const void *k, const void *v, const void *out,
                            const void *dout, int d, const BwdParams &p, cudaStream_t stream);

// Launches the attention kernel.  q/k/v: bf16 row matrices [rows, d].
cudaError_t launch_ring_attn(const void *q, int64_t q_total_rows, const void *k, const void *v,
                             int64_t kv_total_rows, int d, bool out_f32, const AttnParams &p,
                             cudaStream_t stream);

// Row permutation kernels (shard.cu).  mode: 0 shard, 1 unshard (layout, P),
// 2 frame transpose [T,N] -> [N,T], 3 back.  row_bytes: 128, 256 (bf16 rows) or 4 (fp32).
// status: the device status word (bounds checks of the RA_CHECKS build).
cudaError_t launch_row_permute(const void *x, void *y, int64_t BH, int64_t S, int row_bytes,
                               int mode, int64_t a, int64_t b, int layout, int *status,
                               cudaStream_t stream);

// lse_merge kernel (merge.cu).
cudaError_t launch_lse_merge(const float *o_parts, const float *lse_parts, int n, int64_t rows,
                             int d, void *out, float *lse_out, int *status, cudaStream_t stream);

// Watchdog self-test kernel (attn_fwd.cu).
cudaError_t launch_watchdog_selftest(const WatchdogParams &wd, cudaStream_t stream);

// Bounds-check self-test kernel (attn_fwd.cu): checks one index against a
// bound it exceeds, touching no memory through it.
cudaError_t launch_checks_selftest(int *status, cudaStream_t stream);

// Scratch bytes factored_attn uses for these sizes and this P (api.cu): 0
// when every rank chunk of T / P frames fits one tile, otherwise
// factored_attn_workspace(B, H, T, N, d).
size_t factored_scratch_bytes(int B, int H, int T, int N, int d, int P);

// Records `e` as the error ra_last_cuda_error reports; returns RA_ERR_CUDA (api.cu).
int record_cuda_error(cudaError_t e);

}  // namespace ra
