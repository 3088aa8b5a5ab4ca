/*
 * ringattn.h -- C ABI of the GB300 (sm_103a) ring-attention hot path.
 *
 * Ring attention for context parallelism: every one of P ranks keeps its
 * chunk of queries and visits the P key/value blocks in ring order, folding
 * each block's partial attention into a running result with the online
 * softmax ("day 83" blog, "Context parallelism: splitting the sequence";
 * k8ai "Sequence and Context Parallel", "How context parallel works").  Here
 * the P ranks are P sequence chunks of one tensor on one GPU: a ring step is a
 * change of key/value block, not a transfer.
 *
 * Conventions shared by every entry point
 *  - Element types: bf16 (raw 16-bit storage, passed as void*), fp32 (float*).
 *  - Layout [B, H, S, d], row-major, d innermost, contiguous.  d is 64 or 128.
 *  - "Sharded order": rows [r*L, (r+1)*L) of each (b, h) hold rank r's chunk,
 *    L = S / P, in the layout chosen by ra_cp_shard (contiguous, or zigzag
 *    when causal).  Attention inputs and outputs are in sharded order.
 *  - Softmax scale 1/sqrt(d); LSE = natural log of the row's sum of
 *    exp(score), scale included.
 *  - Every device pointer must be 16-byte aligned.  The caller owns all
 *    memory; the library allocates no device memory.
 *  - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *    default stream) and never synchronise, except ra_get_status.
 *  - Return value: RA_OK (0) or a negative RA_ERR_* code.  Argument errors are
 *    detected on the host before anything is launched.  A sizes product of
 *    zero (B*H == 0 or S == 0) is a successful no-op.
 */
#ifndef RINGATTN_H
#define RINGATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RA_OK 0
#define RA_ERR_ARG (-1)     /* null pointer, negative size, bad enum value        */
#define RA_ERR_SHAPE (-2)   /* S % P != 0, S % 2P != 0 for zigzag, d not 64/128   */
#define RA_ERR_ALIGN (-3)   /* a device pointer is not 16-byte aligned            */
#define RA_ERR_CUDA (-4)    /* a CUDA call or launch failed: see ra_last_cuda_error */
#define RA_ERR_TIMEOUT (-5) /* a kernel's bounded wait expired (device watchdog)   */
#define RA_ERR_WORKSPACE (-6) /* workspace missing or smaller than required        */
#define RA_ERR_BOUNDS (-7)  /* a device index fell outside its buffer (RA_CHECKS build) */

#define RA_LAYOUT_CONTIGUOUS 0
#define RA_LAYOUT_ZIGZAG 1

/* Global <-> sharded token index maps (host only, no CUDA).
 * Contiguous ("day 83" blog, "Context parallelism: splitting the sequence"):
 *   rank r holds tokens [r*L, (r+1)*L).
 * Zigzag, the balanced causal split (k8ai "How context parallel works"): the
 *   sequence is cut into 2P chunks of C = S/(2P); rank r holds chunk r then
 *   chunk 2P-1-r.  Sharded row j = r*L + i maps to global token
 *   g = r*C + i (i < C) or (2P-1-r)*C + (i - C) (i >= C).
 * s2g[j] = g and g2s[g] = j, both int64 arrays of S entries owned by the
 * caller (either may be NULL).  Errors: RA_ERR_ARG, RA_ERR_SHAPE. */
int ra_cp_shard_index(int64_t S, int P, int layout, int64_t *s2g, int64_t *g2s);

/* KV block that rank r holds at ring step s: (r - s) mod P (k8ai "Sequence
 * and Context Parallel", ring diagram: after the first exchange rank 0 holds
 * block 3 and rank 1 holds block 0 of four).  Host only.  Returns -1 on bad
 * arguments. */
int ra_ring_source(int P, int rank, int step);

/* Row permutation of a bf16 [BH, S, d] tensor between global and sharded
 * order under the map above: inverse = 0 writes y[j] = x[s2g[j]] (shard),
 * inverse = 1 writes y[g] = x[g2s[g]] (unshard).  x and y must not overlap.
 * Bit-exact copy; 128-bit coalesced loads and stores. */
int ra_cp_shard(const void *x, void *y, int64_t BH, int64_t S, int d, int P, int layout,
                int inverse, void *stream);

/* Frame transpose of a video tensor ("day 83" blog, "The spatial-temporal
 * twist": tokens t*N + n).  bf16 rows of d elements: inverse = 0 maps
 * [BH, T, N, d] -> [BH, N, T, d]; inverse = 1 maps back.  x, y must not
 * overlap. */
int ra_frame_transpose(const void *x, void *y, int64_t BH, int64_t T, int64_t N, int d,
                       int inverse, void *stream);

/* Ring attention forward for all P simulated ranks.
 * q, k, v: bf16 [B, H, S, d] in sharded order (contiguous layout when
 * causal = 0, zigzag when causal = 1).  out: bf16 [B, H, S, d], lse: fp32
 * [B, H, S], both in sharded order.  Rank r's queries visit KV blocks
 * (r - s) mod P for s = 0..P-1; scores are masked by global token position
 * (key <= query) when causal.  Requires S % P == 0 (S % 2P == 0 if causal).
 * The result is exact full attention over the whole sequence (ultralytics
 * glossary, "How Context Parallelism Works").  When
 * non-causal chunks end in a short tile (S/P mod 256 in (0, 128], a multiple
 * of 8, P times it at most 128), every rank's last rows are computed
 * together in rank 0's block order; only the rounding order differs. */
int ring_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                  int H, int64_t S, int d, int P, int causal, void *stream);

/* One rank's share of the ring, for a range of ring steps.
 * q_local: bf16 [B, H, L, d], rank `rank`'s queries (L = S/P); k, v: bf16
 * [B, H, S, d] in sharded order.  Steps step_begin <= s < step_end visit
 * blocks (rank - s) mod P.
 *  out_fp32 = 0: out_local bf16 [B, H, L, d] and lse_local fp32 [B, H, L]
 *                hold attention over the keys of those steps (normalised).
 *  out_fp32 = 1: one partial per step, n = step_end - step_begin:
 *                out_local fp32 [n, B, H, L, d] (normalised per step) and
 *                lse_local fp32 [n, B, H, L]; a row that sees no key in a step
 *                gets O = 0, LSE = -inf.  Merge them with lse_merge.
 * Errors: RA_ERR_ARG if the step range is empty or outside [0, P], or rank is
 * outside [0, P). */
int ring_attn_fwd_rank(const void *q_local, const void *k, const void *v, void *out_local,
                       float *lse_local, int B, int H, int64_t S, int d, int P, int rank,
                       int causal, int step_begin, int step_end, int out_fp32, void *stream);

/* Ring attention with the K/V exchange performed as real copies, overlapped
 * with the attention of the current step: while a rank works on the block it
 * holds, the next block is already travelling, so the transfer time hides
 * behind compute ("day 83" blog, "Context parallelism: splitting the
 * sequence"; k8ai "Sequence and Context Parallel", ring diagram).  Same inputs,
 * outputs and result as ring_attn_fwd.  Every simulated rank r owns a K/V
 * double buffer in `workspace`; at step s the compute stream attends rank r's
 * queries to the block in its current buffer (block (r - s) mod P) while
 * `comm_stream` copies each rank's current block into the next buffer of rank
 * r + 1 (2P device-to-device copies per step).  Each step writes fp32 partials
 * (workspace), merged at the end by the lse_merge kernel on `stream`.  Stacked
 * last rows (as in ring_attn_fwd) read rank 0's current block at every step,
 * so each rank's last rows still meet every block once.
 * comm_stream may equal stream (copies then serialise with compute).
 * comm_stream NULL: no copy calls and no events; each step's launch itself
 * copies the blocks the next step reads (the same 2P ring sends), with warps
 * that the attention leaves idle, and the stream orders the steps.  On one
 * GPU this is the form that overlaps: a device-to-device copy runs on the
 * SMs and cannot start beside a launch that holds all of them.
 * workspace: >= ring_attn_fwd_overlap_workspace(...) bytes, 256-byte aligned,
 * used by this call only.  Events (comm_stream not NULL) are created and
 * released internally. */
int ring_attn_fwd_overlap(const void *q, const void *k, const void *v, void *out, float *lse,
                          int B, int H, int64_t S, int d, int P, int causal, void *workspace,
                          size_t ws_bytes, void *stream, void *comm_stream);

/* Workspace bytes of ring_attn_fwd_overlap (0 on bad arguments). */
size_t ring_attn_fwd_overlap_workspace(int B, int H, int64_t S, int d, int P);

/* Backward pass of ring_attn_fwd (the ring's exchanges recur in the backward
 * pass of every attention layer: k8ai "Sequence and Context Parallel",
 * "Communication profile").  Gradients of the loss with upstream gradient
 * dout = dL/dO:  P_ij = exp(q_i.k_j / sqrt(d) - LSE_i),  D_i = dO_i . O_i,
 *   dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - D_i),
 *   dQ_i = sum_j dS_ij k_j / sqrt(d),  dK_j = sum_i dS_ij q_i / sqrt(d).
 * q, k, v, out (the forward output), dout, dq, dk, dv: bf16 [B, H, S, d] and
 * lse (the forward LSE): fp32 [B, H, S], all in sharded order with the same
 * P and causal flag as the forward.  Rank r's dQ visits the K/V blocks in the
 * forward's ring order; block b's dK/dV gather the query chunks of ranks
 * b, b+1, ... (the order the block travels the ring).  Non-causal chunks
 * whose last 128-row tile is short (a multiple of 8 rows, P times it at most
 * 128) have those rows of every rank (or block) taken together, in rank 0's
 * (block 0's) order; only the rounding order differs.  workspace: at least
 * ring_attn_bwd_workspace(...) bytes (fp32 D), 256-byte aligned, used by this
 * call only.  dq, dk, dv must not overlap the inputs. */
int ring_attn_bwd(const void *q, const void *k, const void *v, const void *out, const float *lse,
                  const void *dout, void *dq, void *dk, void *dv, int B, int H, int64_t S, int d,
                  int P, int causal, void *workspace, size_t ws_bytes, void *stream);

/* Workspace bytes of ring_attn_bwd (0 on bad arguments). */
size_t ring_attn_bwd_workspace(int B, int H, int64_t S);

/* Ulysses all-to-all (k8ai "Sequence and Context Parallel", "An alternative:
 * all-to-all on heads": the tokens are re-split by head for the attention
 * and re-split by sequence afterwards).  Row permutation of a bf16 tensor of
 * B*H*S rows of d elements between two per-rank layouts (P divides H):
 *   sequence-split  [P][B][H][L][d]    rank r holds its L = S/P tokens of every head;
 *   head-split      [P][B][H/P][S][d]  rank r holds heads r*H/P .. of every token
 *                                      (token r*L + i = row i of rank r).
 * inverse = 0: sequence-split -> head-split; 1: back.  Bit-exact copy. */
int ra_ulysses_a2a(const void *x, void *y, int B, int H, int64_t S, int d, int P, int inverse,
                   void *stream);

/* Attention with Ulysses parallelism: q, k, v, out bf16 and lse fp32 in the
 * sequence-split per-rank layout above ([P][B][H][L][d] / [P][B][H][L]);
 * all-to-all to head-split, full attention of every token over all S keys
 * for each rank's H/P heads (causal: key <= query by token position, S even),
 * all-to-all back.  Equals full attention.  Requires H % P == 0 (the degree is
 * at most the number of heads).  workspace: >= ulysses_attn_workspace(...)
 * bytes, 256-byte aligned, used by this call only. */
int ulysses_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                     int H, int64_t S, int d, int P, int causal, void *workspace, size_t ws_bytes,
                     void *stream);

/* Workspace bytes of ulysses_attn_fwd (0 on bad arguments). */
size_t ulysses_attn_workspace(int B, int H, int64_t S, int d);

/* The all-gather and reduce-scatter forms of context parallelism, the two
 * communication patterns the glossary lists beside the ring (ultralytics
 * glossary, "How Context Parallelism Works").  q, k, v, out: bf16 per-rank buffers [P][B][H][L][d]
 * (rank r's L = S/P tokens of every head, in the order ra_cp_shard gives its
 * chunk: contiguous, or zigzag when causal); lse: fp32 [P][B][H][L].  Both
 * equal full attention.
 *  cp_allgather_attn_fwd:     K and V are all-gathered into one rank-major
 *                             copy, then every rank attends its queries to all
 *                             S keys (blocks in ring order, one accumulator).
 *  cp_reducescatter_attn_fwd: queries are all-gathered; each rank's K/V block
 *                             yields a partial (O, LSE) for every query; the
 *                             partials of each query are merged (the reduce)
 *                             and each rank's rows are scattered back.
 * Both stack every rank's short last rows as ring_attn_fwd does (the
 * reduce-scatter form files their partials under the block they read).
 * workspace: >= cp_variant_workspace(...) bytes (either form), 256-byte
 * aligned, used by this call only. */
int cp_allgather_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                          int B, int H, int64_t S, int d, int P, int causal, void *workspace,
                          size_t ws_bytes, void *stream);
int cp_reducescatter_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                              int B, int H, int64_t S, int d, int P, int causal, void *workspace,
                              size_t ws_bytes, void *stream);
size_t cp_variant_workspace(int B, int H, int64_t S, int d, int P);

/* Online-softmax merge of n normalised partials of the same rows ("day 83"
 * blog, "Context parallelism: splitting the sequence"):  M = max_i LSE_i,  w_i = exp(LSE_i - M),
 *   LSE = M + ln(sum w_i),  O = sum w_i O_i / sum w_i;
 * rows whose partials are all empty (LSE = -inf) get O = 0, LSE = -inf.
 * o_parts fp32 [n][rows][d], lse_parts fp32 [n][rows]; out bf16 [rows][d],
 * lse_out fp32 [rows].  1 <= n <= 64. */
int lse_merge(const float *o_parts, const float *lse_parts, int n, int64_t rows, int d,
              void *out, float *lse_out, void *stream);

/* Factored video attention ("day 83" blog, "The spatial-temporal twist").
 * q, k, v: bf16 [B, H, T*N, d], token t*N + n (whole frames contiguous).
 *  spatial:  out_s bf16 [B, H, T*N, d], lse_s fp32 [B, H, T*N]: attention of
 *            each token over the N tokens of its own frame.
 *  temporal: out_t bf16 [B, H, T*N, d], lse_t fp32 [B, H, T*N]: attention of
 *            each token over the T tokens at its spatial position, run as a
 *            ring over P chunks of T/P frames (T % P == 0).  With every
 *            chunk resident on one GPU, adjacent chunks of at most 32 frames
 *            together may share a tile (12-frame chunks at P = 4 are taken
 *            in pairs): the ring then has fewer, longer steps, and the
 *            result differs only in the rounding order of the exact merge.
 * The two outputs are independent (not chained).  workspace: used only when
 * the rank chunks are longer than 128 frames (T / P > 128); then device
 * memory of at least factored_attn_workspace(...) bytes, 256-byte aligned,
 * owned by the caller and used as scratch by this call only, else ignored
 * (it may be null). */
int factored_attn(const void *q, const void *k, const void *v, void *out_s, float *lse_s,
                  void *out_t, float *lse_t, int B, int H, int T, int N, int d, int P,
                  void *workspace, size_t ws_bytes, void *stream);

/* Scratch bytes that suffice for factored_attn at these sizes with any P
 * (0 on bad arguments).  0 when T <= 128.  For T > 128: room for
 * position-major copies of q, k, v and of the temporal output (bf16) and LSE
 * (fp32).  A call only uses them when its rank chunks are longer than 128
 * frames (T / P > 128); with chunks of up to 128 frames the temporal pass
 * reads and writes the frame-major tensors in place, factored_attn checks no
 * workspace and the pointer may be null, whatever this function returns. */
size_t factored_attn_workspace(int B, int H, int T, int N, int d);

/* Size of the fixed device scratch that factored_attn_static works in. */
#define RA_STATIC_SCRATCH_BYTES (64u << 20)

/* factored_attn without any device allocation: the same computation, inputs
 * and outputs as factored_attn, but its scratch is a fixed array of
 * RA_STATIC_SCRATCH_BYTES (64 MiB) compiled into this library, so the caller
 * passes no workspace.  The pages have no counterpart: it exists for callers
 * that may not allocate device memory themselves, for example a host program
 * whose device memory is all handed to its own pool at start-up, or a serving
 * loop in which an allocation (and the synchronisation cudaMalloc implies) is
 * not allowed.
 *  - Limit: any size whose rank chunks hold at most 128 frames (T / P <= 128)
 *    needs no scratch and is accepted.  Longer chunks need
 *    factored_attn_workspace(B,H,T,N,d) <= RA_STATIC_SCRATCH_BYTES: about
 *    65,000 tokens x heads at d = 128 and 130,000 at d = 64; larger sizes
 *    return RA_ERR_WORKSPACE and launch nothing.  Other argument errors are
 *    those of factored_attn.
 *  - The array lives in every GPU that loads the library until the process
 *    exits.  The first call on a device whose sizes need scratch (rank chunks
 *    over 128 frames) looks up the array's device address (once per device,
 *    with that device current); make that call before any stream capture.
 *    The CUDA runtime loads device code lazily by default, so that call is
 *    also when the 64 MiB array is placed in the device's memory: it can fail
 *    there with RA_ERR_CUDA (out of memory) if the caller's own pool has
 *    already taken all device memory, so make it before creating such a pool.
 *    Calls whose sizes need no scratch never look the array up, and under lazy
 *    loading never cause it to be placed in device memory.
 *  - The looked-up address is kept for the life of the process: after
 *    cudaDeviceReset, or after the primary context is destroyed and made
 *    again, this entry point must not be called on that device.
 *  - Nothing in the scratch needs to start at zero (every byte read is first
 *    written by the same call), but all calls share the one array: calls whose
 *    work overlaps on the GPU (other streams, other host threads) race; order
 *    them on one stream or synchronise between them.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
int factored_attn_static(const void *q, const void *k, const void *v, void *out_s, float *lse_s,
                         void *out_t, float *lse_t, int B, int H, int T, int N, int d, int P,
                         void *stream);

/* Synchronises `stream`, then returns and clears the device status word:
 * RA_OK, or RA_ERR_TIMEOUT if a kernel's bounded wait expired since the last
 * call (the kernel then stopped early and its outputs are undefined),
 * RA_ERR_BOUNDS (checked builds only, see below), or RA_ERR_CUDA if the
 * synchronisation failed. */
int ra_get_status(void *stream);

/* Bounded-wait limit of the kernels' barrier waits, in nanoseconds (default
 * 2e9).  Values <= 0 restore the default.  Applies to later launches. */
void ra_set_watchdog_ns(int64_t ns);

/* Folding of factored_attn's temporal ring (process-wide, later calls):
 * 1 (default) lets adjacent rank chunks of at most 32 frames together share
 * a block, so the ring has fewer, longer steps (12-frame chunks at P = 4 run
 * as 2 blocks of 24 frames); 0 runs the ring over the P chunks exactly as
 * given (P steps).  Both give the same result up to rounding order. */
void ra_set_temporal_fold(int enable);

/* Runs a kernel whose only wait can never be satisfied, with the current
 * watchdog limit, to exercise the timeout path: returns RA_OK when launched;
 * ra_get_status then reports RA_ERR_TIMEOUT. */
int ra_watchdog_selftest(void *stream);

/* Bounds-checked builds.  Compiled with -DRA_CHECKS, every kernel checks each
 * global row index and TMA coordinate it computes against the extent of the
 * buffer it addresses, and each TMEM column range against the allocation.
 * A failed check records RA_ERR_BOUNDS in the device status word (read with
 * ra_get_status; the first error since the last read wins) and the access is
 * not made: a store is skipped, a TMA load is redirected to coordinate 0 so
 * that its barrier still completes.  Outputs are then undefined.  The default
 * build compiles no checks in and never reports RA_ERR_BOUNDS.
 * ra_checks_enabled: 1 in a build with the checks, 0 otherwise.
 * ra_checks_selftest: launches a kernel that checks one index against a bound
 * it exceeds, without any memory access through that index; returns RA_OK
 * when launched, after which ra_get_status reports RA_ERR_BOUNDS in a checked
 * build and RA_OK in the default build. */
int ra_checks_enabled(void);
int ra_checks_selftest(void *stream);

/* Text for an RA_* code; the last CUDA error (cudaError_t) seen on RA_ERR_CUDA. */
const char *ra_strerror(int code);
int ra_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* RINGATTN_H */
