// C ABI of the ring-attention library: argument validation, the device
// status word, and the launch of each entry point on the caller's stream.
// Declarations and the contract of every function are in include/ringattn.h.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "ra_internal.h"
#include "ringattn.h"

namespace {

__device__ int g_status;  // first device-side error since the last ra_get_status

std::atomic<int> g_last_cuda_error{0};
std::atomic<int64_t> g_watchdog_ns{2000000000LL};
std::atomic<int> g_temporal_fold{1};

int fail_cuda(cudaError_t e) {
  g_last_cuda_error.store(static_cast<int>(e));
  return RA_ERR_CUDA;
}

int *status_ptr() {
  static int *ptrs[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int *>(p);
  }
  return ptrs[dev];
}

bool watchdog(ra::WatchdogParams *wd) {
  wd->status = status_ptr();
  wd->limit_ns = g_watchdog_ns.load();
  return wd->status != nullptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

float scale_log2(int d) { return static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(d))); }

int check_d(int d) { return (d == 64 || d == 128) ? RA_OK : RA_ERR_SHAPE; }

// Rows per rank of the packed remainder tile for a launch of P ranks'
// chunks of L rows (0: none).  A non-causal chunk ending in a short single
// tile (L mod 256 in (0, 128], a multiple of 8 so the 128-byte swizzle
// phase holds) has every rank's last rows stacked in one query tile when
// they fit: one short unit per head instead of P, and the launch's last
// wave no longer waits for them.
int rem_pack_rows(int64_t L, int P, int causal) {
  const int64_t n_pairs = (L + 255) / 256;
  const int64_t rem = L - (n_pairs - 1) * 256;
  if (causal || n_pairs < 2 || P < 2 || rem <= 0 || rem > 128 || rem % 8 != 0 || P * rem > 128)
    return 0;
  return static_cast<int>(rem);
}

// Largest row count a 2-D tensor map coordinate can address with a tile of
// slack past the end.
constexpr int64_t kMaxRows = (int64_t(1) << 31) - 512;

}  // namespace

int ra::record_cuda_error(cudaError_t e) { return fail_cuda(e); }

extern "C" {

const char *ra_strerror(int code) {
  switch (code) {
    case RA_OK: return "ok";
    case RA_ERR_ARG: return "invalid argument (null pointer, negative size or bad option)";
    case RA_ERR_SHAPE: return "unsupported shape (S % P, S % 2P for zigzag, or d not 64/128)";
    case RA_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case RA_ERR_CUDA: return "CUDA error (see ra_last_cuda_error)";
    case RA_ERR_TIMEOUT: return "device watchdog: a kernel's bounded wait expired";
    case RA_ERR_WORKSPACE: return "workspace missing or too small";
    case RA_ERR_BOUNDS:
      return "bounds check (RA_CHECKS build): a device index fell outside its buffer";
    default: return "unknown error";
  }
}

int ra_last_cuda_error(void) { return g_last_cuda_error.load(); }

void ra_set_watchdog_ns(int64_t ns) { g_watchdog_ns.store(ns > 0 ? ns : 2000000000LL); }

void ra_set_temporal_fold(int enable) { g_temporal_fold.store(enable != 0 ? 1 : 0); }

int ra_cp_shard_index(int64_t S, int P, int layout, int64_t *s2g, int64_t *g2s) {
  if (S < 0 || P <= 0 || (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG))
    return RA_ERR_ARG;
  if (S % P != 0) return RA_ERR_SHAPE;
  if (layout == RA_LAYOUT_ZIGZAG && S % (2 * static_cast<int64_t>(P)) != 0) return RA_ERR_SHAPE;
  const int64_t L = S / P;
  const int64_t C = L / 2;
  for (int64_t j = 0; j < S; ++j) {
    const int64_t r = j / L, i = j % L;
    int64_t g = j;
    if (layout == RA_LAYOUT_ZIGZAG) g = i < C ? r * C + i : (2 * P - 1 - r) * C + (i - C);
    if (s2g) s2g[j] = g;
    if (g2s) g2s[g] = j;
  }
  return RA_OK;
}

int ra_ring_source(int P, int rank, int step) {
  if (P <= 0 || rank < 0 || rank >= P || step < 0) return -1;
  return ((rank - step) % P + P) % P;
}

int ra_cp_shard(const void *x, void *y, int64_t BH, int64_t S, int d, int P, int layout,
                int inverse, void *stream) {
  if (BH < 0 || S < 0 || P <= 0 || (inverse != 0 && inverse != 1) ||
      (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG))
    return RA_ERR_ARG;
  if (check_d(d) != RA_OK || S % P != 0) return RA_ERR_SHAPE;
  if (layout == RA_LAYOUT_ZIGZAG && S % (2 * static_cast<int64_t>(P)) != 0) return RA_ERR_SHAPE;
  if (BH == 0 || S == 0) return RA_OK;
  if (!x || !y) return RA_ERR_ARG;
  if (!aligned16(x) || !aligned16(y)) return RA_ERR_ALIGN;
  if (BH * S > kMaxRows) return RA_ERR_SHAPE;
  int *sw = status_ptr();
  if (sw == nullptr) return fail_cuda(cudaGetLastError());
  cudaError_t e = ra::launch_row_permute(x, y, BH, S, d * 2, inverse ? 1 : 0, P, 0, layout, sw,
                                         as_stream(stream));
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

int ra_frame_transpose(const void *x, void *y, int64_t BH, int64_t T, int64_t N, int d,
                       int inverse, void *stream) {
  if (BH < 0 || T < 0 || N < 0 || (inverse != 0 && inverse != 1)) return RA_ERR_ARG;
  if (check_d(d) != RA_OK) return RA_ERR_SHAPE;
  if (BH == 0 || T == 0 || N == 0) return RA_OK;
  if (!x || !y) return RA_ERR_ARG;
  if (!aligned16(x) || !aligned16(y)) return RA_ERR_ALIGN;
  if (BH * T * N > kMaxRows) return RA_ERR_SHAPE;
  int *sw = status_ptr();
  if (sw == nullptr) return fail_cuda(cudaGetLastError());
  cudaError_t e = ra::launch_row_permute(x, y, BH, T * N, d * 2, inverse ? 3 : 2, T, N, 0, sw,
                                         as_stream(stream));
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

int ring_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                  int H, int64_t S, int d, int P, int causal, void *stream) {
  if (B < 0 || H < 0 || S < 0 || P <= 0 || (causal != 0 && causal != 1)) return RA_ERR_ARG;
  if (check_d(d) != RA_OK || S % P != 0) return RA_ERR_SHAPE;
  if (causal && S % (2 * static_cast<int64_t>(P)) != 0) return RA_ERR_SHAPE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH == 0 || S == 0) return RA_OK;
  if (!q || !k || !v || !out || !lse) return RA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return RA_ERR_ALIGN;
  if (BH * S > kMaxRows || BH > 0x7fffffff) return RA_ERR_SHAPE;
  ra::AttnParams p{};
  const int64_t L = S / P;
  p.BH = static_cast<int>(BH);
  p.G = 1;
  p.n_ranks = P;
  p.n_stepgroups = 1;
  p.n_pairs = static_cast<int>((L + 255) / 256);
  p.q_rows_bh = S;
  p.kv_rows_bh = S;
  p.L = L;
  p.P = P;
  p.rank_begin = 0;
  p.step_begin = 0;
  p.steps_per_group = P;
  p.causal = causal;
  p.rem_pack = rem_pack_rows(L, P, causal);
  p.scale_log2 = scale_log2(d);
  p.out = out;
  p.lse = lse;
  if (!watchdog(&p.wd)) return fail_cuda(cudaGetLastError());
  cudaError_t e = ra::launch_ring_attn(q, BH * S, k, v, BH * S, d, false, p, as_stream(stream));
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

int ring_attn_fwd_rank(const void *q_local, const void *k, const void *v, void *out_local,
                       float *lse_local, int B, int H, int64_t S, int d, int P, int rank,
                       int causal, int step_begin, int step_end, int out_fp32, void *stream) {
  if (B < 0 || H < 0 || S < 0 || P <= 0 || (causal != 0 && causal != 1) ||
      (out_fp32 != 0 && out_fp32 != 1))
    return RA_ERR_ARG;
  if (rank < 0 || rank >= P || step_begin < 0 || step_end > P || step_begin >= step_end)
    return RA_ERR_ARG;
  if (check_d(d) != RA_OK || S % P != 0) return RA_ERR_SHAPE;
  if (causal && S % (2 * static_cast<int64_t>(P)) != 0) return RA_ERR_SHAPE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH == 0 || S == 0) return RA_OK;
  if (!q_local || !k || !v || !out_local || !lse_local) return RA_ERR_ARG;
  if (!aligned16(q_local) || !aligned16(k) || !aligned16(v) || !aligned16(out_local) ||
      !aligned16(lse_local))
    return RA_ERR_ALIGN;
  if (BH * S > kMaxRows || BH > 0x7fffffff) return RA_ERR_SHAPE;
  const int64_t L = S / P;
  const int n = step_end - step_begin;
  ra::AttnParams p{};
  p.BH = static_cast<int>(BH);
  p.G = 1;
  p.n_ranks = 1;
  p.n_pairs = static_cast<int>((L + 255) / 256);
  p.q_rows_bh = L;
  p.kv_rows_bh = S;
  p.L = L;
  p.P = P;
  p.rank_begin = rank;
  p.step_begin = step_begin;
  if (out_fp32) {
    p.n_stepgroups = n;
    p.steps_per_group = 1;
    p.out_part_stride = BH * L * d;
    p.lse_part_stride = BH * L;
  } else {
    p.n_stepgroups = 1;
    p.steps_per_group = n;
  }
  p.causal = causal;
  p.scale_log2 = scale_log2(d);
  p.out = out_local;
  p.lse = lse_local;
  if (!watchdog(&p.wd)) return fail_cuda(cudaGetLastError());
  cudaError_t e =
      ra::launch_ring_attn(q_local, BH * L, k, v, BH * S, d, out_fp32 != 0, p, as_stream(stream));
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

// Workspace of ring_attn_fwd_overlap: two K/V buffers of [P][BH][L][d] bf16
// each (K then V), then fp32 partials [P][BH][S][d] and LSEs [P][BH][S].
static size_t ovl_part(size_t bytes) { return (bytes + 255) & ~static_cast<size_t>(255); }

size_t ring_attn_fwd_overlap_workspace(int B, int H, int64_t S, int d, int P) {
  if (B < 0 || H < 0 || S < 0 || P <= 0 || check_d(d) != RA_OK) return 0;
  const size_t rows = static_cast<size_t>(B) * H * S;
  return 4 * ovl_part(rows * d * 2) + ovl_part(static_cast<size_t>(P) * rows * d * 4) +
         ovl_part(static_cast<size_t>(P) * rows * 4);
}

int ring_attn_fwd_overlap(const void *q, const void *k, const void *v, void *out, float *lse,
                          int B, int H, int64_t S, int d, int P, int causal, void *workspace,
                          size_t ws_bytes, void *stream, void *comm_stream) {
  if (B < 0 || H < 0 || S < 0 || P <= 0 || P > 64 || (causal != 0 && causal != 1))
    return RA_ERR_ARG;
  if (check_d(d) != RA_OK || S % P != 0) return RA_ERR_SHAPE;
  if (causal && S % (2 * static_cast<int64_t>(P)) != 0) return RA_ERR_SHAPE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH == 0 || S == 0) return RA_OK;
  if (!q || !k || !v || !out || !lse) return RA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return RA_ERR_ALIGN;
  if (BH * S > kMaxRows || BH > 0x7fffffff) return RA_ERR_SHAPE;
  const size_t need = ring_attn_fwd_overlap_workspace(B, H, S, d, P);
  if (!workspace || ws_bytes < need) return RA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return RA_ERR_ALIGN;
  cudaStream_t cs = as_stream(stream);
  // Without a comm stream the exchange runs inside the step launches (their
  // idle warps copy the next step's blocks), ordered by the stream alone.
  const bool in_launch = comm_stream == nullptr;
  cudaStream_t xs = in_launch ? cs : as_stream(comm_stream);
  ra::WatchdogParams wd;
  if (!watchdog(&wd)) return fail_cuda(cudaGetLastError());

  const int64_t L = S / P;
  const size_t blk_bytes = static_cast<size_t>(BH * L) * d * 2;  // one rank's block, one tensor
  const size_t buf_bytes = ovl_part(static_cast<size_t>(BH * S) * d * 2);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  uint8_t *kb[2] = {ws, ws + 2 * buf_bytes};
  uint8_t *vb[2] = {ws + buf_bytes, ws + 3 * buf_bytes};
  float *o_parts = reinterpret_cast<float *>(ws + 4 * buf_bytes);
  float *l_parts = reinterpret_cast<float *>(
      ws + 4 * buf_bytes + ovl_part(static_cast<size_t>(P) * BH * S * d * 4));

  cudaEvent_t copied[2] = {}, consumed[2] = {};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 2 && !in_launch; ++i) {
    if ((e = cudaEventCreateWithFlags(&copied[i], cudaEventDisableTiming)) != cudaSuccess)
      return fail_cuda(e);
    if ((e = cudaEventCreateWithFlags(&consumed[i], cudaEventDisableTiming)) != cudaSuccess)
      return fail_cuda(e);
  }
  // The comm stream may not start before inputs written on `stream` are ready.
  cudaEvent_t start = nullptr;
  if (!in_launch) {
    if ((e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming)) != cudaSuccess)
      return fail_cuda(e);
    e = cudaEventRecord(start, cs);
    if (e == cudaSuccess && xs != cs) e = cudaStreamWaitEvent(xs, start, 0);
  }

  for (int s = 0; s < P && e == cudaSuccess; ++s) {
    // ---- comm: ring send for step s + 1 (rank r receives rank r-1's block).
    if (!in_launch && s + 1 < P) {
      const int nb = (s + 1) & 1;
      if (s >= 1) e = cudaStreamWaitEvent(xs, consumed[nb], 0);  // step s-1 read it
      for (int r = 0; r < P && e == cudaSuccess; ++r) {
        const int from = (r + P - 1) % P;
        for (int t = 0; t < 2 && e == cudaSuccess; ++t) {
          uint8_t *dst = (t ? vb[nb] : kb[nb]) + static_cast<size_t>(r) * blk_bytes;
          if (s == 0) {
            const uint8_t *src = static_cast<const uint8_t *>(t ? v : k) +
                                 static_cast<size_t>(from * L) * d * 2;
            e = cudaMemcpy2DAsync(dst, static_cast<size_t>(L) * d * 2, src,
                                  static_cast<size_t>(S) * d * 2, static_cast<size_t>(L) * d * 2,
                                  static_cast<size_t>(BH), cudaMemcpyDeviceToDevice, xs);
          } else {
            const uint8_t *src = (t ? vb[s & 1] : kb[s & 1]) + static_cast<size_t>(from) * blk_bytes;
            e = cudaMemcpyAsync(dst, src, blk_bytes, cudaMemcpyDeviceToDevice, xs);
          }
        }
      }
      if (e == cudaSuccess) e = cudaEventRecord(copied[nb], xs);
    }
    if (e != cudaSuccess) break;
    // ---- compute: step s for every rank, from its current buffer.
    if (!in_launch && s >= 1) e = cudaStreamWaitEvent(cs, copied[s & 1], 0);
    if (e != cudaSuccess) break;
    ra::AttnParams p{};
    p.BH = static_cast<int>(BH);
    p.G = 1;
    p.n_ranks = P;
    p.n_stepgroups = 1;
    p.n_pairs = static_cast<int>((L + 255) / 256);
    p.q_rows_bh = S;
    p.L = L;
    p.P = P;
    p.step_begin = s;
    p.steps_per_group = 1;
    p.causal = causal;
    // Stacked last rows read rank 0's current block for every rank: over the
    // P steps each rank's rows still meet every block once.
    p.rem_pack = rem_pack_rows(L, P, causal);
    p.scale_log2 = scale_log2(d);
    p.out = o_parts + static_cast<size_t>(s) * BH * S * d;
    p.lse = l_parts + static_cast<size_t>(s) * BH * S;
    p.wd = wd;
    const void *ks = k, *vs = v;
    int64_t kv_rows = BH * S;
    if (s == 0) {
      p.kv_rows_bh = S;
    } else {
      p.kv_own = 1;
      p.kv_rows_bh = L;
      p.kv_rank_stride = BH * L;
      ks = kb[s & 1];
      vs = vb[s & 1];
    }
    if (in_launch && s + 1 < P) {
      // The same ring send as the copies above, done by this launch: rank r's
      // next buffer receives rank r - 1's current block (step 0: the inputs,
      // a head pitch of S rows).
      const int nb = (s + 1) & 1;
      p.x_on = 1;
      p.x_ranks = P;
      p.x_bh = static_cast<int>(BH);
      p.xk_src = static_cast<const uint8_t *>(s == 0 ? k : kb[s & 1]);
      p.xv_src = static_cast<const uint8_t *>(s == 0 ? v : vb[s & 1]);
      p.xk_dst = kb[nb];
      p.xv_dst = vb[nb];
      p.x_row_bytes = L * d * 2;
      p.x_src_rank = s == 0 ? L * d * 2 : static_cast<int64_t>(blk_bytes);
      p.x_src_head = s == 0 ? S * d * 2 : L * d * 2;
      p.x_dst_rank = static_cast<int64_t>(blk_bytes);
      p.x_dst_head = L * d * 2;
      p.x_src_span = s == 0 ? BH * S * d * 2 : static_cast<int64_t>(P) * blk_bytes;
      p.x_dst_span = static_cast<int64_t>(P) * blk_bytes;
    }
    e = ra::launch_ring_attn(q, BH * S, ks, vs, kv_rows, d, true, p, cs);
    if (e == cudaSuccess && !in_launch && s >= 1) e = cudaEventRecord(consumed[s & 1], cs);
  }
  if (e == cudaSuccess)
    e = ra::launch_lse_merge(o_parts, l_parts, P, BH * S, d, out, lse, wd.status, cs);
  for (int i = 0; i < 2 && !in_launch; ++i) {
    cudaEventDestroy(copied[i]);
    cudaEventDestroy(consumed[i]);
  }
  if (start) cudaEventDestroy(start);
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

int ra_ulysses_a2a(const void *x, void *y, int B, int H, int64_t S, int d, int P, int inverse,
                   void *stream) {
  if (B < 0 || H < 0 || S < 0 || P <= 0 || (inverse != 0 && inverse != 1)) return RA_ERR_ARG;
  if (check_d(d) != RA_OK || S % P != 0 || H % P != 0) return RA_ERR_SHAPE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH == 0 || S == 0) return RA_OK;
  if (!x || !y) return RA_ERR_ARG;
  if (!aligned16(x) || !aligned16(y)) return RA_ERR_ALIGN;
  if (BH * S > kMaxRows) return RA_ERR_SHAPE;
  int *sw = status_ptr();
  if (sw == nullptr) return fail_cuda(cudaGetLastError());
  cudaError_t e = ra::launch_row_permute(x, y, BH, S, d * 2, inverse ? 5 : 4, P, H, B, sw,
                                         as_stream(stream));
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

size_t ulysses_attn_workspace(int B, int H, int64_t S, int d) {
  if (B < 0 || H < 0 || S < 0 || check_d(d) != RA_OK) return 0;
  const size_t rows = static_cast<size_t>(B) * H * S;
  return 4 * ovl_part(rows * d * 2) + ovl_part(rows * 4);
}

int ulysses_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                     int H, int64_t S, int d, int P, int causal, void *workspace, size_t ws_bytes,
                     void *stream) {
  if (B < 0 || H < 0 || S < 0 || P <= 0 || (causal != 0 && causal != 1)) return RA_ERR_ARG;
  if (check_d(d) != RA_OK || S % P != 0 || H % P != 0) return RA_ERR_SHAPE;
  if (causal && S % 2 != 0) return RA_ERR_SHAPE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH == 0 || S == 0) return RA_OK;
  if (!q || !k || !v || !out || !lse) return RA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return RA_ERR_ALIGN;
  if (BH * S > kMaxRows || BH > 0x7fffffff) return RA_ERR_SHAPE;
  if (!workspace || ws_bytes < ulysses_attn_workspace(B, H, S, d)) return RA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return RA_ERR_ALIGN;
  cudaStream_t st = as_stream(stream);
  ra::WatchdogParams wd;
  if (!watchdog(&wd)) return fail_cuda(cudaGetLastError());
  const size_t tb = ovl_part(static_cast<size_t>(BH * S) * d * 2);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  void *qh = ws, *kh = ws + tb, *vh = ws + 2 * tb, *oh = ws + 3 * tb;
  float *lh = reinterpret_cast<float *>(ws + 4 * tb);
  const void *src[3] = {q, k, v};
  void *dst[3] = {qh, kh, vh};
  cudaError_t e;
  for (int i = 0; i < 3; ++i) {
    e = ra::launch_row_permute(src[i], dst[i], BH, S, d * 2, 4, P, H, B, wd.status, st);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  // Head-split: B*H heads of S tokens in global order; no ring (P = 1).
  ra::AttnParams p{};
  p.BH = static_cast<int>(BH);
  p.G = 1;
  p.n_ranks = 1;
  p.n_stepgroups = 1;
  p.n_pairs = static_cast<int>((S + 255) / 256);
  p.q_rows_bh = S;
  p.kv_rows_bh = S;
  p.L = S;
  p.P = 1;
  p.steps_per_group = 1;
  p.causal = causal;  // zigzag with one rank is the identity order
  p.scale_log2 = scale_log2(d);
  p.out = oh;
  p.lse = lh;
  p.wd = wd;
  e = ra::launch_ring_attn(qh, BH * S, kh, vh, BH * S, d, false, p, st);
  if (e != cudaSuccess) return fail_cuda(e);
  e = ra::launch_row_permute(oh, out, BH, S, d * 2, 5, P, H, B, wd.status, st);
  if (e != cudaSuccess) return fail_cuda(e);
  e = ra::launch_row_permute(lh, lse, BH, S, 4, 5, P, H, B, wd.status, st);
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

// Workspace of the all-gather / reduce-scatter forms: three rank-major bf16
// copies (Q, K, V), then fp32 partials [P][BH][S][d] + LSEs, then a rank-major
// bf16 output and fp32 LSE.
size_t cp_variant_workspace(int B, int H, int64_t S, int d, int P) {
  if (B < 0 || H < 0 || S < 0 || P <= 0 || check_d(d) != RA_OK) return 0;
  const size_t rows = static_cast<size_t>(B) * H * S;
  return 4 * ovl_part(rows * d * 2) + ovl_part(static_cast<size_t>(P) * rows * d * 4) +
         ovl_part(static_cast<size_t>(P) * rows * 4) + ovl_part(rows * 4);
}

static int cp_variant_check(const void *q, const void *k, const void *v, void *out, float *lse,
                            int B, int H, int64_t S, int d, int P, int causal, void *workspace,
                            size_t ws_bytes) {
  if (B < 0 || H < 0 || S < 0 || P <= 0 || P > 64 || (causal != 0 && causal != 1))
    return RA_ERR_ARG;
  if (check_d(d) != RA_OK || S % P != 0) return RA_ERR_SHAPE;
  if (causal && S % (2 * static_cast<int64_t>(P)) != 0) return RA_ERR_SHAPE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH == 0 || S == 0) return 1;  // no-op
  if (!q || !k || !v || !out || !lse) return RA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return RA_ERR_ALIGN;
  if (BH * S > kMaxRows || BH > 0x7fffffff) return RA_ERR_SHAPE;
  if (!workspace || ws_bytes < cp_variant_workspace(B, H, S, d, P)) return RA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return RA_ERR_ALIGN;
  return RA_OK;
}

int cp_allgather_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                          int B, int H, int64_t S, int d, int P, int causal, void *workspace,
                          size_t ws_bytes, void *stream) {
  int rc = cp_variant_check(q, k, v, out, lse, B, H, S, d, P, causal, workspace, ws_bytes);
  if (rc != RA_OK) return rc == 1 ? RA_OK : rc;
  const int64_t BH = static_cast<int64_t>(B) * H, L = S / P;
  cudaStream_t st = as_stream(stream);
  ra::WatchdogParams wd;
  if (!watchdog(&wd)) return fail_cuda(cudaGetLastError());
  const size_t tb = ovl_part(static_cast<size_t>(BH * S) * d * 2);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  void *kg = ws + tb, *vg = ws + 2 * tb;
  cudaError_t e = ra::launch_row_permute(k, kg, BH, S, d * 2, 6, P, H, B, wd.status, st);
  if (e == cudaSuccess) e = ra::launch_row_permute(v, vg, BH, S, d * 2, 6, P, H, B, wd.status, st);
  if (e == cudaSuccess) {
    // Every rank's own queries (buffer r) against every block of the gathered
    // K/V, all ranks in one launch.
    ra::AttnParams p{};
    p.BH = static_cast<int>(BH);
    p.G = 1;
    p.n_ranks = P;
    p.n_stepgroups = 1;
    p.n_pairs = static_cast<int>((L + 255) / 256);
    p.q_rows_bh = L;
    p.q_rank_stride = BH * L;
    p.kv_rows_bh = S;
    p.L = L;
    p.P = P;
    p.rank_begin = 0;
    p.steps_per_group = P;
    p.causal = causal;
    p.rem_pack = rem_pack_rows(L, P, causal);
    p.scale_log2 = scale_log2(d);
    p.out = out;
    p.lse = lse;
    p.wd = wd;
    e = ra::launch_ring_attn(q, BH * S, kg, vg, BH * S, d, false, p, st);
  }
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

int cp_reducescatter_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                              int B, int H, int64_t S, int d, int P, int causal, void *workspace,
                              size_t ws_bytes, void *stream) {
  int rc = cp_variant_check(q, k, v, out, lse, B, H, S, d, P, causal, workspace, ws_bytes);
  if (rc != RA_OK) return rc == 1 ? RA_OK : rc;
  const int64_t BH = static_cast<int64_t>(B) * H, L = S / P;
  cudaStream_t st = as_stream(stream);
  ra::WatchdogParams wd;
  if (!watchdog(&wd)) return fail_cuda(cudaGetLastError());
  const size_t tb = ovl_part(static_cast<size_t>(BH * S) * d * 2);
  const size_t pb = ovl_part(static_cast<size_t>(P) * BH * S * d * 4);
  const size_t lb = ovl_part(static_cast<size_t>(P) * BH * S * 4);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  void *qg = ws, *kg = ws + tb, *vg = ws + 2 * tb, *og = ws + 3 * tb;
  float *o_parts = reinterpret_cast<float *>(ws + 4 * tb);
  float *l_parts = reinterpret_cast<float *>(ws + 4 * tb + pb);
  float *lg = reinterpret_cast<float *>(ws + 4 * tb + pb + lb);
  const void *src[3] = {q, k, v};
  void *dst[3] = {qg, kg, vg};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 3 && e == cudaSuccess; ++i)
    e = ra::launch_row_permute(src[i], dst[i], BH, S, d * 2, 6, P, H, B, wd.status, st);
  if (e == cudaSuccess) {
    // Every (rank, block) pair once; the partial is filed under the block.
    ra::AttnParams p{};
    p.BH = static_cast<int>(BH);
    p.G = 1;
    p.n_ranks = P;
    p.n_stepgroups = P;
    p.n_pairs = static_cast<int>((L + 255) / 256);
    p.q_rows_bh = S;
    p.kv_rows_bh = S;
    p.L = L;
    p.P = P;
    p.steps_per_group = 1;
    p.causal = causal;
    p.part_by_block = 1;
    // Stacked last rows meet rank 0's block of each step and file the
    // partial under that block.
    p.rem_pack = rem_pack_rows(L, P, causal);
    p.scale_log2 = scale_log2(d);
    p.out = o_parts;
    p.lse = l_parts;
    p.out_part_stride = BH * S * d;
    p.lse_part_stride = BH * S;
    p.wd = wd;
    e = ra::launch_ring_attn(qg, BH * S, kg, vg, BH * S, d, true, p, st);
  }
  if (e == cudaSuccess)
    e = ra::launch_lse_merge(o_parts, l_parts, P, BH * S, d, og, lg, wd.status, st);
  if (e == cudaSuccess)
    e = ra::launch_row_permute(og, out, BH, S, d * 2, 7, P, H, B, wd.status, st);
  if (e == cudaSuccess) e = ra::launch_row_permute(lg, lse, BH, S, 4, 7, P, H, B, wd.status, st);
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

size_t ring_attn_bwd_workspace(int B, int H, int64_t S) {
  if (B < 0 || H < 0 || S < 0) return 0;
  return ovl_part(static_cast<size_t>(B) * H * S * 4);
}

int ring_attn_bwd(const void *q, const void *k, const void *v, const void *out, const float *lse,
                  const void *dout, void *dq, void *dk, void *dv, int B, int H, int64_t S, int d,
                  int P, int causal, void *workspace, size_t ws_bytes, void *stream) {
  if (B < 0 || H < 0 || S < 0 || P <= 0 || (causal != 0 && causal != 1)) return RA_ERR_ARG;
  if (check_d(d) != RA_OK || S % P != 0) return RA_ERR_SHAPE;
  if (causal && S % (2 * static_cast<int64_t>(P)) != 0) return RA_ERR_SHAPE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH == 0 || S == 0) return RA_OK;
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return RA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return RA_ERR_ALIGN;
  if (BH * S > kMaxRows || BH > 0x7fffffff) return RA_ERR_SHAPE;
  if (!workspace || ws_bytes < ring_attn_bwd_workspace(B, H, S)) return RA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return RA_ERR_ALIGN;
  ra::BwdParams p{};
  p.BH = static_cast<int>(BH);
  p.P = P;
  p.S = S;
  p.L = S / P;
  p.n_t = static_cast<int>((p.L + 127) / 128);
  p.causal = causal;
  p.scale_log2 = scale_log2(d);
  p.scale = static_cast<float>(1.0 / sqrt(static_cast<double>(d)));
  p.lse = lse;
  p.Dv = static_cast<float *>(workspace);
  p.dq = static_cast<__nv_bfloat16 *>(dq);
  p.dk = static_cast<__nv_bfloat16 *>(dk);
  p.dv = static_cast<__nv_bfloat16 *>(dv);
  if (!watchdog(&p.wd)) return fail_cuda(cudaGetLastError());
  cudaError_t e = ra::launch_attn_bwd(q, k, v, out, dout, d, p, as_stream(stream));
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

int lse_merge(const float *o_parts, const float *lse_parts, int n, int64_t rows, int d, void *out,
              float *lse_out, void *stream) {
  if (n < 1 || n > 64 || rows < 0) return RA_ERR_ARG;
  if (check_d(d) != RA_OK) return RA_ERR_SHAPE;
  if (rows == 0) return RA_OK;
  if (!o_parts || !lse_parts || !out || !lse_out) return RA_ERR_ARG;
  if (!aligned16(o_parts) || !aligned16(out) || !aligned16(lse_parts) || !aligned16(lse_out))
    return RA_ERR_ALIGN;
  int *sw = status_ptr();
  if (sw == nullptr) return fail_cuda(cudaGetLastError());
  cudaError_t e = ra::launch_lse_merge(o_parts, lse_parts, n, rows, d, out, lse_out, sw,
                                       as_stream(stream));
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

// Workspace of factored_attn.  Rank chunks of up to 128 frames (always, when
// T <= 128) are packed: q, k, v are read in place and the temporal output
// written in place, no workspace.  Longer chunks (possible only when
// T > 128) run on position-major copies of q, k, v and write a
// position-major output and LSE that are transposed back: four bf16 parts
// and one fp32 part, each 256-byte aligned.
static size_t ws_part(size_t bytes) { return (bytes + 255) & ~static_cast<size_t>(255); }
constexpr int kPackMaxFrames = 128;

size_t factored_attn_workspace(int B, int H, int T, int N, int d) {
  if (B < 0 || H < 0 || T < 0 || N < 0 || check_d(d) != RA_OK) return 0;
  const size_t rows = static_cast<size_t>(B) * H * T * N;
  return T > kPackMaxFrames ? 4 * ws_part(rows * d * 2) + ws_part(rows * 4) : 0;
}

int factored_attn(const void *q, const void *k, const void *v, void *out_s, float *lse_s,
                  void *out_t, float *lse_t, int B, int H, int T, int N, int d, int P,
                  void *workspace, size_t ws_bytes, void *stream) {
  if (B < 0 || H < 0 || T < 0 || N < 0 || P <= 0) return RA_ERR_ARG;
  if (check_d(d) != RA_OK || T % P != 0) return RA_ERR_SHAPE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t S = static_cast<int64_t>(T) * N;
  if (BH == 0 || S == 0) return RA_OK;
  if (!q || !k || !v || !out_s || !lse_s || !out_t || !lse_t) return RA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out_s) || !aligned16(lse_s) ||
      !aligned16(out_t) || !aligned16(lse_t))
    return RA_ERR_ALIGN;
  if (BH * S > kMaxRows || BH > 0x7fffffff) return RA_ERR_SHAPE;
  const size_t need = ra::factored_scratch_bytes(B, H, T, N, d, P);
  if (need > 0) {
    if (!workspace || ws_bytes < need) return RA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return RA_ERR_ALIGN;
  }
  cudaStream_t st = as_stream(stream);
  ra::WatchdogParams wd;
  if (!watchdog(&wd)) return fail_cuda(cudaGetLastError());
  cudaError_t e;

  // Spatial: T independent N-token problems per (b, h), no ring.
  {
    ra::AttnParams p{};
    p.BH = static_cast<int>(BH);
    p.G = T;
    p.n_ranks = 1;
    p.n_stepgroups = 1;
    p.n_pairs = (N + 255) / 256;
    p.q_rows_bh = S;
    p.q_rows_g = N;
    p.kv_rows_bh = S;
    p.kv_rows_g = N;
    p.L = N;
    p.P = 1;
    p.steps_per_group = 1;
    p.scale_log2 = scale_log2(d);
    p.out = out_s;
    p.lse = lse_s;
    p.wd = wd;
    e = ra::launch_ring_attn(q, BH * S, k, v, BH * S, d, false, p, st);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  // Temporal: N problems of T tokens per (b, h), each a ring over P chunks
  // of T/P frames.  Chunks of up to 128 frames are read from and written to
  // the frame-major tensors in place (packed tiles); longer ones run on
  // position-major copies whose output is transposed back.
  const bool packed = T / P <= kPackMaxFrames;
  const void *tq = q, *tk = k, *tv = v;
  void *oT = out_t;
  float *lT = lse_t;
  if (!packed) {
    // Workspace: [output | q | k | v] position-major (bf16), then the LSE.
    const size_t tbytes = ws_part(static_cast<size_t>(BH * S) * d * 2);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    oT = ws;
    lT = reinterpret_cast<float *>(ws + 4 * tbytes);
    void *dst[3] = {ws + tbytes, ws + 2 * tbytes, ws + 3 * tbytes};
    const void *src[3] = {q, k, v};
    for (int i = 0; i < 3; ++i) {
      e = ra::launch_row_permute(src[i], dst[i], BH, S, d * 2, 2, T, N, 0, wd.status, st);
      if (e != cudaSuccess) return fail_cuda(e);
    }
    tq = dst[0];
    tk = dst[1];
    tv = dst[2];
  }
  {
    ra::AttnParams p{};
    // On one GPU every rank's chunk is resident, so packed tiles may fold f
    // adjacent ranks' chunks (f divides P) into one block of f * T / P
    // frames: the ring then runs over P / f such blocks.  Its merge over
    // steps is exact, so folding changes only the rounding order, and the
    // block-diagonal tile work shrinks by f (each query row of a tile meets
    // one position's keys).  Folding stops at 32 rows per block (the
    // warp-packed tiles) and keeps at least two blocks (a CTA's two query
    // tiles): 12-frame chunks at P = 4 fold in pairs.
    int f = 1;
    if (packed && g_temporal_fold.load())
      for (int c = 2; c <= P / 2; ++c)
        if (P % c == 0 && static_cast<int64_t>(c) * (T / P) <= 32) f = c;
    const int Pr = P / f;  // ring size after folding
    const int64_t L = T / Pr;
    p.BH = static_cast<int>(BH);
    p.G = N;
    p.n_ranks = Pr;
    p.n_stepgroups = 1;
    p.n_pairs = static_cast<int>((L + 255) / 256);
    p.q_rows_bh = S;
    p.q_rows_g = T;
    p.kv_rows_bh = S;
    p.kv_rows_g = T;
    p.L = L;
    if (packed) {
      // Short chunks: one 128-row tile carries the same rank's chunk of
      // floor(128 / L) spatial positions (4-D TMA box over the frame-major
      // tensor), each position's queries masked to its own keys.
      // Chunks of up to 32 frames take 16 or 32 tile rows per position so
      // that every warp's queries and keys share one 32-column chunk.
      const int lrow = L <= 16 ? 16 : L <= 32 ? 32 : static_cast<int>(L);
      const int pack = 128 / lrow < N ? 128 / lrow : N;
      p.pack = pack;
      p.Lf = static_cast<int>(L);
      p.pLrow = lrow;
      p.pN = N;
      p.pT = T;
      p.G = (N + pack - 1) / pack;
      p.L = static_cast<int64_t>(pack) * lrow;
      // Two ranks' chunks per CTA (its two query tiles share the key tiles).
      p.n_ranks = (Pr + 1) / 2;
      p.pack_ranks = Pr;
      p.n_pairs = 1;
      p.pack_frame_major = 1;
    }
    p.P = Pr;
    p.steps_per_group = Pr;
    p.scale_log2 = scale_log2(d);
    p.out = oT;
    p.lse = lT;
    p.wd = wd;
    e = ra::launch_ring_attn(tq, BH * S, tk, tv, BH * S, d, false, p, st);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  if (!packed) {
    e = ra::launch_row_permute(oT, out_t, BH, S, d * 2, 3, T, N, 0, wd.status, st);
    if (e != cudaSuccess) return fail_cuda(e);
    e = ra::launch_row_permute(lT, lse_t, BH, S, 4, 3, T, N, 0, wd.status, st);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  return RA_OK;
}

int ra_get_status(void *stream) {
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return fail_cuda(e);
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_status, sizeof(int));
  if (e != cudaSuccess) return fail_cuda(e);
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
  if (e != cudaSuccess) return fail_cuda(e);
  return v;
}

int ra_checks_enabled(void) {
#ifdef RA_CHECKS
  return 1;
#else
  return 0;
#endif
}

int ra_checks_selftest(void *stream) {
  int *st = status_ptr();
  if (st == nullptr) return fail_cuda(cudaGetLastError());
  cudaError_t e = ra::launch_checks_selftest(st, as_stream(stream));
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

int ra_watchdog_selftest(void *stream) {
  ra::WatchdogParams wd;
  if (!watchdog(&wd)) return fail_cuda(cudaGetLastError());
  cudaError_t e = ra::launch_watchdog_selftest(wd, as_stream(stream));
  return e == cudaSuccess ? RA_OK : fail_cuda(e);
}

}  // extern "C"

// Scratch a factored_attn call with this P actually uses: none while each
// rank chunk (T / P frames) fits one tile, else the full position-major set.
size_t ra::factored_scratch_bytes(int B, int H, int T, int N, int d, int P) {
  if (P > 0 && T >= 0 && T % P == 0 && T / P <= kPackMaxFrames) return 0;
  return factored_attn_workspace(B, H, T, N, d);
}
