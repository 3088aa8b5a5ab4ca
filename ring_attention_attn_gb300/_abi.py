"""ctypes binding of libringattn.so: argument marshalling only.

Every function here has the name of the C entry point it calls (see
include/ringattn.h for the contract).  Tensors are torch CUDA tensors used as
device memory; the current torch stream is passed as the CUDA stream.  There
is no fallback: without the built library, or with CPU tensors, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
# RINGATTN_LIB selects another build of the same library (same ABI).
LIB_PATH = os.environ.get("RINGATTN_LIB") or os.path.join(HERE, "libringattn.so")

RA_OK = 0
ERRORS = {-1: "RA_ERR_ARG", -2: "RA_ERR_SHAPE", -3: "RA_ERR_ALIGN", -4: "RA_ERR_CUDA",
          -5: "RA_ERR_TIMEOUT", -6: "RA_ERR_WORKSPACE", -7: "RA_ERR_BOUNDS"}

# Every symbol include/ringattn.h declares.
EXPORTS = ("ra_cp_shard_index", "ra_ring_source", "ra_cp_shard", "ra_frame_transpose",
           "ring_attn_fwd", "ring_attn_fwd_rank", "ring_attn_fwd_overlap",
           "ring_attn_fwd_overlap_workspace", "ring_attn_bwd", "ring_attn_bwd_workspace",
           "ra_ulysses_a2a", "ulysses_attn_fwd", "ulysses_attn_workspace",
           "cp_allgather_attn_fwd", "cp_reducescatter_attn_fwd", "cp_variant_workspace",
           "lse_merge", "factored_attn",
           "factored_attn_workspace", "factored_attn_static", "ra_get_status",
           "ra_set_watchdog_ns", "ra_set_temporal_fold",
           "ra_watchdog_selftest", "ra_checks_enabled", "ra_checks_selftest", "ra_strerror",
           "ra_last_cuda_error")

_lock = threading.Lock()
_lib = None


class RingAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = lib().ra_strerror(code).decode()
        extra = ""
        if code == -4:
            extra = f" (cudaError {lib().ra_last_cuda_error()})"
        super().__init__(f"{where}: {ERRORS.get(code, code)}: {msg}{extra}")


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run `python -m ring_attention_attn_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            i32, i64, vp, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
            sig = {
                "ra_cp_shard_index": (i32, [i64, i32, i32, vp, vp]),
                "ra_ring_source": (i32, [i32, i32, i32]),
                "ra_cp_shard": (i32, [vp, vp, i64, i64, i32, i32, i32, i32, vp]),
                "ra_frame_transpose": (i32, [vp, vp, i64, i64, i64, i32, i32, vp]),
                "ring_attn_fwd": (i32, [vp, vp, vp, vp, vp, i32, i32, i64, i32, i32, i32, vp]),
                "ring_attn_fwd_rank": (i32, [vp, vp, vp, vp, vp, i32, i32, i64, i32, i32, i32,
                                             i32, i32, i32, i32, vp]),
                "ring_attn_fwd_overlap": (i32, [vp, vp, vp, vp, vp, i32, i32, i64, i32, i32, i32,
                                                vp, sz, vp, vp]),
                "ring_attn_fwd_overlap_workspace": (sz, [i32, i32, i64, i32, i32]),
                "ring_attn_bwd": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i64, i32, i32,
                                        i32, vp, sz, vp]),
                "ring_attn_bwd_workspace": (sz, [i32, i32, i64]),
                "ra_ulysses_a2a": (i32, [vp, vp, i32, i32, i64, i32, i32, i32, vp]),
                "ulysses_attn_fwd": (i32, [vp, vp, vp, vp, vp, i32, i32, i64, i32, i32, i32, vp, sz,
                                           vp]),
                "ulysses_attn_workspace": (sz, [i32, i32, i64, i32]),
                "cp_allgather_attn_fwd": (i32, [vp, vp, vp, vp, vp, i32, i32, i64, i32, i32, i32,
                                                vp, sz, vp]),
                "cp_reducescatter_attn_fwd": (i32, [vp, vp, vp, vp, vp, i32, i32, i64, i32, i32,
                                                    i32, vp, sz, vp]),
                "cp_variant_workspace": (sz, [i32, i32, i64, i32, i32]),
                "lse_merge": (i32, [vp, vp, i32, i64, i32, vp, vp, vp]),
                "factored_attn": (i32, [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                        vp, sz, vp]),
                "factored_attn_workspace": (sz, [i32, i32, i32, i32, i32]),
                "factored_attn_static": (i32, [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                               i32, i32, vp]),
                "ra_get_status": (i32, [vp]),
                "ra_set_watchdog_ns": (None, [i64]),
                "ra_set_temporal_fold": (None, [i32]),
                "ra_watchdog_selftest": (i32, [vp]),
                "ra_checks_enabled": (i32, []),
                "ra_checks_selftest": (i32, [vp]),
                "ra_strerror": (ctypes.c_char_p, [i32]),
                "ra_last_cuda_error": (i32, []),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _check(code: int, where: str):
    if code != RA_OK:
        raise RingAttnError(code, where)


_raw_stream = None


def _stream(stream=None):
    """The given stream, else the current torch stream of the current device
    (read as a raw handle: building a torch Stream object per call costs
    microseconds)."""
    global _raw_stream
    import torch
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _raw_stream is None:
        get = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        dev = getattr(torch._C, "_cuda_getDevice", None)
        _raw_stream = ((lambda: get(dev())) if get is not None and dev is not None
                       else (lambda: torch.cuda.current_stream().cuda_stream))
    return ctypes.c_void_p(_raw_stream())


def _dev(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


# ------------------------------------------------------------------- host --
def ra_cp_shard_index(S: int, P: int, layout: int):
    """(s2g, g2s) int64 numpy maps; layout 0 contiguous, 1 zigzag."""
    s2g = np.empty(max(S, 1), dtype=np.int64)
    g2s = np.empty(max(S, 1), dtype=np.int64)
    _check(lib().ra_cp_shard_index(S, P, layout, s2g.ctypes.data_as(ctypes.c_void_p),
                                   g2s.ctypes.data_as(ctypes.c_void_p)), "ra_cp_shard_index")
    return s2g[:S], g2s[:S]


def ra_ring_source(P: int, rank: int, step: int) -> int:
    r = lib().ra_ring_source(P, rank, step)
    if r < 0:
        raise RingAttnError(-1, "ra_ring_source")
    return r


# ----------------------------------------------------------------- device --
def ra_cp_shard(x, P: int, layout: int, inverse: bool = False, out=None, stream=None):
    """Row permutation [B,H,S,d] bf16 between global and sharded order."""
    import torch
    B, H, S, d = x.shape
    y = torch.empty_like(x) if out is None else out
    _check(lib().ra_cp_shard(_dev(x, torch.bfloat16, "x"), _dev(y, torch.bfloat16, "out"), B * H,
                             S, d, P, layout, int(inverse), _stream(stream)), "ra_cp_shard")
    return y


def ra_frame_transpose(x, T: int, N: int, inverse: bool = False, out=None, stream=None):
    """[B,H,T*N,d] <-> [B,H,N*T,d] row transpose of bf16 video tokens."""
    import torch
    B, H, S, d = x.shape
    y = torch.empty_like(x) if out is None else out
    _check(lib().ra_frame_transpose(_dev(x, torch.bfloat16, "x"), _dev(y, torch.bfloat16, "out"),
                                    B * H, T, N, d, int(inverse), _stream(stream)),
           "ra_frame_transpose")
    return y


def ring_attn_fwd(q, k, v, P: int, causal: bool = False, out=None, lse=None, stream=None):
    """Ring attention over P simulated ranks; q/k/v [B,H,S,d] bf16 in sharded order."""
    import torch
    B, H, S, d = q.shape
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib().ring_attn_fwd(_dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"),
                               _dev(v, torch.bfloat16, "v"), _dev(out, torch.bfloat16, "out"),
                               _dev(lse, torch.float32, "lse"), B, H, S, d, P, int(causal),
                               _stream(stream)), "ring_attn_fwd")
    return out, lse


def ring_attn_fwd_rank(q_local, k, v, P: int, rank: int, causal: bool = False,
                       step_begin: int = 0, step_end: int | None = None, out_fp32: bool = False,
                       out=None, lse=None, stream=None):
    """One rank's queries against ring steps [step_begin, step_end).

    out_fp32=False: (out bf16 [B,H,L,d], lse [B,H,L]) over those steps' keys.
    out_fp32=True: per-step partials (out fp32 [n,B,H,L,d], lse [n,B,H,L]).
    """
    import torch
    B, H, L, d = q_local.shape
    S = k.shape[2]
    step_end = P if step_end is None else step_end
    n = step_end - step_begin
    if out is None:
        out = (torch.empty((n, B, H, L, d), dtype=torch.float32, device=q_local.device)
               if out_fp32 else torch.empty_like(q_local))
    if lse is None:
        shape = (n, B, H, L) if out_fp32 else (B, H, L)
        lse = torch.empty(shape, dtype=torch.float32, device=q_local.device)
    odt = torch.float32 if out_fp32 else torch.bfloat16
    _check(lib().ring_attn_fwd_rank(_dev(q_local, torch.bfloat16, "q_local"),
                                    _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
                                    _dev(out, odt, "out"), _dev(lse, torch.float32, "lse"), B, H,
                                    S, d, P, rank, int(causal), step_begin, step_end,
                                    int(out_fp32), _stream(stream)), "ring_attn_fwd_rank")
    return out, lse


def ring_attn_fwd_overlap_workspace(B: int, H: int, S: int, d: int, P: int) -> int:
    return int(lib().ring_attn_fwd_overlap_workspace(B, H, S, d, P))


def ring_attn_fwd_overlap(q, k, v, P: int, causal: bool = False, workspace=None, out=None,
                          lse=None, stream=None, comm_stream=None):
    """ring_attn_fwd with the ring's K/V exchange done as device copies on
    `comm_stream`, overlapped with each step's attention (sharded order).
    comm_stream None: each step's launch copies the next step's blocks itself
    (no copy calls, no events)."""
    import torch
    B, H, S, d = q.shape
    need = ring_attn_fwd_overlap_workspace(B, H, S, d, P)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    comm = _stream(comm_stream) if comm_stream is not None else None
    _check(lib().ring_attn_fwd_overlap(_dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"),
                                       _dev(v, torch.bfloat16, "v"),
                                       _dev(out, torch.bfloat16, "out"),
                                       _dev(lse, torch.float32, "lse"), B, H, S, d, P, int(causal),
                                       _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                                       _stream(stream), comm), "ring_attn_fwd_overlap")
    return out, lse


def ring_attn_bwd_workspace(B: int, H: int, S: int) -> int:
    return int(lib().ring_attn_bwd_workspace(B, H, S))


def ring_attn_bwd(q, k, v, out, lse, dout, P: int, causal: bool = False, workspace=None,
                  grads=None, stream=None):
    """Gradients (dq, dk, dv) of ring_attn_fwd for upstream gradient dout
    (all [B,H,S,d] bf16, sharded order; lse fp32 [B,H,S] from the forward)."""
    import torch
    B, H, S, d = q.shape
    need = ring_attn_bwd_workspace(B, H, S)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    dq, dk, dv = grads if grads is not None else (torch.empty_like(q), torch.empty_like(k),
                                                  torch.empty_like(v))
    bf = torch.bfloat16
    _check(lib().ring_attn_bwd(_dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"),
                               _dev(out, bf, "out"), _dev(lse, torch.float32, "lse"),
                               _dev(dout, bf, "dout"), _dev(dq, bf, "dq"), _dev(dk, bf, "dk"),
                               _dev(dv, bf, "dv"), B, H, S, d, P, int(causal),
                               _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                               _stream(stream)), "ring_attn_bwd")
    return dq, dk, dv


def ra_ulysses_a2a(x, B: int, H: int, S: int, P: int, inverse: bool = False, out=None,
                   stream=None):
    """Ulysses all-to-all: sequence-split [P,B,H,S/P,d] <-> head-split [P,B,H/P,S,d]."""
    import torch
    d = x.shape[-1]
    shape = (P, B, H, S // P, d) if inverse else (P, B, H // P, S, d)
    y = torch.empty(shape, dtype=x.dtype, device=x.device) if out is None else out
    _check(lib().ra_ulysses_a2a(_dev(x, torch.bfloat16, "x"), _dev(y, torch.bfloat16, "out"), B, H,
                                S, d, P, int(inverse), _stream(stream)), "ra_ulysses_a2a")
    return y


def ulysses_attn_workspace(B: int, H: int, S: int, d: int) -> int:
    return int(lib().ulysses_attn_workspace(B, H, S, d))


def ulysses_attn_fwd(q, k, v, B: int, H: int, S: int, P: int, causal: bool = False,
                     workspace=None, out=None, lse=None, stream=None):
    """Attention with Ulysses parallelism; q/k/v sequence-split [P,B,H,S/P,d] bf16.
    Returns out (same layout) and lse [P,B,H,S/P]."""
    import torch
    d = q.shape[-1]
    need = ulysses_attn_workspace(B, H, S, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib().ulysses_attn_fwd(_dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"),
                                  _dev(v, torch.bfloat16, "v"), _dev(out, torch.bfloat16, "out"),
                                  _dev(lse, torch.float32, "lse"), B, H, S, d, P, int(causal),
                                  _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                                  _stream(stream)), "ulysses_attn_fwd")
    return out, lse


def cp_variant_workspace(B: int, H: int, S: int, d: int, P: int) -> int:
    return int(lib().cp_variant_workspace(B, H, S, d, P))


def _cp_variant(fn, name, q, k, v, B, H, S, P, causal, workspace, out, lse, stream):
    import torch
    d = q.shape[-1]
    need = cp_variant_workspace(B, H, S, d, P)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device) if lse is None else lse
    _check(fn(_dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"),
              _dev(v, torch.bfloat16, "v"), _dev(out, torch.bfloat16, "out"),
              _dev(lse, torch.float32, "lse"), B, H, S, d, P, int(causal),
              _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)), name)
    return out, lse


def cp_allgather_attn_fwd(q, k, v, B: int, H: int, S: int, P: int, causal: bool = False,
                          workspace=None, out=None, lse=None, stream=None):
    """All-gather form: per-rank buffers [P,B,H,S/P,d]; K/V gathered, then local attention."""
    return _cp_variant(lib().cp_allgather_attn_fwd, "cp_allgather_attn_fwd", q, k, v, B, H, S, P,
                       causal, workspace, out, lse, stream)


def cp_reducescatter_attn_fwd(q, k, v, B: int, H: int, S: int, P: int, causal: bool = False,
                              workspace=None, out=None, lse=None, stream=None):
    """Reduce-scatter form: per-rank buffers; per-block partials merged per query."""
    return _cp_variant(lib().cp_reducescatter_attn_fwd, "cp_reducescatter_attn_fwd", q, k, v, B,
                       H, S, P, causal, workspace, out, lse, stream)


def lse_merge(o_parts, lse_parts, out=None, lse_out=None, stream=None):
    """Merge n fp32 partials [n, ..., d] / [n, ...] into bf16 out and fp32 lse."""
    import torch
    n, d = o_parts.shape[0], o_parts.shape[-1]
    rows = o_parts[0].numel() // d
    out = torch.empty(o_parts.shape[1:], dtype=torch.bfloat16, device=o_parts.device) \
        if out is None else out
    lse_out = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device) \
        if lse_out is None else lse_out
    _check(lib().lse_merge(_dev(o_parts, torch.float32, "o_parts"),
                           _dev(lse_parts, torch.float32, "lse_parts"), n, rows, d,
                           _dev(out, torch.bfloat16, "out"), _dev(lse_out, torch.float32, "lse_out"),
                           _stream(stream)), "lse_merge")
    return out, lse_out


def factored_attn_workspace(B: int, H: int, T: int, N: int, d: int) -> int:
    return int(lib().factored_attn_workspace(B, H, T, N, d))


def factored_attn(q, k, v, T: int, N: int, P: int, workspace=None, outs=None, stream=None):
    """Spatial (within frame) and temporal (across frames, ring over P) attention.

    Returns (out_s, lse_s, out_t, lse_t).  workspace: uint8 CUDA tensor of at
    least factored_attn_workspace(...) bytes, needed only when the rank chunks
    exceed 128 frames (T / P > 128; allocated here if None).
    """
    import torch
    B, H, S, d = q.shape
    chunks_fit = P > 0 and T % P == 0 and T // P <= 128
    need = 0 if chunks_fit else factored_attn_workspace(B, H, T, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if outs is None:
        outs = (torch.empty_like(q), torch.empty((B, H, S), dtype=torch.float32, device=q.device),
                torch.empty_like(q), torch.empty((B, H, S), dtype=torch.float32, device=q.device))
    out_s, lse_s, out_t, lse_t = outs
    _check(lib().factored_attn(_dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"),
                               _dev(v, torch.bfloat16, "v"), _dev(out_s, torch.bfloat16, "out_s"),
                               _dev(lse_s, torch.float32, "lse_s"),
                               _dev(out_t, torch.bfloat16, "out_t"),
                               _dev(lse_t, torch.float32, "lse_t"), B, H, T, N, d, P,
                               _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                               _stream(stream)), "factored_attn")
    return out_s, lse_s, out_t, lse_t


def factored_attn_static(q, k, v, T: int, N: int, P: int, outs, stream=None):
    """factored_attn working in the library's fixed device scratch (no workspace
    argument, no device allocation by the library).  `outs` = (out_s, lse_s,
    out_t, lse_t), caller-allocated like factored_attn's outputs."""
    import torch
    B, H, S, d = q.shape
    out_s, lse_s, out_t, lse_t = outs
    _check(lib().factored_attn_static(_dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"),
                                      _dev(v, torch.bfloat16, "v"),
                                      _dev(out_s, torch.bfloat16, "out_s"),
                                      _dev(lse_s, torch.float32, "lse_s"),
                                      _dev(out_t, torch.bfloat16, "out_t"),
                                      _dev(lse_t, torch.float32, "lse_t"), B, H, T, N, d, P,
                                      _stream(stream)), "factored_attn_static")
    return out_s, lse_s, out_t, lse_t


def ra_get_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status code."""
    return int(lib().ra_get_status(_stream(stream)))


def ra_set_watchdog_ns(ns: int):
    lib().ra_set_watchdog_ns(int(ns))


def ra_set_temporal_fold(enable: bool):
    """Fold short adjacent temporal chunks into fewer ring blocks (default on)."""
    lib().ra_set_temporal_fold(int(bool(enable)))


def ra_watchdog_selftest(stream=None):
    _check(lib().ra_watchdog_selftest(_stream(stream)), "ra_watchdog_selftest")


def ra_checks_enabled() -> bool:
    """True when the loaded library was built with the device bounds checks."""
    return bool(lib().ra_checks_enabled())


def ra_checks_selftest(stream=None):
    _check(lib().ra_checks_selftest(_stream(stream)), "ra_checks_selftest")
