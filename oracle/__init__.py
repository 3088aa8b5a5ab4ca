"""fp64 CPU oracle for ring attention: TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference legs import this package.  It shares no code with the CUDA path and
is never called by it.  Each function below restates a definition from the
pages on context parallelism; the arithmetic lives in ``attn_ref.c`` (plain
fp64 loops, OpenMP over query rows) and, for tiny shapes, in ``brute.py``
(pure Python).

Citations (page title, section):
  * full attention is the target of the ring method -- ultralytics glossary
    "Context Parallelism", "How Context Parallelism Works" (the ring's answer
    is exact full attention);
  * ring schedule and online-softmax accumulation -- "day 83" blog, "Context
    parallelism: splitting the sequence"; k8ai "Sequence and Context
    Parallel", "How context parallel works" (ring diagram);
  * balanced causal chunking -- k8ai, "How context parallel works", read as
    zigzag (2P chunks, rank r holds chunks r and 2P-1-r);
  * factored spatial / temporal attention -- "day 83" blog, "The
    spatial-temporal twist";
  * the backward pass (the ring's exchanges recur in the backward pass of
    every attention layer, k8ai "Communication profile"; the glossary's
    example calls .backward()) -- the gradients of the full-attention
    definition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, fp64, OpenMP) into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def configure(lib):
    """Declare the C signatures on a loaded oracle library (also used by the
    mutation tests, which load deliberately broken copies of the oracle)."""
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.oracle_threads.restype = i32
    lib.oracle_shard_index.argtypes = [i64, i64, i32, vp, vp]
    lib.oracle_attention.argtypes = [vp, vp, vp, i64, i64, i64, i64, i32, i64, vp, i64, vp, vp]
    lib.oracle_factored.argtypes = [vp, vp, vp, i64, i64, i64, i64, i32, vp, i64, vp, vp]
    lib.oracle_ring_attention.argtypes = [vp, vp, vp, i64, i64, i64, i64, i32, vp, vp, i64, vp,
                                          vp]
    lib.oracle_lse_merge.argtypes = [vp, vp, i64, i64, i64, vp, vp]
    lib.oracle_attention_bwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, vp, vp, vp]
    lib.oracle_attention_bwd.restype = i32
    lib.oracle_ring_source.argtypes = [i64, i64, i64]
    lib.oracle_ring_source.restype = i64
    for f in ("oracle_shard_index", "oracle_attention", "oracle_factored",
              "oracle_ring_attention", "oracle_lse_merge"):
        getattr(lib, f).restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = configure(ctypes.CDLL(build()))
    return _lib


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().oracle_threads())


def _bits(x) -> np.ndarray:
    """bf16 tensor (torch) or uint16 array -> contiguous uint16 bit patterns."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16, x.dtype
    return x.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, int(r.size)


def shard_index(S: int, P: int, layout: int):
    """(s2g, g2s) int64 maps for layout 0 = contiguous, 1 = zigzag."""
    s2g = np.empty(max(S, 1), dtype=np.int64)
    g2s = np.empty(max(S, 1), dtype=np.int64)
    rc = _load().oracle_shard_index(S, P, layout, _ptr(s2g), _ptr(g2s))
    if rc != 0:
        raise ValueError(f"bad shard arguments S={S} P={P} layout={layout}")
    return s2g[:S], g2s[:S]


def ring_source(P: int, r: int, s: int) -> int:
    """KV block that rank r holds at ring step s."""
    return int(_load().oracle_ring_source(P, r, s))


def flat_rows(B: int, H: int, S: int, per_head_rows) -> np.ndarray:
    """Flat row indices bh*S + i for the same per-head rows in every head."""
    per = np.asarray(per_head_rows, dtype=np.int64)
    return (np.arange(B * H, dtype=np.int64)[:, None] * S + per[None, :]).reshape(-1)


def attention(q, k, v, causal: bool = False, q_offset: int = 0, rows=None):
    """Full softmax attention in fp64 (the definition).

    q: [B,H,Sq,d] bf16, k/v: [B,H,Skv,d] bf16, global order; query i sits at
    global position q_offset + i.  Returns (o, lse): [B,H,Sq,d], [B,H,Sq]
    float64 for all rows, or [n,d], [n] for the flat rows given.
    """
    B, H, Sq, d = q.shape
    Skv = k.shape[2]
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    r, n = _rows(rows)
    n_out = n if r is not None else B * H * Sq
    o = np.empty((max(n_out, 1), d))
    lse = np.empty(max(n_out, 1))
    rc = _load().oracle_attention(_ptr(qb), _ptr(kb), _ptr(vb), B * H, Sq, Skv, d, int(causal),
                                  q_offset, _ptr(r) if r is not None else None, n, _ptr(o),
                                  _ptr(lse))
    if rc != 0:
        raise MemoryError("oracle_attention failed")
    o, lse = o[:n_out], lse[:n_out]
    if r is None:
        return o.reshape(B, H, Sq, d), lse.reshape(B, H, Sq)
    return o, lse


def factored(q, k, v, T: int, N: int, which: str, rows=None):
    """Factored video attention: which='spatial' (within a frame) or 'temporal'.

    q/k/v: [B,H,T*N,d] bf16, token index t*N + n.
    """
    B, H, S, d = q.shape
    assert S == T * N
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    r, n = _rows(rows)
    n_out = n if r is not None else B * H * S
    o = np.empty((max(n_out, 1), d))
    lse = np.empty(max(n_out, 1))
    w = {"spatial": 0, "temporal": 1}[which]
    _load().oracle_factored(_ptr(qb), _ptr(kb), _ptr(vb), B * H, T, N, d, w,
                            _ptr(r) if r is not None else None, n, _ptr(o), _ptr(lse))
    o, lse = o[:n_out], lse[:n_out]
    if r is None:
        return o.reshape(B, H, S, d), lse.reshape(B, H, S)
    return o, lse


def ring_attention(q, k, v, P: int, causal: bool = False, order=None, rows=None):
    """Ring attention, step by step with the online-softmax fold (fp64).

    Global-order q/k/v [B,H,S,d]; causal implies the zigzag layout.  order:
    optional [P][P] int table (block visited by rank r at step s).
    """
    B, H, S, d = q.shape
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    r, n = _rows(rows)
    n_out = n if r is not None else B * H * S
    o = np.empty((max(n_out, 1), d))
    lse = np.empty(max(n_out, 1))
    ordr = None
    if order is not None:
        ordr = np.ascontiguousarray(np.asarray(order, dtype=np.int64).reshape(P, P))
    rc = _load().oracle_ring_attention(_ptr(qb), _ptr(kb), _ptr(vb), B * H, S, d, P,
                                       int(causal), _ptr(ordr) if ordr is not None else None,
                                       _ptr(r) if r is not None else None, n, _ptr(o),
                                       _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_ring_attention: bad arguments")
    o, lse = o[:n_out], lse[:n_out]
    if r is None:
        return o.reshape(B, H, S, d), lse.reshape(B, H, S)
    return o, lse


def attention_bwd(q, k, v, dout, causal: bool = False):
    """fp64 gradients (dq, dk, dv) of full attention for upstream gradient dout.

    q, k, v, dout: [B,H,S,d] bf16 in global order; returns float64 arrays of
    the same shape.
    """
    B, H, S, d = q.shape
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    dq = np.empty((B, H, S, d))
    dk = np.empty((B, H, S, d))
    dv = np.empty((B, H, S, d))
    rc = _load().oracle_attention_bwd(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), B * H, S, d,
                                      int(causal), _ptr(dq), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise MemoryError("oracle_attention_bwd failed")
    return dq, dk, dv


def lse_merge(o_parts, lse_parts):
    """Merge n normalised partials: o_parts [n,rows,d], lse_parts [n,rows] -> (o, lse)."""
    op = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    lp = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64))
    n, rows, d = op.shape
    o = np.empty((max(rows, 1), d))
    lse = np.empty(max(rows, 1))
    _load().oracle_lse_merge(_ptr(op), _ptr(lp), n, rows, d, _ptr(o), _ptr(lse))
    return o[:rows], lse[:rows]
