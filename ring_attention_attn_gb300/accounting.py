"""Algorithmic FLOP and byte counts for the ring-attention hot path.

Host-side arithmetic used by the benchmark's roofline figures and pinned, in
the tests, to the numbers the pages print for their worked examples ("day 83"
blog, "What the numbers look like" and "The communication pattern"; the
ultralytics glossary, "How Context Parallelism Works").

Conventions: an attention score costs 2*d FLOPs for q.k and 2*d for p.v, so
4*d FLOPs per visible (query, key) pair; only visible pairs count (causal
masks halve the work, padded tile work is never counted).
"""
from __future__ import annotations


def tokens(frames: int, per_frame: int) -> int:
    """Video tokens: frames x spatial tokens per frame (frame-major order)."""
    return frames * per_frame


def spatial_tokens(height: int, width: int, downsample: int) -> int:
    """Latent tokens of one frame after `downsample`x spatial reduction."""
    return (height // downsample) * (width // downsample)


def per_rank(S: int, P: int) -> int:
    """Tokens each of P ranks holds when S tokens are split along the sequence."""
    return S // P


def scores_per_head(S: int) -> int:
    """Entries of the full S x S attention matrix of one head."""
    return S * S


def attn_matrix_bytes(S: int, elem_bytes: int = 2) -> int:
    """Bytes of a materialised S x S score matrix of one head."""
    return S * S * elem_bytes


def kv_bytes_per_step(L: int, d: int, heads: int = 1, elem_bytes: int = 2) -> int:
    """K and V bytes one rank sends per ring step: 2 tensors of L x d per head."""
    return 2 * L * d * elem_bytes * heads


def ring_pass_bytes(L: int, d: int, heads: int, P: int, elem_bytes: int = 2) -> int:
    """KV bytes one rank sends over a full ring pass (P - 1 steps)."""
    return kv_bytes_per_step(L, d, heads, elem_bytes) * (P - 1)


def transfer_seconds(n_bytes: float, gb_per_s: float) -> float:
    return n_bytes / (gb_per_s * 1e9)


def causal_pairs(S: int) -> int:
    """Visible (query, key) pairs of a causal S-token sequence: S(S+1)/2."""
    return S * (S + 1) // 2


def attention_flops(BH: int, Sq: int, Skv: int, d: int, causal: bool = False) -> int:
    """FLOPs of softmax attention (4*d per visible score).  For causal the
    query and key sets are the same S tokens."""
    if causal:
        assert Sq == Skv
        return 4 * d * BH * causal_pairs(Sq)
    return 4 * d * BH * Sq * Skv


def factored_flops(BH: int, T: int, N: int, d: int):
    """(spatial, temporal) FLOPs of factored video attention."""
    spatial = 4 * d * BH * T * N * N
    temporal = 4 * d * BH * N * T * T
    return spatial, temporal


def attention_io_bytes(BH: int, Sq: int, Skv: int, d: int, out_bytes: int = 2) -> int:
    """Compulsory HBM bytes of one attention call: q, k, v read once (bf16),
    out written once (`out_bytes` per element) and an fp32 LSE per query."""
    return BH * (Sq * d * 2 + 2 * Skv * d * 2 + Sq * d * out_bytes + Sq * 4)


def merge_bytes(n: int, rows: int, d: int) -> int:
    """Compulsory HBM bytes of lse_merge: n fp32 partials (O and LSE) read,
    bf16 O and fp32 LSE written."""
    return n * rows * d * 4 + n * rows * 4 + rows * d * 2 + rows * 4


def shard_bytes(BH: int, S: int, d: int) -> int:
    """A bf16 row permutation reads and writes every element once."""
    return 2 * BH * S * d * 2
