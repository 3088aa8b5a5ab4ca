"""GB300-native (sm_103a) ring attention hot path for context parallelism.

The compute runs in libringattn.so (hand-written CUDA: tcgen05/TMEM/TMA
attention kernel, coalesced permutation and merge kernels); this package is
its thin Python binding plus host-side FLOP/byte accounting.
"""
from . import accounting  # noqa: F401
from ._abi import (  # noqa: F401
    EXPORTS,
    RingAttnError,
    cp_allgather_attn_fwd,
    cp_reducescatter_attn_fwd,
    cp_variant_workspace,
    factored_attn,
    factored_attn_static,
    factored_attn_workspace,
    lib,
    lse_merge,
    ra_cp_shard,
    ra_cp_shard_index,
    ra_frame_transpose,
    ra_get_status,
    ra_ring_source,
    ra_set_watchdog_ns,
    ra_set_temporal_fold,
    ra_ulysses_a2a,
    ra_watchdog_selftest,
    ra_checks_enabled,
    ra_checks_selftest,
    ring_attn_fwd,
    ring_attn_bwd,
    ring_attn_bwd_workspace,
    ring_attn_fwd_overlap,
    ring_attn_fwd_overlap_workspace,
    ring_attn_fwd_rank,
    ulysses_attn_fwd,
    ulysses_attn_workspace,
)
