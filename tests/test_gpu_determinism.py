"""Repeated calls give bit-identical results: every kernel folds its tiles in
a fixed order and the persistent walks are static, so any difference between
two runs on the same inputs would mean a race (a barrier phase miscounted, a
buffer reused too early)."""
import pytest
import torch

import ring_attention_attn_gb300 as ra

pytestmark = pytest.mark.gpu

REPEATS = 6


def _rnd(g, *shape):
    return torch.randn(*shape, device="cuda", generator=g).bfloat16()


def _same_every_time(fn):
    ref = [x.clone() for x in fn()]
    for _ in range(REPEATS):
        got = fn()
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0


def test_factored_persistent_passes_are_deterministic():
    g = torch.Generator(device="cuda").manual_seed(5)
    q, k, v = (_rnd(g, 1, 8, 24 * 900, 128) for _ in range(3))
    _same_every_time(lambda: ra.factored_attn(q, k, v, 24, 900, 2))


def test_persistent_causal_partials_are_deterministic():
    g = torch.Generator(device="cuda").manual_seed(6)
    q = _rnd(g, 1, 40, 512, 128)
    k, v = _rnd(g, 1, 40, 4096, 128), _rnd(g, 1, 40, 4096, 128)
    _same_every_time(lambda: ra.ring_attn_fwd_rank(q, k, v, 8, 0, causal=True, out_fp32=True))


def test_overlapped_ring_and_backward_are_deterministic():
    g = torch.Generator(device="cuda").manual_seed(7)
    B, H, S, d, P = 1, 8, 4096, 128, 4
    q, k, v, do = (_rnd(g, B, H, S, d) for _ in range(4))
    ws = torch.empty(ra.ring_attn_fwd_overlap_workspace(B, H, S, d, P), dtype=torch.uint8,
                     device="cuda")
    comm = torch.cuda.Stream()
    _same_every_time(lambda: ra.ring_attn_fwd_overlap(q, k, v, P, workspace=ws, comm_stream=comm))
    # the exchange inside the step launches: a block copied while the same
    # launch reads the other buffer
    _same_every_time(lambda: ra.ring_attn_fwd_overlap(q, k, v, P, workspace=ws))
    o, lse = ra.ring_attn_fwd(q, k, v, P)
    _same_every_time(lambda: ra.ring_attn_bwd(q, k, v, o, lse, do, P))


@pytest.mark.parametrize("B,H,S,d,P,causal", [(1, 8, 4096, 128, 4, False), (1, 4, 4096, 64, 2, True),
                                              (2, 3, 1320, 128, 5, False)])
def test_overlap_exchange_forms_are_bit_identical(B, H, S, d, P, causal):
    """The ring sends done by the step launches and the same sends as device
    copies on a comm stream move identical bytes into identical buffers, and
    the step launches compute the same partials: the outputs must agree bit
    for bit (a copy landing late or in the wrong place would show)."""
    g = torch.Generator(device="cuda").manual_seed(11 + P)
    q, k, v = (_rnd(g, B, H, S, d) for _ in range(3))
    if causal:
        q, k, v = (ra.ra_cp_shard(x, P, 1) for x in (q, k, v))
    o1, l1 = ra.ring_attn_fwd_overlap(q, k, v, P, causal=causal, comm_stream=torch.cuda.Stream())
    o2, l2 = ra.ring_attn_fwd_overlap(q, k, v, P, causal=causal)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal,d,H,S", [(True, 64, 4, 4096), (False, 128, 4, 4096),
                                         (True, 64, 18, 2048), (False, 128, 18, 2048)])
def test_split_units_are_deterministic(causal, d, H, S):
    """Launches of fewer query-tile pairs than SMs run as split units (the two
    softmax warpgroups alternate key tiles and merge through shared memory):
    the exchange and the "both accumulators read" barrier must leave no race.
    With at most as many split units as SMs (H = 4) each runs on a CTA pair,
    whose second CTA hands its state over in the first CTA's K/V slots: the
    two barriers of that hand-over must leave none either."""
    g = torch.Generator(device="cuda").manual_seed(8 + d + H)
    q, k, v = (_rnd(g, 1, H, S, d) for _ in range(3))
    if causal:
        q, k, v = (ra.ra_cp_shard(x, 2, 1) for x in (q, k, v))
    _same_every_time(lambda: ra.ring_attn_fwd(q, k, v, 2, causal=causal))
