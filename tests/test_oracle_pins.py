"""Pins for the fp64 oracle: checks against facts the pages and mathematics fix.

None of these compares the oracle with itself: each one checks it against an
independent restatement (pure-Python brute force, a torch float64 softmax,
closed forms, invariants the pages state, exact special cases).
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import brute

TOL = 1e-12


def _np(t):
    return t.double().numpy()


# 1. Brute force on tiny shapes -------------------------------------------------
@pytest.mark.parametrize("S", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("d", [4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(S, d, causal):
    q, k, v = synth.make_custom((1, 2, S, d), (1, 2, S, d), seed=100 + 10 * S + d)
    o, lse = oracle.attention(q, k, v, causal=causal)
    for h in range(2):
        O, L = brute.attention(q[0, h].float().tolist(), k[0, h].float().tolist(),
                               v[0, h].float().tolist(), causal)
        assert np.max(np.abs(o[0, h] - np.array(O))) <= TOL
        assert np.max(np.abs(lse[0, h] - np.array(L))) <= TOL


def test_brute_force_rectangular_offset():
    """Queries at a global offset against a longer key sequence (causal)."""
    q, k, v = synth.make_custom((1, 1, 5, 4), (1, 1, 12, 4), seed=7)
    off = 6
    o, lse = oracle.attention(q, k, v, causal=True, q_offset=off)
    K, V = k[0, 0].float().tolist(), v[0, 0].float().tolist()
    for i in range(5):
        n = off + i + 1
        O, L = brute.attention([q[0, 0, i].float().tolist()], K[:n], V[:n], causal=False)
        assert np.max(np.abs(o[0, 0, i] - np.array(O[0]))) <= TOL
        assert abs(lse[0, 0, i] - L[0]) <= TOL


# 2. Ring equals full attention (ultralytics glossary; day 83 blog) ---------------
@pytest.mark.parametrize("P", [1, 2, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [48, 64])
def test_ring_equals_full(P, causal, S):
    q, k, v = synth.make_custom((1, 2, S, 16), (1, 2, S, 16), seed=200 + P + S)
    of, lf = oracle.attention(q, k, v, causal=causal)
    orr, lr = oracle.ring_attention(q, k, v, P, causal=causal)
    assert np.max(np.abs(of - orr)) <= TOL
    assert np.max(np.abs(lf - lr)) <= TOL


# 3. Chunked online-softmax merge equals one-shot softmax (day 83 blog) ------------
@pytest.mark.parametrize("causal", [False, True])
def test_chunked_merge_equals_one_shot(causal):
    S, d = 40, 8
    q, k, v = synth.make_custom((1, 1, S, d), (1, 1, S, d), seed=300)
    of, lf = oracle.attention(q, k, v, causal=causal)
    bounds = [0, 1, 8, 8, 20, 21, 40]  # chunk sizes 1, 7, 0 (empty), 12, 1, 19
    os_, ls_ = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        o_i, l_i = oracle.attention(q, k[:, :, a:b], v[:, :, a:b], causal=causal, q_offset=-a)
        os_.append(o_i[0, 0])
        ls_.append(l_i[0, 0])
    assert np.all(np.isneginf(ls_[2]))  # the empty chunk
    if causal:
        assert np.isneginf(ls_[3][0])  # row 0 sees nothing in keys [8, 20)
    om, lm = oracle.lse_merge(np.stack(os_), np.stack(ls_))
    assert np.max(np.abs(om - of[0, 0])) <= TOL
    assert np.max(np.abs(lm - lf[0, 0])) <= TOL


def test_merge_all_empty_and_single():
    o = np.zeros((3, 4, 5))
    lse = np.full((3, 4), -np.inf)
    om, lm = oracle.lse_merge(o, lse)
    assert np.all(om == 0.0) and np.all(np.isneginf(lm))
    rng = np.random.default_rng(1)
    o1 = rng.standard_normal((1, 6, 5))
    l1 = rng.standard_normal((1, 6))
    om, lm = oracle.lse_merge(o1, l1)
    assert np.max(np.abs(om - o1[0])) <= TOL and np.max(np.abs(lm - l1[0])) <= TOL


def test_merge_closed_form_two_parts():
    """Two partials with equal LSE: output is their mean, LSE rises by ln 2."""
    rng = np.random.default_rng(2)
    o = rng.standard_normal((2, 3, 4))
    l = np.tile(rng.standard_normal(3), (2, 1))
    om, lm = oracle.lse_merge(o, l)
    assert np.max(np.abs(om - o.mean(0))) <= TOL
    assert np.max(np.abs(lm - (l[0] + math.log(2)))) <= TOL


# 4. Order invariance of the non-causal ring -------------------------------------
def test_order_invariance_all_permutations():
    P, S = 4, 32
    q, k, v = synth.make_custom((1, 1, S, 8), (1, 1, S, 8), seed=400)
    base_o, base_l = oracle.ring_attention(q, k, v, P)
    for perm in itertools.permutations(range(P)):
        order = [[(perm[s] + r) % P for s in range(P)] for r in range(P)]
        o, l = oracle.ring_attention(q, k, v, P, order=order)
        assert np.max(np.abs(o - base_o)) <= TOL
        assert np.max(np.abs(l - base_l)) <= TOL


# 5. Q = 0 closed form ---------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_mean_of_values(causal):
    S, d = 24, 8
    _, k, v = synth.make_custom((1, 2, S, d), (1, 2, S, d), seed=500)
    q = torch.zeros((1, 2, S, d), dtype=torch.bfloat16)
    o, lse = oracle.attention(q, k, v, causal=causal)
    V = _np(v)
    for i in range(S):
        n = i + 1 if causal else S
        assert np.max(np.abs(o[0, :, i] - V[0, :, :n].mean(axis=1))) <= TOL
        assert np.max(np.abs(lse[0, :, i] - math.log(n))) <= TOL


# 6. Special cases ----------------------------------------------------------------
def test_causal_row_zero():
    q, k, v = synth.make_custom((1, 3, 16, 8), (1, 3, 16, 8), seed=600)
    o, lse = oracle.attention(q, k, v, causal=True)
    Q, K, V = _np(q), _np(k), _np(v)
    assert np.max(np.abs(o[0, :, 0] - V[0, :, 0])) <= TOL
    expect = (Q[0, :, 0] * K[0, :, 0]).sum(-1) / math.sqrt(8)
    assert np.max(np.abs(lse[0, :, 0] - expect)) <= TOL


def test_values_all_ones():
    q, k, _ = synth.make_custom((1, 2, 20, 8), (1, 2, 20, 8), seed=601)
    v = torch.ones((1, 2, 20, 8), dtype=torch.bfloat16)
    for causal in (False, True):
        o, _ = oracle.attention(q, k, v, causal=causal)
        assert np.max(np.abs(o - 1.0)) <= TOL


def test_duplicated_keys_raise_lse_by_ln2():
    q, k, v = synth.make_custom((1, 2, 12, 8), (1, 2, 12, 8), seed=602)
    o1, l1 = oracle.attention(q, k, v)
    o2, l2 = oracle.attention(q, torch.cat([k, k], 2), torch.cat([v, v], 2))
    assert np.max(np.abs(o1 - o2)) <= TOL
    assert np.max(np.abs(l2 - l1 - math.log(2))) <= TOL


@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_float64_softmax(causal):
    """Cross-check with a library routine (torch float64 softmax/logsumexp)."""
    S, d = 512, 64
    q, k, v = synth.make_custom((1, 2, S, d), (1, 2, S, d), seed=603)
    o, lse = oracle.attention(q, k, v, causal=causal)
    Q, K, V = q.double(), k.double(), v.double()
    s = Q @ K.transpose(-1, -2) / math.sqrt(d)
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(S, S, dtype=torch.bool), 1), float("-inf"))
    ref_o = torch.softmax(s, -1) @ V
    ref_l = torch.logsumexp(s, -1)
    assert np.max(np.abs(o - ref_o.numpy())) <= 1e-12
    assert np.max(np.abs(lse - ref_l.numpy())) <= 1e-12


def test_ring_with_one_rank_is_plain_attention():
    q, k, v = synth.make_custom((1, 2, 30, 8), (1, 2, 30, 8), seed=604)
    o1, l1 = oracle.ring_attention(q, k, v, 1)
    o2, l2 = oracle.attention(q, k, v)
    assert np.max(np.abs(o1 - o2)) <= TOL and np.max(np.abs(l1 - l2)) <= TOL


def test_sampled_rows_match_full_rows():
    q, k, v = synth.make_custom((1, 2, 40, 8), (1, 2, 40, 8), seed=605)
    of, lf = oracle.attention(q, k, v, causal=True)
    rows = oracle.flat_rows(1, 2, 40, [0, 7, 39])
    o, l = oracle.attention(q, k, v, causal=True, rows=rows)
    assert np.array_equal(o, of.reshape(-1, 8)[rows])
    assert np.array_equal(l, lf.reshape(-1)[rows])


# 7. Shard maps (day 83 blog contiguous split; k8ai balanced causal split) --------
def test_zigzag_tiny_map():
    s2g, g2s = oracle.shard_index(8, 2, 1)
    # C = 2: rank 0 holds chunks 0 and 3, rank 1 holds chunks 1 and 2
    assert s2g.tolist() == [0, 1, 6, 7, 2, 3, 4, 5]
    assert g2s.tolist() == [0, 1, 4, 5, 6, 7, 2, 3]
    s2g, _ = oracle.shard_index(8, 2, 0)
    assert s2g.tolist() == list(range(8))


@pytest.mark.parametrize("S,P", [(4096, 2), (48, 4), (64, 8), (16, 8)])
def test_zigzag_is_a_permutation_with_two_chunks_per_rank(S, P):
    s2g, g2s = oracle.shard_index(S, P, 1)
    assert sorted(s2g.tolist()) == list(range(S))
    assert np.array_equal(g2s[s2g], np.arange(S))
    C, L = S // (2 * P), S // P
    for r in range(P):
        mine = s2g[r * L:(r + 1) * L]
        assert mine[:C].tolist() == list(range(r * C, (r + 1) * C))
        c2 = 2 * P - 1 - r
        assert mine[C:].tolist() == list(range(c2 * C, (c2 + 1) * C))


def test_zigzag_balances_causal_work():
    S, P = 4096, 2
    L = S // P
    for layout, expect in ((1, [4195328, 4195328]), (0, [2098176, 6292480])):
        s2g, _ = oracle.shard_index(S, P, layout)
        pairs = [int((s2g[r * L:(r + 1) * L] + 1).sum()) for r in range(P)]
        assert pairs == expect


def test_shard_index_rejects_bad_sizes():
    with pytest.raises(ValueError):
        oracle.shard_index(10, 4, 0)
    with pytest.raises(ValueError):
        oracle.shard_index(12, 4, 1)


# 8. Factored attention locality (day 83 blog, "The spatial-temporal twist") ------
def test_factored_spatial_is_local_to_frame():
    T, N, d = 6, 10, 8
    q, k, v = synth.make_custom((1, 2, T * N, d), (1, 2, T * N, d), seed=800)
    o, l = oracle.factored(q, k, v, T, N, "spatial")
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 3 * N:] = k2[:, :, 3 * N:] * -2
    v2[:, :, 3 * N:] = v2[:, :, 3 * N:] + 1
    o2, l2 = oracle.factored(q, k2, v2, T, N, "spatial")
    assert np.array_equal(o[:, :, :3 * N], o2[:, :, :3 * N])
    assert np.array_equal(l[:, :, :3 * N], l2[:, :, :3 * N])
    assert not np.array_equal(o[:, :, 3 * N:], o2[:, :, 3 * N:])
    # each frame on its own is plain attention
    for t in range(T):
        sl = slice(t * N, (t + 1) * N)
        of, lf = oracle.attention(q[:, :, sl], k[:, :, sl], v[:, :, sl])
        assert np.max(np.abs(of - o[:, :, sl])) <= TOL
        assert np.max(np.abs(lf - l[:, :, sl])) <= TOL


def test_factored_temporal_across_frames():
    T, N, d = 8, 5, 8
    q, k, v = synth.make_custom((1, 2, T * N, d), (1, 2, T * N, d), seed=801)
    o, l = oracle.factored(q, k, v, T, N, "temporal")
    # temporal attention at position n = plain attention over the frames' tokens n
    tr = lambda x: x.reshape(1, 2, T, N, d).transpose(2, 3).contiguous()  # [B,H,N,T,d]
    qt, kt, vt = (tr(x).reshape(1, 2 * N, T, d) for x in (q, k, v))
    ot, lt = oracle.attention(qt, kt, vt)
    ot = ot.reshape(1, 2, N, T, d).transpose(0, 1, 3, 2, 4)
    lt = lt.reshape(1, 2, N, T).transpose(0, 1, 3, 2)
    assert np.max(np.abs(ot.reshape(1, 2, T * N, d) - o)) <= TOL
    assert np.max(np.abs(lt.reshape(1, 2, T * N) - l)) <= TOL
    # ... and as a ring over P = 4 chunks of frames
    orr, lr = oracle.ring_attention(qt, kt, vt, 4)
    assert np.max(np.abs(orr.reshape(1, 2, N, T, d).transpose(0, 1, 3, 2, 4).reshape(1, 2, T * N, d) - o)) <= TOL
    # perturbing another spatial position leaves position 0 untouched
    k2 = k.clone().reshape(1, 2, T, N, d)
    k2[..., 1:, :] *= 3
    o2, _ = oracle.factored(q, k2.reshape(1, 2, T * N, d), v, T, N, "temporal")
    pos0 = np.arange(T) * N
    assert np.array_equal(o[:, :, pos0], o2[:, :, pos0])
