"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances: max |O_gpu - O_ref| <= 1e-2 and max |LSE_gpu - LSE_ref| <= 1e-3
(bf16 inputs, fp32 accumulation, bf16 output); index maps and permutations
bit-exact.  Outputs are un-sharded with the oracle's own index map before
comparison, so the check does not rely on the CUDA permutation.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
import ring_attention_attn_gb300 as ra

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


def _shard_host(x, P, layout):
    """Global -> sharded order using the oracle's map (CPU)."""
    s2g, _ = oracle.shard_index(x.shape[2], P, layout)
    return x[:, :, torch.from_numpy(s2g)].contiguous()


def _unshard_host(y, P, layout):
    _, g2s = oracle.shard_index(y.shape[2], P, layout)
    return y[:, :, torch.from_numpy(g2s)].contiguous()


def _cmp(o_gpu, lse_gpu, o_ref, lse_ref, o_tol=O_TOL, lse_tol=LSE_TOL):
    o_gpu = o_gpu.double().cpu().numpy().reshape(o_ref.shape)
    lse_gpu = lse_gpu.double().cpu().numpy().reshape(lse_ref.shape)
    eo = np.max(np.abs(o_gpu - o_ref)) if o_ref.size else 0.0
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse_gpu)), "-inf pattern of LSE differs"
    el = np.max(np.abs(lse_gpu[fin] - lse_ref[fin])) if fin.any() else 0.0
    assert eo <= o_tol, f"max|dO| = {eo:.3e}"
    assert el <= lse_tol, f"max|dLSE| = {el:.3e}"
    return eo, el


def _run_ring(q, k, v, P, causal):
    layout = 1 if causal else 0
    qs, ks, vs = (_shard_host(x, P, layout).cuda() for x in (q, k, v))
    out, lse = ra.ring_attn_fwd(qs, ks, vs, P, causal=causal)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    return (_unshard_host(out.cpu(), P, layout),
            _unshard_host(lse.cpu().unsqueeze(-1), P, layout).squeeze(-1))


# ----------------------------------------------------------- permutations --
@pytest.mark.parametrize("S,P,layout,d", [(4096, 2, 1, 64), (1024, 4, 0, 64), (48, 4, 1, 128),
                                          (14400, 4, 0, 128), (600, 3, 1, 128), (16, 8, 1, 64)])
def test_cp_shard_bit_exact(S, P, layout, d):
    x, _, _ = synth.make_custom((2, 3, S, d), (1, 1, 1, d), seed=S + P)
    y = ra.ra_cp_shard(x.cuda(), P, layout)
    assert torch.equal(y.cpu().view(torch.int16), _shard_host(x, P, layout).view(torch.int16))
    back = ra.ra_cp_shard(y, P, layout, inverse=True)
    assert torch.equal(back.cpu().view(torch.int16), x.view(torch.int16))


def test_cp_shard_index_matches_oracle():
    for S, P, layout in [(4096, 2, 1), (1024, 4, 0), (600, 3, 1), (432000, 8, 0), (64, 8, 1)]:
        a = ra.ra_cp_shard_index(S, P, layout)
        b = oracle.shard_index(S, P, layout)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("T,N,d", [(48, 900, 128), (5, 7, 64)])
def test_frame_transpose_bit_exact(T, N, d):
    x, _, _ = synth.make_custom((1, 3, T * N, d), (1, 1, 1, d), seed=T * N)
    y = ra.ra_frame_transpose(x.cuda(), T, N)
    ref = x.reshape(1, 3, T, N, d).transpose(2, 3).reshape(1, 3, T * N, d)
    assert torch.equal(y.cpu().view(torch.int16), ref.view(torch.int16))
    back = ra.ra_frame_transpose(y, T, N, inverse=True)
    assert torch.equal(back.cpu().view(torch.int16), x.view(torch.int16))


# ------------------------------------------------------------------ merge --
@pytest.mark.parametrize("n,rows,d,empty_rows,empty_parts",
                         [(8, 1000, 128, 3, 2), (3, 777, 64, 1, 1), (1, 50, 128, 0, 0),
                          (17, 300, 64, 5, 9)])
def test_lse_merge(n, rows, d, empty_rows, empty_parts):
    o, l = synth.make_partials(n, rows, d, seed=n * rows, empty_rows=empty_rows,
                               empty_parts=empty_parts)
    om, lm = ra.lse_merge(o.cuda(), l.cuda())
    ro, rl = oracle.lse_merge(o.double().numpy(), l.double().numpy())
    _cmp(om, lm, ro, rl)
    assert torch.all(om[:empty_rows].float() == 0)


# -------------------------------------------------------------- attention --
def test_ring_c1_full():
    w = synth.WORKLOADS["c1"]
    q, k, v = synth.make_qkv(w)
    o, l = _run_ring(q, k, v, w.P, w.causal)
    ro, rl = oracle.attention(q, k, v, causal=False)
    _cmp(o, l, ro, rl)


def test_ring_c2_causal_zigzag_full():
    w = synth.WORKLOADS["c2"]
    q, k, v = synth.make_qkv(w)
    o, l = _run_ring(q, k, v, w.P, w.causal)
    ro, rl = oracle.attention(q, k, v, causal=True)
    _cmp(o, l, ro, rl)


CASES = [
    # B, H, S, d, P, causal  -- ragged tails, tiny chunks, P = 1, C not a tile multiple
    (1, 2, 1000, 64, 4, False),
    (2, 1, 520, 128, 2, False),
    (1, 1, 8, 64, 2, False),
    (1, 2, 300, 128, 1, False),
    (1, 1, 1, 128, 1, False),
    (1, 2, 600, 128, 3, True),
    (1, 1, 1024, 128, 4, True),
    (2, 2, 520, 64, 2, True),
    (1, 1, 16, 64, 8, True),
    (1, 3, 2048, 128, 8, False),
    # chunks ending in a short tile whose rows all ranks stack in one tile
    (1, 2, 1088, 64, 4, False),   # 272-row chunks: 4 x 16 rows
    (1, 3, 888, 128, 3, False),   # 296-row chunks: 3 x 40 rows
    (2, 1, 2112, 64, 8, False),   # 264-row chunks: 8 x 8 rows
    (1, 1, 656, 128, 2, False),   # 328-row chunks: 2 x 72 rows do not fit
    # at least as many query-tile pairs as SMs: pair units (fewer run as split
    # units, one query tile each, key tiles alternating between warpgroups;
    # when the split units fit the 152 SMs, each runs on a pair of CTAs that
    # take alternate key tiles)
    (1, 40, 2048, 64, 2, True),
    (1, 24, 2048, 128, 4, True),
    (1, 40, 2048, 128, 2, False),
    (1, 18, 2048, 64, 2, True),   # 144 pairs, 288 split units: one CTA each
    (1, 18, 2048, 128, 2, False),
    (1, 3, 384, 64, 1, False),    # 3 key tiles: CTA 0 takes 2 (one per warpgroup), CTA 1 one
    (1, 2, 128, 128, 1, True),    # one key tile: the second CTA meets none
    (1, 5, 1920, 64, 3, True),    # causal 640-row chunks: 1 to 15 key tiles per query tile
]


@pytest.mark.parametrize("B,H,S,d,P,causal", CASES)
def test_ring_small_cases(B, H, S, d, P, causal):
    q, k, v = synth.make_custom((B, H, S, d), (B, H, S, d), seed=S * 7 + d + P)
    o, l = _run_ring(q, k, v, P, causal)
    ro, rl = oracle.attention(q, k, v, causal=causal)
    _cmp(o, l, ro, rl)


@pytest.mark.parametrize("d,causal", [(64, False), (128, False), (64, True)])
def test_ring_rescale_every_tile(d, causal):
    """Scores that rise tile by tile: channel 0 holds 4 in every query and
    round(6.5 t sqrt(d) / 4) in the keys of key tile t, so each tile's scores
    sit ~6.5 (9.4 in log2 units) above the previous tile's while their spread
    within the tile stays that of the random channels.  Row maxima then jump
    past the lazy-rescale threshold (2^8) at nearly every tile, and O is
    rescaled each time.  Split units (fewer query-tile pairs than SMs), where
    at d = 64 without the mask three S buffers let a warpgroup reach a tile
    before its previous PV is issued."""
    B, H, S, P = 1, 2, 1024, 1
    q, k, v = synth.make_custom((B, H, S, d), (B, H, S, d), seed=77 + d + causal)
    q, k = q.clone(), k.clone()
    q[..., 0] = 4.0
    k[..., 0] = (torch.arange(S) // 128).float().mul(6.5 * d ** 0.5 / 4).round().bfloat16()
    o, l = _run_ring(q, k, v, P, causal)
    ro, rl = oracle.attention(q, k, v, causal=causal)
    _cmp(o, l, ro, rl)


def _c3_rows(w):
    """One row in every 128-row query tile of every rank chunk and head of the
    14,400-token workload (2,784 rows, the lane rotating from tile to tile),
    plus the first and last row of each chunk."""
    rows = synth.tile_rows(w.B * w.H, w.S, w.L)
    edge = oracle.flat_rows(w.B, w.H, w.S, synth.sample_rows(w, 2 * w.P))
    return np.unique(np.concatenate([rows, edge]))


def test_ring_c3_every_row():
    """The 14,400-token workload through the ring, every output row (345,600
    rows, 2.5 TFLOP of fp64: about a minute on 16 host cores)."""
    w = synth.WORKLOADS["c3"]
    q, k, v = synth.make_qkv(w)
    o, l = _run_ring(q, k, v, w.P, w.causal)
    ro, rl = oracle.attention(q, k, v)
    _cmp(o, l, ro, rl)


@pytest.mark.parametrize("causal", [False, True])
def test_rank_partials_and_merge(causal):
    B, H, S, d, P, rank = 1, 2, 4096, 128, 8, 3
    layout = 1 if causal else 0
    q, k, v = synth.make_custom((B, H, S, d), (B, H, S, d), seed=55 + causal)
    qs, ks, vs = (_shard_host(x, P, layout) for x in (q, k, v))
    L = S // P
    q_local = qs[:, :, rank * L:(rank + 1) * L].contiguous().cuda()
    kd, vd = ks.cuda(), vs.cuda()
    parts, lparts = ra.ring_attn_fwd_rank(q_local, kd, vd, P, rank, causal=causal, out_fp32=True)
    fused, lfused = ra.ring_attn_fwd_rank(q_local, kd, vd, P, rank, causal=causal)
    merged, lmerged = ra.lse_merge(parts, lparts)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    s2g, _ = oracle.shard_index(S, P, layout)
    gq = s2g[rank * L:(rank + 1) * L]
    # every per-step partial against the oracle on that block's keys
    for s in range(P):
        src = oracle.ring_source(P, rank, s)
        blk = torch.from_numpy(s2g[src * L:(src + 1) * L])
        kb, vb = k[:, :, blk], v[:, :, blk]
        ro = np.empty((B, H, L, d))
        rl = np.empty((B, H, L))
        qg = q[:, :, torch.from_numpy(gq)]
        if causal:
            # keys of this block visible to each query: global key <= global query
            for i in range(L):
                vis = torch.from_numpy(np.nonzero(s2g[src * L:(src + 1) * L] <= gq[i])[0])
                oi, li = oracle.attention(qg[:, :, i:i + 1], kb[:, :, vis], vb[:, :, vis])
                ro[:, :, i], rl[:, :, i] = oi[:, :, 0], li[:, :, 0]
        else:
            ro, rl = oracle.attention(qg, kb, vb)
        _cmp(parts[s], lparts[s], ro, rl)
    ro, rl = oracle.attention(q, k, v, causal=causal, rows=oracle.flat_rows(B, H, S, gq))
    _cmp(merged, lmerged, ro, rl)
    _cmp(fused, lfused, ro, rl)
    assert (merged.float() - fused.float()).abs().max().item() <= 4e-3


@pytest.mark.parametrize("d", [64, 128])
def test_persistent_units_with_empty_steps(d):
    """Short units (4 key tiles) and more units than SMs: CTAs walk several
    units each.  Causal zigzag per-step partials of rank 0 make the pairs of
    its first chunk empty for every block but its own (they see no key), so
    the walk mixes empty and full units; every partial, merged, must match
    the oracle."""
    B, H, S, P, rank = 1, 40, 4096, 8, 0
    q, k, v = synth.make_custom((B, H, S, d), (B, H, S, d), seed=91 + d)
    qs, ks, vs = (_shard_host(x, P, 1) for x in (q, k, v))
    L = S // P
    q_local = qs[:, :, rank * L:(rank + 1) * L].contiguous().cuda()
    parts, lparts = ra.ring_attn_fwd_rank(q_local, ks.cuda(), vs.cuda(), P, rank, causal=True,
                                          out_fp32=True)
    merged, lmerged = ra.lse_merge(parts, lparts)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    # first chunk of rank 0 (global tokens 0..255) sees only its own block
    C = S // (2 * P)
    lp = lparts.cpu()
    assert torch.isinf(lp[1:, :, :, :C]).all() and (lp[1:, :, :, :C] < 0).all()
    assert (parts.cpu()[1:, :, :, :C] == 0).all()
    s2g, _ = oracle.shard_index(S, P, 1)
    gq = s2g[rank * L:(rank + 1) * L]
    pick = np.array([0, 1, C - 1, C, C + 1, L - 1, 77, 300])
    rows = oracle.flat_rows(B, H, S, gq[pick])
    ro, rl = oracle.attention(q, k, v, causal=True, rows=rows)
    mo = merged.reshape(B, H, L, d)[:, :, torch.from_numpy(pick)].reshape(-1, d)
    ml = lmerged.reshape(B, H, L)[:, :, torch.from_numpy(pick)].reshape(-1)
    _cmp(mo, ml, ro, rl)


@pytest.mark.parametrize("out_fp32", [False, True])
def test_outputs_at_16_byte_offsets(out_fp32):
    """Outputs that are only 16-byte aligned take the 16-byte store path;
    the values must equal those written to aligned buffers bit for bit."""
    B, H, S, d, P = 1, 2, 1000, 128, 4
    q, k, v = (x.cuda() for x in synth.make_custom((B, H, S, d), (B, H, S, d), seed=123))
    if out_fp32:
        L = S // P
        ql = q[:, :, :L].contiguous()
        want, lwant = ra.ring_attn_fwd_rank(ql, k, v, P, 0, out_fp32=True)
        buf = torch.empty(want.numel() + 4, dtype=torch.float32, device="cuda")
        lbuf = torch.empty(lwant.numel() + 4, dtype=torch.float32, device="cuda")
        got = buf[4:].view(want.shape)
        lgot = lbuf[4:].view(lwant.shape)
        assert got.data_ptr() % 32 == 16
        ra.ring_attn_fwd_rank(ql, k, v, P, 0, out_fp32=True, out=got, lse=lgot)
    else:
        want, lwant = ra.ring_attn_fwd(q, k, v, P)
        buf = torch.empty(want.numel() + 8, dtype=torch.bfloat16, device="cuda")
        lbuf = torch.empty(lwant.numel() + 4, dtype=torch.float32, device="cuda")
        got = buf[8:].view(want.shape)
        lgot = lbuf[4:].view(lwant.shape)
        assert got.data_ptr() % 32 == 16
        ra.ring_attn_fwd(q, k, v, P, out=got, lse=lgot)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    assert torch.equal(got, want)
    assert torch.equal(lgot, lwant)


def test_rank_step_subrange():
    B, H, S, d, P, rank = 1, 1, 2048, 64, 4, 2
    q, k, v = synth.make_custom((B, H, S, d), (B, H, S, d), seed=77)
    L = S // P
    qd, kd, vd = q[:, :, rank * L:(rank + 1) * L].contiguous().cuda(), k.cuda(), v.cuda()
    o, l = ra.ring_attn_fwd_rank(qd, kd, vd, P, rank, step_begin=1, step_end=3)
    blocks = [oracle.ring_source(P, rank, s) for s in (1, 2)]
    idx = torch.cat([torch.arange(b * L, (b + 1) * L) for b in blocks])
    ro, rl = oracle.attention(q[:, :, rank * L:(rank + 1) * L], k[:, :, idx], v[:, :, idx])
    _cmp(o, l, ro, rl)


def test_c5_full_size_every_tile():
    """One rank's 54,000 queries against 432,000 keys: per-step partials +
    lse_merge (the benchmark's launch configuration) and the fused call, on
    two rows of every 128-row query tile of every head (3,376 rows, two lane
    rotations over all 128 softmax threads) plus the chunk's first and last
    rows."""
    w = synth.WORKLOADS["c5"]
    q, k, v = synth.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    parts, lparts = ra.ring_attn_fwd_rank(qd, kd, vd, w.P, 0, out_fp32=True)
    o, l = ra.lse_merge(parts, lparts)
    fo, fl = ra.ring_attn_fwd_rank(qd, kd, vd, w.P, 0)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    rows = np.unique(np.concatenate([synth.tile_rows(w.B * w.H, w.L, w.L),
                                     synth.tile_rows(w.B * w.H, w.L, w.L, salt=61),
                                     oracle.flat_rows(w.B, w.H, w.L, synth.sample_rows(w, 12))]))
    ro, rl = oracle.attention(q, k, v, rows=rows)
    _cmp(o.reshape(-1, w.d)[rows.tolist()], l.reshape(-1)[rows.tolist()], ro, rl)
    _cmp(fo.reshape(-1, w.d)[rows.tolist()], fl.reshape(-1)[rows.tolist()], ro, rl)
    assert (o.float() - fo.float()).abs().max().item() <= 2e-3


# ------------------------------------------------- overlapped ring copies --
# exchange: "stream" = copies on a comm stream, "same" = copies serialised on
# the compute stream, "launch" = no comm stream, the step launches copy
@pytest.mark.parametrize("B,H,S,d,P,causal,exchange",
                         [(1, 2, 2048, 128, 4, False, "stream"), (1, 2, 4096, 64, 2, True, "stream"),
                          (2, 1, 1200, 128, 3, True, "same"), (1, 3, 1000, 64, 8, False, "stream"),
                          (1, 2, 1088, 128, 4, False, "stream"),  # stacked last rows
                          (1, 2, 2048, 128, 4, False, "launch"), (1, 2, 4096, 64, 2, True, "launch"),
                          (2, 1, 1200, 128, 3, True, "launch"), (1, 3, 1000, 64, 8, False, "launch"),
                          (1, 2, 1088, 128, 4, False, "launch")])
def test_overlap_ring_matches_oracle_and_fused(B, H, S, d, P, causal, exchange):
    layout = 1 if causal else 0
    q, k, v = synth.make_custom((B, H, S, d), (B, H, S, d), seed=S + 11 * P + causal)
    qs, ks, vs = (_shard_host(x, P, layout).cuda() for x in (q, k, v))
    comm = {"stream": torch.cuda.Stream(), "same": torch.cuda.current_stream(),
            "launch": None}[exchange]
    o, l = ra.ring_attn_fwd_overlap(qs, ks, vs, P, causal=causal, comm_stream=comm)
    fo, fl = ra.ring_attn_fwd(qs, ks, vs, P, causal=causal)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    assert (o.float() - fo.float()).abs().max().item() <= 4e-3
    assert (l - fl).abs().max().item() <= 1e-4
    ro, rl = oracle.attention(q, k, v, causal=causal)
    _cmp(_unshard_host(o.cpu(), P, layout), _unshard_host(l.cpu().unsqueeze(-1), P, layout).squeeze(-1),
         ro, rl)


# ----------------------------------------------------- Ulysses (all-to-all) --
def _seq_split(x, P):
    B, H, S, d = x.shape
    return x.reshape(B, H, P, S // P, d).permute(2, 0, 1, 3, 4).contiguous()


@pytest.mark.parametrize("B,H,S,d,P", [(1, 4, 512, 64, 2), (2, 8, 1200, 128, 4), (1, 2, 96, 128, 2)])
def test_ulysses_all_to_all_bit_exact(B, H, S, d, P):
    x, _, _ = synth.make_custom((B, H, S, d), (1, 1, 1, 1), seed=H * S)
    xs = _seq_split(x, P)
    y = ra.ra_ulysses_a2a(xs.cuda(), B, H, S, P)
    L, Hp = S // P, H // P
    ref = xs.reshape(P, B, P, Hp, L, d).permute(2, 1, 3, 0, 4, 5).reshape(P, B, Hp, S, d)
    assert torch.equal(y.cpu().view(torch.int16), ref.view(torch.int16))
    back = ra.ra_ulysses_a2a(y, B, H, S, P, inverse=True)
    assert torch.equal(back.cpu().view(torch.int16), xs.view(torch.int16))


@pytest.mark.parametrize("B,H,S,d,P,causal", [(1, 4, 1024, 64, 2, False), (1, 8, 1200, 128, 4, True),
                                              (2, 4, 600, 128, 4, False)])
def test_ulysses_attention_matches_oracle(B, H, S, d, P, causal):
    q, k, v = synth.make_custom((B, H, S, d), (B, H, S, d), seed=S + H + P)
    o, l = ra.ulysses_attn_fwd(*(_seq_split(x, P).cuda() for x in (q, k, v)), B, H, S, P,
                               causal=causal)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    o = o.cpu().permute(1, 2, 0, 3, 4).reshape(B, H, S, d)
    l = l.cpu().permute(1, 2, 0, 3).reshape(B, H, S)
    ro, rl = oracle.attention(q, k, v, causal=causal)
    _cmp(o, l, ro, rl)


# ------------------------------------------ all-gather / reduce-scatter forms --
def _per_rank(x, P, layout):
    B, H, S, d = x.shape
    return _shard_host(x, P, layout).reshape(B, H, P, S // P, d).permute(2, 0, 1, 3, 4).contiguous()


@pytest.mark.parametrize("form", ["allgather", "reducescatter"])
@pytest.mark.parametrize("B,H,S,d,P,causal", [(1, 2, 1024, 128, 4, False), (1, 2, 2048, 64, 2, True),
                                              (2, 1, 600, 128, 3, True), (1, 3, 1000, 64, 8, False),
                                              (1, 2, 1088, 128, 4, False)])  # stacked last rows
def test_allgather_reducescatter_forms_match_oracle(form, B, H, S, d, P, causal):
    layout = 1 if causal else 0
    q, k, v = synth.make_custom((B, H, S, d), (B, H, S, d), seed=S + 5 * P + causal)
    fn = ra.cp_allgather_attn_fwd if form == "allgather" else ra.cp_reducescatter_attn_fwd
    o, l = fn(*(_per_rank(x, P, layout).cuda() for x in (q, k, v)), B, H, S, P, causal=causal)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    o = _unshard_host(o.cpu().permute(1, 2, 0, 3, 4).reshape(B, H, S, d), P, layout)
    l = _unshard_host(l.cpu().permute(1, 2, 0, 3).reshape(B, H, S, 1), P, layout).squeeze(-1)
    ro, rl = oracle.attention(q, k, v, causal=causal)
    _cmp(o, l, ro, rl)


# ---------------------------------- every CP form at 14,400 tokens (sampled) --
@pytest.mark.parametrize("form", ["overlap", "ulysses", "allgather", "reducescatter"])
def test_cp_forms_c3_every_tile(form):
    """The 14,400-token workload (3,600-row chunks: each rank's last 16 rows
    stacked into one tile) through every context-parallel form, on the rows
    the ring test checks (one per query tile, chunk and head)."""
    w = synth.WORKLOADS["c3"]
    q, k, v = synth.make_qkv(w)
    B, H, S, d, P = w.B, w.H, w.S, w.d, w.P
    if form == "overlap":
        o, l = ra.ring_attn_fwd_overlap(q.cuda(), k.cuda(), v.cuda(), P,
                                        comm_stream=torch.cuda.Stream())
        o, l = o.cpu(), l.cpu()
    else:
        fn = {"ulysses": ra.ulysses_attn_fwd, "allgather": ra.cp_allgather_attn_fwd,
              "reducescatter": ra.cp_reducescatter_attn_fwd}[form]
        o, l = fn(*(_seq_split(x, P).cuda() for x in (q, k, v)), B, H, S, P)
        o = o.cpu().permute(1, 2, 0, 3, 4).reshape(B, H, S, d)
        l = l.cpu().permute(1, 2, 0, 3).reshape(B, H, S)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    rows = _c3_rows(w)
    ro, rl = oracle.attention(q, k, v, rows=rows)
    _cmp(o.reshape(-1, d)[rows], l.reshape(-1)[rows], ro, rl)


# ---------------------------------------------------------------- factored --
@pytest.mark.parametrize("B,H,T,N,d,P", [(1, 2, 8, 50, 64, 4),    # 2-frame chunks fold in pairs
                                          (1, 2, 68, 20, 64, 4),   # 17-frame chunks: 2 rank pairs
                                          (1, 1, 24, 30, 128, 6),  # 4-frame chunks fold by 3
                                          (1, 2, 80, 7, 64, 5),    # P = 5: no fold, last unpaired
                                          (1, 2, 12, 50, 64, 3),   # odd P: last rank unpaired
                                          (2, 1, 6, 70, 128, 1),   # one rank
                                          (1, 3, 24, 40, 128, 2),
                                          (1, 2, 40, 9, 64, 2),    # 20-frame chunks: 32 rows each
                                          (1, 1, 48, 5, 128, 1),   # 48-frame chunks: 2 per tile
                                          (1, 1, 260, 3, 64, 2),   # 130-frame chunks: not packed
                                          (1, 2, 130, 4, 128, 1)])
@pytest.mark.parametrize("fold", [True, False])
def test_factored_small_full(B, H, T, N, d, P, fold):
    q, k, v = synth.make_custom((B, H, T * N, d), (B, H, T * N, d), seed=99 + T + P)
    ra.ra_set_temporal_fold(fold)
    try:
        os_, ls, ot, lt = ra.factored_attn(q.cuda(), k.cuda(), v.cuda(), T, N, P)
    finally:
        ra.ra_set_temporal_fold(True)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    ro, rl = oracle.factored(q, k, v, T, N, "spatial")
    _cmp(os_, ls, ro, rl)
    ro, rl = oracle.factored(q, k, v, T, N, "temporal")
    _cmp(ot, lt, ro, rl)


@pytest.mark.parametrize("fold", [True, False])
def test_factored_c4_every_tile(fold):
    """48 frames x 900 tokens, H = 24: spatial and temporal outputs on every
    token (1,036,800 rows each) with the ring's four 12-frame chunks folded
    into two blocks (the default); as four steps, the temporal output on
    every token and the spatial one (the same launch either way) on one
    token of every 128-row query tile of every frame and head."""
    w = synth.WORKLOADS["c4"]
    q, k, v = synth.make_qkv(w)
    ra.ra_set_temporal_fold(fold)
    try:
        os_, ls, ot, lt = ra.factored_attn(q.cuda(), k.cuda(), v.cuda(), w.T, w.N, w.P)
    finally:
        ra.ra_set_temporal_fold(True)
    torch.cuda.synchronize()
    assert ra.ra_get_status() == 0
    if fold:
        ro, rl = oracle.factored(q, k, v, w.T, w.N, "spatial")
        _cmp(os_, ls, ro, rl)
    else:
        rows = synth.tile_rows(w.B * w.H * w.T, w.N, w.N)
        ro, rl = oracle.factored(q, k, v, w.T, w.N, "spatial", rows=rows)
        _cmp(os_.reshape(-1, w.d)[rows.tolist()], ls.reshape(-1)[rows.tolist()], ro, rl)
    ro, rl = oracle.factored(q, k, v, w.T, w.N, "temporal")
    _cmp(ot, lt, ro, rl)


# ---------------------------------------------------------- edge + status --
def test_empty_inputs_are_noops():
    z = torch.empty((1, 0, 64, 64), dtype=torch.bfloat16, device="cuda")
    out, lse = ra.ring_attn_fwd(z, z, z, 2)
    z2 = torch.empty((1, 1, 0, 64), dtype=torch.bfloat16, device="cuda")
    ra.ring_attn_fwd(z2, z2, z2, 2)
    assert ra.ra_get_status() == 0


def test_watchdog_reports_timeout():
    ra.ra_set_watchdog_ns(1_000_000)  # 1 ms
    try:
        ra.ra_watchdog_selftest()
        assert ra.ra_get_status() == -5
        assert ra.ra_get_status() == 0  # cleared by the read
    finally:
        ra.ra_set_watchdog_ns(0)
    # the context is still usable afterwards
    q, k, v = synth.make_custom((1, 1, 256, 64), (1, 1, 256, 64), seed=3)
    o, l = _run_ring(q, k, v, 2, False)
    ro, rl = oracle.attention(q, k, v)
    _cmp(o, l, ro, rl)
