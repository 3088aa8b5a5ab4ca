"""Golden values the pages print, checked against the oracle's ring schedule
and the byte / FLOP calculators that the benchmark's roofline figures use."""
import os

import pytest

import oracle
from ring_attention_attn_gb300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


def test_ring_schedule_matches_diagram():
    """k8ai "How context parallel works": ring diagram for 4 GPUs."""
    seen = 0
    for step, rank, block in _rows("ring_schedule_p4.txt"):
        assert oracle.ring_source(4, int(rank), int(step)) == int(block)
        seen += 1
    assert seen == 8


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_every_rank_sees_every_block_once(P):
    """P steps bring each block to each rank exactly once (day 83 blog, "Context
    parallelism: splitting the sequence")."""
    for r in range(P):
        assert sorted(oracle.ring_source(P, r, s) for s in range(P)) == list(range(P))
    # rank 0 of an 8-way ring visits 0, 7, 6, ..., 1
    if P == 8:
        assert [oracle.ring_source(8, 0, s) for s in range(8)] == [0, 7, 6, 5, 4, 3, 2, 1]


def _value(name):
    for row in _rows("page_figures.txt"):
        if row[0] == name:
            return float(row[1]), float(row[2])
    raise KeyError(name)


def _close(got, name):
    want, rel = _value(name)
    assert abs(got - want) <= rel * abs(want) + 1e-12, (name, got, want)


def test_token_counts():
    _close(acc.tokens(16, 900), "tokens_16_frames")
    _close(acc.tokens(48, 900), "tokens_48_frames")
    _close(acc.scores_per_head(43200), "scores_per_head_43200")
    _close(acc.per_rank(43200, 4), "per_gpu_43200_p4")
    _close(acc.per_rank(32000, 4), "per_gpu_32000_p4")
    _close(acc.spatial_tokens(720, 1280, 16), "spatial_tokens_720p")
    _close(acc.tokens(24 * 5, acc.spatial_tokens(720, 1280, 16)), "total_tokens_5s_24fps")
    _close(acc.attn_matrix_bytes(432000), "attn_bytes_432000")
    _close(acc.per_rank(432000, 8), "per_gpu_432000_p8")


def test_communication_figures():
    L, d = 54000, 128
    _close(acc.kv_bytes_per_step(L, d), "kv_bytes_per_step_head")
    # the page rounds to 27.6 MB per head before multiplying by 32 and by 7
    _close(acc.kv_bytes_per_step(L, d, heads=32), "kv_bytes_per_step_32h")
    _close(acc.ring_pass_bytes(L, d, heads=32, P=8), "kv_bytes_ring_pass_p8")
    _close(acc.transfer_seconds(acc.ring_pass_bytes(L, d, 32, 8), 450), "kv_seconds_450gbs")


def test_flop_counts_of_the_workloads():
    assert acc.attention_flops(2, 1024, 1024, 64) == 536870912          # c1
    assert acc.attention_flops(4, 4096, 4096, 64, causal=True) == 8592031744  # c2
    assert acc.causal_pairs(4096) == 2 * 4195328
    assert acc.attention_flops(24, 14400, 14400, 128) == 2548039680000   # c3
    sp, tp = acc.factored_flops(24, 48, 900, 128)                        # c4
    assert (sp, tp) == (477757440000, 25480396800)
    assert acc.attention_flops(4, 54000, 432000, 128) == 47775744000000  # c5
    assert acc.merge_bytes(8, 216000, 128) == 947808000
