"""Property tests of the library's host logic against the oracle over random
shapes: the shard index maps (bit-exact, both layouts), the ring schedule,
and argument validation that must reject every shape the layouts cannot
split.  CPU only; no device memory is touched."""
import ctypes

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
import ring_attention_attn_gb300 as ra  # noqa: E402
from ring_attention_attn_gb300 import _abi  # noqa: E402


@settings(max_examples=200, deadline=None)
@given(P=st.integers(1, 16), chunks=st.integers(1, 64), layout=st.sampled_from([0, 1]))
def test_shard_maps_match_oracle(P, chunks, layout):
    S = 2 * P * chunks if layout == 1 else P * chunks
    a = ra.ra_cp_shard_index(S, P, layout)
    b = oracle.shard_index(S, P, layout)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # s2g and g2s are inverse permutations
    assert np.array_equal(a[1][a[0]], np.arange(S))


@settings(max_examples=200, deadline=None)
@given(P=st.integers(1, 64), r=st.integers(0, 63), s=st.integers(0, 200))
def test_ring_source_matches_oracle(P, r, s):
    r = r % P
    assert ra.ra_ring_source(P, r, s) == oracle.ring_source(P, r, s)


@settings(max_examples=200, deadline=None)
@given(P=st.integers(1, 16), S=st.integers(1, 5000))
def test_shapes_the_layouts_cannot_split_are_rejected(P, S):
    L = _abi.lib()
    vp = ctypes.c_void_p
    good, s = vp(256), vp(0)  # never dereferenced when validation fails
    for causal in (0, 1):
        bad = S % P != 0 or (causal and S % (2 * P) != 0)
        if bad:
            assert L.ring_attn_fwd(good, good, good, good, good, 1, 1, S, 64, P, causal, s) == -2
    # the index maps reject the same shapes, on the host
    s2g = np.empty(S, dtype=np.int64)
    rc = L.ra_cp_shard_index(S, P, 1, s2g.ctypes.data_as(vp), None)
    assert (rc == 0) == (S % (2 * P) == 0)
