"""CPU checks of the C ABI: the library loads without a GPU, exports every
symbol the header declares, and its host-side logic (index maps, ring
schedule, argument validation) is exact."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import ring_attention_attn_gb300 as ra
from ring_attention_attn_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ringattn.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, re.M)))


def test_library_exports_every_declared_symbol():
    names = _declared()
    assert "ring_attn_fwd" in names and "lse_merge" in names and "factored_attn" in names
    lib = ctypes.CDLL(_abi.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(_abi.EXPORTS) == names


@pytest.mark.parametrize("S,P,layout", [(4096, 2, 1), (1024, 4, 0), (600, 3, 1), (16, 8, 1),
                                        (432000, 8, 0), (0, 4, 1)])
def test_shard_index_bit_exact_against_oracle(S, P, layout):
    a = ra.ra_cp_shard_index(S, P, layout)
    b = oracle.shard_index(S, P, layout)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_ring_source_matches_oracle():
    for P in (1, 2, 3, 4, 8):
        for r in range(P):
            for s in range(2 * P):
                assert ra.ra_ring_source(P, r, s) == oracle.ring_source(P, r, s)


def test_argument_errors_are_reported_before_any_launch():
    L = _abi.lib()
    vp = ctypes.c_void_p
    good = vp(256)       # never dereferenced: validation fails first
    odd = vp(256 + 8)    # not 16-byte aligned
    nul = vp(0)
    s = vp(0)
    # d unsupported, S % P, zigzag S % 2P
    assert L.ring_attn_fwd(good, good, good, good, good, 1, 1, 1024, 96, 4, 0, s) == -2
    assert L.ring_attn_fwd(good, good, good, good, good, 1, 1, 1000, 64, 3, 0, s) == -2
    assert L.ring_attn_fwd(good, good, good, good, good, 1, 1, 1004, 64, 4, 1, s) == -2
    # null pointer, negative sizes, bad flag
    assert L.ring_attn_fwd(nul, good, good, good, good, 1, 1, 1024, 64, 4, 0, s) == -1
    assert L.ring_attn_fwd(good, good, good, good, good, -1, 1, 1024, 64, 4, 0, s) == -1
    assert L.ring_attn_fwd(good, good, good, good, good, 1, 1, 1024, 64, 4, 2, s) == -1
    # misaligned
    assert L.ring_attn_fwd(good, odd, good, good, good, 1, 1, 1024, 64, 4, 0, s) == -3
    # empty sizes are no-ops even with null pointers
    assert L.ring_attn_fwd(nul, nul, nul, nul, nul, 0, 4, 1024, 64, 4, 0, s) == 0
    assert L.ring_attn_fwd(nul, nul, nul, nul, nul, 1, 4, 0, 64, 4, 0, s) == 0
    # rank entry point: rank / step range
    assert L.ring_attn_fwd_rank(good, good, good, good, good, 1, 1, 1024, 64, 4, 4, 0, 0, 4, 0, s) == -1
    assert L.ring_attn_fwd_rank(good, good, good, good, good, 1, 1, 1024, 64, 4, 0, 0, 2, 2, 0, s) == -1
    assert L.ring_attn_fwd_rank(good, good, good, good, good, 1, 1, 1024, 64, 4, 0, 0, 0, 5, 0, s) == -1
    # merge: n range, d
    assert L.lse_merge(good, good, 0, 10, 64, good, good, s) == -1
    assert L.lse_merge(good, good, 65, 10, 64, good, good, s) == -1
    assert L.lse_merge(good, good, 2, 10, 32, good, good, s) == -2
    # shard / transpose
    assert L.ra_cp_shard(good, good, 1, 12, 64, 4, 1, 0, s) == -2
    assert L.ra_cp_shard(good, good, 1, 16, 64, 4, 2, 0, s) == -1
    assert L.ra_frame_transpose(good, odd, 1, 4, 4, 64, 0, s) == -3
    # factored: T % P; workspace too small or missing (chunks over 128 frames)
    assert L.factored_attn(good, good, good, good, good, good, good, 1, 1, 10, 9, 64, 4,
                           good, 1 << 30, s) == -2
    assert L.factored_attn(good, good, good, good, good, good, good, 1, 1, 136, 9, 64, 1,
                           good, 16, s) == -6
    assert L.factored_attn(good, good, good, good, good, good, good, 1, 1, 136, 9, 64, 1,
                           nul, 0, s) == -6


def test_sizes_beyond_the_addressable_rows_are_rejected():
    """Row indices are 32-bit in the tensor maps and index math: B*H*S rows
    must stay below 2^31 - 512; larger inputs fail on the host."""
    L = _abi.lib()
    vp = ctypes.c_void_p
    good, s = vp(256), vp(0)
    S = 1 << 27  # 2^27 tokens x 16 heads = 2^31 rows
    assert L.ring_attn_fwd(good, good, good, good, good, 1, 16, S, 64, 1, 0, s) == -2
    assert L.ring_attn_fwd_rank(good, good, good, good, good, 1, 16, S, 64, 8, 0, 0, 0, 8, 1, s) == -2
    assert L.ra_cp_shard(good, good, 16, S, 64, 1, 0, 0, s) == -2
    assert L.ra_frame_transpose(good, good, 16, 1 << 14, 1 << 13, 64, 0, s) == -2
    assert L.ra_ulysses_a2a(good, good, 1, 16, S, 64, 2, 0, s) == -2


def test_workspace_size():
    """None for T <= 128 (in place); for T > 128 position-major q, k, v, output
    (bf16) and LSE (fp32)."""
    part = lambda b: (b + 255) // 256 * 256
    assert ra.factored_attn_workspace(1, 24, 48, 900, 128) == 0
    assert ra.factored_attn_workspace(1, 24, 128, 900, 128) == 0
    rows = 2 * 3 * 130 * 7
    assert ra.factored_attn_workspace(2, 3, 130, 7, 64) == 4 * part(rows * 128) + part(rows * 4)
    assert ra.factored_attn_workspace(1, 24, 48, 900, 96) == 0


def test_strerror_covers_codes():
    L = _abi.lib()
    for code in range(0, -7, -1):
        assert L.ra_strerror(code).decode() != "unknown error"


def test_python_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        ra.ring_attn_fwd(x, x, x, 2)


def test_checked_build_compiles_and_exports_the_same_symbols():
    """The RA_CHECKS build (device bounds checks) builds from the same sources
    and exports the header's symbols; it says so through ra_checks_enabled."""
    from ring_attention_attn_gb300 import build as ra_build
    path = ra_build.build(checks=True)
    lib = ctypes.CDLL(path)
    for n in _declared():
        assert hasattr(lib, n), n
    lib.ra_checks_enabled.restype = ctypes.c_int
    assert lib.ra_checks_enabled() == 1
    assert _abi.lib().ra_checks_enabled() == 0
