"""The pins must catch plausible oracle mistakes.

Each case compiles a copy of the oracle source with one planted mistake (a
dropped term, a wrong sign or index, a swapped operand) into a temporary
library, swaps it in for the real one, and checks that at least one pin
fails.  Mistakes are planted in the oracle on the CPU only.
"""
import contextlib
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_bwd as bwd
import test_oracle_pins as pins
import test_page_figures as figures

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_ref.c")

MUTANTS = {
    "scale_1_over_d": ("1.0 / sqrt((double)d)", "1.0 / (double)d",
                       [lambda: pins.test_brute_force_tiny(8, 8, False)]),
    "causal_off_by_one": ("count = q_offset + i + 1;", "count = q_offset + i;",
                          [lambda: pins.test_brute_force_tiny(8, 4, True)]),
    "values_read_from_keys": ("const uint16_t *vrow = V + (start + t * stride) * d;",
                              "const uint16_t *vrow = K + (start + t * stride) * d;",
                              [lambda: pins.test_brute_force_tiny(3, 4, False)]),
    "lse_log2": ("double L = m + log(z);", "double L = m + log2(z);",
                 [lambda: pins.test_brute_force_tiny(16, 8, False)]),
    "merge_weight_sign": ("double w = exp(lse_parts[i * rows + r] - M);",
                          "double w = exp(M - lse_parts[i * rows + r]);",
                          [lambda: pins.test_chunked_merge_equals_one_shot(False)]),
    "ring_fold_drops_rescale": ("acc[c] = acc[c] * a + accb[c] * b;",
                                "acc[c] = acc[c] * a + accb[c];",
                                [lambda: pins.test_ring_equals_full(4, False, 64)]),
    "ring_direction": ("return ((r - s) % P + P) % P;", "return ((r + s) % P + P) % P;",
                       [figures.test_ring_schedule_matches_diagram]),
    "zigzag_wrong_mirror": ("int64_t chunk = (i < C) ? r : (2 * P - 1 - r);",
                            "int64_t chunk = (i < C) ? r : (P + r);",
                            [lambda: pins.test_zigzag_is_a_permutation_with_two_chunks_per_rank(48, 4),
                             pins.test_zigzag_balances_causal_work]),
    "bwd_ds_drops_d": ("double ds = P[j] * (dP[j] - D);", "double ds = P[j] * dP[j];",
                       [lambda: bwd.test_against_torch_float64_autograd(False)]),
    "bwd_dk_unscaled": ("dK[j * d + c] += scale * ds * widen_bf16(Q[i * d + c]);",
                        "dK[j * d + c] += ds * widen_bf16(Q[i * d + c]);",
                        [lambda: bwd.test_finite_differences_against_brute_force(False)]),
    "bwd_dv_from_dp": ("dV[j * d + c] += P[j] * widen_bf16(dO[i * d + c]);",
                       "dV[j * d + c] += dP[j] * widen_bf16(dO[i * d + c]);",
                       [lambda: bwd.test_finite_differences_against_brute_force(True)]),
    "temporal_stride_wrong": ("attend(q + flat * d, Kh, Vh, d, pos, T, N, scale",
                              "attend(q + flat * d, Kh, Vh, d, pos, T, 1, scale",
                              [pins.test_factored_temporal_across_frames]),
}


@contextlib.contextmanager
def _mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib_path = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", str(path), "-o",
                    str(lib_path), "-lm"], check=True)
    lib = oracle.configure(ctypes.CDLL(str(lib_path)))
    saved = oracle._load()
    oracle._lib = lib
    try:
        yield
    finally:
        oracle._lib = saved


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new, checks = MUTANTS[name]
    with _mutant(tmp_path, name, old, new):
        failures = 0
        for check in checks:
            try:
                check()
            except (AssertionError, ValueError):
                failures += 1
        assert failures > 0, f"no pin caught mutant {name}"
