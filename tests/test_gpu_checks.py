"""The bounds-checked build (-DRA_CHECKS): every kernel checks the global
row indices, TMA coordinates and TMEM columns it computes, and a failed check
is reported as RA_ERR_BOUNDS (-7) instead of an out-of-range access.

Small cases of every entry point run on that build in a child process (the
binding picks its library once per process) and must leave the device status
at 0 and match the oracle.  The default build compiles no checks in: its
self-test reports nothing."""
import os
import subprocess
import sys

import pytest

import ring_attention_attn_gb300 as ra
from ring_attention_attn_gb300 import build as ra_build

pytestmark = pytest.mark.gpu

TESTS = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_reports_no_bounds_error_on_every_entry_point():
    lib = ra_build.build(checks=True)
    env = dict(os.environ, RINGATTN_LIB=lib)
    r = subprocess.run([sys.executable, os.path.join(TESTS, "checks_child.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr


def test_default_build_has_no_checks_compiled_in():
    assert not ra.ra_checks_enabled()
    ra.ra_checks_selftest()
    assert ra.ra_get_status() == 0
