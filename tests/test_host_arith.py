"""CPU checks of the host/device arithmetic in csrc/common.cuh (udiv, the stream-K partition,
the workspace layout) and of its segment validity rule against the oracle's, through a small
host program built with nvcc (tests/host_checks.cu)."""
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import sdpa_varlen_oracle as O  # noqa: E402


@pytest.fixture(scope="module")
def host_checks(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path_factory.mktemp("hc") / "host_checks")
    src = os.path.join(ROOT, "tests", "host_checks.cu")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-o", exe, src], check=True, capture_output=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    return out.returncode, out.stdout


def test_division_partition_and_workspace_layout(host_checks):
    rc, out = host_checks
    fails = [ln for ln in out.splitlines() if ln.startswith("FAIL")]
    assert rc == 0 and not fails, "\n".join(fails[:20])
    assert "failures 0" in out


def test_segment_validity_rule_matches_the_oracle(host_checks):
    _, out = host_checks
    rows = [ln.split()[1:] for ln in out.splitlines() if ln.startswith("SEG ")]
    assert len(rows) == 3 * 4 * 3 * 6 * 4
    for r in rows:
        qs, ql, col, ke, T, nrows, cols, w, bits = (int(x) for x in r)
        want = O.segment_status(np.array([qs, ql, col, ke]), T, nrows, cols, w)
        assert bits == want, (qs, ql, col, ke, w, bits, want)


def test_the_static_entry_fallback_case_needs_the_reduced_grid(host_checks):
    """The case tests/test_zz_no_alloc.py runs to reach the allocation-free entry's reduced
    grid: its scratch does not fit the 32 MiB array at the general grid (two split-K CTAs
    per SM on a 152-SM GB300) but fits at one CTA per SM."""
    _, out = host_checks
    need = {int(g): int(b) for g, b in (ln.split()[1:] for ln in out.splitlines() if ln.startswith("STATIC_NEED"))}
    cap = 32 << 20
    assert need[304] > cap >= need[152], need
