"""The tensor-memory (tcgen05) partition kernels on every shape they accept:
a child process forces one of them (PA_VERIFY_KERNEL=tc: rows on the MMA's
M dimension; tk: keys on M) for 1..64 query rows per KV head, head_dim 64 /
128, bf16 / f16 and u8 caches, windows and ragged tails, and each case is
compared with the fp64 oracle (<= 2e-3) and its gather trace bit-exactly."""
import json
import os
import subprocess
import sys

import pytest

from pa_testing import TOL

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("kernel", ["tc", "tk"])
def test_forced_tensor_memory_path_matches_oracle(kernel):
    env = dict(os.environ, PA_VERIFY_KERNEL=kernel)
    proc = subprocess.run([sys.executable, os.path.join(HERE, "tc_forced_cases.py")], env=env,
                          capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-3000:]
    rows = [json.loads(line) for line in proc.stdout.splitlines() if line.startswith("{")]
    assert len(rows) == 12
    for r in rows:
        assert r["bits"] == 0, r
        assert r["trace_ok"], r
        if r["excess"] is None:
            assert r["err"] <= TOL, r
        else:  # short-context edge case: the derived bf16 bound (see pa_testing.derived_tolerance)
            assert r["excess"] <= 0.0, r


def test_forced_partitions_of_odd_half_stages():
    """704-key partitions: the u8 keys-on-M kernel's 128-key stages end
    half filled inside a partition (its keys past the partition's end belong
    to the next one and must not count); every forced case must still match."""
    env = dict(os.environ, PA_VERIFY_KERNEL="tk", PA_VERIFY_PART_TOKENS="704")
    proc = subprocess.run([sys.executable, os.path.join(HERE, "tc_forced_cases.py")], env=env,
                          capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-3000:]
    rows = [json.loads(line) for line in proc.stdout.splitlines() if line.startswith("{")]
    assert len(rows) == 12
    assert any(r["kernel"] == 4 for r in rows)
    for r in rows:
        assert r["bits"] == 0, r
        assert r["trace_ok"], r
        if r["excess"] is None:
            assert r["err"] <= TOL, r
        else:
            assert r["excess"] <= 0.0, r
