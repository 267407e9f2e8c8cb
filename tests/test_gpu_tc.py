"""Each partition kernel on shapes the default choice would send elsewhere: a
child process forces one (PA_VERIFY_KERNEL=tc: the 16-bit rows-on-M
tensor-memory kernel; mma: the warp-level kernel, 16-bit and u8) for 1..64
query rows per KV head, head_dim 64 / 128, bf16 / f16 and u8 caches, windows
and ragged tails, and each case is compared with the fp64 oracle (<= 2e-3)
and its gather trace bit-exactly."""
import json
import os
import subprocess
import sys

import pytest

from pa_testing import TOL

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("kernel", ["tc", "mma"])
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


def test_small_forced_partitions():
    """384-key partitions (three 128-key stages of the u8 kernel, six 64-key
    stages of the 16-bit one): many partitions per sequence, partition ends
    inside pages of 32 and 64 tokens' neighbours; every case must still
    match, and the u8 tensor-memory kernel must be among the kernels run."""
    env = dict(os.environ, PA_VERIFY_PART_TOKENS="384")
    env.pop("PA_VERIFY_KERNEL", None)
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
