"""The cooperative form of canvas attention against the oracle: the attention
parity and failure cases re-run in a child process (the library reads the
switch once per process) with DG_ATTN_COOP=1, which zeroes the split
counters with a memset and launches the kernel cooperatively instead of as
the programmatic dependent of a counter reset kernel."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_cooperative_attention_matches_the_oracle():
    env = dict(os.environ, DG_ATTN_COOP="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        "tests/test_gpu_parity.py", "tests/test_gpu_failure.py", "-k", "attn or append or withheld"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
