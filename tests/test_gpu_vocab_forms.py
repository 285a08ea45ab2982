"""The other forms of the vocabulary step against the oracle: the vocabulary
parity cases re-run in a child process (the library reads the switch once
per process) with DG_VOCAB_SINGLE_SM=1, which selects vocab_main (one CTA per
role unit), the form used where two-CTA clusters cannot be placed, and with
DG_VOCAB_COOP=1, the paired form launched cooperatively."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("switch", ["DG_VOCAB_SINGLE_SM=1", "DG_VOCAB_COOP=1"])
def test_vocab_form_matches_the_oracle(switch):
    key, val = switch.split("=")
    env = dict(os.environ, **{key: val})
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        "tests/test_gpu_parity.py", "-k", "vocab"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
