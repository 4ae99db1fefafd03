"""The tcgen05 form of the cluster attention (DF_ATTN_TC=1): the bf16 parity
and lossless tests again, in a child process with the switch on (the library
reads it once per process).  The 27B-class width has five query heads per KV
head and keeps the mma.sync kernel, so it is left out here."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_tcgen05_attention_parity_and_lossless():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    env = dict(os.environ, DF_ATTN_TC="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_bf16.py", "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider", "-k", "not 27b"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "failed" not in r.stdout
