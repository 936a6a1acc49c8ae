"""The Saguaro sampler's two decision kernels against the oracle: one warp
per row (the default from eight rows per SM on) and one CTA per row, each
forced on every case of tests/_sampler_case.py (greedy rows, whole-row passes,
error rows, partial CTAs; fp32 and bf16) in a fresh process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_50_gb300 import _build
    _build.build()


@pytest.mark.parametrize("warp", ["1", "0"])
def test_sampler_paths_match_oracle(built, warp):
    p = subprocess.run([sys.executable, "-m", "tests._sampler_case"], cwd=ROOT,
                       env=dict(os.environ, SPECV_SAMPLE_WARP=warp), capture_output=True, text=True,
                       timeout=900)
    assert p.returncode == 0 and "sampler case ok" in p.stdout, p.stdout[-2000:] + p.stderr[-3000:]
