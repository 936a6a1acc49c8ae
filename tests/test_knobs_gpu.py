"""The tuning variables select other code paths of the same library: the
persistent producer-warp statistics kernel (SPECV_PERSIST), the chunk-local
draw forced on or off (SPECV_LOCAL_DRAW), ring depths (SPECV_STAGES,
SPECV_STAGES_B), chunk lengths (SPECV_ITERS) and cluster sizes
(SPECV_CLUSTER).  Each setting runs tests/_knob_case.py (an SSD round, the
Saguaro sampler and MSS against the oracle) in a fresh process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SETTINGS = [
    {"SPECV_PERSIST": "1"},
    {"SPECV_LOCAL_DRAW": "0"},
    {"SPECV_LOCAL_DRAW": "1"},
    {"SPECV_STAGES": "3"},
    {"SPECV_STAGES": "4", "SPECV_STAGES_B": "3"},
    {"SPECV_ITERS": "1"},
    {"SPECV_ITERS": "16"},
    {"SPECV_CLUSTER": "1"},
    {"SPECV_CLUSTER": "16"},
]


@pytest.fixture(scope="module")
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_50_gb300 import _build
    _build.build()


@pytest.mark.parametrize("env", SETTINGS, ids=lambda e: ",".join(f"{k}={v}" for k, v in e.items()))
def test_tuning_setting_keeps_parity(built, env):
    p = subprocess.run([sys.executable, "-m", "tests._knob_case"], cwd=ROOT,
                       env=dict(os.environ, **env), capture_output=True, text=True, timeout=600)
    assert p.returncode == 0 and "knob case ok" in p.stdout, p.stdout[-2000:] + p.stderr[-3000:]
