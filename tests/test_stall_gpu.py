"""Failure detection on the device without a fault: every wait of the kernels
on a bulk copy is bounded (about a second of device time), after which the
row is flagged SPECV_ROW_DEVICE_TIMEOUT and the kernel returns.  The test hook
SPECV_TEST_STALL makes one such wait run out by arming a ring barrier for 16
bytes more than its copy brings (a barrier that nothing completes): "A:0" in
the row-statistics kernel (item 0 = batch row 0, position 0, chunk 0), "B:<b>"
in the decision kernel's residual pass of a batch row b that rejects a draft.
Each case runs tests/_stall_case.py in a fresh process."""
import os
import subprocess
import sys

import pytest

import oracle
from speculative_decoding_verification_50_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_50_gb300 import _build
    _build.build()


def rejecting_row():
    """A sampled batch row of the stall case whose round rejects a draft, so
    that the decision kernel runs the residual pass through its ring."""
    from tests._stall_case import SPEC
    d = wl.generate(SPEC)
    o = oracle.verify(d["target"], d["draft"], d["tokens"], d["temperature"], d["uniforms"],
                      lib=oracle.load(oracle.build()))
    rows = [b for b in range(SPEC.B)
            if d["temperature"][b] > 0 and o["accept_len"][b] < SPEC.K and o["boundary"][b] == 0]
    assert rows, o["accept_len"]
    return rows[0]


def run_case(stall, row):
    p = subprocess.run([sys.executable, "-m", "tests._stall_case", str(row)], cwd=ROOT,
                       env=dict(os.environ, SPECV_TEST_STALL=stall), capture_output=True,
                       text=True, timeout=300)
    assert p.returncode == 0 and "stall case ok" in p.stdout, p.stdout[-2000:] + p.stderr[-3000:]
    print(p.stdout.strip())


def test_statistics_wait_runs_out(built):
    run_case("A:0", 0)


def test_decision_wait_runs_out(built):
    b = rejecting_row()
    run_case(f"B:{b}", b)
