"""bench.py's host logic on CPU: the layouts it hands to the library (packed
rows by per-row draft counts, the sampler's rows, MSS nodes) and the
algorithmic bytes the roofline divides by.  Checked against the unpacked
generator output and against the byte counts of the configurations."""
import dataclasses
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_verification_50_gb300 import workloads as wl  # noqa: E402


def small(name, **kw):
    spec, _ = bench.WORKLOADS[name]
    return dataclasses.replace(spec, **{"B": 6, "V": 40, **kw})


def test_algorithmic_bytes_of_the_configurations():
    """The byte counts of the benchmark plan: B(2K+1)V s for verification,
    B(2K+2)V s for the fused SSD round."""
    ab = bench.algorithmic_bytes(wl.SPECS["cfg5"])
    assert ab["verify"] == 2_647_130_112
    ab = bench.algorithmic_bytes(wl.SPECS["cfg4"])
    assert ab["verify"] == 73_875_456 and ab["predict"] == 41_041_920 and ab["step_fused"] == 82_083_840
    assert bench.algorithmic_bytes(wl.SPECS["cfg3"])["verify"] == 147_750_912
    assert bench.algorithmic_bytes(wl.SPECS["cfg1"])["verify"] == 147_456
    assert bench.algorithmic_bytes(wl.SPECS["cfg2a"])["verify"] == 2_821_632
    spec, _ = bench.WORKLOADS["cfg5-ssd"]
    assert bench.lay_out(wl.generate(dataclasses.replace(spec, B=1, V=64)),
                         dataclasses.replace(spec, B=1, V=64), None)["bytes"] == 18 * 64 * 4


def test_draft_counts_depend_on_the_row_only():
    K = 8
    full = bench.draft_counts(0, 40, K)
    assert ((full >= 0) & (full <= K)).all() and len(set(full.tolist())) > 3
    assert np.array_equal(bench.draft_counts(10, 5, K), full[10:15])


def test_ragged_layout_packs_rows_by_count():
    spec = small("cfg5-ragged")
    data = wl.generate(spec)
    lay = bench.lay_out(data, spec, "ragged", first_row=3)
    kb = bench.draft_counts(3, spec.B, spec.K)
    assert np.array_equal(lay["cu"], np.cumsum(kb))
    t0 = d0 = 0
    for b in range(spec.B):
        k = int(kb[b])
        assert np.array_equal(lay["target"][t0 + 0:t0 + k + 1], data["target"][b, :k + 1])
        assert np.array_equal(lay["draft"][d0:d0 + k], data["draft"][b, :k])
        assert np.array_equal(lay["tokens"][d0:d0 + k], data["tokens"][b, :k])
        # uniforms: the row's k accept uniforms, then its bonus uniform
        assert np.array_equal(lay["uniforms"][t0:t0 + k], data["uniforms"][b, :k])
        assert lay["uniforms"][t0 + k] == data["uniforms"][b, -1]
        t0 += k + 1
        d0 += k
    assert lay["target"].shape[0] == t0 == lay["rows"]
    assert lay["bytes"] == int((2 * kb + 1).sum()) * spec.V * spec.elem_bytes


def test_sampler_layout_takes_every_draft_row():
    spec = small("cfg5-sample")
    data = wl.generate(spec)
    lay = bench.lay_out(data, spec, "sample")
    n = spec.B * (spec.K + 1)
    assert lay["draft"].shape == (n, spec.V) and lay["rows"] == n
    assert np.array_equal(lay["draft"][spec.K + 1], data["draft"][1, 0])
    assert np.array_equal(lay["temperature"], np.repeat(data["temperature"], spec.K + 1))
    assert np.array_equal(lay["uniforms"], data["uniforms"].reshape(-1))
    assert lay["bytes"] == n * spec.V * spec.elem_bytes


def test_no_draft_and_mss_layouts():
    spec = small("cfg5-nodraft")
    lay = bench.lay_out(wl.generate(spec), spec, "nodraft")
    assert lay["draft"] is None and lay["bytes"] == spec.B * (spec.K + 1) * spec.V * spec.elem_bytes
    spec = small("cfg5-mss")
    data = bench.gen_data(spec, list(range(5)), "mss", "cfg5-mss")
    lay = bench.lay_out(data, spec, "mss")
    assert lay["tokens"].shape == (5, bench.MSS_M["cfg5-mss"]) and lay["rows"] == 5
    assert lay["bytes"] == 2 * 5 * spec.V * spec.elem_bytes


def test_clock_summary_reports_median_and_throttle_reasons():
    """The clocks object of the bench line from nvidia-smi's CSV samples:
    median SM clock under load, the maximum, and every throttle reason seen
    active (a rejected run shows hw_slowdown or a thermal slowdown)."""
    class Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s = bench.ClockSampler(None)
    s.proc = Done()
    s.lines = [
        "0, 2070, 2070, 900.1, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1100.0, Active, Not Active, Not Active, Not Active",
        "garbled line",
        "0, [N/A], 2070, 0, Not Active, Not Active, Not Active, Not Active",
    ]
    c = s.stop()
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0 and c["samples"] == 3
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert bench.ClockSampler(None).stop()["reasons"] == ["nvidia-smi unavailable"]
