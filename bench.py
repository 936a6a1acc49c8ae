#!/usr/bin/env python3
"""Throughput of the verification / outcome-prediction hot path on GB300.

One step = one pass of the whole hot path over one batch through the C ABI:
specv_ssd_round (row statistics, accept test, residual/bonus draw, top-F
outcome keys at every lookahead and the hit check, fused over one read of the
logits) for the SSD workloads, specv_verify for the verify-only ones.

Default workload "cfg5-ssd": B=256, K=8, V=152064, fp32 Zipf-like logits
(config 5) with the draft logits at K+1 lookaheads so the step also predicts
F=6 outcome keys per lookahead and checks the hit (the full SSD round).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Under torchrun (N > 1) every rank runs its own batch (weak scaling: batch
rows r*B .. (r+1)*B-1 of one global batch); no collective touches the data
path; the timed region is bracketed by barriers and the max over ranks is
reported.  Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from speculative_decoding_verification_50_gb300 import workloads as wl  # noqa: E402

METRIC = "verify rows/s (B·(K+1) vocab rows) and achieved HBM GB/s vs GB300 peak"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    "cfg5-ssd": (dataclasses.replace(wl.SPECS["cfg5"], name="cfg5-ssd", ssd=True, F=6),
                 "config 5 (B=256, K=8, V=152064, fp32 Zipf-like logits) as a full SSD round: "
                 "verify + top-6 outcome keys at K+1 lookaheads + hit check"),
    "cfg5-ssd-geo": (dataclasses.replace(wl.SPECS["cfg5"], name="cfg5-ssd-geo", ssd=True, F=6),
                     "config 5 as a full SSD round with the Theorem 12 geometric fan-out "
                     "(a=0.5, r=1, 54 keys over the K+1 lookaheads) + hit check"),
    "cfg5-ssd-saguaro": (dataclasses.replace(wl.SPECS["cfg5"], name="cfg5-ssd-saguaro", ssd=True, F=6),
                         "config 5 as a full SSD round whose drafts came from Saguaro sampling "
                         "sigma_{6,0.3} (q = sigma in the accept test and the residual)"),
    "cfg5-sample": (dataclasses.replace(wl.SPECS["cfg5"], name="cfg5-sample", ssd=True),
                    "Saguaro draft-side sampling sigma_{6,0.3} of the B*(K+1) = 2304 draft rows "
                    "of a config 5 round (V=152064 fp32), one token per row"),
    "cfg5-ragged": (dataclasses.replace(wl.SPECS["cfg5"], name="cfg5-ragged"),
                    "config 5 with per-row draft counts K_b in 0..8 (seeded), rows packed "
                    "by cu_num_draft_tokens, verify only"),
    "cfg5-nodraft": (dataclasses.replace(wl.SPECS["cfg5"], name="cfg5-nodraft"),
                     "config 5 without draft logits (SPECV_NO_DRAFT_PROBS), verify only"),
    "cfg5-mss": (dataclasses.replace(wl.SPECS["cfg5"], name="cfg5-mss", B=2048),
                 "multi-step speculative sampling (MSS) at 2048 token-tree nodes, 3 candidate "
                 "children each drawn from q, config 5 logits (V=152064 fp32)"),
    "cfg5": (wl.SPECS["cfg5"], "config 5 (B=256, K=8, V=152064, fp32 Zipf-like logits), verify only"),
    "cfg4": (wl.SPECS["cfg4"], "config 4 (B=32, K=4, V=128256, bf16, F=6): verify + predict + hit"),
    "cfg3": (wl.SPECS["cfg3"], "config 3 (B=64, K=4, V=128256, bf16, T in {0,0.6,1}), verify only"),
    "cfg2a": (wl.SPECS["cfg2a"], "config 2a (B=1, K=5, V=128256, bf16, greedy), verify only"),
    "cfg2b": (wl.SPECS["cfg2b"], "config 2b (B=1, K=5, V=128256, bf16, T=0.7), verify only"),
    "cfg1": (wl.SPECS["cfg1"], "config 1 (B=1, K=4, V=4096, fp32, T=1), verify only"),
    "cfg4-predict": (wl.SPECS["cfg4"], "config 4's draft rows (B=32, K+1=5, V=128256, bf16, F=6) "
                                       "through the separate calls: specv_predict_outcomes, then "
                                       "specv_check_hit on a fixed outcome"),
}

# Workloads in another layout: rows packed by per-row draft counts, or
# verification without draft logits.
LAYOUT = {"cfg5-ragged": "ragged", "cfg5-nodraft": "nodraft", "cfg5-sample": "sample",
          "cfg5-mss": "mss", "cfg4-predict": "predict"}

# Candidates per token-tree node of the MSS workloads.
MSS_M = {"cfg5-mss": 3}

# Saguaro sampling (F_s, C) of the drafts (SSD rounds) or of the sampler.
SAGUARO = {"cfg5-ssd-saguaro": (6, 0.3), "cfg5-sample": (6, 0.3)}

# Workloads whose keys follow the geometric fan-out: (acceptance rate a,
# power-law exponent r, key budget over the K+1 lookaheads).
GEOMETRIC = {"cfg5-ssd-geo": (0.5, 1.0, 54)}

KERNEL_DIR = os.path.join(ROOT, "speculative_decoding_verification_50_gb300", "csrc")
# Sources of the row-statistics kernel, the one the roofline reports on.
# kernel A's sources and the host code that sizes its chunks: a recorded DRAM
# traffic figure holds only for the code it was captured with
KERNEL_SRCS = ("stats_kernel.cuh", "specv_device.cuh", "specv_common.cuh", "specv_api.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ---------------------------------------------------------------------------
# distributed plumbing (also exercised by tests/test_bench_dist.py on gloo)

def dist_env() -> tuple:
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_rows(rank: int, world: int, B: int) -> list:
    """Weak scaling: rank r owns rows r*B .. r*B+B-1 of a global batch."""
    return list(range(rank * B, (rank + 1) * B))


def reduce_max(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------

def measured_peak() -> tuple:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SRCS:
        with open(os.path.join(KERNEL_DIR, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """ncu DRAM bytes per verify launch recorded for this kernel source, or None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(workload)
    except Exception:
        return None
    if not rec or rec.get("kernel_hash") != kernel_hash():
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS),
               "--format=csv,noheader,nounits", "-lms", "50"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(torch, dev) -> str | None:
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        return "GPU-" + str(u)
    except Exception:
        return None


def algorithmic_bytes(spec) -> dict:
    s = spec.elem_bytes
    verify = spec.B * (2 * spec.K + 1) * spec.V * s
    predict = spec.B * (spec.K + 1) * spec.V * s if spec.F else 0
    fused = spec.B * (2 * spec.K + 2) * spec.V * s if spec.F else verify
    return dict(verify=verify, predict=predict, step_fused=fused)


def draft_counts(first_row: int, n: int, K: int) -> np.ndarray:
    """Seeded per-row draft counts in 0..K; row b's count depends on b only."""
    return np.array([np.random.default_rng((20261202, b)).integers(0, K + 1)
                     for b in range(first_row, first_row + n)], np.int64)


def gen_data(spec, rows, mode, workload: str) -> dict:
    """Seeded inputs of the given batch rows (token-tree nodes for MSS)."""
    if mode == "mss":
        return wl.generate_mss(spec, MSS_M[workload], rows=rows)
    return wl.generate(spec, rows=rows)


def lay_out(data, spec, mode, first_row: int = 0) -> dict:
    """The call's inputs in the workload's layout, with its target rows (the
    metric's rows) and its algorithmic bytes (every row it must normalise)."""
    if mode == "mss":  # one target and one draft row per node; a node is a metric row
        n, s = data["target"].shape[0], spec.elem_bytes
        return dict(target=data["target"], draft=data["draft"], tokens=data["candidates"],
                    temperature=data["temperature"], uniforms=data["uniforms"], cu=None,
                    rows=n, bytes=2 * n * spec.V * s)
    B, K, V, s = data["tokens"].shape[0], spec.K, spec.V, spec.elem_bytes
    lay = dict(target=data["target"], draft=data["draft"], tokens=data["tokens"],
               temperature=data["temperature"], uniforms=data["uniforms"], cu=None)
    if mode == "ragged":
        kb = draft_counts(first_row, B, K)
        lay.update(
            cu=np.cumsum(kb).astype(np.int32),
            target=np.concatenate([data["target"][b, :kb[b] + 1] for b in range(B)]),
            draft=np.concatenate([data["draft"][b, :kb[b]] for b in range(B)]),
            tokens=np.concatenate([data["tokens"][b, :kb[b]] for b in range(B)]).astype(np.int32),
            uniforms=np.concatenate([np.append(data["uniforms"][b, :kb[b]], data["uniforms"][b, -1])
                                     for b in range(B)]).astype(np.float32))
        lay.update(rows=int((kb + 1).sum()), bytes=int((2 * kb + 1).sum()) * V * s)
    elif mode == "nodraft":
        lay.update(draft=None, rows=B * (K + 1), bytes=B * (K + 1) * V * s)
    elif mode == "predict":  # the draft rows at K+1 lookaheads, ranked once
        lay.update(target=None, rows=B * (K + 1), bytes=B * (K + 1) * V * s)
    elif mode == "sample":  # every draft row of the round, one draw each
        rows = data["draft"].reshape(-1, V)
        n = rows.shape[0]
        lay.update(target=None, draft=rows, tokens=np.zeros(0, np.int32),
                   temperature=np.repeat(data["temperature"], K + 1).astype(np.float32),
                   uniforms=np.resize(data["uniforms"].reshape(-1), n).astype(np.float32),
                   rows=n, bytes=n * V * s)
    else:
        ab = algorithmic_bytes(dataclasses.replace(spec, B=B))
        lay.update(rows=B * (K + 1), bytes=ab["step_fused"] if spec.F else ab["verify"])
    return lay


def time_oracle(lay, spec, nthreads: int, mode=None, saguaro=None) -> float:
    import oracle
    t0 = time.perf_counter()
    if mode == "mss":
        oracle.mss(lay["target"], lay["draft"], lay["tokens"], lay["temperature"], lay["uniforms"],
                   nthreads=nthreads)
        return time.perf_counter() - t0
    if mode == "sample":
        oracle.saguaro_sample(lay["draft"], lay["temperature"], *saguaro, lay["uniforms"])
        return time.perf_counter() - t0
    if mode == "predict":
        p = oracle.predict(lay["draft"], lay["tokens"], spec.F, nthreads=nthreads)
        n = np.zeros(lay["tokens"].shape[0], np.int32)
        oracle.check_hit(p["keys"], n, np.zeros((n.size, spec.K + 1), np.int32))
        return time.perf_counter() - t0
    if mode == "ragged":
        oracle.verify_ragged(lay["target"], lay["draft"], lay["cu"], lay["tokens"],
                             lay["temperature"], lay["uniforms"], spec.K, nthreads=nthreads)
        return time.perf_counter() - t0
    o = oracle.verify(lay["target"], lay["draft"], lay["tokens"], lay["temperature"],
                      lay["uniforms"], nthreads=nthreads, no_draft=(mode == "nodraft"),
                      saguaro=saguaro)
    if spec.F:
        p = oracle.predict(lay["draft"], lay["tokens"], spec.F, nthreads=nthreads)
        oracle.check_hit(p["keys"], o["accept_len"], o["out_tokens"])
    return time.perf_counter() - t0


def oracle_threads(mode, cores: int, rows: int) -> int:
    """Threads the oracle runs on: OpenMP over batch rows (or nodes), except
    the sampler's, which is one loop."""
    return 1 if mode == "sample" else max(1, min(cores, rows))


def cpu_baseline(spec, budget_s: float = 12.0, mode=None, saguaro=None, workload: str = "") -> dict:
    """The oracle on a bounded sample of the workload, on this host's cores."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    rows = list(range(min(spec.B, max(1, cores))))
    lay = lay_out(gen_data(spec, rows, mode, workload), spec, mode)
    t = time_oracle(lay, spec, cores, mode, saguaro)
    per_row = t / len(rows)
    # one batch row alone: the loops run on one thread (parallel over rows only)
    one = lay_out(gen_data(spec, [0], mode, workload), spec, mode)
    single = one["rows"] / time_oracle(one, spec, 1, mode, saguaro)
    n = int(min(spec.B, max(len(rows), budget_s / max(per_row, 1e-6))))
    if n > len(rows):
        lay = lay_out(gen_data(spec, list(range(n)), mode, workload), spec, mode)
        t = time_oracle(lay, spec, cores, mode, saguaro)
    value = lay["rows"] / t
    return {"value": value, "unit": "rows/s", "cores": oracle_threads(mode, cores, n), "kind": "oracle",
            "single_thread_value": round(single, 2),
            "sample": f"{n} of {spec.B} batch rows of {spec.name} "
                      f"({'MSS' if mode == 'mss' else 'verify+predict+hit' if spec.F else 'verify'}), "
                      f"fp64 C, {'one thread' if mode == 'sample' else 'OpenMP over rows'}, "
                      f"{t:.1f} s"}


# ---------------------------------------------------------------------------
# host placement of the pinned input buffers (the end-to-end figure is bound
# by the host-to-device link)

def numa_nodes() -> list:
    import glob
    return sorted(int(os.path.basename(n)[4:]) for n in glob.glob("/sys/devices/system/node/node[0-9]*"))


def pages_node(addr: int) -> dict:
    """Pages per NUMA node of the mapping holding host address `addr`
    (from /proc/self/numa_maps), e.g. {"N0": 65536}; {} if not found."""
    try:
        with open("/proc/self/numa_maps") as f:
            maps = f.read().splitlines()
        with open("/proc/self/maps") as f:
            ranges = f.read().splitlines()
    except OSError:
        return {}
    for ln in ranges:
        lo, hi = (int(x, 16) for x in ln.split()[0].split("-"))
        if lo <= addr < hi:
            for m in maps:
                if int(m.split()[0], 16) == lo:
                    return {kv.split("=")[0]: int(kv.split("=")[1]) for kv in m.split()[2:]
                            if kv.startswith("N") and "=" in kv}
    return {}


def gpu_numa_node(torch, dev):
    p = torch.cuda.get_device_properties(dev)
    bus = getattr(p, "pci_bus_id", None)
    dom = getattr(p, "pci_domain_id", 0)
    devid = getattr(p, "pci_device_id", None)
    if bus is None or devid is None:
        return None
    path = f"/sys/bus/pci/devices/{dom:04x}:{bus:02x}:{devid:02x}.0/numa_node"
    try:
        with open(path) as f:
            return int(f.read().strip())
    except (OSError, ValueError):
        return None


# ---------------------------------------------------------------------------

# The configurations timed after the headline in the default run (one GPU).
SIDE_CONFIGS = ("cfg1", "cfg2a", "cfg2b", "cfg3", "cfg4")


def prepare(name, args, torch, sv, dev, rank, world, batch=0):
    """Inputs, outputs and one call of workload `name` on this rank's shard."""
    spec, desc = WORKLOADS[name]
    if batch:
        spec = dataclasses.replace(spec, B=batch)
        desc += f" [B overridden to {batch}]"
    fanout = None
    if name in GEOMETRIC:
        fanout, _ = sv.specv_geometric_fanout(spec.K, *GEOMETRIC[name], max_f=32)
        spec = dataclasses.replace(spec, F=max(1, max(fanout)))
        desc += f" [F_k = {fanout}]"
    mode = LAYOUT.get(name)
    saguaro = SAGUARO.get(name)
    data = gen_data(spec, shard_rows(rank, world, spec.B), mode, name)
    lay = lay_out(data, spec, mode, first_row=rank * spec.B)
    B, K, V, F = spec.B, spec.K, spec.V, spec.F
    is_bf16 = spec.dtype == wl.BF16

    def host_logits(a):
        t = torch.from_numpy(a)
        return t.view(torch.bfloat16) if is_bf16 else t

    h = dict(target=host_logits(lay["target"]).pin_memory() if lay["target"] is not None else None,
             draft=host_logits(lay["draft"]).pin_memory() if lay["draft"] is not None else None,
             tok=torch.from_numpy(lay["tokens"]).pin_memory(),
             temp=torch.from_numpy(lay["temperature"]).pin_memory(),
             unif=torch.from_numpy(lay["uniforms"]).pin_memory(),
             cu=torch.from_numpy(lay["cu"]).pin_memory() if lay["cu"] is not None else None)
    d = {k: (v.to(dev) if v is not None else None) for k, v in h.items()}
    pq_shape = (max(1, h["tok"].numel()),) if mode == "ragged" else \
        (lay["rows"],) if mode == "sample" else (B, K)
    i32 = dict(dtype=torch.int32, device=dev)
    n_out = lay["rows"] if mode == "sample" else B
    outs = dict(accept_len=torch.empty(B, **i32), out_tokens=torch.empty((B, K + 1), **i32),
                p_draft=torch.empty(pq_shape, dtype=torch.float32, device=dev),
                q_draft=torch.empty(pq_shape, dtype=torch.float32, device=dev),
                row_status=torch.empty(n_out, **i32))
    lib = sv.load_library()
    code = sv.SPECV_BF16 if is_bf16 else sv.SPECV_FP32
    ws = torch.empty(max(1, lib.specv_verify_workspace_bytes(B, K, V, code)), dtype=torch.uint8, device=dev)
    s_tok = None
    if mode == "sample":
        ws = torch.empty(max(1, lib.specv_saguaro_workspace_bytes(lay["rows"], V, saguaro[0], code)),
                         dtype=torch.uint8, device=dev)
        s_tok = torch.empty(lay["rows"], **i32)
    if mode == "mss":
        Mc = MSS_M[name]
        outs = dict(accepted=torch.empty(B, **i32), out_token=torch.empty(B, **i32),
                    accept_prob=torch.empty((B, Mc), dtype=torch.float32, device=dev),
                    row_status=torch.empty(B, **i32))
        ws = torch.empty(max(1, lib.specv_mss_workspace_bytes(B, Mc, V, code)), dtype=torch.uint8, device=dev)
    keys = key_logits = hit = None
    if mode == "predict":  # a fixed outcome to check against: one verification of the batch
        t_dev = host_logits(data["target"]).to(dev)
        v = sv.specv_verify(t_dev, d["draft"][:, :K], d["tok"], d["temp"], d["unif"])
        fixed_n, fixed_tok = v["accept_len"], v["out_tokens"]
        del t_dev
    if F:
        keys = torch.empty((B, K + 1, F), **i32)
        key_logits = torch.empty((B, K + 1, F), dtype=torch.float32, device=dev)
        hit = torch.empty(B, dtype=torch.uint8, device=dev)
        ws = torch.empty(max(1, lib.specv_ssd_workspace_bytes(B, K, V, F, code)), dtype=torch.uint8, device=dev)
    if mode == "predict":
        ws = torch.empty(max(1, lib.specv_predict_workspace_bytes(B, K, V, F, code)), dtype=torch.uint8,
                         device=dev)
    ws.zero_()
    stream = torch.cuda.current_stream(dev)
    launches = [0]
    per_call = [0]  # our launches in the last call

    def call(ev=None):
        if ev is not None:
            sv.specv_set_split_event(ev[1])  # recorded between the call's two launches
            ev[0].record(stream)
        if mode == "predict":  # a4 then a5 through their own entry points
            sv.specv_predict_outcomes(d["draft"], d["tok"], F, keys=keys, key_logits=key_logits,
                                      row_status=outs["row_status"], workspace=ws)
            n_pred = sv.last_launch_count()
            sv.specv_check_hit(keys, fixed_n, fixed_tok, hit=hit)
            per_call[0] = n_pred + sv.last_launch_count()
            launches[0] += per_call[0]
            if ev is not None:
                ev[2].record(stream)
                sv.specv_set_split_event(None)
            return
        if mode == "sample":
            sv.specv_saguaro_sample(d["draft"], d["temp"], *saguaro, d["unif"], tokens=s_tok,
                                    q=outs["q_draft"], row_status=outs["row_status"], workspace=ws)
        elif mode == "mss":
            sv.specv_mss_verify(d["target"], d["draft"], d["tok"], d["temp"], d["unif"], workspace=ws, **outs)
        elif F:  # the fused SSD round: verify + outcome keys + hit in one pass
            sv.specv_ssd_round(d["target"], d["draft"], d["tok"], d["temp"], d["unif"], F, keys=keys,
                               key_logits=key_logits, hit=hit, workspace=ws, fanout=fanout,
                               saguaro=saguaro, **outs)
        elif mode == "ragged":
            sv.specv_verify_ragged(d["target"], d["draft"], d["cu"], d["tok"], d["temp"], d["unif"], K,
                                   workspace=ws, **outs)
        else:
            sv.specv_verify(d["target"], d["draft"], d["tok"], d["temp"], d["unif"], workspace=ws, **outs)
        per_call[0] = sv.last_launch_count()
        launches[0] += per_call[0]
        if ev is not None:
            ev[2].record(stream)
            sv.specv_set_split_event(None)

    in_bytes = sum(t.numel() * t.element_size() for t in (d["target"], d["draft"]) if t is not None)
    return dict(name=name, spec=spec, desc=desc, mode=mode, saguaro=saguaro, fanout=fanout, lay=lay,
                h=h, d=d, outs=outs, keys=keys, hit=hit, s_tok=s_tok, call=call, launches=launches,
                per_call=per_call,
                in_bytes=in_bytes, stream=stream, is_bf16=is_bf16)


def make_flush(torch, dev):
    """Between timed calls whose inputs fit in L2 (outside their events):
    write a buffer twice the L2, then read another as large, so the call
    starts with an L2 of clean, unrelated lines rather than paying for the
    flush's write-backs."""
    fw = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    fr = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        fw.zero_()
        fr.sum()
    return flush


def submit_us(torch, w, barrier) -> float:
    """Host time to enqueue one call (Python, ctypes, the library's checks),
    measured with the GPU kept busy so the host never waits for it."""
    barrier()
    torch.cuda._sleep(50_000_000)  # about 25 ms of GPU time: the host runs ahead
    t0 = time.perf_counter()
    for _ in range(20):
        w["call"]()
    dt = (time.perf_counter() - t0) / 20
    barrier()
    return dt * 1e6


def gpu_wait(torch, us: float) -> None:
    """A GPU-side wait of about `us` microseconds (at up to 2.1 GHz) queued
    before a timed group of calls, so every call of the group is on the
    stream before the GPU reaches it: the events then time the GPU's work,
    not the host's enqueueing."""
    torch.cuda._sleep(int(us * 2100))


def time_calls(torch, w, steps, reps, flush, barrier, t_sub):
    """K steps of `reps` calls each; returns (per-call ms of each step, our
    kernel launches).  Inputs that fit in L2 are timed call by call with an
    L2 flush before each (outside the events); larger inputs back to back."""
    stream, call, launches = w["stream"], w["call"], w["launches"]
    launches[0] = 0
    barrier()
    per_step = []
    if flush is None:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for k in range(steps):
            gpu_wait(torch, 1.5 * reps * t_sub + 20)
            ev[k][0].record(stream)
            for _ in range(reps):
                call()
            ev[k][1].record(stream)
        barrier()
        per_step = [e[0].elapsed_time(e[1]) / reps for e in ev]
    else:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps * reps)]
        for k in range(steps * reps):
            flush()
            gpu_wait(torch, 1.5 * t_sub + 20)
            ev[k][0].record(stream)
            call()
            ev[k][1].record(stream)
        barrier()
        t = [e[0].elapsed_time(e[1]) for e in ev]
        per_step = [sum(t[k * reps:(k + 1) * reps]) / reps for k in range(steps)]
    return per_step, launches[0]


def time_split(torch, w, n, flush, barrier, t_sub):
    """n calls with an event between the call's two launches: per-call
    (call ms, first-launch ms, second-launch ms)."""
    stream, call = w["stream"], w["call"]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for e in evs:  # create the events (a torch event exists once recorded)
        e[1].record(stream)
    barrier()
    for k in range(n):
        if flush is not None:
            flush()
        gpu_wait(torch, 1.5 * t_sub + 20)
        call(evs[k])
    barrier()
    return ([e[0].elapsed_time(e[2]) for e in evs], [e[0].elapsed_time(e[1]) for e in evs],
            [e[1].elapsed_time(e[2]) for e in evs])


def measure(torch, w, steps, warmup, target_s, barrier, dev, peak):
    """The headline timing of one workload: `steps` steps, each the mean of
    enough repeated calls that the timed region lasts about target_s."""
    for _ in range(warmup):
        w["call"]()
    barrier()
    flush = make_flush(torch, dev) if w["in_bytes"] <= L2_BYTES else None
    if flush is not None:
        flush()
        barrier()
    t_sub = submit_us(torch, w, barrier)
    # a short probe of the call time sets the repeats per step
    probe, _ = time_calls(torch, w, 2, 3, flush, barrier, t_sub)
    t_call = max(1e-3, min(probe))
    reps = max(1, int(np.ceil(target_s * 1e3 / (steps * t_call))))
    if flush is None:  # keep each step's queued wait short
        reps = min(reps, max(1, int(20_000 / max(t_sub, 1.0))))
    per_step, launches = time_calls(torch, w, steps, reps, flush, barrier, t_sub)
    ms_call = statistics.mean(per_step)
    hot = None
    if flush is not None:  # the same calls back to back, inputs left in L2
        hs, _ = time_calls(torch, w, max(1, steps // 4), reps, None, barrier, t_sub)
        hot = statistics.mean(hs)
    n_split = min(steps * reps, 2000)
    call_ms, first_ms, second_ms = time_split(torch, w, n_split, flush, barrier, t_sub)
    kb = w["lay"]["bytes"]
    f_ms, s_ms = statistics.mean(first_ms), statistics.mean(second_ms)
    dominant = 0 if f_ms >= s_ms else 1  # the longer of the two timed parts
    return dict(per_step=per_step, reps=reps, launches=launches, ms=ms_call, hot=hot,
                call_ms=call_ms, first_ms=first_ms, second_ms=second_ms, dominant=dominant,
                kernel_ms=max(f_ms, s_ms), stream_ms=f_ms, submit_us=t_sub,
                gbs=kb / (ms_call / 1e3) / 1e9, frac=kb / (ms_call / 1e3) / 1e9 / peak)


def spawn_ranks(args, argv) -> int:
    """`--gpus N` outside torchrun: start N ranks of this script on this
    node, one per local GPU (NCCL for the two timing reductions; gloo on the
    host with --dry-run), and return the worst exit code.  Rank 0 prints."""
    n = args.gpus
    if not args.dry_run:
        import torch
        have = torch.cuda.device_count() if torch.cuda.is_available() else 0
        if have < n:
            print(json.dumps({"error": f"--gpus {n} asks for {n} GPUs; this node has {have}"}), flush=True)
            return 2
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE=str(n), LOCAL_RANK=str(r),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__)] + list(argv), env=env))
    rc = 0
    for p in procs:
        rc = max(rc, p.wait())
    return rc


def run_dry(args) -> None:
    """The multi-rank plumbing on the host (gloo, no GPU, no kernels): process
    group, barriers, the max over ranks of a stand-in step time and the sum of
    the shards' rows.  Prints a line marked dry_run; it measures nothing."""
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1:
        dist.init_process_group("gloo")
    spec, desc = WORKLOADS[args.workload]
    rows = float(len(shard_rows(rank, world, spec.B)) * (spec.K + 1))
    t0 = time.perf_counter()
    if world > 1:
        dist.barrier()
    dt = time.perf_counter() - t0
    ms = reduce_max(dt * 1e3, world)
    rows_total = reduce_sum(rows, world)
    if rank == 0:
        print(json.dumps({"dry_run": True, "metric": METRIC, "value": None, "unit": "rows/s",
                          "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": None, "scaling": "weak",
                          "rows_per_step_all_ranks": rows_total, "barrier_ms_max": round(ms, 3),
                          "config": {"workload": f"{args.workload}: {desc}", "B_per_gpu": spec.B}}),
              flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_ours(args) -> None:
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from speculative_decoding_verification_50_gb300 import _build
    _build.build()
    import speculative_decoding_verification_50_gb300 as sv
    sv.load_library()

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    peak, peak_kind = measured_peak()
    w = prepare(args.workload, args, torch, sv, dev, rank, world, batch=args.batch)
    spec, lay, mode, outs = w["spec"], w["lay"], w["mode"], w["outs"]
    B, K, V, F = spec.B, spec.K, spec.V, spec.F
    flush = make_flush(torch, dev) if w["in_bytes"] <= L2_BYTES else None
    for _ in range(args.warmup):
        w["call"]()
    barrier()

    sampler = ClockSampler(gpu_uuid(torch, dev))
    sampler.start()
    # the GPU idled while the sampler started: a few untimed calls bring its
    # clocks back up before the timed region
    for _ in range(3):
        if flush is not None:
            flush()
        w["call"]()
    m = measure(torch, w, args.steps, 0, args.timed_s, barrier, dev, peak)
    clocks = sampler.stop()
    ms_step = reduce_max(m["ms"], world, dev)
    rows_total = reduce_sum(float(lay["rows"]), world, dev)
    value = rows_total / (ms_step / 1e3)

    # end to end: host inputs in pinned memory, copies inside the timed region
    e2e_steps = max(2, min(args.steps, 10))
    h, d = w["h"], w["d"]
    hold = dict(n=torch.empty(B, dtype=torch.int32).pin_memory(),
                ot=torch.empty((B, K + 1), dtype=torch.int32).pin_memory(),
                keys=torch.empty((B, K + 1, F), dtype=torch.int32).pin_memory() if F else None,
                hit=torch.empty(B, dtype=torch.uint8).pin_memory() if F else None,
                st=torch.empty(lay["rows"], dtype=torch.int32).pin_memory() if mode == "sample" else None,
                tm=torch.empty(B, dtype=torch.int32).pin_memory() if mode == "mss" else None)

    def h2d_only():
        for k in ("target", "draft", "cu", "tok", "temp", "unif"):
            if d[k] is not None:
                d[k].copy_(h[k], non_blocking=True)

    def d2h_reads():
        if mode == "sample":
            hold["st"].copy_(w["s_tok"], non_blocking=True)
        elif mode == "mss":
            hold["n"].copy_(outs["accepted"], non_blocking=True)
            hold["tm"].copy_(outs["out_token"], non_blocking=True)
        elif mode == "predict":
            pass  # keys and hit below
        else:
            hold["n"].copy_(outs["accept_len"], non_blocking=True)
            hold["ot"].copy_(outs["out_tokens"], non_blocking=True)
        if F:
            hold["keys"].copy_(w["keys"], non_blocking=True)
            hold["hit"].copy_(w["hit"], non_blocking=True)

    def e2e_step():
        h2d_only()
        w["call"]()
        d2h_reads()

    # the host link alone: the same host-to-device copies, nothing else
    h2d_ms = []
    for _ in range(2):
        h2d_only()
        barrier()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(w["stream"])
        for _ in range(e2e_steps):
            h2d_only()
        c1.record(w["stream"])
        barrier()
        h2d_ms.append(c0.elapsed_time(c1) / e2e_steps)
    h2d_ms = min(h2d_ms)
    e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(w["stream"])
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(w["stream"])
    barrier()
    e2e_ms = reduce_max(e0.elapsed_time(e1), world, dev) / e2e_steps
    # the same steps again with an event between their phases (host-to-device
    # copies, the call, the device-to-host reads): where a slow step's time goes
    ph = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(e2e_steps)]
    barrier()
    for ev in ph:
        ev[0].record(w["stream"])
        h2d_only()
        ev[1].record(w["stream"])
        w["call"]()
        ev[2].record(w["stream"])
        d2h_reads()
        ev[3].record(w["stream"])
    barrier()
    phases = {name: round(statistics.mean(e[i].elapsed_time(e[i + 1]) for e in ph), 4)
              for i, name in enumerate(("h2d_ms", "call_ms", "d2h_ms"))}
    h2d_each = [e[0].elapsed_time(e[1]) for e in ph]
    phases["h2d_ms_min_max"] = [round(min(h2d_each), 4), round(max(h2d_each), 4)]
    h2d = sum(t.numel() * t.element_size() for t in h.values() if t is not None)
    d2h = (hold["st"].numel() * 4 if mode == "sample" else 2 * B * 4 if mode == "mss" else
           hold["keys"].numel() * 4 + hold["hit"].numel() if mode == "predict" else
           hold["n"].numel() * 4 + hold["ot"].numel() * 4 +
           ((hold["keys"].numel() * 4 + hold["hit"].numel()) if F else 0))
    big = h["target"] if h["target"] is not None else h["draft"]
    placement = {"numa_nodes": numa_nodes(), "gpu_numa_node": gpu_numa_node(torch, dev),
                 "pinned_input_pages": pages_node(big.data_ptr()),
                 "cpu_affinity": len(os.sched_getaffinity(0))}

    # the other configurations, after the headline (one GPU, default run)
    side = {}
    if world == 1 and args.workload == "cfg5-ssd" and not args.batch and not args.no_configs:
        side_sampler = ClockSampler(gpu_uuid(torch, dev))
        side_sampler.start()
        for name in SIDE_CONFIGS:
            ws_ = prepare(name, args, torch, sv, dev, 0, 1)
            ms_ = measure(torch, ws_, max(5, args.steps // 2), 3, 0.15, barrier, dev, peak)
            kb = ws_["lay"]["bytes"]
            side[name] = {
                "workload": WORKLOADS[name][1],
                "rows": ws_["lay"]["rows"], "algorithmic_bytes": kb,
                "ms": round(ms_["ms"], 5),
                "rows_per_s": round(ws_["lay"]["rows"] / (ms_["ms"] / 1e3), 1),
                "gbs_algorithmic": round(ms_["gbs"], 1), "frac": round(ms_["frac"], 4),
                **({"ms_hot": round(ms_["hot"], 5),
                    "frac_hot": round(kb / (ms_["hot"] / 1e3) / 1e9 / peak, 4)} if ms_["hot"] else {}),
                "timing": "cold: L2 flushed before each call" if ms_["hot"] else "back to back",
                "first_launch_ms": round(statistics.mean(ms_["first_ms"]), 5),
                "second_launch_ms": round(statistics.mean(ms_["second_ms"]), 5),
                # launch 1 alone: the logits' bytes over its split-event time
                "launch1_frac": round(kb / (ms_["stream_ms"] / 1e3) / 1e9 / peak, 4),
                "host_submit_us": round(ms_["submit_us"], 1),
                "calls_timed": len(ms_["per_step"]) * ms_["reps"],
            }
            del ws_
        side_clocks = side_sampler.stop()

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    def outcome_summary() -> dict:
        """What the last call decided (the workload's acceptance and hit rates)."""
        if mode == "sample":
            return {"rows_sampled": int(lay["rows"])}
        if mode == "predict":
            return {"hit_rate": round(float(w["hit"].float().mean().item()), 4)}
        if mode == "mss":
            acc = outs["accepted"].cpu().numpy()
            return {"candidate_accepted_rate": round(float((acc >= 0).mean()), 4),
                    "accepted_index_hist": np.bincount(acc + 1, minlength=MSS_M[args.workload] + 1).tolist()}
        n = outs["accept_len"].cpu().numpy()
        dd = {"mean_accept_len": round(float(n.mean()), 4),
              "accept_len_hist": np.bincount(n, minlength=K + 1).tolist()}
        if F:
            dd["hit_rate"] = round(float(w["hit"].float().mean().item()), 4)
        return dd

    def decision_reread() -> int | None:
        """Logit bytes the decision kernel reads again in the last call: a
        sampled batch row that rejected draft n reads target and draft row n,
        one that accepted all K drafts at most target row K (less when its draw
        is chunk-local); greedy rows read none.  Strided verification and SSD
        rounds only."""
        if mode is not None or d["draft"] is None:
            return None
        n = outs["accept_len"].cpu().numpy()
        T = np.asarray(lay["temperature"]).reshape(-1)[:len(n)]
        es = d["target"].element_size()
        rows = np.where(T > 0, np.where(n < K, 2, 1), 0)
        return int(rows.sum()) * V * es

    kernel_bytes = lay["bytes"]
    # The roofline's kernel is launch 1, the one that streams every logit once
    # (its algorithmic bytes are the logits), timed apart from the call's
    # other launches by the split event, on the launching stream.  Where the
    # later launches take longer (small, latency-bound batches), the line says
    # so under "dominant_launch".
    k_ms = m["stream_ms"]
    achieved = kernel_bytes / (k_ms / 1e3) / 1e9
    call_gbs = kernel_bytes / (ms_step / 1e3) / 1e9
    traffic = recorded_traffic(args.workload)
    kname = (f"launch 1 of {w['per_call'][0]} "
             f"({'bf16' if w['is_bf16'] else 'fp32'} {mode or ('ssd' if F else 'verify')}): "
             "streams every logit once")
    f_mean, s_mean = statistics.mean(m["first_ms"]), statistics.mean(m["second_ms"])
    # the decision kernel's own bytes and rate (launch 2, split event)
    reread = decision_reread()
    decision_line = None
    if reread is not None and s_mean > 0:
        dgbs = reread / (s_mean / 1e3) / 1e9
        decision_line = {"reread_bytes": reread, "ms": round(s_mean, 5), "gbs": round(dgbs, 1),
                         "frac": round(dgbs / peak, 4),
                         "note": "rows of the rejected position read again (at most one row "
                                 "after a full acceptance); records and candidates not counted"}
    dominant = {"launch": "1" if m["dominant"] == 0 else f"2..{w['per_call'][0]}",
                "share_of_split_call": round(max(f_mean, s_mean) / (f_mean + s_mean), 4)}
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "repeats_per_step": m["reps"],
        "ms_x_sm_mhz": round(ms_step * clocks["sm_mhz"], 2) if clocks.get("sm_mhz") else None,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; see workloads.py)",
        "config": {
            "workload": f"{args.workload}: {w['desc']}",
            "B_per_gpu": B, "K": K, "V": V, "logits": spec.dtype, "F": F,
            **({"M": MSS_M[args.workload], "nodes": B} if mode == "mss" else {}),
            **({"fanout": w["fanout"]} if w["fanout"] else {}),
            "rows_per_step_per_gpu": lay["rows"],
            "step": (f"one call; each of the {args.steps} timed steps is the mean of "
                     f"{m['reps']} calls"),
            "l2": (f"inputs {w['in_bytes'] / 1e9:.2f} GB > {L2_BYTES / 2**20:.0f} MiB L2, no flush"
                   if w["in_bytes"] > L2_BYTES else
                   f"inputs {w['in_bytes'] / 1e6:.1f} MB fit in L2: between timed calls (outside "
                   f"their events) a {2 * L2_BYTES / 2**20:.0f} MiB buffer is written, then "
                   f"another as large is read"),
        },
        "roofline": {
            "bound": "hbm",
            "kernel": kname,
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_kind": (f"of {peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                          else "of fallback"),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": kernel_bytes,
            "avg_launch_ms": round(k_ms, 5),
            "dominant_launch": dominant,
        },
        "call": {"api": ("specv_predict_outcomes + specv_check_hit" if mode == "predict" else
                         "specv_saguaro_sample" if mode == "sample" else
                         "specv_mss_verify" if mode == "mss" else
                         "specv_ssd_round" if F else "specv_verify"),
                 "launches": w["per_call"][0],
                 "ms": round(ms_step, 5),
                 **({"ms_hot": round(m["hot"], 5)} if m["hot"] is not None else {}),
                 "ms_split": round(statistics.mean(m["call_ms"]), 5),
                 "ms_split_p10_p50_p90": [round(float(x), 5) for x in
                                          np.percentile(m["call_ms"], [10, 50, 90])],
                 "first_launch_ms": round(statistics.mean(m["first_ms"]), 5),
                 "second_launch_ms": round(statistics.mean(m["second_ms"]), 5),
                 "host_submit_us": round(m["submit_us"], 1),
                 "gbs_algorithmic": round(call_gbs, 1), "frac": round(call_gbs / peak, 4)},
        "e2e": {"value": round(rows_total / (e2e_ms / 1e3), 1), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "h2d_copy_ms": round(h2d_ms, 4),
                "phases_in_step": phases,
                "h2d_gbs": round(h2d / (h2d_ms / 1e3) / 1e9, 1),
                "host_placement": placement},
        "outcome": outcome_summary(),
        **({"decision": decision_line} if decision_line else {}),
        "gpu_launches": m["launches"],
        "clocks": clocks,
    }
    if side:
        line["configs"] = side
        line["configs_clocks"] = side_clocks
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, mode=mode, saguaro=w["saguaro"], workload=args.workload)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args) -> None:
    """The oracle (CPU, fp64) as the reference arm, on a bounded sample."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    spec, desc = WORKLOADS[args.workload]
    mode = LAYOUT.get(args.workload)
    saguaro = SAGUARO.get(args.workload)
    if args.workload in GEOMETRIC:  # the oracle's cost does not depend on the split of F
        spec = dataclasses.replace(spec, F=16)
    cores = os.cpu_count() or 1
    probe = lay_out(gen_data(spec, [0], mode, args.workload), spec, mode)
    time_oracle(probe, spec, 1, mode, saguaro)  # the first call pays for loading
    t_row = time_oracle(probe, spec, 1, mode, saguaro)
    # whole run (warm-up + timed) within about a minute, but at least one batch
    # row per core so that every core has work
    per_step = 60.0 / max(1, args.steps + args.warmup)
    n = int(max(min(cores, spec.B), min(spec.B, per_step / max(t_row, 1e-6) * cores)))
    lay = lay_out(gen_data(spec, list(range(n)), mode, args.workload), spec, mode)
    for _ in range(args.warmup):
        time_oracle(lay, spec, cores, mode, saguaro)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time_oracle(lay, spec, cores, mode, saguaro)
    dt = (time.perf_counter() - t0) / args.steps
    value = lay["rows"] / dt
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 2), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; see workloads.py)",
        "config": {"workload": f"{args.workload}: {desc}", "B_per_gpu": spec.B, "K": spec.K,
                   "V": spec.V, "logits": spec.dtype, "F": spec.F,
                   "sample_rows_per_step": n},
        "cpu_baseline": {"value": round(value, 2), "unit": "rows/s", "cores": oracle_threads(mode, cores, n),
                         "kind": "oracle",
                         "sample": f"{n} of {spec.B} batch rows per step, fp64 C oracle, "
                                   f"{'one thread' if mode == 'sample' else 'OpenMP over rows'}"},
        "e2e": {"value": round(value, 2), "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="cfg5-ssd", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the configurations timed after the headline")
    ap.add_argument("--timed-s", type=float, default=1.2,
                    help="length of the headline's timed region (repeats per step)")
    ap.add_argument("--dry-run", action="store_true",
                    help="host-only run of the multi-rank plumbing (gloo, no GPU, no kernels)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override B (smaller cases for profiling captures)")
    argv = sys.argv[1:] if argv is None else list(argv)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_ranks(args, argv))
    if args.dry_run:
        run_dry(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
