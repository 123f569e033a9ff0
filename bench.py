"""Benchmark of the single-token gated delta-rule decode step on GB300.

Default workload: the packed GDN decode over a slot pool, B=256 request rows, H=16 q/k heads,
HV=32 value heads, K=V=128, bf16 mixed_qkv / a / b / out, fp32 state [256, 32, 128, 128] (1.07 GB,
larger than the 129 MB L2, so every step streams the state from HBM: no L2 flush is needed), and
int32 cache indices that are a seeded permutation of the pool. One step = one
gdn_decode_step_indexed call = one kernel launch.

Prints one JSON line: state GB/s (the metric: 2*B*HV*V*K*4 bytes per step over the step time),
us/step, the roofline of the step kernel against the measured HBM copy bandwidth, an end-to-end
figure through the public API with host buffers, the fp64 CPU oracle timed on a bounded sample on
the host cores, and the SM clocks sampled during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload packed|buffered|fused] [--B 256] [--L 16] [--T 128]

Under torchrun (N > 1) each rank runs its own full workload on its own GPU (independent
replicas: the decode has no exchange step) and rank 0 reports the aggregate over ranks.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-step state HBM GB/s (% of GB300 peak), µs/step at B=256 HV=32 K=V=128"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ------------------------------------------------------------------------------------------------
# environment helpers
# ------------------------------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sources_hash(files) -> str:
    """Hash of the kernel sources with comments and blank lines removed, so that a comment edit
    does not orphan a traffic record taken on the same code."""
    h = hashlib.sha256()
    for rel in files:
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        h.update("\n".join(lines).encode())
    return h.hexdigest()[:16]


KERNEL_FILES = {
    "step": ["ssm_recurrent_decode_gb300/csrc/step_kernel.cu", "ssm_recurrent_decode_gb300/csrc/gdn_tile.cuh",
             "ssm_recurrent_decode_gb300/csrc/gdn_common.cuh"],
    "step_bf16": ["ssm_recurrent_decode_gb300/csrc/step_stage_bf16.cu", "ssm_recurrent_decode_gb300/csrc/gdn_pipe.cuh",
                  "ssm_recurrent_decode_gb300/csrc/gdn_tile.cuh", "ssm_recurrent_decode_gb300/csrc/gdn_common.cuh"],
    "buffered": ["ssm_recurrent_decode_gb300/csrc/buffered_pipe.cu", "ssm_recurrent_decode_gb300/csrc/gdn_pipe.cuh",
                 "ssm_recurrent_decode_gb300/csrc/gdn_tile.cuh", "ssm_recurrent_decode_gb300/csrc/gdn_common.cuh"],
    "fused": ["ssm_recurrent_decode_gb300/csrc/fused_pipe.cu", "ssm_recurrent_decode_gb300/csrc/gdn_pipe.cuh",
              "ssm_recurrent_decode_gb300/csrc/gdn_tile.cuh", "ssm_recurrent_decode_gb300/csrc/gdn_common.cuh",
              "ssm_recurrent_decode_gb300/csrc/gdn_chain.cuh"],
    "mamba": ["ssm_recurrent_decode_gb300/csrc/mamba_kernel.cu", "ssm_recurrent_decode_gb300/csrc/gdn_common.cuh"],
    "front": ["ssm_recurrent_decode_gb300/csrc/front.cu", "ssm_recurrent_decode_gb300/csrc/gemv_kernel.cu",
              "ssm_recurrent_decode_gb300/csrc/gemv_tc.cu", "ssm_recurrent_decode_gb300/csrc/fused_pipe.cu",
              "ssm_recurrent_decode_gb300/csrc/fused_kernel.cu", "ssm_recurrent_decode_gb300/csrc/gdn_chain.cuh"],
    "gemv": ["ssm_recurrent_decode_gb300/csrc/gemv_kernel.cu", "ssm_recurrent_decode_gb300/csrc/gemv_tc.cu",
             "ssm_recurrent_decode_gb300/csrc/gemv_internal.h", "ssm_recurrent_decode_gb300/csrc/gdn_cluster.cuh",
             "ssm_recurrent_decode_gb300/csrc/gdn_pipe.cuh", "ssm_recurrent_decode_gb300/csrc/gdn_common.cuh",
             "ssm_recurrent_decode_gb300/csrc/gdn_chain.cuh"],
}


def measured_traffic(kernel: str, workload_key: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on the kernel as it is
    now (the capture records a hash of the kernel's sources); else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(workload_key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("sources_hash") != kernel_sources_hash(KERNEL_FILES[kernel]):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples (every 200 ms) of this GPU's SM clock and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = self._smi_id(device_index)
        self.proc = None
        self.window = None

    @staticmethod
    def _smi_id(device_index):
        import torch
        try:
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            return u if u.startswith("GPU-") else f"GPU-{u}"
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            return vis.split(",")[device_index] if vis else str(device_index)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", self.dev], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 9:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if self.window and self.window[0] - 0.1 <= r[0] <= self.window[1] + 0.1]
        use = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


# ------------------------------------------------------------------------------------------------
# the fp64 CPU oracle as a baseline (bounded samples of the same workload)
# ------------------------------------------------------------------------------------------------
class OracleSampler:
    """The fp64 CPU oracle on single (slot, value head) tiles of the packed workload. Inputs come
    from gdn_synth and are prepared once; run() times only the oracle calls."""

    def __init__(self, H, HV, K, V, seed):
        import gdn_synth as syn
        import oracle
        self.oracle, self.H, self.HV, self.K, self.V = oracle, H, HV, K, V
        d = syn.packed_inputs(2, H, HV, K, V, "bf16", seed, 0)
        x = syn.bf16_bits_to_f32(d["mixed_qkv"]).astype(np.float64)
        self.a = syn.bf16_bits_to_f32(d["a"]).astype(np.float64)
        self.b = syn.bf16_bits_to_f32(d["b"]).astype(np.float64)
        self.A_log, self.dt_bias = d["A_log"], d["dt_bias"]
        self.q, self.k, self.v = oracle.split_packed(x, H, HV, K, V)
        self.pool = [(r, hv, syn.state_tile_values(seed, HV, V, K, r, hv).astype(np.float64)[None, None])
                     for r in range(2) for hv in range(4)]
        self.done = 0

    def run(self, n_tiles=None, budget_s=float("inf")):
        """Process n_tiles tiles (or until budget_s seconds of oracle time); returns (tiles, s)."""
        G = self.HV // self.H
        tiles, spent = 0, 0.0
        while spent < budget_s and (n_tiles is None or tiles < n_tiles):
            row, hv, S0 = self.pool[self.done % len(self.pool)]
            S = S0.copy()
            h = hv // G
            t0 = time.perf_counter()
            g, beta = self.oracle.gdn_gates(self.a[row:row + 1, hv:hv + 1], self.b[row:row + 1, hv:hv + 1],
                                            self.A_log[hv:hv + 1], self.dt_bias[hv:hv + 1])
            self.oracle.delta_step(self.q[row:row + 1, h:h + 1], self.k[row:row + 1, h:h + 1],
                                   self.v[row:row + 1, hv:hv + 1], g, beta, S, scale=self.K ** -0.5)
            spent += time.perf_counter() - t0
            tiles += 1
            self.done += 1
        return tiles, spent


def cpu_model() -> str:
    """The host CPU's model name as /proc/cpuinfo gives it (x86 "model name"; Arm "CPU part"
    codes with the implementer), else the platform string."""
    import platform
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = (x.strip() for x in line.split(":", 1))
                    fields.setdefault(k, v)
        if "model name" in fields:
            return fields["model name"]
        if "CPU part" in fields:
            return f"implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    except OSError:
        pass
    return platform.processor() or platform.machine()


def _oracle_worker(H, HV, K, V, seed, budget_s, barrier, results):
    """One process of the all-cores oracle timing: prepares its inputs, waits for the others, runs
    the oracle for budget_s seconds and reports its tile count."""
    sampler = OracleSampler(H, HV, K, V, seed)
    sampler.run(n_tiles=2)
    barrier.wait(timeout=300)
    results.put(sampler.run(budget_s=budget_s)[0])


def cpu_baseline(H, HV, K, V, seed, budget_s=10.0):
    """The fp64 oracle on one host thread, then split over (slot, value head) tiles on every core
    the process may use: one spawned process per core (started with spawn, so that no child
    inherits a CUDA context), all released together."""
    import multiprocessing as mp
    tiles, spent = OracleSampler(H, HV, K, V, seed).run(budget_s=budget_s)
    state_bytes = tiles * 2 * V * K * 4
    cores = len(os.sched_getaffinity(0))
    procs = []
    try:
        ctx = mp.get_context("spawn")
        barrier, results = ctx.Barrier(cores + 1), ctx.Queue()
        procs = [ctx.Process(target=_oracle_worker,
                             args=(H, HV, K, V, seed + 1 + i, budget_s / 2, barrier, results))
                 for i in range(cores)]
        for p in procs:
            p.start()
        barrier.wait(timeout=300)
        t0 = time.perf_counter()
        counts = [results.get(timeout=300) for _ in procs]
        wall = time.perf_counter() - t0
        for p in procs:
            p.join(timeout=60)
        all_cores = {"value": round(sum(counts) * 2 * V * K * 4 / wall / 1e9, 4), "unit": "GB/s",
                     "cores": cores,
                     "sample": f"{sum(counts)} tiles over {cores} processes, {wall:.1f} s wall"}
    except Exception as e:   # the single-thread figure stands on its own
        for p in procs:
            p.kill()
        all_cores = {"value": None, "cores": cores, "unavailable": f"{type(e).__name__}: {e}"}
    return {"value": round(state_bytes / spent / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "cpu": cpu_model(),
            "sample": f"{tiles} (slot, value head) tiles of the packed decode (H={H}, HV={HV}, "
                      f"K={K}, V={V}, bf16 inputs), fp64 C oracle, one thread, {spent:.1f} s",
            "all_cores": all_cores}


def packed_workload_config(B, H, HV, K, V, state_dtype="f32"):
    """The packed decode workload as both arms name it: the `workload` text and its sizes."""
    sbytes = 4 if state_dtype == "f32" else 2
    return (f"gdn packed decode over a slot pool: B={B} H={H} HV={HV} K=V={K}, bf16 mixed_qkv/a/b/out, "
            f"{state_dtype} state [{B},{HV},{V},{K}], permuted int32 cache indices",
            {"B": B, "H": H, "HV": HV, "K": K, "V": V, "input_dtype": "bf16", "state_dtype": state_dtype,
             "state_bytes_per_step": 2 * B * HV * V * K * sbytes})


# ------------------------------------------------------------------------------------------------
# byte counts that the pages print figures for (checked against them in tests/golden/)
# ------------------------------------------------------------------------------------------------
def mamba_page_bytes(B, D, N):
    """Bytes per Mamba-1 decode step by the page's own model: each (row, channel) program moves five
    N-vectors of fp32 (A row, B, C, old and new state) and about six fp32 scalars, B D (20 N + 24)
    ("Triton decode kernel + MBU analysis", Microbench, bytes-moved model)."""
    return B * D * (20 * N + 24)


def gemv_weight_bytes(N, Kd):
    """Bytes of one bf16 projection weight [N, Kd], read once per decode call."""
    return N * Kd * 2


def state_tile_bytes(V, K, state_dtype="f32"):
    """Bytes of one (slot, head) state tile [V, K] as stored."""
    return V * K * (4 if state_dtype == "f32" else 2)


def fused_layer_bytes(T, heads, D):
    """Device bytes of one fused-KDA layer's tensors at T tokens with T + 8 slots: the fp32 state
    pool, the bf16 conv state, x, raw_g, raw_beta, output gate and output, and the fp32 parameters
    (conv weights, A_log, dt_bias, norm weight), as the fused workload allocates them."""
    dim, slots = heads * D, T + 8
    return (slots * heads * D * D * 4 + slots * 3 * dim * 3 * 2 + T * 3 * dim * 2 + T * dim * 2
            + T * heads * 2 + T * dim * 2 + T * dim * 2 + 3 * dim * 4 * 4 + heads * 4 + dim * 4 + D * 4)


def cpu_baseline_buffered(H, HV, K, V, L, seed, budget_s=10.0):
    """The fp64 oracle's buffered decode on one host thread: whole L-step cycles of one request
    row (all HV value heads, bf16 inputs and rings) until budget_s seconds of oracle time, counted
    with the GPU line's mean state traffic, (1 + 1/L) V K 4 bytes per (row, value head) and step."""
    import gdn_synth as syn
    import oracle
    f64 = lambda bits: syn.bf16_bits_to_f32(bits).astype(np.float64)
    S = syn.normal_f32(seed, syn.Tag.STATE, 0, (1, HV, V, K), 1.0).astype(np.float64)
    d_c, k_c, g_c = np.zeros((1, HV, L, V)), np.zeros((1, H, L, K)), np.zeros((1, HV, L))
    steps = []
    for p in range(L):
        d = syn.packed_inputs(1, H, HV, K, V, "bf16", seed, p)
        q, k, v = oracle.split_packed(f64(d["mixed_qkv"]), H, HV, K, V)
        g, beta = oracle.gdn_gates(f64(d["a"]), f64(d["b"]), d["A_log"], d["dt_bias"])
        steps.append((q, k, v, g, beta))
    done, spent = 0, 0.0
    while spent < budget_s or done % L:
        p = done % L
        q, k, v, g, beta = steps[p]
        t0 = time.perf_counter()
        oracle.gdn_buffered(q, k, v, g, beta, S, d_c, k_c, g_c, np.array([p], np.int32), L=L,
                            ring_bf16=True, scale=K ** -0.5)
        spent += time.perf_counter() - t0
        done += 1
    traffic = done * HV * (1 + 1 / L) * V * K * 4
    return {"value": round(traffic / spent / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"{done // L} whole {L}-step cycles of one request row ({HV} value heads, H={H}, "
                      f"K={K}, V={V}, bf16 inputs and rings), fp64 C oracle, one thread, {spent:.1f} s"}


def cpu_baseline_fused(heads, D, seed, budget_s=10.0):
    """The fp64 oracle's fused KDA decode on one host thread: single-token calls (every head) until
    budget_s seconds of oracle time, counted with the GPU line's state bytes, 2 D^2 4 per
    (token, head)."""
    import gdn_synth as syn
    import oracle
    f64 = lambda bits: syn.bf16_bits_to_f32(bits).astype(np.float64)
    ins = syn.fused_inputs(1, heads, D, 2, seed)
    S = syn.normal_f32(seed, syn.Tag.STATE, 0, (2, heads, D, D), 1.0).astype(np.float64)
    cs = f64(ins["conv_state"]).reshape(2, 3 * heads * D, 3)
    args = (f64(ins["x"]), ins["conv_w"], cs, f64(ins["raw_g"]), f64(ins["raw_beta"]), ins["A_log"],
            ins["dt_bias"], S, f64(ins["out_gate"]), ins["norm_w"])
    idx = np.array([1], np.int32)
    calls, spent = 0, 0.0
    while spent < budget_s or calls == 0:
        t0 = time.perf_counter()
        oracle.fused_kda(*args, idx=idx, pad_slot=0)
        spent += time.perf_counter() - t0
        calls += 1
    return {"value": round(calls * heads * 2 * D * D * 4 / spent / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "cpu": cpu_model(),
            "sample": f"{calls} single-token calls ({heads} heads x {D}, conv update, per-key decay, "
                      f"gated RMSNorm), fp64 C oracle, one thread, {spent:.1f} s"}


def _oracle_calls(call, budget_s):
    """Times `call()` (one oracle invocation) repeatedly until budget_s seconds of oracle time,
    at least once; returns (calls, seconds)."""
    calls, spent = 0, 0.0
    while spent < budget_s or calls == 0:
        t0 = time.perf_counter()
        call()
        spent += time.perf_counter() - t0
        calls += 1
    return calls, spent


def cpu_baseline_mamba(D, N, seed, budget_s=10.0):
    """The fp64 oracle's Mamba-1 decode on one host thread: one request row (D channels, fp32
    inputs) per call until budget_s seconds, counted with the line's bytes model B D (20 N + 24)."""
    import gdn_synth as syn
    import oracle
    m = syn.mamba_inputs(1, D, N, "f32", seed)
    h = m["h"].astype(np.float64)
    calls, spent = _oracle_calls(lambda: oracle.mamba_decode(m["x"], m["dt"], m["A"], m["Bm"], m["Cm"], h,
                                                            Dskip=m["Dskip"], z=m["z"]), budget_s)
    return {"value": round(calls * mamba_page_bytes(1, D, N) / spent / 1e9, 4), "unit": "GB/s",
            "cores": 1, "kind": "oracle", "cpu": cpu_model(),
            "sample": f"{calls} single-row calls (D={D}, N={N}, fp32, D skip and silu(z) gate), fp64 C "
                      f"oracle, one thread, {spent:.1f} s"}


def cpu_baseline_gemv(T, N, Kd, seed, budget_s=10.0, rows=256):
    """The fp64 oracle's projection on one host thread: `rows` of the N weight rows (a bounded
    sample; the full fp64 matrix would take N Kd 8 bytes) against T token rows per call until
    budget_s seconds, counted with the line's bf16 weight bytes for those rows."""
    import gdn_synth as syn
    import oracle
    rows = min(rows, N)
    x = syn.bf16_bits_to_f32(syn.f32_to_bf16_bits(syn.normal_f32(seed, syn.Tag.X, 0, (T, Kd), 1.0)))
    W = syn.bf16_bits_to_f32(syn.f32_to_bf16_bits(syn.normal_f32(seed, syn.Tag.CONV_W, 0, (rows, Kd), 0.02)))
    x, W = x.astype(np.float64), W.astype(np.float64)
    calls, spent = _oracle_calls(lambda: oracle.gemv(x, W), budget_s)
    return {"value": round(calls * gemv_weight_bytes(rows, Kd) / spent / 1e9, 4), "unit": "GB/s",
            "cores": 1, "kind": "oracle", "cpu": cpu_model(),
            "sample": f"{calls} calls on {rows} of the {N} weight rows (Kd={Kd}, T={T}), fp64 C oracle, "
                      f"one thread, {spent:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    H, HV, K, V, B = 16, 32, 128, 128, args.B
    # size each step's sample so that warm-up plus timed steps stay within about 90 s
    sampler = OracleSampler(H, HV, K, V, 1)
    probe_tiles, probe_s = sampler.run(budget_s=1.0)
    t_tile = probe_s / probe_tiles
    tiles_per_step = int(max(1, min(B * HV, 90.0 / ((args.steps + args.warmup) * t_tile))))
    for _ in range(args.warmup):
        sampler.run(tiles_per_step)
    spent = 0.0
    for _ in range(args.steps):
        spent += sampler.run(tiles_per_step)[1]
    state_bytes = args.steps * tiles_per_step * 2 * V * K * 4
    value = state_bytes / spent / 1e9
    name, sizes = packed_workload_config(B, H, HV, K, V)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(spent / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, **sizes},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{tiles_per_step} of the {B * HV} (slot, value head) tiles per step "
                                   f"through the fp64 C oracle, one thread"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------------
# GPU arm: shared timing harness
# ------------------------------------------------------------------------------------------------
def max_over_ranks(values, world):
    """Element-wise maximum of a list of floats over all ranks (gloo all-reduce); identity at N=1."""
    import torch
    t = torch.tensor(values, dtype=torch.float64)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


class Harness:
    def __init__(self, args):
        import torch
        self.torch = torch
        self.args = args
        self.rank, self.world, local = dist_env()
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
        self.dev = torch.device("cuda", local)
        torch.cuda.set_device(self.dev)
        self.stream = torch.cuda.current_stream(self.dev)

    def barrier(self):
        self.torch.cuda.synchronize(self.dev)
        if self.world > 1:
            self.torch.distributed.barrier()

    def time_steps(self, step, steps, warmup, sample_clocks=True):
        """warm-up, then `steps` calls of step(i) bracketed by barrier + synchronize, timed with
        CUDA events on the launching stream. Returns (ms per step, clocks record)."""
        torch = self.torch
        for i in range(warmup):
            step(i)
        clocks = ClockSampler(self.dev.index) if sample_clocks else None
        if clocks:
            clocks.start()
        self.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        e0.record(self.stream)
        for i in range(steps):
            step(i)
        e1.record(self.stream)
        self.barrier()
        t1 = time.time()
        if clocks:
            clocks.mark(t0, t1)
        return e0.elapsed_time(e1) / steps, (clocks.stop() if clocks else None)

    def time_graph(self, step, steps, warmup, per_graph, min_replays=20, min_region_s=0.5):
        """Warm up eagerly, capture `per_graph` calls of step(i) into one CUDA graph, and time
        replays of it, each replay between its own pair of CUDA events on the replay stream
        (barrier + synchronize on both sides of the timed region). At least `min_replays` replays,
        at least `steps` calls, and at least `min_region_s` seconds of replays (so that the clock
        sampler sees several samples inside the timed region). Returns (median ms per call over
        the replays, calls timed, clocks record) and leaves the spread in self.spread. Replaying a
        graph takes the host's per-call cost out of the measurement, which otherwise dominates at
        small batches."""
        torch = self.torch
        for i in range(warmup):
            step(i)
        self.barrier()
        s = torch.cuda.Stream(self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(per_graph):
                step(i)
        # one untimed replay warms the graph and sizes the timed region
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            g.replay()
            ea.record(s)
            g.replay()
            eb.record(s)
        self.barrier()
        est_ms = max(ea.elapsed_time(eb), 1e-3)
        reps = max(min_replays, -(-steps // per_graph), int(np.ceil(min_region_s * 1e3 / est_ms)))
        reps = min(reps, 200000)
        if self.world > 1:   # every rank replays the same number of times
            (reps_f,) = max_over_ranks([float(reps)], self.world)
            reps = int(reps_f)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        clocks = ClockSampler(self.dev.index)
        clocks.start()
        self.barrier()
        t0 = time.time()
        with torch.cuda.stream(s):
            ev[0].record(s)
            for r in range(reps):
                g.replay()
                ev[r + 1].record(s)
        self.barrier()
        t1 = time.time()
        clocks.mark(t0, t1)
        per_call = [ev[r].elapsed_time(ev[r + 1]) / per_graph for r in range(reps)]
        med = statistics.median(per_call)
        total = ev[0].elapsed_time(ev[reps])
        self.spread = {"replays": reps, "calls_per_replay": per_graph,
                       "us_median": round(med * 1e3, 3), "us_min": round(min(per_call) * 1e3, 3),
                       "us_max": round(max(per_call) * 1e3, 3),
                       "us_mean": round(total / (reps * per_graph) * 1e3, 3),
                       "timed_region_s": round(total * 1e-3, 3)}
        return med, reps * per_graph, clocks.stop()

    def finish(self, line):
        if self.rank == 0 and line is not None:
            if getattr(self.args, "capture", None) is not None:
                self.args.capture.append(line)     # a secondary row of the default run
            else:
                print(json.dumps(line), flush=True)
        if self.world > 1:
            self.torch.distributed.destroy_process_group()
        return 0


def roofline(achieved_bytes_per_launch, ms, kernel, traffic_key):
    peak, src = hbm_peak()
    ach = achieved_bytes_per_launch / (ms * 1e-3) / 1e9
    r = {"bound": "hbm", "achieved": round(ach, 2), "peak": peak, "unit": "GB/s",
         "frac": round(ach / peak, 4), "peak_source": f"{src} (hbm copy, burst)",
         "frac_of_nominal": round(ach / NOMINAL_HBM_GBS, 4),
         "traffic": measured_traffic(kernel, traffic_key),
         "algorithmic_bytes_per_launch": int(achieved_bytes_per_launch)}
    if ach > peak:
        r["frac_above_1"] = ("the measured peak is a torch copy_ (read + write) of one buffer; this "
                             "kernel streams its reads and writes faster than that copy, so the "
                             "copy figure is not a ceiling here: frac_of_nominal is against 7.9 TB/s")
    return r


def base_line(h, value, ms, steps, warmup, workload, config, kernel_launches):
    line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": h.world,
            "steps": steps, "warmup": warmup, "ms_per_step": round(ms, 6),
            "us_per_step": round(ms * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload, **config, "parallelism": f"replicas x{h.world}"},
            "gpu_launches": kernel_launches}
    spread = getattr(h, "spread", None)
    if spread is not None:
        # value and ms_per_step are the median over replays; steps counts every call timed, which
        # is at least --steps (more when 20 replays or 0.5 s of replays need more calls)
        line["steps_requested"] = h.args.steps
        line["timing_spread"] = spread
    return line


# ------------------------------------------------------------------------------------------------
# workloads
# ------------------------------------------------------------------------------------------------
def packed_workload(B, H, HV, K, V, seed, device, layer=0, state_dtype="f32"):
    import torch
    import gdn_synth as syn
    width = 2 * H * K + HV * V
    x = torch.empty((B, width), dtype=torch.bfloat16, device=device)
    a = torch.empty((B, HV), dtype=torch.bfloat16, device=device)
    b = torch.empty((B, HV), dtype=torch.bfloat16, device=device)
    A_log = torch.empty(HV, dtype=torch.float32, device=device)
    dt_bias = torch.empty(HV, dtype=torch.float32, device=device)
    state = torch.empty((B, HV, V, K), dtype=torch.bfloat16 if state_dtype == "bf16" else torch.float32,
                        device=device)
    r = syn.GdnRecipe()
    syn.fill_normal_(x, seed, syn.Tag.QKV, 0, r.qkv_std, layer)
    syn.fill_normal_(a, seed, syn.Tag.A, 0, r.a_std, layer)
    syn.fill_normal_(b, seed, syn.Tag.B, 0, r.b_std, layer)
    syn.fill_normal_(A_log, seed, syn.Tag.A_LOG, 0, r.A_log_std, layer)
    syn.fill_normal_(dt_bias, seed, syn.Tag.DT_BIAS, 0, r.dt_bias_std, layer)
    syn.fill_normal_(state, seed, syn.Tag.STATE, 0, r.state_std, layer)
    idx = torch.from_numpy(syn.permutation(seed + 7919 * layer, B)).to(device)
    out = torch.empty((B, 1, HV, V), dtype=torch.bfloat16, device=device)
    return dict(x=x, a=a, b=b, A_log=A_log, dt_bias=dt_bias, state=state, idx=idx, out=out)


def inplace_stream_gbs(buf, h, reps=20):
    """Context for the roofline: a plain in-place read-modify-write stream over the same buffer as
    the state (torch's elementwise multiply by 1.0: every element read and written once, values
    unchanged), timed with CUDA events on this GPU in the same run; median of `reps`."""
    torch = h.torch
    nbytes = 2 * buf.numel() * buf.element_size()
    for _ in range(3):
        buf.mul_(1.0)
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(h.stream)
        buf.mul_(1.0)
        e1.record(h.stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    med = statistics.median(times)
    return {"value": round(nbytes / (med * 1e-3) / 1e9, 1), "unit": "GB/s",
            "how": f"torch in-place multiply by 1.0 over the {buf.numel() * buf.element_size() / 1e9:.2f} GB "
                   f"state buffer (read + write), median of {reps} CUDA-event timings in this run; "
                   f"context for the roofline, not its peak"}


def packed_io_bytes(B, H, HV, K, V):
    """Bytes of the step's inputs and outputs besides the state: mixed_qkv, a, b, A_log, dt_bias,
    cache indices, out."""
    return B * (2 * H * K + HV * V) * 2 + 2 * B * HV * 2 + 2 * HV * 4 + B * 4 + B * HV * V * 2


def l2_bytes(dev):
    import torch
    try:
        return int(torch.cuda.get_device_properties(dev).L2_cache_size)
    except Exception:
        return 129 * 1024 * 1024


def pool_count(state_bytes, dev):
    """Independent state pools to rotate through so that one pass over them is at least four
    times the L2 size: a small pool would otherwise be served from L2 on the next call. A state
    of three L2 sizes or more streams from HBM on its own."""
    l2 = l2_bytes(dev)
    if state_bytes >= 3 * l2:
        return 1
    return max(1, -(-4 * l2 // state_bytes))


def run_packed(args):
    import ssm_recurrent_decode_gb300 as gdn
    h = Harness(args)
    torch = h.torch
    gdn.lib()
    B, H, HV, K, V = args.B, 16, 32, 128, 128
    sbytes = 2 if args.state_dtype == "bf16" else 4
    w = packed_workload(B, H, HV, K, V, seed=1234 + h.rank, device=h.dev, state_dtype=args.state_dtype)
    import gdn_synth as syn
    n_pools = pool_count(B * HV * V * K * sbytes, h.dev)
    pools = [w["state"]]
    for p in range(1, n_pools):
        s = torch.empty_like(w["state"])
        syn.fill_normal_(s, 1234 + h.rank, syn.Tag.STATE, 0, 1.0, layer=p)
        pools.append(s)
    q, k, v = gdn.split_mixed_qkv(w["x"], H, HV, K, V)
    calls = [gdn.gdn_decode_step_indexed(q, k, v, pool, w["out"], w["idx"], H=H, a=w["a"], b=w["b"],
                                         A_log=w["A_log"], dt_bias=w["dt_bias"], prepare=True)
             for pool in pools]

    def step(i):
        calls[i % n_pools]()

    per_graph = max(64, n_pools)
    ms, steps, clk = h.time_graph(step, args.steps, args.warmup, per_graph)

    # End to end through the public API, with host buffers: every step copies its inputs from
    # pinned host memory and its output back to pinned host memory. Copies run on their own
    # streams over two sets of device buffers, so step i's compute overlaps step i+1's input copy
    # and step i-1's output copy (events order each buffer's reuse).
    hx = w["x"].cpu().pin_memory()
    ha, hb = w["a"].cpu().pin_memory(), w["b"].cpu().pin_memory()
    hout = [torch.empty(w["out"].shape, dtype=w["out"].dtype).pin_memory() for _ in range(2)]
    dev_in = [(w["x"], w["a"], w["b"]), tuple(torch.empty_like(t) for t in (w["x"], w["a"], w["b"]))]
    dev_out = [w["out"], torch.empty_like(w["out"])]
    e2e_calls = []
    for j in range(2):
        qj, kj, vj = gdn.split_mixed_qkv(dev_in[j][0], H, HV, K, V)
        e2e_calls.append(gdn.gdn_decode_step_indexed(qj, kj, vj, pools[0], dev_out[j], w["idx"], H=H,
                                                     a=dev_in[j][1], b=dev_in[j][2], A_log=w["A_log"],
                                                     dt_bias=w["dt_bias"], prepare=True))
    s_comp = torch.cuda.current_stream(h.dev)
    s_in, s_out = torch.cuda.Stream(h.dev), torch.cuda.Stream(h.dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        for i in range(n):
            j = i % 2
            if i >= 2:
                s_in.wait_event(ev_done[j])        # step i-2 has consumed this input set
            with torch.cuda.stream(s_in):
                for d_t, h_t in zip(dev_in[j], (hx, ha, hb)):
                    d_t.copy_(h_t, non_blocking=True)
                ev_in[j].record(s_in)
            s_comp.wait_event(ev_in[j])
            if i >= 2:
                s_comp.wait_event(ev_out[j])       # step i-2's output has been copied out
            e2e_calls[j](s_comp.cuda_stream)
            ev_done[j].record(s_comp)
            s_out.wait_event(ev_done[j])
            with torch.cuda.stream(s_out):
                hout[j].copy_(dev_out[j], non_blocking=True)
                ev_out[j].record(s_out)

    e2e_steps = max(2, min(steps, 2000))
    e2e_run(4)
    h.barrier()
    t0 = time.perf_counter()
    e2e_run(e2e_steps)
    h.barrier()
    ms_e2e = (time.perf_counter() - t0) * 1e3 / e2e_steps
    h2d = (hx.numel() + ha.numel() + hb.numel()) * 2
    d2h = hout[0].numel() * 2
    ms, ms_e2e = max_over_ranks([ms, ms_e2e], h.world)
    if h.rank != 0:
        return h.finish(None)

    state_bytes = 2 * B * HV * V * K * sbytes
    gbs = h.world * state_bytes / (ms * 1e-3) / 1e9
    peak, _ = hbm_peak()
    name, sizes = packed_workload_config(B, H, HV, K, V, args.state_dtype)
    assert sizes["state_bytes_per_step"] == state_bytes
    line = base_line(
        h, gbs, ms, steps, args.warmup, name,
        {**sizes, "state_pools": n_pools,
         "l2": (f"state of {state_bytes / 2 / 1e9:.2f} GB read per step, larger than the L2: no flush "
                f"between steps" if n_pools == 1 else
                f"{n_pools} state pools rotated, at least 4x the L2 size per pass"),
         "timing": f"CUDA-graph replays of {per_graph} calls; e2e: prepared calls with copies"},
        steps)
    line["pct_of_peak"] = round(100 * gbs / h.world / peak, 2)            # of the measured copy bandwidth
    line["pct_of_nominal_peak"] = round(100 * gbs / h.world / NOMINAL_HBM_GBS, 2)  # of 7.9 TB/s
    if not getattr(args, "secondary_row", False):
        line["stream_reference"] = inplace_stream_gbs(pools[0], h)
    line["roofline"] = roofline(state_bytes + packed_io_bytes(B, H, HV, K, V), ms,
                                "step_bf16" if args.state_dtype == "bf16" else "step",
                                f"packed_B{B}" + ("_bf16state" if args.state_dtype == "bf16" else ""))
    if not getattr(args, "secondary_row", False):
        line["cpu_baseline"] = cpu_baseline(H, HV, K, V, seed=7, budget_s=args.cpu_budget)
    line["e2e"] = {"value": round(h.world * state_bytes / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                   "us_per_step": round(ms_e2e * 1e3, 3), "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h,
                   "how": "prepared gdn_decode_step_indexed calls; per step a pinned-host -> device "
                          "copy of mixed_qkv, a, b and a device -> pinned-host copy of out, on copy "
                          "streams overlapping the neighbouring steps; host wall clock between "
                          "synchronizations"}
    line["clocks"] = clk
    return h.finish(line)


def run_buffered(args):
    """Buffered output-only decode at the packed shapes: every step reads the checkpoint tile,
    appends d/k/g records, and the step at write_pos == L-1 folds the ring and writes the tile.
    The timed loop runs whole cycles (all L phases, every row at the same phase), so the mean is
    the exact cycle average; each phase is also timed on its own."""
    import ssm_recurrent_decode_gb300 as gdn
    h = Harness(args)
    torch = h.torch
    gdn.lib()
    B, H, HV, K, V, L = args.B, 16, 32, 128, 128, args.L
    w = packed_workload(B, H, HV, K, V, seed=4321 + h.rank, device=h.dev)
    q, k, v = gdn.split_mixed_qkv(w["x"], H, HV, K, V)
    d_cache = torch.zeros((B, HV, L, V), dtype=torch.bfloat16, device=h.dev)
    k_cache = torch.zeros((B, H, L, K), dtype=torch.bfloat16, device=h.dev)
    g_cache = torch.zeros((B, HV, L), dtype=torch.float32, device=h.dev)
    pos = [torch.full((B,), p, dtype=torch.int32, device=h.dev) for p in range(L)]
    calls = [gdn.gdn_decode_buffered(q, k, v, w["state"], w["out"], d_cache, k_cache, g_cache, pos[p],
                                     cache_indices=w["idx"], H=H, a=w["a"], b=w["b"],
                                     A_log=w["A_log"], dt_bias=w["dt_bias"], kernel=args.kernel,
                                     prepare=True)
             for p in range(L)]

    def step(i):
        calls[i % L]()

    warm = max(args.warmup, L)
    warm = ((warm + L - 1) // L) * L
    per_graph = L * max(1, 64 // L)
    ms, steps, clk = h.time_graph(step, max(L, args.steps), warm, per_graph)
    # per-phase times: events around each call of a cycle, averaged over cycles
    cycles = max(1, min(50, steps // L))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(cycles * L)]
    h.barrier()
    for i in range(cycles * L):
        ev[i][0].record(h.stream)
        calls[i % L](h.stream.cuda_stream)
        ev[i][1].record(h.stream)
    h.barrier()
    phase_ms = [statistics.mean(ev[c * L + p][0].elapsed_time(ev[c * L + p][1]) for c in range(cycles))
                for p in range(L)]
    (ms,) = max_over_ranks([ms], h.world)
    if h.rank != 0:
        return h.finish(None)
    S = B * HV * V * K * 4
    state_traffic = (1 + 1 / L) * S
    ring_append = B * (HV * V * 2 + H * K * 2 + HV * 4)
    ring_read_mean = B * (HV * V * 2 + H * K * 2 + HV * 4) * (L - 1) / 2
    io = packed_io_bytes(B, H, HV, K, V)
    gbs = h.world * state_traffic / (ms * 1e-3) / 1e9
    line = base_line(
        h, gbs, ms, steps, warm,
        f"gdn buffered output-only decode: B={B} H={H} HV={HV} K=V={K}, L={L}, bf16 rings, "
        f"fp32 checkpoint state, all phases timed", {"B": B, "H": H, "HV": HV, "K": K, "V": V, "L": L,
        "timing": f"CUDA-graph replays of {per_graph} calls (whole cycles); phase times: direct calls",
        "state_bytes_per_step_mean": state_traffic,
        "packed_equivalent_state_GBs": round(2 * S / (ms * 1e-3) / 1e9, 2)}, steps)
    line["roofline"] = roofline(state_traffic + ring_append + ring_read_mean + io, ms, "buffered",
                                f"buffered_B{B}_L{L}")
    if not getattr(args, "secondary_row", False):
        line["cpu_baseline"] = cpu_baseline_buffered(H, HV, K, V, L, seed=8, budget_s=args.cpu_budget)
    line["phase_us"] = [round(p * 1e3, 2) for p in phase_ms]
    line["flush_over_nonflush"] = (round(phase_ms[-1] / statistics.mean(phase_ms[:-1]), 3)
                                   if L > 1 else None)
    line["clocks"] = clk
    return h.finish(line)


def fused_workload(T, heads, D, seed, device, layout="DS"):
    import numpy as np
    import torch
    import gdn_synth as syn
    num_slots = T + 8
    dim = heads * D
    ins = syn.fused_inputs(T, heads, D, num_slots, seed)
    bf = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)
    state = torch.empty((num_slots, heads, D, D), dtype=torch.float32, device=device)
    syn.fill_normal_(state, seed, syn.Tag.STATE, 0, 1.0)
    cs = bf(ins["conv_state"])
    if layout == "SD":
        cs = cs.transpose(1, 2).contiguous().transpose(1, 2)
    return dict(x=bf(ins["x"]), conv_w=torch.from_numpy(ins["conv_w"]).to(device), conv_state=cs,
                raw_g=bf(ins["raw_g"]), raw_beta=bf(ins["raw_beta"]),
                A_log=torch.from_numpy(ins["A_log"]).to(device),
                dt_bias=torch.from_numpy(ins["dt_bias"]).to(device), state=state,
                idx=torch.arange(1, T + 1, dtype=torch.int32, device=device),
                out_gate=bf(ins["out_gate"]), norm_w=torch.from_numpy(ins["norm_w"]).to(device),
                out=torch.empty((T, heads, D), dtype=torch.bfloat16, device=device), dim=dim)


def run_fused(args):
    """Fused KDA decode (conv update -> per-key-decay delta step -> gated RMSNorm), 96 heads of
    128, T tokens, T+8 slots, slot 0 the NULL slot."""
    import ssm_recurrent_decode_gb300 as gdn
    h = Harness(args)
    gdn.lib()
    T, heads, D = args.T, 96, 128
    w = fused_workload(T, heads, D, seed=555 + h.rank, device=h.dev, layout=args.layout)
    import gdn_synth as syn
    n_pools = pool_count(T * heads * D * D * 4, h.dev)
    pools = [w["state"]]
    for p in range(1, n_pools):
        s = h.torch.empty_like(w["state"])
        syn.fill_normal_(s, 555 + h.rank, syn.Tag.STATE, 0, 1.0, layer=p)
        pools.append(s)
    calls = [gdn.gdn_decode_fused(w["x"], w["conv_w"], w["conv_state"], w["raw_g"], w["raw_beta"],
                                  w["A_log"], w["dt_bias"], pool, w["idx"], w["out_gate"],
                                  w["norm_w"], w["out"], pad_slot_id=0, gate_kind="kda",
                                  kda_gate_form=0, gate_act="silu", kernel=args.kernel, prepare=True)
             for pool in pools]

    def step(i):
        calls[i % n_pools]()

    per_graph = max(64, n_pools)
    ms, steps, clk = h.time_graph(step, args.steps, args.warmup, per_graph)
    (ms,) = max_over_ranks([ms], h.world)
    if h.rank != 0:
        return h.finish(None)
    dim = w["dim"]
    state_bytes = 2 * T * heads * D * D * 4
    io = (T * 3 * dim * 2            # x
          + 2 * T * 3 * dim * 3 * 2  # conv state read + write
          + 3 * dim * 4 * 4          # conv weights
          + T * dim * 2 * 2          # raw_g, out_gate
          + T * heads * 2 + heads * 4 + dim * 4 + D * 4 + T * 4
          + T * dim * 2)             # out
    gbs = h.world * state_bytes / (ms * 1e-3) / 1e9
    line = base_line(
        h, gbs, ms, steps, args.warmup,
        f"fused KDA decode: T={T} tokens, {heads} heads x {D}, conv width 4 ({args.layout} conv "
        f"state), per-key decay bounded at -5, gated RMSNorm with silu",
        {"T": T, "heads": heads, "head_dim": D, "state_bytes_per_step": state_bytes,
         "state_pools": n_pools, "kernel": args.kernel,
         "l2": f"{n_pools} state pool(s) rotated, at least 4x the L2 size per pass",
         "timing": f"CUDA-graph replays of {per_graph} calls"}, steps)
    line["roofline"] = roofline(state_bytes + io, ms, "fused", f"fused_T{T}")
    if not getattr(args, "secondary_row", False):
        line["cpu_baseline"] = cpu_baseline_fused(heads, D, seed=9, budget_s=args.cpu_budget)
    line["clocks"] = clk
    return h.finish(line)


def stack_decode(layers=48, B=256, H=16, HV=48, K=128, V=128, steps=1000, seed=2024, pairs=8,
                 heads_per_pair=2, device=None, verbose=False, chained=True, sample_clocks=False):
    """The stacked decode under CUDA graphs: `layers` independent state pools, one graph that
    draws fresh seeded inputs for every layer on the device (keyed by seed, layer and a device step
    counter), and one graph of `layers` decode calls, replayed `steps` times (chained: every layer
    after the first through gdn_decode_step_indexed_chained, so that its launch overlaps the
    previous layer's tail). Afterwards the fp64 oracle replays `pairs` sampled (layer, slot)
    pairs, on `heads_per_pair` q/k heads each (all their value heads), through every step and the
    drift of the GPU state against it is measured. Returns a dict of timings and errors."""
    import torch
    import gdn_synth as syn
    import oracle
    import ssm_recurrent_decode_gb300 as gdn
    dev = device or torch.device("cuda", torch.cuda.current_device())
    r = syn.GdnRecipe()
    G = HV // H
    width = 2 * H * K + HV * V
    ctr = torch.zeros(1, dtype=torch.int32, device=dev)
    L = []
    for l in range(layers):
        w = packed_workload(B, H, HV, K, V, seed, dev, layer=l)
        L.append(w)

    def gen():
        for l, w in enumerate(L):
            syn.fill_normal_(w["x"], seed, syn.Tag.QKV, 0, r.qkv_std, l, step_ptr=ctr)
            syn.fill_normal_(w["a"], seed, syn.Tag.A, 0, r.a_std, l, step_ptr=ctr)
            syn.fill_normal_(w["b"], seed, syn.Tag.B, 0, r.b_std, l, step_ptr=ctr)
        syn.add_i32_(ctr, 1)

    views = [gdn.split_mixed_qkv(w["x"], H, HV, K, V) for w in L]

    def decode():
        sid = torch.cuda.current_stream(dev).cuda_stream
        for l, ((q, k, v), w) in enumerate(zip(views, L)):
            gdn.gdn_decode_step_indexed(q, k, v, w["state"], w["out"], w["idx"], H=H, a=w["a"],
                                        b=w["b"], A_log=w["A_log"], dt_bias=w["dt_bias"], stream=sid,
                                        chained=chained and l > 0)

    # one eager pass loads every kernel before capture; then the pools are reset to step 0
    gen()
    decode()
    torch.cuda.synchronize(dev)
    for l, w in enumerate(L):
        syn.fill_normal_(w["state"], seed, syn.Tag.STATE, 0, r.state_std, l)
    ctr.zero_()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    g_gen, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_gen, stream=s):
        gen()
    with torch.cuda.graph(g_dec, stream=s):
        decode()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = None
    if sample_clocks:   # SM clocks and throttle reasons during the timed steps
        sampler = ClockSampler(dev.index)
        sampler.start()
    t_start = time.time()
    with torch.cuda.stream(s):
        w0.record(s)
        for i in range(steps):
            g_gen.replay()
            ev[i][0].record(s)
            g_dec.replay()
            ev[i][1].record(s)
        w1.record(s)
    torch.cuda.synchronize(dev)
    clocks = None
    if sampler is not None:
        sampler.mark(t_start, time.time())
        clocks = sampler.stop()
    dec_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = w0.elapsed_time(w1)

    # sampled (layer, slot) pairs, replayed by the oracle from the initial tiles
    rng = np.random.default_rng(seed)
    picks = []
    for _ in range(pairs):
        l = int(rng.integers(layers)); b = int(rng.integers(B)); h0 = int(rng.integers(H - heads_per_pair + 1))
        picks.append((l, b, h0))
    drift, out_err = 0.0, 0.0
    for l, b, h0 in picks:
        slot = int(L[l]["idx"][b].item())
        hvs = list(range(h0 * G, (h0 + heads_per_pair) * G))
        S = np.stack([syn.state_tile_values(seed, HV, V, K, slot, hv, r.state_std, l) for hv in hvs])[None].astype(np.float64)
        A_log = syn.normal_f32(seed, syn.Tag.A_LOG, 0, (HV,), r.A_log_std, l).astype(np.float64)[hvs]
        dt_bias = syn.normal_f32(seed, syn.Tag.DT_BIAS, 0, (HV,), r.dt_bias_std, l).astype(np.float64)[hvs]
        f64 = lambda x: syn.bf16_bits_to_f32(syn.f32_to_bf16_bits(x)).astype(np.float64)
        for step in range(steps):
            x = f64(syn.normal_f32(seed, syn.Tag.QKV, step, (width,), r.qkv_std, l, start=b * width))
            av = f64(syn.normal_f32(seed, syn.Tag.A, step, (HV,), r.a_std, l, start=b * HV))[hvs]
            bv = f64(syn.normal_f32(seed, syn.Tag.B, step, (HV,), r.b_std, l, start=b * HV))[hvs]
            q = x[:H * K].reshape(H, K)[h0:h0 + heads_per_pair][None]
            k = x[H * K:2 * H * K].reshape(H, K)[h0:h0 + heads_per_pair][None]
            v = x[2 * H * K:].reshape(HV, V)[hvs][None]
            g, beta = oracle.gdn_gates(av[None], bv[None], A_log, dt_bias)
            o, _ = oracle.delta_step(q, k, v, g, beta, S, scale=K ** -0.5)
        got_S = L[l]["state"][slot, hvs[0]:hvs[-1] + 1].cpu().numpy()
        drift = max(drift, float(np.max(np.abs(got_S - S[0]) / np.maximum(1.0, np.abs(S[0])))))
        got_o = L[l]["out"][b, 0, hvs[0]:hvs[-1] + 1].float().cpu().numpy()
        out_err = max(out_err, float(np.max(np.abs(got_o - o[0]) / np.maximum(1.0, np.abs(o[0])))))
        if verbose:
            print(f"pair layer={l} slot={slot} heads={h0}..{h0 + heads_per_pair - 1}: drift so far {drift:.3g}")
    return {"dec_ms_per_step": statistics.mean(dec_ms), "dec_ms_median": statistics.median(dec_ms),
            "total_ms_per_step": total_ms / steps, "drift": drift, "last_out_err": out_err,
            "picks": picks, "state_bytes_per_step": 2 * layers * B * HV * V * K * 4, "clocks": clocks}


def run_stack(args):
    h = Harness(args)
    import ssm_recurrent_decode_gb300 as gdn
    gdn.lib()
    layers, B, H, HV, K, V = args.layers, args.B, 16, 48, 128, 128
    steps = args.steps
    res = stack_decode(layers, B, H, HV, K, V, steps=steps, device=h.dev, pairs=args.pairs,
                       chained=not args.no_chain, sample_clocks=True)
    ms = res["dec_ms_median"]
    (ms,) = max_over_ranks([ms], h.world)
    if h.rank != 0:
        return h.finish(None)
    state_bytes = res["state_bytes_per_step"]
    gbs = h.world * state_bytes / (ms * 1e-3) / 1e9
    line = base_line(
        h, gbs, ms, steps, 1,
        f"{layers}-layer stacked gdn decode under CUDA graphs: B={B} H={H} HV={HV} K=V={K}, an "
        f"fp32 state pool per layer ({layers * B * HV * V * K * 4 / 1e9:.1f} GB), fresh device-drawn "
        f"bf16 inputs every step", {"layers": layers, "B": B, "H": H, "HV": HV, "K": K, "V": V,
                                     "state_bytes_per_step": state_bytes,
                                     "chained_layers": not args.no_chain}, steps * layers)
    line["per_layer_us"] = round(ms * 1e3 / layers, 3)
    line["clocks"] = res["clocks"]
    line["with_input_generation_ms_per_step"] = round(res["total_ms_per_step"], 4)
    line["drift_vs_oracle"] = {"max_rel_state_err": res["drift"], "last_step_out_err": res["last_out_err"],
                               "pairs": [list(p) for p in res["picks"]], "steps": steps,
                               "bar": 1e-4}
    line["roofline"] = roofline(state_bytes / layers + packed_io_bytes(B, H, HV, K, V),
                                ms / layers, "step", f"packed_HV{HV}_B{B}")
    return h.finish(line)


def run_mamba(args):
    """Mamba-1 selective-scan decode ("Triton decode kernel + MBU analysis"): B rows, D channels,
    N state entries, fp32 inputs and state. Bandwidth by the page's bytes model B*D*(20N+24)."""
    import torch
    import gdn_synth as syn
    import ssm_recurrent_decode_gb300 as gdn
    h = Harness(args)
    gdn.lib()
    B, D, N = args.B, args.D, args.N
    m = syn.mamba_inputs(B, D, N, "f32", 77 + h.rank)
    t = {k: torch.from_numpy(np.ascontiguousarray(v)).to(h.dev) for k, v in m.items()}
    state_bytes = B * D * N * 4
    n_pools = pool_count(state_bytes, h.dev)
    pools = [t["h"]] + [t["h"].clone() for _ in range(n_pools - 1)]
    y = torch.empty((B, D), dtype=torch.float32, device=h.dev)
    calls = [gdn.mamba_selective_scan_decode(t["x"], t["dt"], t["A"], t["Bm"], t["Cm"], pool, y,
                                             Dskip=t["Dskip"], z=t["z"], prepare=True) for pool in pools]

    def step(i):
        calls[i % n_pools]()

    per_graph = max(64, n_pools)
    ms, steps, clk = h.time_graph(step, args.steps, args.warmup, per_graph)
    (ms,) = max_over_ranks([ms], h.world)
    if h.rank != 0:
        return h.finish(None)
    page_bytes = mamba_page_bytes(B, D, N)
    gbs = h.world * page_bytes / (ms * 1e-3) / 1e9
    line = base_line(
        h, gbs, ms, steps, args.warmup,
        f"Mamba-1 selective-scan decode: B={B} D={D} N={N}, fp32 inputs and state, with D skip and "
        f"silu(z) gate", {"B": B, "D": D, "N": N, "bytes_model": "B*D*(20N+24)",
                          "bytes_per_step": page_bytes, "state_pools": n_pools,
                          "timing": f"CUDA-graph replays of {per_graph} calls",
                          "context": "the page's Triton kernel on an A10G: 60.5 / 59.6 / 58.4 us at "
                                     "B = 1 / 4 / 8, D = 1536, N = 16 (launch-bound)"}, steps)
    min_bytes = 2 * B * D * N * 4 + D * N * 4 + 2 * B * N * 4 + 4 * B * D * 4 + D * 4
    line["roofline"] = roofline(min_bytes, ms, "mamba", f"mamba_B{B}_D{D}_N{N}")
    if not getattr(args, "secondary_row", False):
        line["cpu_baseline"] = cpu_baseline_mamba(D, N, seed=78, budget_s=args.cpu_budget)
    line["clocks"] = clk
    return h.finish(line)


def run_gemv(args):
    """Decode projection ("Optimization Log", Kernel 3: BF16 GEMV with split-K) at one of the
    page's shapes, synthetic bf16 weights N(0, 0.02^2); bandwidth = weight bytes per call / time."""
    import torch
    import gdn_synth as syn
    import ssm_recurrent_decode_gb300 as gdn
    h = Harness(args)
    gdn.lib()
    T, N, Kd = args.T, args.gemv_n, args.gemv_k
    x = torch.empty((T, Kd), dtype=torch.bfloat16, device=h.dev)
    syn.fill_normal_(x, 91, syn.Tag.X, 0, 1.0)
    w_bytes = gemv_weight_bytes(N, Kd)
    n_pools = pool_count(w_bytes, h.dev)
    Ws = []
    for p in range(n_pools):
        W = torch.empty((N, Kd), dtype=torch.bfloat16, device=h.dev)
        syn.fill_normal_(W, 91, syn.Tag.CONV_W, 0, 0.02, layer=p)
        Ws.append(W)
    y = torch.empty((T, N), dtype=torch.bfloat16, device=h.dev)
    splits = args.gemv_splits or gdn.lib().gdn_gemv_default_splits(T, N, Kd)
    ws = gdn.gemv_workspace(T, N, Kd, splits, device=h.dev)
    calls = [gdn.gdn_gemv_bf16(x, W, y, splits=splits, workspace=ws, prepare=True) for W in Ws]

    def step(i):
        calls[i % n_pools]()

    per_graph = max(64, n_pools)
    ms, steps, clk = h.time_graph(step, args.steps, args.warmup, per_graph)
    (ms,) = max_over_ranks([ms], h.world)
    if h.rank != 0:
        return h.finish(None)
    gbs = h.world * w_bytes / (ms * 1e-3) / 1e9
    passes = (T + 15) // 16                   # token rows per pass over W: 16 (one when T = 1)
    line = base_line(
        h, gbs, ms, steps, args.warmup,
        f"decode projection GEMV: T={T} token rows, W [{N}, {Kd}] bf16 ({w_bytes / 1e6:.0f} MB), "
        f"fp32 accumulation, {splits} K split(s)",
        {"T": T, "N": N, "Kd": Kd, "splits": splits, "weight_pools": n_pools,
         "timing": f"CUDA-graph replays of {per_graph} calls; roofline over the whole call "
                   f"(the K ranges are added inside a thread-block cluster up to 8 ranges, by a "
                   f"second launch beyond)"},
        steps * (passes + (1 if gdn.lib().gdn_gemv_workspace_bytes(T, N, splits) > 0 else 0)))
    line["metric"] = "decode projection weight-stream GB/s"
    # algorithmic bytes: W once, x, y (any split-K exchange is the kernel's overhead)
    io = T * Kd * 2 + T * N * 2
    line["roofline"] = roofline(w_bytes + io, ms, "gemv", f"gemv_T{T}_N{N}_K{Kd}")
    if not getattr(args, "secondary_row", False):
        line["cpu_baseline"] = cpu_baseline_gemv(T, N, Kd, seed=92, budget_s=args.cpu_budget)
    line["clocks"] = clk
    return h.finish(line)


def run_front(args):
    """One DeltaNet layer's decode forward (gdn_decode_front): input projection -> conv update,
    delta step, gated RMSNorm -> output projection, at the Optimization Log's model width 5120 with
    32 heads of 128 (GDN gate), T tokens; synthetic bf16 weights N(0, 1/fan_in)."""
    import numpy as np
    import torch
    import gdn_synth as syn
    import ssm_recurrent_decode_gb300 as gdn
    h = Harness(args)
    gdn.lib()
    T, hidden, heads, D = args.T, args.hidden, 32, 128
    dim = heads * D
    P = gdn.front_proj_width(heads, D, "gdn")
    seed = 777 + h.rank
    num_slots = T + 8
    ins = syn.fused_inputs(T, heads, D, num_slots, seed)
    dev = h.dev
    conv_w = torch.from_numpy(ins["conv_w"]).to(dev)
    conv_state = torch.from_numpy(ins["conv_state"].view(np.int16)).view(torch.bfloat16).to(dev)
    A_log = torch.from_numpy(ins["A_log"]).to(dev)
    dt_bias = torch.from_numpy(np.ascontiguousarray(ins["dt_bias"][:heads])).to(dev)
    norm_w = torch.from_numpy(ins["norm_w"]).to(dev)
    idx = torch.arange(1, T + 1, dtype=torch.int32, device=dev)
    x = torch.empty((T, hidden), dtype=torch.bfloat16, device=dev)
    syn.fill_normal_(x, seed, syn.Tag.X, 0, 1.0)
    z = torch.empty((T, P), dtype=torch.bfloat16, device=dev)
    o = torch.empty((T, dim), dtype=torch.bfloat16, device=dev)
    y = torch.empty((T, hidden), dtype=torch.bfloat16, device=dev)
    w_bytes = (P * hidden + hidden * dim) * 2
    state_bytes = num_slots * heads * D * D * 4
    n_pools = pool_count(w_bytes + state_bytes, dev)
    layers = []
    for p in range(n_pools):               # independent layers (weights and state), rotated
        W_in = torch.empty((P, hidden), dtype=torch.bfloat16, device=dev)
        W_out = torch.empty((hidden, dim), dtype=torch.bfloat16, device=dev)
        syn.fill_normal_(W_in, seed, syn.Tag.CONV_W, 1, hidden ** -0.5, layer=p)
        syn.fill_normal_(W_out, seed, syn.Tag.CONV_W, 2, dim ** -0.5, layer=p)
        st = torch.empty((num_slots, heads, D, D), dtype=torch.float32, device=dev)
        syn.fill_normal_(st, seed, syn.Tag.STATE, 0, 1.0, layer=p)
        layers.append((W_in, W_out, st))
    calls = [gdn.gdn_decode_front(x, W_in, W_out, z, o, y, conv_w, conv_state, A_log, dt_bias, st,
                                  idx, norm_w, pad_slot_id=0, gate_kind="gdn", kernel=args.kernel,
                                  prepare=True)
             for W_in, W_out, st in layers]
    in_splits = gdn.lib().gdn_gemv_default_splits(T, P, hidden)
    out_splits = gdn.lib().gdn_gemv_default_splits(T, hidden, dim)

    def step(i):
        calls[i % n_pools]()

    per_graph = max(64, n_pools)
    ms, steps, clk = h.time_graph(step, args.steps, args.warmup, per_graph)
    (ms,) = max_over_ranks([ms], h.world)
    if h.rank != 0:
        return h.finish(None)
    tile_bytes = 2 * T * heads * D * D * 4            # each token's state tile read and written
    io = (T * hidden * 2 + 2 * T * P * 2               # x; z written and read
          + 2 * T * 3 * dim * 3 * 2 + 3 * dim * 4 * 4  # conv state read + write, conv weights
          + 2 * T * dim * 2 + T * hidden * 2           # o written and read, y
          + heads * 8 + D * 4 + T * 4)
    total = w_bytes + tile_bytes + io
    gbs = h.world * total / (ms * 1e-3) / 1e9
    line = base_line(
        h, gbs, ms, steps, args.warmup,
        f"DeltaNet layer decode front: T={T}, hidden {hidden}, {heads} heads x {D} (GDN gate), "
        f"in_proj [{P}, {hidden}] + conv + step + gated RMSNorm + out_proj [{hidden}, {dim}], bf16 "
        f"weights ({w_bytes / 1e6:.0f} MB)",
        {"T": T, "hidden": hidden, "heads": heads, "head_dim": D, "proj_width": P,
         "in_splits": in_splits, "out_splits": out_splits, "weight_bytes": w_bytes,
         "layers_rotated": n_pools, "timing": f"CUDA-graph replays of {per_graph} calls (3 launches each)"},
        steps * 3)
    line["metric"] = "decode layer front GB/s (weights, state, activations)"
    line["roofline"] = roofline(total, ms, "front", f"front_T{T}")
    line["roofline"]["scope"] = "whole call: input projection, fused decode, output projection"
    line["clocks"] = clk
    return h.finish(line)


# Secondary rows measured by the default run after the headline (one GPU, rank 0 only): the
# other hot-path rows at their workload sizes, each with its own timing and roofline, summarised in
# the headline's JSON line under "secondary" (no CPU baseline, no end-to-end leg).
SECONDARY_ROWS = [
    ("packed_B256_bf16_state", {"workload": "packed", "B": 256, "state_dtype": "bf16"}),
    ("packed_B16", {"workload": "packed", "B": 16}),
    ("buffered_B256_L16", {"workload": "buffered", "B": 256, "L": 16}),
    ("fused_kda_T128", {"workload": "fused", "T": 128}),
    ("fused_kda_T8", {"workload": "fused", "T": 8}),
    ("stack48_B16_chained", {"workload": "stack", "B": 16, "layers": 48, "steps": 50, "pairs": 2}),
    ("mamba_B1024_N16", {"workload": "mamba", "B": 1024, "N": 16}),
    ("mamba_B1024_N64", {"workload": "mamba", "B": 1024, "N": 64}),
    ("gemv_17408x5120_T8", {"workload": "gemv", "T": 8}),
    ("front_T1", {"workload": "front", "T": 1}),
]


def secondary_summary(line):
    r = line.get("roofline", {})
    out = {"workload": line["config"].get("workload"), "metric": line["metric"], "value": line["value"],
           "unit": line["unit"], "us_per_call": line["us_per_step"], "roofline_frac": r.get("frac"),
           "roofline_achieved": r.get("achieved"), "timing_spread": line.get("timing_spread"),
           "clocks": line.get("clocks")}
    for k in ("drift_vs_oracle", "per_layer_us", "state_traffic_gbs"):
        if k in line:
            out[k] = line[k]
    return out


def run_default_with_secondary(args):
    """The headline (packed B=256) line, then the secondary rows, printed as one JSON line."""
    import copy
    captured = []
    args.capture = captured
    run_packed(args)
    line = captured[0]
    secondary = {}
    t0 = time.time()
    for name, over in SECONDARY_ROWS:
        a2 = copy.copy(args)
        for k, v in over.items():
            setattr(a2, k, v)
        if "steps" not in over:
            a2.steps = 20
        a2.warmup = max(3, min(args.warmup, 5))
        a2.secondary_row = True
        a2.capture = []
        try:
            {"packed": run_packed, "buffered": run_buffered, "fused": run_fused, "stack": run_stack,
             "mamba": run_mamba, "gemv": run_gemv, "front": run_front}[a2.workload](a2)
            secondary[name] = secondary_summary(a2.capture[0])
        except Exception as e:   # a failed secondary row is reported, never hides the headline
            secondary[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
    line["secondary"] = secondary
    line["secondary_wall_s"] = round(time.time() - t0, 1)
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["packed", "buffered", "fused", "stack", "mamba", "gemv", "front"],
                   default="packed")
    p.add_argument("--B", type=int, default=256)
    p.add_argument("--L", type=int, default=16)
    p.add_argument("--T", type=int, default=128)
    p.add_argument("--layout", choices=["DS", "SD"], default="DS")
    p.add_argument("--kernel", choices=["auto", "tile", "pipe", "stage"], default="auto",
                   help="kernel family of the buffered, fused and front workloads")
    p.add_argument("--state-dtype", choices=["f32", "bf16"], default="f32")
    p.add_argument("--D", type=int, default=1536)
    p.add_argument("--hidden", type=int, default=5120, help="model width of the front workload")
    p.add_argument("--gemv-n", type=int, default=17408)
    p.add_argument("--gemv-k", type=int, default=5120)
    p.add_argument("--gemv-splits", type=int, default=0, help="K ranges (0: the library's choice)")
    p.add_argument("--N", type=int, default=16)
    p.add_argument("--layers", type=int, default=48)
    p.add_argument("--pairs", type=int, default=8)
    p.add_argument("--no-chain", action="store_true",
                   help="stack workload: ordinary launches for every layer (no programmatic overlap)")
    p.add_argument("--cpu-budget", type=float, default=10.0)
    p.add_argument("--no-secondary", action="store_true",
                   help="default workload only: skip the secondary rows measured after the headline")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if (args.workload == "packed" and args.B == 256 and args.state_dtype == "f32" and not args.no_secondary
            and dist_env()[1] == 1):
        return run_default_with_secondary(args)
    return {"packed": run_packed, "buffered": run_buffered, "fused": run_fused,
            "stack": run_stack, "mamba": run_mamba, "gemv": run_gemv,
            "front": run_front}[args.workload](args)


if __name__ == "__main__":
    sys.exit(main())
