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
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-step state HBM GB/s (% of GB300 peak), µs/step at B=256 HV=32 K=V=128"
FALLBACK_HBM_GBS = 6800.0
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
    h = hashlib.sha256()
    for rel in files:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


KERNEL_FILES = {
    "step": ["ssm_recurrent_decode_gb300/csrc/step_kernel.cu", "ssm_recurrent_decode_gb300/csrc/gdn_tile.cuh",
             "ssm_recurrent_decode_gb300/csrc/gdn_common.cuh"],
    "buffered": ["ssm_recurrent_decode_gb300/csrc/buffered_kernel.cu", "ssm_recurrent_decode_gb300/csrc/gdn_tile.cuh",
                 "ssm_recurrent_decode_gb300/csrc/gdn_common.cuh"],
    "fused": ["ssm_recurrent_decode_gb300/csrc/fused_kernel.cu", "ssm_recurrent_decode_gb300/csrc/gdn_tile.cuh",
              "ssm_recurrent_decode_gb300/csrc/gdn_common.cuh"],
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


def cpu_baseline(H, HV, K, V, seed, budget_s=10.0):
    tiles, spent = OracleSampler(H, HV, K, V, seed).run(budget_s=budget_s)
    state_bytes = tiles * 2 * V * K * 4
    return {"value": round(state_bytes / spent / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{tiles} (slot, value head) tiles of the packed decode (H={H}, HV={HV}, "
                      f"K={K}, V={V}, bf16 inputs), fp64 C oracle, one thread, {spent:.1f} s"}


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
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(spent / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"gdn packed decode B={B} H={H} HV={HV} K=V={K}, fp64 CPU oracle on "
                               f"{tiles_per_step} (slot, value head) tiles per step",
                   "B": B, "H": H, "HV": HV, "K": K, "V": V},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{tiles_per_step} tiles per step, one thread"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------
def packed_workload(B, H, HV, K, V, seed, device):
    import torch
    import gdn_synth as syn
    width = 2 * H * K + HV * V
    x = torch.empty((B, width), dtype=torch.bfloat16, device=device)
    a = torch.empty((B, HV), dtype=torch.bfloat16, device=device)
    b = torch.empty((B, HV), dtype=torch.bfloat16, device=device)
    A_log = torch.empty(HV, dtype=torch.float32, device=device)
    dt_bias = torch.empty(HV, dtype=torch.float32, device=device)
    state = torch.empty((B, HV, V, K), dtype=torch.float32, device=device)
    r = syn.GdnRecipe()
    syn.fill_normal_(x, seed, syn.Tag.QKV, 0, r.qkv_std)
    syn.fill_normal_(a, seed, syn.Tag.A, 0, r.a_std)
    syn.fill_normal_(b, seed, syn.Tag.B, 0, r.b_std)
    syn.fill_normal_(A_log, seed, syn.Tag.A_LOG, 0, r.A_log_std)
    syn.fill_normal_(dt_bias, seed, syn.Tag.DT_BIAS, 0, r.dt_bias_std)
    syn.fill_normal_(state, seed, syn.Tag.STATE, 0, r.state_std)
    idx = torch.from_numpy(syn.permutation(seed, B)).to(device)
    out = torch.empty((B, 1, HV, V), dtype=torch.bfloat16, device=device)
    return dict(x=x, a=a, b=b, A_log=A_log, dt_bias=dt_bias, state=state, idx=idx, out=out)


def run_packed(args):
    import torch
    import ssm_recurrent_decode_gb300 as gdn
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    gdn.lib()
    B, H, HV, K, V = args.B, 16, 32, 128, 128
    w = packed_workload(B, H, HV, K, V, seed=1234 + rank, device=dev)
    q, k, v = gdn.split_mixed_qkv(w["x"], H, HV, K, V)
    stream = torch.cuda.current_stream(dev)

    def step():
        gdn.gdn_decode_step_indexed(q, k, v, w["state"], w["out"], w["idx"], H=H, a=w["a"],
                                    b=w["b"], A_log=w["A_log"], dt_bias=w["dt_bias"],
                                    stream=stream.cuda_stream)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    clocks = ClockSampler(dev.index)
    clocks.start()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    t1 = time.time()
    clocks.mark(t0, t1)
    ms = e0.elapsed_time(e1) / args.steps
    clk = clocks.stop()

    # end to end through the public API: pinned host inputs in, output back to pinned host memory
    hx = torch.empty_like(w["x"], device="cpu").pin_memory().copy_(w["x"].cpu())
    ha = torch.empty_like(w["a"], device="cpu").pin_memory().copy_(w["a"].cpu())
    hb = torch.empty_like(w["b"], device="cpu").pin_memory().copy_(w["b"].cpu())
    hout = torch.empty_like(w["out"], device="cpu").pin_memory()
    e2e_steps = max(1, min(args.steps, 2000))

    def e2e_step():
        w["x"].copy_(hx, non_blocking=True)
        w["a"].copy_(ha, non_blocking=True)
        w["b"].copy_(hb, non_blocking=True)
        step()
        hout.copy_(w["out"], non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    ms_e2e = e0.elapsed_time(e1) / e2e_steps
    h2d = hx.numel() * 2 + ha.numel() * 2 + hb.numel() * 2
    d2h = hout.numel() * 2

    times = torch.tensor([ms, ms_e2e], dtype=torch.float64)
    if world > 1:
        torch.distributed.all_reduce(times, op=torch.distributed.ReduceOp.MAX)
    ms, ms_e2e = float(times[0]), float(times[1])
    if rank != 0:
        torch.distributed.destroy_process_group()
        return 0

    state_bytes = 2 * B * HV * V * K * 4
    io_bytes = (B * (2 * H * K + HV * V) * 2 + 2 * B * HV * 2 + 2 * HV * 4 + B * 4
                + B * HV * V * 2)
    gbs = world * state_bytes / (ms * 1e-3) / 1e9
    peak, peak_src = hbm_peak()
    achieved = (state_bytes + io_bytes) / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "us_per_step": round(ms * 1e3, 3), "pct_of_peak": round(100 * gbs / world / peak, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"gdn packed decode over a slot pool: B={B} H={H} HV={HV} K=V={K}, "
                               f"bf16 mixed_qkv/a/b/out, fp32 state [{B},{HV},{V},{K}], "
                               f"permuted int32 cache indices",
                   "B": B, "H": H, "HV": HV, "K": K, "V": V, "input_dtype": "bf16",
                   "state_dtype": "f32", "state_bytes_per_step": state_bytes,
                   "l2": "state larger than L2 (1.07 GB vs 129 MB): no flush between steps",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_src} (hbm copy)",
                     "traffic": measured_traffic("step", f"packed_B{B}"),
                     "algorithmic_bytes_per_launch": state_bytes + io_bytes},
        "cpu_baseline": cpu_baseline(H, HV, K, V, seed=7, budget_s=args.cpu_budget),
        "e2e": {"value": round(world * state_bytes / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(ms_e2e * 1e3, 3), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["packed"], default="packed")
    p.add_argument("--B", type=int, default=256)
    p.add_argument("--cpu-budget", type=float, default=10.0)
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_packed(args)


if __name__ == "__main__":
    sys.exit(main())
