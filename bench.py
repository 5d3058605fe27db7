"""Throughput benchmark of the FLARE mixer forward (encode + merge + decode).

One step = one flare_fwd call over one batch of the c2_bf16 workload (FLARE
forward, bf16, B=4 H=8 D=64 M=128 N=65536, R=8 ragged shards, 5% padded
tokens): the split-KV encoder with its fused log-sum-exp merge, then the
local decode of every token. Inputs are seeded synthetic tensors resident in
HBM; K and V (256 MiB each) exceed the 129 MB L2, so no flush is needed.

Prints one JSON line (rank 0). Under torchrun each rank runs an independent
replica of the workload on its own GPU (weak scaling, no collective on the
data path); the reported time is the max over ranks.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (the oracle is the reference implementation here).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FLARE encode+decode tokens/s at 1 GB300; % of roofline (HBM GB/s or tensor-pipe)"
UNIT = "tokens/s"
WORKLOAD = "c2_bf16"
PROFILE_SUMMARY = {  # kernel -> committed ncu summary holding its DRAM traffic
    "encoder": os.path.join(ROOT, "profiles", "encoder_c2_bf16.md"),
    "decode": os.path.join(ROOT, "profiles", "decode_c2_bf16.md"),
}
KERNEL_SOURCES = {   # files whose content the profiled traffic belongs to
    "encoder": ["tc_encoder.cuh", "tc_ptx.cuh", "tc_kernels.cu"],
    "decode": ["tc_decode.cuh", "tc_ptx.cuh", "tc_kernels.cu"],
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        p = os.path.join(ROOT, "latent_query_split_gb300", "csrc", name)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def _profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it still
    describes the current kernel source (else None)."""
    path = PROFILE_SUMMARY[kernel]
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.TemporaryFile(mode="w+")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.out.read())) if len(r) >= 9]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_oracle_sample(w, inputs, max_heads=None):
    """Time the fp64 oracle on a bounded sample: encode + decode of every token
    for the first `max_heads` (b, h) pairs. Returns (tokens/s, description, threads)."""
    import numpy as np
    import torch

    import oracle
    heads = max_heads or 2
    K = inputs["K"][0:1, :, :heads].contiguous().cpu()
    V = inputs["V"][0:1, :, :heads].contiguous().cpu()
    Q = inputs["Q"][:heads].contiguous().cpu()
    mask = None if inputs["mask"] is None else inputs["mask"][0:1].cpu()
    oracle.build()
    t0 = time.perf_counter()
    Z, L = oracle.encode(Q, K, V, mask)
    oracle.decode(Q, Z, K)
    dt = time.perf_counter() - t0
    # one token slot of the workload carries H heads; the sample did `heads` of them
    equiv_tokens = w.N * heads / w.H
    desc = (f"encode (M={w.M} latents, all {w.N} tokens) + decode of all {w.N} tokens for "
            f"{heads} of {w.B * w.H} (batch, head) pairs = {equiv_tokens:.0f} token-equivalents")
    return equiv_tokens / dt, desc, oracle.num_threads(), dt


def run_reference(args, w):
    import torch
    from latent_query_split_gb300 import workloads
    world, rank, _ = _dist_env()
    if rank != 0:
        return 0
    inputs = workloads.make_inputs(w, device="cpu")
    for _ in range(args.warmup):
        cpu_oracle_sample(w, inputs, max_heads=1)
    vals, secs = [], 0.0
    for _ in range(args.steps):
        v, desc, cores, dt = cpu_oracle_sample(w, inputs, max_heads=1)
        vals.append(v)
        secs += dt
    value = statistics.median(vals)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "impl": "reference",
            "config": {"workload": f"{w.name}: FLARE fwd bf16 inputs, B{w.B} H{w.H} D{w.D} "
                                   f"M{w.M} N{w.N} R{w.R}, 5% padded slots; one step = a "
                                   f"bounded sample (one batch-head pair)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--kernel", choices=["auto", "simt", "tensor"], default="auto")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)

    from latent_query_split_gb300 import workloads
    w = workloads.CONFIGS[WORKLOAD]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    import torch.distributed as dist
    from latent_query_split_gb300 import flare

    world, rank, local = _dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    inputs = workloads.make_inputs(w.scaled(seed=w.seed + rank), device=dev)
    Q, K, V, mask, off = inputs["Q"], inputs["K"], inputs["V"], inputs["mask"], inputs["offsets"]
    B, N, H, D, M = w.B, w.N, w.H, w.D, w.M
    Y = torch.empty_like(K)
    Z = torch.empty((B, H, M, D), dtype=torch.float32, device=dev)
    L = torch.empty((B, H, M), dtype=torch.float32, device=dev)
    dims = flare.make_dims(Q, K, None, args.kernel)
    ws_bytes = flare.flare_workspace_bytes(flare.FLARE_OP_FWD, dims, off)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(ev=None):
        # encoder (+ fused merge) and decode, each bracketed by events on `stream`
        with torch.cuda.stream(stream):
            if ev is not None:
                ev[0].record(stream)
            flare.flare_encoder_fwd(Q, K, V, mask, off, Z=Z, L=L, workspace=ws,
                                    kernel=args.kernel, stream=stream)
            if ev is not None:
                ev[1].record(stream)
            flare.flare_decode_fwd(Q, Z, K, Y=Y, kernel=args.kernel, stream=stream)
            if ev is not None:
                ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    flare.flare_device_status(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clock_info = clocks.stop()
    flare.flare_device_status(stream)
    elapsed_ms = start.elapsed_time(end)
    enc_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    dec_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    ms_per_step = elapsed_ms / args.steps
    tokens_per_step = B * N * world
    value = tokens_per_step / (ms_per_step * 1e-3)

    # end to end through the public API with host buffers (pinned), copies timed
    hK, hV = K.cpu().pin_memory(), V.cpu().pin_memory()
    hQ = Q.cpu().pin_memory()
    hmask = mask.cpu().pin_memory() if mask is not None else None
    hY = torch.empty(Y.shape, dtype=Y.dtype).pin_memory()
    dK, dV, dQ = torch.empty_like(K), torch.empty_like(V), torch.empty_like(Q)
    dmask = torch.empty_like(mask) if mask is not None else None
    h2d = sum(t.numel() * t.element_size() for t in (hK, hV, hQ) + ((hmask,) if hmask is not None else ()))
    d2h = hY.numel() * hY.element_size()

    def e2e_step():
        with torch.cuda.stream(stream):
            dK.copy_(hK, non_blocking=True)
            dV.copy_(hV, non_blocking=True)
            dQ.copy_(hQ, non_blocking=True)
            if dmask is not None:
                dmask.copy_(hmask, non_blocking=True)
            flare.flare_fwd(dQ, dK, dV, dmask, off, Y=Y, Z=Z, L=L, workspace=ws,
                            kernel=args.kernel, stream=stream)
            hY.copy_(Y, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    if world > 1:
        dist.barrier()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e2.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = s2.elapsed_time(e2) / e2e_steps
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    flare.flare_device_status(stream)

    # roofline of the dominant kernel (algorithmic bytes: K,V read by the
    # encoder; K read + Y written by the decode; each byte counted once)
    hbm_gbs, _, peak_kind = _peaks()
    tok_bytes = B * N * H * D * K.element_size()
    dominant = "encoder" if enc_ms >= dec_ms else "decode"
    kern_ms = enc_ms if dominant == "encoder" else dec_ms
    algo_bytes = 2 * tok_bytes
    achieved = algo_bytes / (kern_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "traffic": _profiled_traffic(dominant),
                "kernel": dominant, "peak_source": peak_kind,
                "encoder_ms": enc_ms, "decode_ms": dec_ms,
                "encoder_frac": algo_bytes / (enc_ms * 1e-3) / 1e9 / hbm_gbs,
                "decode_frac": algo_bytes / (dec_ms * 1e-3) / 1e9 / hbm_gbs}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded, on device)",
            "config": {"workload": f"{w.name}: FLARE fwd bf16 B{B} H{H} D{D} M{M} N{N} R{w.R} "
                                   f"ragged shards, 5% padded slots",
                       "kernel": args.kernel, "tokens_per_step": tokens_per_step,
                       "l2": "inputs larger than L2 (K, V 256 MiB each), no flush",
                       "parallelism": f"{world} independent replicas" if world > 1 else "1 GPU"},
            "clocks": clock_info,
            "e2e": {"value": tokens_per_step / (e2e_ms * 1e-3), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms},
            "gpu_launches": 2 * args.steps,
            "roofline": roofline}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        hin = {"K": K, "V": V, "Q": Q, "mask": mask}
        v, desc, cores, _ = cpu_oracle_sample(w, hin, max_heads=2)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
