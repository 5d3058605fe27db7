"""Throughput benchmark of the FLARE / FLARE++ token mixer on one GB300.

One step = one pass of the hot path over one batch of a named workload
(latent_query_split_gb300.workloads.CONFIGS), inputs resident in HBM:
  c4_long_bf16 (default)  FLARE forward bf16, B=1 H=8 D=128 M=64 N=4194304,
                     R=64 ragged shards, 1% of keys x8: the split-KV encoder
                     with its log-sum-exp merge, then the local decode of
                     every token (the largest FLARE encode+decode workload)
  c2_bf16            the same forward, B=4 H=8 D=64 M=128 N=65536, R=8
                     ragged shards, 5% padded tokens
  c1_fp32_small      the same forward on the small fp32 workload
  c3_pp_bf16         FLARE++ forward (encoder twice, then the decode)
  c5_bwd_bf16        global-normaliser encoder backward (dQ, dK, dV)
  c5_decbwd_bf16     decode backward (dQ, dZ, dK) on the shapes of c5
  c5_mixbwd_bf16     FLARE mixer backward on the shapes of c5
  c5_ppbwd_bf16      FLARE++ mixer backward on the shapes of c5
--n N runs a workload's structure at N tokens (small cases for profilers).
Token tensors of c2-c5 are 256 MiB or more each (larger than the 129 MB L2),
so no flush is needed between steps; c1 flushes L2 between steps.

Prints one JSON line (rank 0). Under torchrun (N > 1 GPUs) the FLARE forward
workloads run context-parallel by default (--mode cp): every rank holds its
own slice of N tokens of one problem of N x ranks tokens and a replica of the
latent queries, the ranks all-gather their partial (O_r, L_r) over NCCL and
each merges them and decodes its own tokens (weak scaling: the tokens per GPU
are fixed). --mode replicas, and every other workload, runs an independent
replica per GPU with no collective on the data path. The reported time is the
max over ranks.

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
DEFAULT_WORKLOAD = "c4_long_bf16"
# library sources whose content a committed ncu traffic figure belongs to
KERNEL_SOURCES = {
    "encoder": ["tc_encoder.cuh", "tc_ptx.cuh", "tc_host.cuh", "tc_kernels.cu"],
    "decode": ["tc_decode.cuh", "tc_ptx.cuh", "tc_host.cuh", "tc_kernels.cu"],
    "encoder_bwd": ["tc_backward.cuh", "tc_ptx.cuh", "tc_host.cuh", "tc_bwd_launch.cu",
                    "simt_kernels.cu"],
    "flare_pp_fwd": ["tc_encoder.cuh", "tc_decode.cuh", "tc_ptx.cuh", "tc_host.cuh", "tc_kernels.cu"],
    "decode_bwd": ["tc_decode_bwd.cuh", "tc_backward.cuh", "tc_ptx.cuh", "tc_host.cuh",
                   "tc_bwd_launch.cu", "simt_decode_bwd.cu"],
    "flare_bwd": ["tc_decode_bwd.cuh", "tc_backward.cuh", "tc_ptx.cuh", "tc_host.cuh",
                  "tc_bwd_launch.cu", "simt_decode_bwd.cu", "simt_kernels.cu", "flare_api.cu"],
    "flare_pp_bwd": ["tc_decode_bwd.cuh", "tc_backward.cuh", "tc_ptx.cuh", "tc_host.cuh",
                     "tc_bwd_launch.cu", "simt_decode_bwd.cu", "simt_kernels.cu", "flare_api.cu"],
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


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary
    profiles/<kernel>_<workload>.md, if it still describes the current kernel
    source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
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


def replica_workload(w, rank: int):
    """The workload rank `rank` runs: the same shapes, its own seed (each rank
    is an independent replica; no data moves between ranks)."""
    return w.scaled(seed=w.seed + rank)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest `value` over all ranks (the slowest rank's time); the
    identity on one rank."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_replica: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every replica's tokens over the slowest rank's step time."""
    return tokens_per_replica * world / (ms_per_step * 1e-3)


def describe(w) -> str:
    what = {"flare_fwd": "FLARE fwd (encoder + merge + decode)",
            "flare_pp_fwd": "FLARE++ fwd (encoder x2 + decode)",
            "encoder_bwd": "encoder bwd (dQ, dK, dV)",
            "decode_bwd": "decode bwd (dQ, dZ, dK)",
            "flare_bwd": "FLARE mixer bwd (decode bwd + encoder bwd; dQ, dK, dV)",
            "flare_pp_bwd": "FLARE++ mixer bwd (decode bwd + two encoder bwd)"}[w.kind]
    extra = []
    if w.pad_frac:
        extra.append(f"{w.pad_frac:.0%} padded slots")
    if w.empty_shards:
        extra.append(f"empty shards {list(w.empty_shards)}")
    if w.padded_shard:
        extra.append(f"shard {w.padded_shard[1]} of batch {w.padded_shard[0]} all padding")
    if w.key_boost_frac:
        extra.append(f"{w.key_boost_frac:.0%} of keys x{w.key_boost:g}")
    return (f"{w.name}: {what} {w.dtype} B{w.B} H{w.H} D{w.D} M{w.M} N{w.N} R{w.R} "
            f"{'equal' if w.equal_shards else 'ragged'} shards" +
            ("".join(", " + e for e in extra)))


# ---- algorithmic work per step (each required byte counted once) --------------
def algorithmic(w, elem):
    """Per-phase algorithmic (bytes, flops) of one step.

    A pass over one (b, h) streams 2*N*D elements (K and V read, or K read and
    Y written) and does 4*M*N*D flops (two GEMM-shaped products); the backward
    reads K, V and writes dK, dV (4*N*D elements) with 10*M*N*D flops."""
    bh = w.B * w.H
    tok = bh * w.N * w.D * elem
    pass_flops = 4.0 * bh * w.M * w.N * w.D
    if w.kind == "flare_fwd":
        return {"encoder": (2 * tok, pass_flops), "decode": (2 * tok, pass_flops)}
    if w.kind == "flare_pp_fwd":    # the whole call, and one encoder pass and the decode alone
        return {"flare_pp_fwd": (6 * tok, 3 * pass_flops), "encoder": (2 * tok, pass_flops),
                "decode": (2 * tok, pass_flops)}
    if w.kind == "decode_bwd":      # K, dY read, dK written; five GEMM-shaped products
        return {"decode_bwd": (3 * tok, 2.5 * pass_flops)}
    if w.kind == "flare_bwd":       # decode bwd, then encoder bwd reading the old dK too
        return {"flare_bwd": (8 * tok, 5 * pass_flops)}
    if w.kind == "flare_pp_bwd":    # ... plus the query-synthesis encoder bwd
        return {"flare_pp_bwd": (12 * tok, 7.5 * pass_flops)}
    return {"encoder_bwd": (4 * tok, 2.5 * pass_flops)}


def algorithmic_exps(w):
    """Exponentials per step and phase (one per latent-token pair and pass):
    the third, diagnostic ceiling beside HBM and the tensor pipe."""
    pair = float(w.B * w.H * w.M * w.N)
    passes = {"flare_fwd": None, "flare_pp_fwd": 3, "decode_bwd": 1, "flare_bwd": 2,
              "flare_pp_bwd": 3, "encoder_bwd": 1}[w.kind]
    if passes is None:
        return {"encoder": pair, "decode": pair}
    if w.kind == "flare_pp_fwd":
        return {w.kind: passes * pair, "encoder": pair, "decode": pair}
    return {w.kind: passes * pair}


# Phases that stand for several kernels (a whole composite call): reported,
# but the roofline's dominant kernel is taken among the single-kernel phases,
# weighted by how often a step launches each.
COMPOSITE_PHASES = {"flare_pp_fwd": {"encoder": 2, "decode": 1}}


def dominant_phase(phase_ms, kind):
    """The phase whose kernel takes the largest share of a step."""
    calls = COMPOSITE_PHASES.get(kind)
    if calls is None:
        return max(phase_ms, key=phase_ms.get)
    return max(calls, key=lambda k: phase_ms[k] * calls[k])


def cpu_model() -> str:
    """The host CPU's model string (for the CPU baseline's record)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model", "CPU part"):
            for line in info.splitlines():
                if line.startswith(key) and ":" in line:
                    val = line.split(":", 1)[1].strip()
                    arm = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1",
                           "0xd0c": "Arm Neoverse-N1", "0xd49": "Arm Neoverse-N2"}
                    return f"{arm[val]} (CPU part {val})" if val in arm else val
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


# ---- the fp64 oracle on a bounded sample --------------------------------------
def cpu_oracle_sample(w, inputs, pairs=1):
    """Time the fp64 oracle on `pairs` (batch, head) pairs of the workload (every
    token of each). Returns (tokens/s, description, threads, seconds)."""
    import oracle
    b = 0
    hs = slice(0, pairs)
    mask = None if inputs["mask"] is None else inputs["mask"][b:b + 1].cpu()
    tok = lambda x: x[b:b + 1, :, hs].contiguous().cpu()    # noqa: E731
    oracle.build()
    if w.kind == "flare_fwd":
        Q, K, V = inputs["Q"][hs].contiguous().cpu(), tok(inputs["K"]), tok(inputs["V"])
        t0 = time.perf_counter()
        Z, L = oracle.encode(Q, K, V, mask)
        oracle.decode(Q, Z, K)
        dt = time.perf_counter() - t0
        what = "encode + decode"
    elif w.kind == "flare_pp_fwd":
        Qs = inputs["Qseed"][hs].contiguous().cpu()
        Kt, Vt, K, V = (tok(inputs[k]) for k in ("Kt", "Vt", "K", "V"))
        t0 = time.perf_counter()
        oracle.flare_pp_fwd(Qs, Kt, Vt, K, V, mask)
        dt = time.perf_counter() - t0
        what = "FLARE++ forward (two encodes + decode)"
    elif w.kind == "decode_bwd":
        Q, K, dY = inputs["Q"][hs].contiguous().cpu(), tok(inputs["K"]), tok(inputs["dY"])
        Z = inputs["Z"][b:b + 1, hs].contiguous().cpu()
        t0 = time.perf_counter()
        oracle.decode_bwd(Q, Z, K, dY)
        dt = time.perf_counter() - t0
        what = "decode backward"
    elif w.kind == "flare_bwd":
        Q, K, V, dY = (inputs["Q"][hs].contiguous().cpu(), tok(inputs["K"]), tok(inputs["V"]),
                       tok(inputs["dY"]))
        Z, L = oracle.encode(Q, K, V, mask)        # forward statistics, not timed
        t0 = time.perf_counter()
        oracle.flare_bwd(Q, K, V, mask, Z, L, dY)
        dt = time.perf_counter() - t0
        what = "FLARE mixer backward"
    elif w.kind == "flare_pp_bwd":
        Qs = inputs["Qseed"][hs].contiguous().cpu()
        Kt, Vt, K, V, dY = (tok(inputs[k]) for k in ("Kt", "Vt", "K", "V", "dY"))
        Qd, L1, Z, L2, _ = oracle.flare_pp_fwd(Qs, Kt, Vt, K, V, mask)   # not timed
        t0 = time.perf_counter()
        oracle.flare_pp_bwd(Qs, Kt, Vt, K, V, mask, Qd, L1, Z, L2, dY)
        dt = time.perf_counter() - t0
        what = "FLARE++ mixer backward"
    else:
        Q, K, V = inputs["Q"][hs].contiguous().cpu(), tok(inputs["K"]), tok(inputs["V"])
        dZ = inputs["dZ"][b:b + 1, hs].contiguous().cpu()
        Z, L = oracle.encode(Q, K, V, mask)        # forward statistics, not timed
        t0 = time.perf_counter()
        oracle.encode_bwd(Q, K, V, mask, Z, L, dZ)
        dt = time.perf_counter() - t0
        what = "encoder backward"
    equiv = w.N * pairs / w.H       # a token slot of the workload carries H heads
    desc = (f"{what} of all {w.N} tokens (M={w.M}) for {pairs} of {w.B * w.H} "
            f"(batch, head) pairs = {equiv:.0f} token-equivalents")
    return equiv / dt, desc, oracle.num_threads(), dt


def run_reference(args, w):
    from latent_query_split_gb300 import workloads
    world, rank, _ = _dist_env()
    if rank != 0:
        return 0
    inputs = workloads.make_inputs(w, device="cpu")
    for _ in range(args.warmup):
        cpu_oracle_sample(w, inputs)
    vals, secs = [], 0.0
    desc, cores = "", 0
    for _ in range(args.steps):
        v, desc, cores, dt = cpu_oracle_sample(w, inputs)
        vals.append(v)
        secs += dt
    value = statistics.median(vals)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "impl": "reference",
            "config": {"workload": describe(w) + "; one step = a bounded sample "
                                                 "(one batch-head pair)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc, "cpu": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---- one step of the hot path through the public API --------------------------
class Step:
    """Builds the phases of one step (each a call of the public API) for a
    workload, over device tensors."""

    def __init__(self, w, inp, dev, kernel, stream, ex=None):
        import torch
        from latent_query_split_gb300 import flare
        self.w, self.inp, self.kernel, self.stream = w, inp, kernel, stream
        self.ex = ex            # context-parallel exchange (FLARE forward over ranks), or None
        B, N, H, D, M = w.B, w.N, w.H, w.D, w.M
        f32 = dict(dtype=torch.float32, device=dev)
        self.off = inp["offsets"]
        self.Z = torch.empty((B, H, M, D), **f32)
        self.L = torch.empty((B, H, M), **f32)
        pp = w.kind in ("flare_pp_fwd", "flare_pp_bwd")
        Qref = inp["Qseed"] if pp else inp["Q"]
        dims = flare.make_dims(Qref, inp["K"], None, kernel)
        op = {"flare_fwd": flare.FLARE_OP_FWD, "flare_pp_fwd": flare.FLARE_OP_PP_FWD,
              "encoder_bwd": flare.FLARE_OP_ENCODER_BWD,
              "decode_bwd": flare.FLARE_OP_DECODE_BWD, "flare_bwd": flare.FLARE_OP_BWD,
              "flare_pp_bwd": flare.FLARE_OP_PP_BWD}[w.kind]
        nbytes = flare.flare_workspace_bytes(op, dims, None if w.kind == "decode_bwd" else self.off)
        if w.kind in ("flare_bwd", "flare_pp_bwd"):   # the forward that saves the statistics
            fop = flare.FLARE_OP_PP_FWD if pp else flare.FLARE_OP_ENCODER_FWD
            nbytes = max(nbytes, flare.flare_workspace_bytes(fop, dims, self.off))
        self.ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
        if w.kind == "flare_fwd":
            self.Y = torch.empty_like(inp["K"])
        elif w.kind == "flare_pp_fwd":
            self.Y = torch.empty_like(inp["K"])
            self.Qd, self.L1 = torch.empty((B, H, M, D), **f32), torch.empty((B, H, M), **f32)
            self.Qe, self.L1e = torch.empty_like(self.Qd), torch.empty_like(self.L1)
        elif w.kind == "decode_bwd":
            self.dQ, self.dZ = torch.empty((B, H, M, D), **f32), torch.empty((B, H, M, D), **f32)
            self.dK = torch.empty_like(inp["K"])
        elif w.kind == "flare_bwd":
            self.dQ = torch.empty((B, H, M, D), **f32)
            self.dK, self.dV = torch.empty_like(inp["K"]), torch.empty_like(inp["V"])
            flare.flare_encoder_fwd(inp["Q"], inp["K"], inp["V"], inp["mask"], self.off,
                                    Z=self.Z, L=self.L, workspace=self.ws, kernel=kernel,
                                    stream=stream)
        elif w.kind == "flare_pp_bwd":
            self.Qd, self.L1 = torch.empty((B, H, M, D), **f32), torch.empty((B, H, M), **f32)
            self.dQs = torch.empty((B, H, M, D), **f32)
            self.dKt, self.dVt = torch.empty_like(inp["Kt"]), torch.empty_like(inp["Vt"])
            self.dK, self.dV = torch.empty_like(inp["K"]), torch.empty_like(inp["V"])
            Y = torch.empty_like(inp["K"])
            flare.flare_pp_fwd(inp["Qseed"], inp["Kt"], inp["Vt"], inp["K"], inp["V"], inp["mask"],
                               self.off, Y=Y, Qdyn=self.Qd, L1=self.L1, Z=self.Z, L2=self.L,
                               workspace=self.ws, kernel=kernel, stream=stream)
            del Y
        else:
            self.dQ = torch.empty((B, H, M, D), **f32)
            self.dK, self.dV = torch.empty_like(inp["K"]), torch.empty_like(inp["V"])
            # the saved forward statistics the backward consumes (not timed)
            flare.flare_encoder_fwd(inp["Q"], inp["K"], inp["V"], inp["mask"], self.off,
                                    Z=self.Z, L=self.L, workspace=self.ws, kernel=kernel,
                                    stream=stream)

    def full_step(self, inp=None):
        """One step through the one-call public API of the workload."""
        from latent_query_split_gb300 import flare
        x = inp or self.inp
        w, k, st, off = self.w, self.kernel, self.stream, self.off
        if w.kind == "flare_fwd" and self.ex is not None:
            from latent_query_split_gb300 import cp
            cp.cp_fwd(self.ex, x["Q"], x["K"], x["V"], x["mask"], off, Y=self.Y, Z=self.Z,
                      L=self.L, workspace=self.ws, kernel=k, stream=st)
        elif w.kind == "flare_fwd":
            flare.flare_fwd(x["Q"], x["K"], x["V"], x["mask"], off, Y=self.Y, Z=self.Z, L=self.L,
                            workspace=self.ws, kernel=k, stream=st)
        else:
            # the composite call alone when the phases list adds its parts
            for _, fn in self.phases(inp)[:1 if w.kind in COMPOSITE_PHASES else None]:
                fn()

    def phases(self, inp=None):
        """[(name, callable)]: the step's parts as separate public calls (for
        the per-kernel roofline); `inp` overrides the input tensors."""
        from latent_query_split_gb300 import flare
        x = inp or self.inp
        w, k, st, off = self.w, self.kernel, self.stream, self.off
        if w.kind == "flare_fwd":
            return [("encoder", lambda: flare.flare_encoder_fwd(
                        x["Q"], x["K"], x["V"], x["mask"], off, Z=self.Z, L=self.L,
                        workspace=self.ws, kernel=k, stream=st)),
                    ("decode", lambda: flare.flare_decode_fwd(
                        x["Q"], self.Z, x["K"], Y=self.Y, kernel=k, stream=st))]
        if w.kind == "flare_pp_fwd":
            # the whole call; then the query-synthesis encoder pass (Q~ over
            # K~, V~) and the decode (Q(X), Z over K) alone, for their rooflines
            return [("flare_pp_fwd", lambda: flare.flare_pp_fwd(
                        x["Qseed"], x["Kt"], x["Vt"], x["K"], x["V"], x["mask"], off, Y=self.Y,
                        Qdyn=self.Qd, L1=self.L1, Z=self.Z, L2=self.L, workspace=self.ws,
                        kernel=k, stream=st)),
                    ("encoder", lambda: flare.flare_encoder_fwd(
                        x["Qseed"], x["Kt"], x["Vt"], x["mask"], off, Z=self.Qe, L=self.L1e,
                        workspace=self.ws, kernel=k, stream=st)),
                    ("decode", lambda: flare.flare_decode_fwd(
                        self.Qd, self.Z, x["K"], Y=self.Y, kernel=k, stream=st))]
        if w.kind == "decode_bwd":
            return [("decode_bwd", lambda: flare.flare_decode_bwd(
                        x["Q"], x["Z"], x["K"], x["dY"], dQ=self.dQ, dZ=self.dZ, dK=self.dK,
                        workspace=self.ws, kernel=k, stream=st))]
        if w.kind == "flare_bwd":
            return [("flare_bwd", lambda: flare.flare_bwd(
                        x["Q"], x["K"], x["V"], x["mask"], off, x.get("Zs", self.Z),
                        x.get("Ls", self.L), x["dY"], dQ=self.dQ, dK=self.dK, dV=self.dV,
                        workspace=self.ws, kernel=k, stream=st))]
        if w.kind == "flare_pp_bwd":
            return [("flare_pp_bwd", lambda: flare.flare_pp_bwd(
                        x["Qseed"], x["Kt"], x["Vt"], x["K"], x["V"], x["mask"], off,
                        x.get("Qds", self.Qd), x.get("L1s", self.L1), x.get("Zs", self.Z),
                        x.get("Ls", self.L), x["dY"], dQseed=self.dQs, dKt=self.dKt,
                        dVt=self.dVt, dK=self.dK, dV=self.dV, workspace=self.ws, kernel=k,
                        stream=st))]
        return [("encoder_bwd", lambda: flare.flare_encoder_bwd(
                    x["Q"], x["K"], x["V"], x["mask"], off, x.get("Zs", self.Z),
                    x.get("Ls", self.L), x["dZ"], dQ=self.dQ, dK=self.dK, dV=self.dV,
                    workspace=self.ws, kernel=k, stream=st))]

    def inputs_for_e2e(self):
        """Names of the device inputs a user copies in each step, and the
        outputs read back."""
        if self.w.kind == "flare_fwd":
            return ["Q", "K", "V", "mask"], [self.Y]
        if self.w.kind == "flare_pp_fwd":
            return ["Qseed", "Kt", "Vt", "K", "V", "mask"], [self.Y]
        if self.w.kind == "decode_bwd":
            return ["Q", "Z", "K", "dY"], [self.dQ, self.dZ, self.dK]
        if self.w.kind == "flare_bwd":
            return ["Q", "K", "V", "mask", "Zs", "Ls", "dY"], [self.dQ, self.dK, self.dV]
        if self.w.kind == "flare_pp_bwd":
            return (["Qseed", "Kt", "Vt", "K", "V", "mask", "Qds", "L1s", "Zs", "Ls", "dY"],
                    [self.dQs, self.dKt, self.dVt, self.dK, self.dV])
        return ["Q", "K", "V", "mask", "Zs", "Ls", "dZ"], [self.dQ, self.dK, self.dV]


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--kernel", choices=["auto", "simt", "tensor"], default="auto")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", choices=["auto", "cp", "replicas"], default="auto",
                    help="multi-GPU layout: context-parallel token slices (FLARE forward) or "
                         "independent replicas; auto = cp for the FLARE forward")
    ap.add_argument("--n", type=int, default=None,
                    help="run the workload's structure at N tokens (small cases for profiler captures)")
    args = ap.parse_args(argv)

    from latent_query_split_gb300 import workloads
    if args.workload not in workloads.CONFIGS:
        raise SystemExit(f"unknown workload {args.workload}: {sorted(workloads.CONFIGS)}")
    w = workloads.CONFIGS[args.workload]
    if args.n is not None:
        w = w.scaled(N=args.n)
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

    mode = args.mode
    if mode == "auto":
        mode = "cp" if w.kind == "flare_fwd" else "replicas"
    if mode == "cp" and w.kind != "flare_fwd":
        raise SystemExit("--mode cp runs the FLARE forward workloads")
    cp_on = mode == "cp" and world > 1
    inp = workloads.make_inputs(replica_workload(w, rank), device=dev)
    ex = None
    if cp_on:
        # one problem of N x world tokens: this rank's slice is its own draw,
        # the latent queries are rank 0's on every rank
        from latent_query_split_gb300 import cp
        dist.broadcast(inp["Q"], src=0)
        ex = cp.Exchange()
    stream = torch.cuda.Stream(device=dev)
    runner = Step(w, inp, dev, args.kernel, stream, ex)
    phases = runner.phases()
    # an L2 flush between steps for workloads whose tensors fit in L2
    elem = inp["K"].element_size()
    small = w.B * w.N * w.H * w.D * elem < (256 << 20)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if small else None

    def step():
        with torch.cuda.stream(stream):
            runner.full_step()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    flare.flare_device_status(stream)

    # the timed region: whole steps through the one-call API, events at its ends
    # (small workloads: every step bracketed by events after an L2 flush)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)] if flush is not None else None
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    launches0 = flare.flare_launch_count()
    start.record(stream)
    for i in range(args.steps):
        if step_evs is not None:
            with torch.cuda.stream(stream):
                flush.fill_(1)
                step_evs[i][0].record(stream)
        step()
        if step_evs is not None:
            step_evs[i][1].record(stream)
    end.record(stream)
    launches = flare.flare_launch_count() - launches0
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clock_info = clocks.stop()
    flare.flare_device_status(stream)
    elapsed_ms = start.elapsed_time(end)
    if step_evs is not None:    # the flush is not the mixer's work
        elapsed_ms = sum(a.elapsed_time(b) for a, b in step_evs)
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    ms_per_step = elapsed_ms / args.steps

    # per-phase times for the roofline: each phase alone, timed with events
    phase_ms = {}
    reps = max(3, min(args.steps, 200))
    for name, fn in phases:
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            pe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(reps)]
            for a, b in pe:
                if flush is not None:
                    flush.fill_(1)
                a.record(stream)
                fn()
                b.record(stream)
        torch.cuda.synchronize(dev)
        phase_ms[name] = statistics.mean(a.elapsed_time(b) for a, b in pe)
    flare.flare_device_status(stream)
    tokens_per_step = w.B * w.N * world
    value = weak_scaling_value(w.B * w.N, world, ms_per_step)

    # end to end through the public API with host buffers (pinned), copies timed:
    # every step copies its inputs in and reads its result back; the copy-in
    # of step i + 1 (on a copy stream, into the other of two device input
    # sets) overlaps step i, as a training or serving loop prefetches its
    # next batch
    e2e_in, e2e_out = runner.inputs_for_e2e()
    host = {}
    sets = [dict(inp), dict(inp)]
    extra = {"Zs": runner.Z, "Ls": runner.L, "Qds": getattr(runner, "Qd", None),
             "L1s": getattr(runner, "L1", None)}
    for name in e2e_in:
        t = extra[name] if name in extra else inp[name]
        if t is None:
            continue
        host[name] = t.cpu().pin_memory()
        for st_ in sets:
            st_[name] = torch.empty_like(t)
    hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in e2e_out]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in hout)
    cstream = torch.cuda.Stream(device=dev)
    h2d_ev = [torch.cuda.Event(), torch.cuda.Event()]
    done_ev = [torch.cuda.Event(), torch.cuda.Event()]

    def copy_in(i):
        k = i % 2
        with torch.cuda.stream(cstream):
            if i >= 2:
                cstream.wait_event(done_ev[k])       # step i - 2 has read this set
            for name, t in host.items():
                sets[k][name].copy_(t, non_blocking=True)
            h2d_ev[k].record(cstream)

    def compute(i):
        k = i % 2
        with torch.cuda.stream(stream):
            stream.wait_event(h2d_ev[k])
            runner.full_step(sets[k])
            done_ev[k].record(stream)
            for h, d in zip(hout, e2e_out):
                h.copy_(d, non_blocking=True)

    def e2e_run(n, start_ev=None):
        with torch.cuda.stream(cstream):
            if start_ev is not None:
                cstream.wait_event(start_ev)
            copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)

    big = h2d > (8 << 30)
    e2e_run(1 if big else 3)
    torch.cuda.synchronize(dev)
    e2e_steps = 3 if big else max(3, min(args.steps, args.e2e_steps))
    if world > 1:
        dist.barrier()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    e2e_run(e2e_steps, s2)
    e2.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = s2.elapsed_time(e2) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    flare.flare_device_status(stream)

    # roofline of the dominant phase: algorithmic bytes / its event time
    hbm_gbs, bf16_tf, peak_kind = _peaks()
    algo = algorithmic(w, elem)
    exps = algorithmic_exps(w)
    # ex2 ceiling: 32 results per clock per SM (measured on this part), at the sampled SM clock
    sm_mhz = clock_info.get("sm_mhz") or clock_info.get("sm_max_mhz") or 2070.0
    exp_peak = 32.0 * torch.cuda.get_device_properties(dev).multi_processor_count * sm_mhz * 1e6
    dominant = dominant_phase(phase_ms, w.kind)
    per_phase = {}
    for name, ms in phase_ms.items():
        b, f = algo[name]
        per_phase[name] = {"ms": ms, "hbm_frac": b / (ms * 1e-3) / 1e9 / hbm_gbs,
                           "tensor_frac": f / (ms * 1e-3) / 1e12 / bf16_tf,
                           "exp_frac": exps[name] / (ms * 1e-3) / exp_peak,
                           "algo_bytes": b, "algo_flops": f, "algo_exps": exps[name]}
    bytes_dom = algo[dominant][0]
    achieved = bytes_dom / (phase_ms[dominant] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "traffic": profiled_traffic(dominant, w.name),
                "kernel": dominant, "peak_source": peak_kind,
                "timing": "each phase alone, CUDA events on its stream, mean of "
                          f"{reps} calls", "phases": per_phase}

    dt_name = {"f32": "f32", "bf16": "bf16"}[w.dtype]
    # token slots include padding; the rate over valid (unpadded) tokens too
    valid_frac = 1.0 if inp["mask"] is None else float(inp["mask"].float().mean().item())
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dt_name,
            "data": "synthetic (seeded, on device)",
            "config": {"workload": describe(w), "kernel": args.kernel,
                       "tokens_per_step": tokens_per_step,
                       "valid_token_fraction": valid_frac,
                       "l2": ("512 MiB L2 flush between steps (not timed)" if flush is not None
                              else "inputs larger than L2 (token tensors >= 256 MiB), no flush"),
                       "parallelism": (("context-parallel over %d GPUs: %d tokens per GPU, "
                                        "NCCL all-gather of (O_r, L_r), merge and decode on "
                                        "every rank" % (world, w.N)) if cp_on else
                                       f"{world} independent replicas" if world > 1 else "1 GPU")},
            "clocks": clock_info,
            "e2e": {"value": tokens_per_step / (e2e_ms * 1e-3), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms,
                    "copies": "each step's inputs copied in from pinned host memory (step i + 1's "
                              "on a second stream, overlapping step i) and its result read back"},
            "gpu_launches": launches,
            "valid_tokens_per_s": value * valid_frac,
            "roofline": roofline}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, cores, _ = cpu_oracle_sample(w, inp, pairs=1 if w.N > 1 << 20 else 2)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc, "cpu": cpu_model()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
