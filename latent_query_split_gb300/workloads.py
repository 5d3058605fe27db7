"""Seeded synthetic workloads for the FLARE / FLARE++ token mixer.

This module only draws random inputs (values, shard offsets, padding masks);
it holds none of the mixer's arithmetic, so both the CUDA path and the fp64
oracle take their inputs from here.

Shapes follow the appendix "FLARE++: Low-rank attention with dynamic attention
routing" (context-parallel section): token tensors [B, N, H, D] (C = H*D
channels of the per-token projections), the replicated latent queries or seeds
[H, M, D], R token shards with unequal sizes and padding excluded by a mask.

The eight named workloads:
  c1_fp32_small  FLARE fwd fp32, B1 H2 D32 M16 N1024, R4 equal shards, N(0,1)
  c2_bf16        FLARE fwd bf16, B4 H8 D64 M128 N65536, R8 shards of length
                 ~U[0.5,1.5]*N/R summing to N, 5% padded slots; K,V ~ N(0,1),
                 Q ~ N(0, 0.5^2)
  c3_pp_bf16     FLARE++ fwd bf16, B2 H16 D64 M256 N262144, R16; seeds
                 ~ N(0, 0.02^2), K~,V~,K,V ~ N(0,1)
  c4_long_bf16   FLARE fwd bf16, B1 H8 D128 M64 N4194304, R64; 1% of tokens
                 have their whole key (all heads) scaled by 8
  c5_bwd_bf16    encoder bwd bf16, B2 H8 D64 M128 N131072, R8 with shards 2
                 and 5 empty, shard 3 of batch element 1 all padding; dZ ~ N(0,1)
  c5_decbwd_bf16 decode bwd bf16 on the shapes of c5_bwd_bf16 (no mask: the
                 decode has none); Z, dY ~ N(0,1)
  c5_mixbwd_bf16 FLARE mixer bwd bf16 (decode bwd, then encoder bwd adding
                 into dQ, dK) on the shapes, shards and mask of c5_bwd_bf16;
                 Q ~ N(0, 0.5^2), dY ~ N(0,1); Z, L from the forward
  c5_ppbwd_bf16  FLARE++ mixer bwd bf16 on the same shapes, shards and mask;
                 seeds ~ N(0, 0.02^2), K~,V~,K,V,dY ~ N(0,1); Q(X), L1, Z, L2
                 from the forward
N(0, sigma) is read with sigma the standard deviation.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "flare_fwd" | "flare_pp_fwd" | "encoder_bwd" | "decode_bwd"
                         # | "flare_bwd" | "flare_pp_bwd"
    dtype: str           # "f32" | "bf16"
    B: int
    H: int
    M: int
    N: int
    D: int
    R: int
    seed: int
    q_std: float = 1.0           # std of Q (or of the FLARE++ seeds)
    pad_frac: float = 0.0        # padded fraction of token slots per batch element
    key_boost_frac: float = 0.0  # fraction of tokens whose key is scaled
    key_boost: float = 1.0
    empty_shards: Sequence[int] = field(default_factory=tuple)
    padded_shard: Optional[tuple] = None   # (batch element, shard) fully padded
    equal_shards: bool = False

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def scaled(self, **kw) -> "Workload":
        """Same structure at other sizes (for parity cases the oracle can finish)."""
        return dataclasses.replace(self, **kw)


CONFIGS: Dict[str, Workload] = {
    "c1_fp32_small": Workload("c1_fp32_small", "flare_fwd", "f32", B=1, H=2, M=16,
                              N=1024, D=32, R=4, seed=1001, equal_shards=True),
    "c2_bf16": Workload("c2_bf16", "flare_fwd", "bf16", B=4, H=8, M=128, N=65536,
                        D=64, R=8, seed=1002, q_std=0.5, pad_frac=0.05),
    "c3_pp_bf16": Workload("c3_pp_bf16", "flare_pp_fwd", "bf16", B=2, H=16, M=256,
                           N=262144, D=64, R=16, seed=1003, q_std=0.02),
    "c4_long_bf16": Workload("c4_long_bf16", "flare_fwd", "bf16", B=1, H=8, M=64,
                             N=4194304, D=128, R=64, seed=1004,
                             key_boost_frac=0.01, key_boost=8.0),
    "c5_bwd_bf16": Workload("c5_bwd_bf16", "encoder_bwd", "bf16", B=2, H=8, M=128,
                            N=131072, D=64, R=8, seed=1005, empty_shards=(2, 5),
                            padded_shard=(1, 3)),
    "c5_decbwd_bf16": Workload("c5_decbwd_bf16", "decode_bwd", "bf16", B=2, H=8, M=128,
                               N=131072, D=64, R=8, seed=1006),
    "c5_mixbwd_bf16": Workload("c5_mixbwd_bf16", "flare_bwd", "bf16", B=2, H=8, M=128,
                               N=131072, D=64, R=8, seed=1007, q_std=0.5, empty_shards=(2, 5),
                               padded_shard=(1, 3)),
    "c5_ppbwd_bf16": Workload("c5_ppbwd_bf16", "flare_pp_bwd", "bf16", B=2, H=8, M=128,
                              N=131072, D=64, R=8, seed=1008, q_std=0.02, empty_shards=(2, 5),
                              padded_shard=(1, 3)),
}


def shard_offsets(N: int, R: int, rng: np.random.Generator, equal: bool = False,
                  empty: Sequence[int] = ()) -> List[int]:
    """Offsets [0, ..., N] of R contiguous shards.

    Non-empty shards get lengths drawn as u ~ U[0.5, 1.5], rescaled to sum to
    N and floored; the last non-empty shard absorbs the remainder. Shards
    listed in `empty` get length 0.
    """
    live = [r for r in range(R) if r not in set(empty)]
    lens = [0] * R
    if equal:
        for i, r in enumerate(live):
            lens[r] = N // len(live) + (1 if i < N % len(live) else 0)
    elif live:
        u = rng.uniform(0.5, 1.5, size=len(live))
        share = np.floor(u / u.sum() * N).astype(np.int64)
        for r, n in zip(live, share):
            lens[r] = int(n)
        lens[live[-1]] += N - sum(lens)
    off = [0]
    for n in lens:
        off.append(off[-1] + n)
    assert off[-1] == N
    return off


def make_mask(w: Workload, offsets: Sequence[int], rng: np.random.Generator):
    """uint8 [B, N] key-padding mask (1 = valid) or None when nothing is padded."""
    if w.pad_frac <= 0.0 and w.padded_shard is None:
        return None
    mask = np.ones((w.B, w.N), dtype=np.uint8)
    if w.pad_frac > 0.0:
        npad = int(round(w.pad_frac * w.N))
        for b in range(w.B):
            mask[b, rng.choice(w.N, size=npad, replace=False)] = 0
    if w.padded_shard is not None:
        b, r = w.padded_shard
        mask[b, offsets[r]:offsets[r + 1]] = 0
    return mask


def make_inputs(w: Workload, device="cpu") -> dict:
    """Draw every input of workload `w` on `device` (deterministic in w.seed).

    Returns a dict with the token tensors ("K", "V", and "Kt", "Vt" for
    FLARE++), the latent query ("Q", or "Qseed"), host "offsets" (list of R+1
    ints), "mask" (uint8 [B,N] tensor on `device`, or None), "scale" (None =
    D^-1/2), "dZ" for the encoder backward, "Z" (fp32 [B,H,M,D]) and "dY"
    (token-shaped) for the decode backward, and "dY" for the mixer backward
    passes (their forward statistics come from the forward, not from here).
    """
    rng = np.random.default_rng(w.seed)
    offsets = shard_offsets(w.N, w.R, rng, equal=w.equal_shards, empty=w.empty_shards)
    mask_np = make_mask(w, offsets, rng)
    boosted = None
    if w.key_boost_frac > 0.0:
        boosted = np.sort(rng.choice(w.N, size=int(round(w.key_boost_frac * w.N)),
                                     replace=False))
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    dt = w.torch_dtype

    def normal(shape, std=1.0):
        x = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(dt)

    tok = (w.B, w.N, w.H, w.D)
    out = {"offsets": offsets, "scale": None,
           "mask": None if mask_np is None else torch.from_numpy(mask_np).to(dev)}
    if w.kind in ("flare_pp_fwd", "flare_pp_bwd"):
        out["Qseed"] = normal((w.H, w.M, w.D), w.q_std)
        out["Kt"] = normal(tok)
        out["Vt"] = normal(tok)
    else:
        out["Q"] = normal((w.H, w.M, w.D), w.q_std)
    K = normal(tok)
    if boosted is not None:
        idx = torch.from_numpy(boosted).to(dev)
        K[:, idx] *= w.key_boost     # power of two: exact in bf16
    out["K"] = K
    out["V"] = normal(tok)
    if w.kind == "encoder_bwd":
        out["dZ"] = torch.randn((w.B, w.H, w.M, w.D), generator=g, device=dev,
                                dtype=torch.float32)
    if w.kind == "decode_bwd":
        out["Z"] = torch.randn((w.B, w.H, w.M, w.D), generator=g, device=dev,
                               dtype=torch.float32)
        out["dY"] = normal(tok)
    if w.kind in ("flare_bwd", "flare_pp_bwd"):
        out["dY"] = normal(tok)
    out["boosted_tokens"] = boosted
    return out


def token_sample(w: Workload, count: int, seed: int = 0) -> np.ndarray:
    """Seeded sample of flat token slots b*N + n (for checks at full size)."""
    rng = np.random.default_rng(w.seed * 7919 + seed)
    total = w.B * w.N
    count = min(count, total)
    return np.sort(rng.choice(total, size=count, replace=False)).astype(np.int64)
