"""The seeded input recipe of the named workloads (host logic, no GPU).

Checks that the generators produce the structure the workloads state: R
contiguous shards summing to N with lengths proportional to U[0.5, 1.5]
draws, the listed empty shards, the exact padded count per batch element, the
fully padded (batch element, shard) of the backward workloads, and the 1%
of keys scaled by 8 in the long-context workload; and that every draw is a
pure function of the seed.
"""
import dataclasses

import numpy as np
import pytest
import torch

from latent_query_split_gb300 import workloads as wl


def _offsets(w):
    rng = np.random.default_rng(w.seed)
    return wl.shard_offsets(w.N, w.R, rng, equal=w.equal_shards, empty=w.empty_shards), rng


@pytest.mark.parametrize("name", sorted(wl.CONFIGS))
def test_shards_are_contiguous_and_cover_every_token(name):
    w = wl.CONFIGS[name]
    off, _ = _offsets(w)
    assert len(off) == w.R + 1 and off[0] == 0 and off[-1] == w.N
    lens = np.diff(off)
    assert (lens >= 0).all()
    for r in range(w.R):
        assert (lens[r] == 0) == (r in set(w.empty_shards))


@pytest.mark.parametrize("name", ["c2_bf16", "c3_pp_bf16", "c4_long_bf16", "c5_bwd_bf16"])
def test_unequal_shard_lengths_follow_the_uniform_draw(name):
    w = wl.CONFIGS[name]
    off, _ = _offsets(w)
    lens = np.diff(off)
    live = [r for r in range(w.R) if r not in set(w.empty_shards)]
    # the same draw as the generator: lengths are floor(u / sum(u) * N), the
    # last live shard taking the remainder (fewer than one token per shard)
    u = np.random.default_rng(w.seed).uniform(0.5, 1.5, size=len(live))
    share = np.floor(u / u.sum() * w.N).astype(np.int64)
    assert list(lens[live[:-1]]) == list(share[:-1])
    assert 0 <= lens[live[-1]] - share[-1] < len(live)
    # lengths within a factor 3 of each other (1.5 / 0.5), up to the remainder
    assert lens[live].max() <= 3 * lens[live].min() + len(live)


def test_equal_shards_of_the_small_workload():
    w = wl.CONFIGS["c1_fp32_small"]
    off, _ = _offsets(w)
    assert list(np.diff(off)) == [w.N // w.R] * w.R


def test_padding_count_is_exact_per_batch_element():
    w = wl.CONFIGS["c2_bf16"]
    off, rng = _offsets(w)
    mask = wl.make_mask(w, off, rng)
    assert mask.shape == (w.B, w.N) and mask.dtype == np.uint8
    npad = int(round(w.pad_frac * w.N))
    for b in range(w.B):
        assert int((mask[b] == 0).sum()) == npad
    # padding is spread over the sequence, not one block
    assert len(np.unique(np.nonzero(mask[0] == 0)[0] * w.R // w.N)) == w.R


@pytest.mark.parametrize("name", ["c5_bwd_bf16", "c5_mixbwd_bf16", "c5_ppbwd_bf16"])
def test_backward_workloads_pad_one_whole_shard(name):
    w = wl.CONFIGS[name]
    off, rng = _offsets(w)
    mask = wl.make_mask(w, off, rng)
    b, r = w.padded_shard
    assert off[r + 1] > off[r]
    assert (mask[b, off[r]:off[r + 1]] == 0).all()
    # everything else is valid, so every latent row keeps valid keys globally
    rest = mask.copy()
    rest[b, off[r]:off[r + 1]] = 1
    assert (rest == 1).all()
    for bb in range(w.B):
        assert mask[bb].sum() > 0


def test_unpadded_workloads_have_no_mask():
    for name in ["c1_fp32_small", "c3_pp_bf16", "c4_long_bf16", "c5_decbwd_bf16"]:
        w = wl.CONFIGS[name]
        off, rng = _offsets(w)
        assert wl.make_mask(w, off, rng) is None


def test_key_boost_scales_whole_keys_by_eight():
    base = wl.CONFIGS["c4_long_bf16"]
    w = base.scaled(N=4096, H=2, D=128, M=64, R=4)
    plain = dataclasses.replace(w, key_boost_frac=0.0, key_boost=1.0)
    a = wl.make_inputs(w)
    p = wl.make_inputs(plain)
    idx = a["boosted_tokens"]
    assert len(idx) == int(round(w.key_boost_frac * w.N)) and len(np.unique(idx)) == len(idx)
    others = np.setdiff1d(np.arange(w.N), idx)
    # a power of two is exact in bf16: boosted keys are the plain draw times 8
    assert torch.equal(a["K"][:, idx].float(), 8.0 * p["K"][:, idx].float())
    assert torch.equal(a["K"][:, others], p["K"][:, others])
    assert torch.equal(a["V"], p["V"]) and torch.equal(a["Q"], p["Q"])


@pytest.mark.parametrize("name", sorted(wl.CONFIGS))
def test_inputs_are_a_function_of_the_seed(name):
    w = wl.CONFIGS[name].scaled(N=512, R=min(wl.CONFIGS[name].R, 8))
    if w.padded_shard is not None and w.padded_shard[1] >= w.R:
        w = dataclasses.replace(w, padded_shard=None)
    w = dataclasses.replace(w, empty_shards=tuple(r for r in w.empty_shards if r < w.R - 1))
    a, b = wl.make_inputs(w), wl.make_inputs(w)
    assert a["offsets"] == b["offsets"]
    for k, v in a.items():
        if isinstance(v, torch.Tensor):
            assert torch.equal(v, b[k]), k
            assert v.dtype in (torch.float32, torch.bfloat16, torch.uint8), k
    tok = (w.B, w.N, w.H, w.D)
    assert tuple(a["K"].shape) == tok and a["K"].dtype == w.torch_dtype
    q = a["Qseed"] if "Qseed" in a else a["Q"]
    assert tuple(q.shape) == (w.H, w.M, w.D)


def test_query_standard_deviation_reading():
    # N(0, sigma) read with sigma the standard deviation: c2's Q ~ N(0, 0.5)
    w = wl.CONFIGS["c2_bf16"].scaled(H=8, M=128, D=64, N=256)
    q = wl.make_inputs(w)["Q"].float()
    assert abs(q.std().item() - 0.5) < 0.02
    s = wl.make_inputs(wl.CONFIGS["c3_pp_bf16"].scaled(N=256, R=4))["Qseed"].float()
    assert abs(s.std().item() - 0.02) < 0.002
