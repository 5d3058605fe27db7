"""bench.py's algorithmic work per step (host logic, no GPU).

The roofline fraction divides these byte and flop counts by the measured
time, so they are pinned here to the per-(b, h) forms: a forward pass streams
K and V (or K in, Y out), 2·N·D elements, with two GEMM-shaped products of
2·M·N·D flops each; the encoder backward reads K, V and writes dK, dV with
five such products; the decode backward reads K, dY and writes dK. The
expected totals below are those forms evaluated for the named workloads.
"""
import pytest

import bench
from latent_query_split_gb300 import workloads as wl

MB = 1e6


def _alg(name):
    w = wl.CONFIGS[name]
    return bench.algorithmic(w, 4 if w.dtype == "f32" else 2)


def test_flare_forward_counts_each_byte_once():
    a = _alg("c2_bf16")
    # B4 H8 N65536 D64 bf16: 2 tensors x 268.4 MB per pass
    assert a["encoder"][0] == a["decode"][0] == 536870912
    assert a["encoder"][1] == a["decode"][1] == 4.0 * 4 * 8 * 128 * 65536 * 64
    assert a["encoder"][1] / 1e9 == pytest.approx(68.72, abs=0.01)


def test_long_context_and_small_workloads():
    a = _alg("c4_long_bf16")
    assert a["encoder"][0] / 1e9 == pytest.approx(17.18, abs=0.01)
    assert (a["encoder"][1] + a["decode"][1]) / 1e12 == pytest.approx(2.2, abs=0.01)
    s = _alg("c1_fp32_small")
    assert s["encoder"][0] == 2 * 1 * 2 * 1024 * 32 * 4          # fp32 elements
    assert (s["encoder"][0] + s["decode"][0]) / MB == pytest.approx(1.05, abs=0.01)


def test_flare_pp_forward_is_three_passes():
    al = _alg("c3_pp_bf16")
    a = al["flare_pp_fwd"]
    assert a[0] / 1e9 == pytest.approx(3 * 2.147, abs=0.01)
    assert a[1] / 1e12 == pytest.approx(1.65, abs=0.01)
    # one encoder pass and the decode, timed alone: a third each
    assert al["encoder"][0] == al["decode"][0] == a[0] / 3
    assert al["encoder"][1] == al["decode"][1] == a[1] / 3


def test_dominant_kernel_of_a_composite_step():
    # the FLARE++ step launches the encoder twice and the decode once
    ms = {"flare_pp_fwd": 1.6, "encoder": 0.5, "decode": 0.55}
    assert bench.dominant_phase(ms, "flare_pp_fwd") == "encoder"
    ms["decode"] = 1.1
    assert bench.dominant_phase(ms, "flare_pp_fwd") == "decode"
    assert bench.dominant_phase({"encoder": 0.1, "decode": 0.2}, "flare_fwd") == "decode"


def test_backward_counts():
    e = _alg("c5_bwd_bf16")["encoder_bwd"]
    assert e[0] / 1e9 == pytest.approx(1.074, abs=0.001)        # K, V read; dK, dV written
    assert e[1] / 1e9 == pytest.approx(171.8, abs=0.1)           # 10·M·N·D per (b, h)
    d = _alg("c5_decbwd_bf16")["decode_bwd"]
    assert d[0] == 3 * 2 * 8 * 131072 * 64 * 2                   # K, dY read; dK written
    assert d[1] == e[1]
    m = _alg("c5_mixbwd_bf16")["flare_bwd"]
    assert m[0] == d[0] + e[0] + 2 * 8 * 131072 * 64 * 2         # + the old dK read back
    assert m[1] == d[1] + e[1]
    p = _alg("c5_ppbwd_bf16")["flare_pp_bwd"]
    assert p[0] == m[0] + e[0]                                   # + the query-synthesis encoder
    assert p[1] == m[1] + e[1]


def test_exponentials_one_per_latent_token_pair_and_pass():
    w = wl.CONFIGS["c2_bf16"]
    pair = w.B * w.H * w.M * w.N
    assert bench.algorithmic_exps(w) == {"encoder": pair, "decode": pair}
    w3 = wl.CONFIGS["c3_pp_bf16"]
    assert bench.algorithmic_exps(w3)["flare_pp_fwd"] / 1e9 == pytest.approx(3 * 2.147, abs=0.01)
    w5 = wl.CONFIGS["c5_mixbwd_bf16"]
    assert bench.algorithmic_exps(w5)["flare_bwd"] == 2 * w5.B * w5.H * w5.M * w5.N


def test_every_workload_has_kernel_sources_for_its_phases():
    for name, w in wl.CONFIGS.items():
        for phase in _alg(name):
            assert phase in bench.KERNEL_SOURCES, (name, phase)
            assert len(bench.kernel_source_hash(phase)) == 16
