"""GPU parity of every entry point against the fp64 oracle at sizes the oracle
finishes in seconds: several tiles, ragged tails, ragged/empty/padded shards,
both kernel families, and the degenerate cases of the method."""
import math

import numpy as np
import pytest
import torch

import oracle
from latent_query_split_gb300 import flare
from parity import assert_close, assert_L_close, max_err

pytestmark = pytest.mark.gpu

KERNELS = ["simt", "tensor"]


def _call(fn, *a, **kw):
    try:
        return fn(*a, **kw)
    except flare.FlareError as e:
        if e.status == flare.FLARE_ERR_UNSUPPORTED and kw.get("kernel") == "tensor":
            pytest.skip(f"no tensor-core kernel: {e}")
        raise


def _problem(seed, B, H, M, N, D, dtype, offsets, pad=0.1, q_std=0.5, replicated=True, dev="cuda"):
    g = torch.Generator(device="cpu").manual_seed(seed)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    Q = (torch.randn((H, M, D) if replicated else (B, H, M, D), generator=g) * q_std).to(dt)
    K = torch.randn((B, N, H, D), generator=g).to(dt)
    V = torch.randn((B, N, H, D), generator=g).to(dt)
    mask = (torch.rand((B, N), generator=g) > pad).to(torch.uint8) if pad > 0 else None
    return Q.to(dev), K.to(dev), V.to(dev), None if mask is None else mask.to(dev)


CASES = [
    # B, H, M, N, D, offsets, dtype
    (2, 2, 16, 1000, 32, [0, 250, 500, 750, 1000], "f32"),
    (2, 2, 64, 3001, 64, [0, 700, 700, 2000, 3001], "bf16"),
    (1, 3, 128, 5000, 64, [0, 1234, 1300, 4999, 5000], "bf16"),
    (2, 2, 256, 2600, 64, [0, 1000, 2600], "bf16"),
    (1, 2, 64, 2100, 128, [0, 129, 2100], "bf16"),
    (1, 2, 128, 1500, 128, [0, 1500], "f32"),
    (2, 1, 37, 777, 40, [0, 300, 777], "f32"),
    (1, 2, 128, 2048, 64, [0, 512, 1024, 1536, 2048], "f32"),
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}M{c[2]}N{c[3]}D{c[4]}{c[6]}")
def test_encoder_shards_and_merge(cuda_device, kernel, case):
    B, H, M, N, D, off, dt = case
    Q, K, V, mask = _problem(1, B, H, M, N, D, dt, off)
    O_r, L_r, Z, L = _call(flare.flare_encoder_fwd, Q, K, V, mask, off, shard_outputs=True,
                           kernel=kernel)
    flare.flare_device_status()
    Zo, Lo = oracle.encode(Q, K, V, mask)
    Oo, Lro = oracle.encode_shards(Q, K, V, mask, off)
    assert_close("Z", Z, Zo, dt)
    assert_L_close("L", L, Lo)
    assert_close("O_r", O_r, Oo, dt)
    assert_L_close("L_r", L_r, Lro)
    # the standalone merge over the per-shard outputs gives the fused result
    Zm, Lm = flare.flare_lse_merge(O_r, L_r)
    assert_close("Z(merge)", Zm, Zo, dt)
    assert_L_close("L(merge)", Lm, Lo)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}M{c[2]}N{c[3]}D{c[4]}{c[6]}")
def test_flare_fwd_and_decode(cuda_device, kernel, case):
    B, H, M, N, D, off, dt = case
    Q, K, V, mask = _problem(2, B, H, M, N, D, dt, off)
    Y, Z, L = _call(flare.flare_fwd, Q, K, V, mask, off, kernel=kernel)
    flare.flare_device_status()
    Zo, Lo, Yo = oracle.flare_fwd(Q, K, V, mask)
    assert_close("Z", Z, Zo, dt)
    assert_L_close("L", L, Lo)
    assert_close("Y", Y, Yo, dt)
    # decode alone, on the oracle's own Z (fp32), against the oracle decode
    Zf = torch.from_numpy(Zo).float().to(K.device)
    Y2 = _call(flare.flare_decode_fwd, Q, Zf, K, kernel=kernel)
    assert_close("Y(decode)", Y2, oracle.decode(Q, Zf, K), dt)


@pytest.mark.parametrize("kernel", KERNELS)
def test_per_batch_query(cuda_device, kernel):
    B, H, M, N, D = 2, 2, 128, 1800, 64
    off = [0, 900, 1800]
    Q, K, V, mask = _problem(3, B, H, M, N, D, "bf16", off, replicated=False)
    Y, Z, L = _call(flare.flare_fwd, Q, K, V, mask, off, kernel=kernel)
    Zo, Lo, Yo = oracle.flare_fwd(Q, K, V, mask)
    assert_close("Z", Z, Zo, "bf16")
    assert_L_close("L", L, Lo)
    assert_close("Y", Y, Yo, "bf16")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dt,M,D", [("f32", 16, 32), ("bf16", 256, 64), ("bf16", 64, 128)])
def test_flare_pp_fwd(cuda_device, kernel, dt, M, D):
    B, H, N = 2, 2, 2500
    off = [0, 600, 600, 2500]
    g = torch.Generator().manual_seed(4)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    Qs = (torch.randn((H, M, D), generator=g) * 0.02).to(tdt).cuda()
    Kt, Vt, K, V = (torch.randn((B, N, H, D), generator=g).to(tdt).cuda() for _ in range(4))
    mask = (torch.rand((B, N), generator=g) > 0.1).to(torch.uint8).cuda()
    Y, Qd, L1, Z, L2 = _call(flare.flare_pp_fwd, Qs, Kt, Vt, K, V, mask, off, kernel=kernel)
    flare.flare_device_status()
    Qdo, L1o, Zo, L2o, Yo = oracle.flare_pp_fwd(Qs, Kt, Vt, K, V, mask)
    assert_close("Q(X)", Qd, Qdo, dt)
    assert_L_close("L1", L1, L1o)
    assert_close("Z", Z, Zo, dt)
    assert_L_close("L2", L2, L2o)
    assert_close("Y", Y, Yo, dt)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dt,M,D,N", [("f32", 16, 32, 700), ("bf16", 128, 64, 3000),
                                      ("bf16", 64, 128, 1100), ("bf16", 64, 128, 9000),
                                      ("bf16", 128, 128, 3000), ("bf16", 256, 64, 900)])
def test_encoder_bwd(cuda_device, kernel, dt, M, D, N):
    B, H = 2, 2
    off = [0, 200, 200, N]
    Q, K, V, mask = _problem(5, B, H, M, N, D, dt, off, q_std=1.0)
    mask[1, 200:] = 0                         # batch element 1: only shard 0 is live
    g = torch.Generator().manual_seed(6)
    dZ = torch.randn((B, H, M, D), generator=g).cuda()
    Zo, Lo = oracle.encode(Q, K, V, mask)
    Zf = torch.from_numpy(Zo).float().cuda()
    Lf = torch.from_numpy(Lo).float().cuda()
    dQ, dK, dV = _call(flare.flare_encoder_bwd, Q, K, V, mask, off, Zf, Lf, dZ, kernel=kernel)
    flare.flare_device_status()
    dQo, dKo, dVo = oracle.encode_bwd(Q, K, V, mask, Zf, Lf, dZ)
    assert_close("dQ", dQ, dQo, dt)
    assert_close("dK", dK, dKo, dt)
    assert_close("dV", dV, dVo, dt)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("M,replicated", [(128, True), (64, True), (128, False), (256, True), (256, False)])
def test_encoder_bwd_multi_tile_spans(cuda_device, kernel, M, replicated):
    """Enough 128-token tiles that each persistent CTA walks several tiles and
    crosses (b, h) boundaries, so dQ is assembled from several partial pieces;
    rows with a global L of -inf contribute nothing; repeated runs agree bit
    for bit (the pieces are summed in a fixed order). M = 256 runs as two
    passes of 128 latent rows, the second adding its dK and dV shares."""
    B, H, N, D = 2, 3, 20000, 64
    off = [0, 5000, 5000, N]
    Q, K, V, mask = _problem(16, B, H, M, N, D, "bf16", off, q_std=1.0, replicated=replicated)
    mask[1, 12000:] = 0
    g = torch.Generator().manual_seed(17)
    dZ = torch.randn((B, H, M, D), generator=g).cuda()
    Zo, Lo = oracle.encode(Q, K, V, mask)
    Lo[0, 1, :5] = -math.inf
    Zo[0, 1, :5] = 0.0
    Zf = torch.from_numpy(Zo).float().cuda()
    Lf = torch.from_numpy(Lo).float().cuda()
    dQ, dK, dV = _call(flare.flare_encoder_bwd, Q, K, V, mask, off, Zf, Lf, dZ, kernel=kernel)
    flare.flare_device_status()
    dQo, dKo, dVo = oracle.encode_bwd(Q, K, V, mask, Zf, Lf, dZ)
    assert_close("dQ", dQ, dQo, "bf16")
    assert_close("dK", dK, dKo, "bf16")
    assert_close("dV", dV, dVo, "bf16")
    pad = mask == 0
    assert dK[pad].abs().max().item() == 0.0 and dV[pad].abs().max().item() == 0.0
    dQ2, dK2, dV2 = _call(flare.flare_encoder_bwd, Q, K, V, mask, off, Zf, Lf, dZ, kernel=kernel)
    assert torch.equal(dQ, dQ2) and torch.equal(dK, dK2) and torch.equal(dV, dV2)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dt,M,D,N,replicated", [("f32", 16, 32, 700, True), ("bf16", 128, 64, 3000, True),
                                                 ("bf16", 64, 64, 2100, False), ("bf16", 64, 128, 1100, True),
                                                 ("bf16", 256, 64, 900, True), ("bf16", 256, 64, 9000, False),
                                                 ("bf16", 64, 128, 9000, False), ("bf16", 128, 128, 3000, True),
                                                 ("f32", 37, 40, 333, False)])
def test_decode_bwd(cuda_device, kernel, dt, M, D, N, replicated):
    B, H = 2, 2
    Q, K, _, _ = _problem(18, B, H, M, N, D, dt, [0, N], pad=0, q_std=1.0, replicated=replicated)
    g = torch.Generator().manual_seed(19)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    Z = torch.randn((B, H, M, D), generator=g).cuda()
    dY = torch.randn((B, N, H, D), generator=g).to(tdt).cuda()
    dQ, dZ, dK = _call(flare.flare_decode_bwd, Q, Z, K, dY, kernel=kernel)
    flare.flare_device_status()
    dQo, dZo, dKo = oracle.decode_bwd(Q, Z, K, dY)
    # dQ and dZ add one bf16-rounded product per token, so their rounding
    # error grows like sqrt(N): past a few thousand tokens they are held to
    # the full-size bound, 2e-2 of max(1, largest reference magnitude)
    many = dt == "bf16" and N > 4096
    for name, dev, ref in (("dQ", dQ, dQo), ("dZ", dZ, dZo)):
        err, scale = max_err(dev, ref)
        print(f"{name}: max abs err {err:.3e}, max |ref| {scale:.3e}")
        assert_close(name, dev, ref, dt, atol=2e-2 * max(1.0, scale) if many else None)
    assert_close("dK", dK, dKo, dt)
    # two runs agree bit for bit (fixed-order sums)
    dQ2, dZ2, dK2 = _call(flare.flare_decode_bwd, Q, Z, K, dY, kernel=kernel)
    assert torch.equal(dQ, dQ2) and torch.equal(dZ, dZ2) and torch.equal(dK, dK2)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("M,D,replicated", [(128, 64, True), (256, 64, False), (256, 64, True),
                                            (64, 128, False), (128, 128, False)])
def test_decode_bwd_multi_tile_spans(cuda_device, kernel, M, D, replicated):
    """Enough 128-token tiles that each persistent CTA walks several tiles
    and crosses (b, h) boundaries: the pipelines' barriers go through many
    phases (the M = 256 statistics kernel hands each tile's partial row
    statistics from one warp to another), and dQ, dZ are assembled from
    several pieces; repeated runs agree bit for bit."""
    B, H, N = 2, 3, 20000
    Q, K, _, _ = _problem(20, B, H, M, N, D, "bf16", [0, N], pad=0, q_std=1.0, replicated=replicated)
    g = torch.Generator().manual_seed(21)
    Z = torch.randn((B, H, M, D), generator=g).cuda()
    dY = torch.randn((B, N, H, D), generator=g).to(torch.bfloat16).cuda()
    dQ, dZ, dK = _call(flare.flare_decode_bwd, Q, Z, K, dY, kernel=kernel)
    flare.flare_device_status()
    dQo, dZo, dKo = oracle.decode_bwd(Q, Z, K, dY)
    for name, dev, ref in (("dQ", dQ, dQo), ("dZ", dZ, dZo)):
        err, scale = max_err(dev, ref)
        print(f"{name}: max abs err {err:.3e}, max |ref| {scale:.3e}")
        # one bf16-rounded product per token: the full-size bound (see test_decode_bwd)
        assert_close(name, dev, ref, "bf16", atol=2e-2 * max(1.0, scale))
    assert_close("dK", dK, dKo, "bf16")
    dQ2, dZ2, dK2 = _call(flare.flare_decode_bwd, Q, Z, K, dY, kernel=kernel)
    assert torch.equal(dQ, dQ2) and torch.equal(dZ, dZ2) and torch.equal(dK, dK2)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dt,M,D,N,replicated", [("f32", 16, 32, 700, True), ("bf16", 128, 64, 3000, True),
                                                 ("bf16", 64, 64, 2100, False), ("bf16", 256, 64, 900, True),
                                                 ("bf16", 128, 64, 20000, True), ("bf16", 64, 128, 4000, False),
                                                 ("bf16", 128, 128, 2500, True)])
def test_flare_bwd(cuda_device, kernel, dt, M, D, N, replicated):
    """FLARE mixer backward: the decode's shares of dQ and dK are written
    first and the encoder's are added in place (dK read back and summed in
    fp32); padded tokens keep the decode's dK and get no dV. The 20000-token
    case walks several tiles per CTA across (b, h) boundaries."""
    B, H = 2, 3 if N > 10000 else 2
    off = [0, N // 4, N // 4, N]
    Q, K, V, mask = _problem(30, B, H, M, N, D, dt, off, q_std=1.0, replicated=replicated)
    mask[1, N // 2:] = 0
    g = torch.Generator().manual_seed(31)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    dY = torch.randn((B, N, H, D), generator=g).to(tdt).cuda()
    Zo, Lo = oracle.encode(Q, K, V, mask)
    Zf = torch.from_numpy(Zo).float().cuda()
    Lf = torch.from_numpy(Lo).float().cuda()
    dQ, dK, dV = _call(flare.flare_bwd, Q, K, V, mask, off, Zf, Lf, dY, kernel=kernel)
    flare.flare_device_status()
    dQo, dKo, dVo = oracle.flare_bwd(Q, K, V, mask, Zf, Lf, dY)
    assert_close("dQ", dQ, dQo, dt)
    assert_close("dK", dK, dKo, dt)
    assert_close("dV", dV, dVo, dt)
    pad = mask == 0
    assert dV[pad].abs().max().item() == 0.0
    dQ2, dK2, dV2 = _call(flare.flare_bwd, Q, K, V, mask, off, Zf, Lf, dY, kernel=kernel)
    assert torch.equal(dQ, dQ2) and torch.equal(dK, dK2) and torch.equal(dV, dV2)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dt,M,D,N", [("f32", 16, 32, 700), ("bf16", 128, 64, 2500), ("bf16", 64, 64, 5000),
                                      ("bf16", 256, 64, 2500), ("bf16", 64, 128, 3000), ("bf16", 128, 128, 2000)])
def test_flare_pp_bwd(cuda_device, kernel, dt, M, D, N):
    """FLARE++ mixer backward from the oracle's forward statistics: the seeds'
    gradient, the four token gradients and the summed gradient of Q(X)."""
    B, H = 2, 2
    off = [0, 600, 600, N]
    g = torch.Generator().manual_seed(32)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    Qs = (torch.randn((H, M, D), generator=g) * 0.5).to(tdt).cuda()
    Kt, Vt, K, V, dY = (torch.randn((B, N, H, D), generator=g).to(tdt).cuda() for _ in range(5))
    mask = (torch.rand((B, N), generator=g) > 0.1).to(torch.uint8).cuda()
    Qdo, L1o, Zo, L2o, _ = oracle.flare_pp_fwd(Qs, Kt, Vt, K, V, mask)
    Qd, L1, Z, L2 = (torch.from_numpy(x).float().cuda() for x in (Qdo, L1o, Zo, L2o))
    out = _call(flare.flare_pp_bwd, Qs, Kt, Vt, K, V, mask, off, Qd, L1, Z, L2, dY, want_dQdyn=True,
                kernel=kernel)
    flare.flare_device_status()
    # the device rounds Q(X) to bf16 as an operand: the oracle takes the same values
    Qd_op = Qd.to(tdt).float() if dt == "bf16" else Qd
    ref = oracle.flare_pp_bwd(Qs, Kt, Vt, K, V, mask, Qd_op, L1, Z, L2, dY)
    # encoder 1's c = <dZ1, Z1> uses the unrounded Q(X)
    ref1 = oracle.encode_bwd(Qs, Kt, Vt, mask, Qd, L1, ref[5])
    for name, dev, r in zip(("dQseed", "dKt", "dVt", "dK", "dV", "dQdyn"), out,
                            (ref1[0], ref1[1], ref1[2]) + tuple(ref[3:])):
        assert_close(name, dev, r, dt)
    out2 = _call(flare.flare_pp_bwd, Qs, Kt, Vt, K, V, mask, off, Qd, L1, Z, L2, dY, want_dQdyn=True,
                 kernel=kernel)
    assert all(torch.equal(x, y) for x, y in zip(out, out2))


# ---- edge cases ------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", KERNELS)
def test_empty_and_masked_rows(cuda_device, kernel):
    """Rows with no valid key anywhere return L = -inf, Z = 0 (never NaN); an
    empty shard returns L_r = -inf, O_r = 0."""
    B, H, M, N, D = 3, 2, 64, 1000, 64
    off = [0, 0, 400, 400, 1000]
    Q, K, V, mask = _problem(7, B, H, M, N, D, "bf16", off)
    mask[0] = 0                      # batch element 0: every row empty
    mask[1, 400:] = 0                # batch element 1: shard 3 all padding
    O_r, L_r, Z, L = _call(flare.flare_encoder_fwd, Q, K, V, mask, off, shard_outputs=True,
                           kernel=kernel)
    Zo, Lo = oracle.encode(Q, K, V, mask)
    assert_close("Z", Z, Zo, "bf16")
    assert_L_close("L", L, Lo)
    assert torch.all(L[0] == -math.inf) and torch.all(Z[0] == 0)
    assert torch.all(L_r[[0, 2]] == -math.inf) and torch.all(O_r[[0, 2]] == 0)
    assert torch.all(L_r[3, 1] == -math.inf)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("N", [1, 127, 129])
def test_tiny_token_counts(cuda_device, kernel, N):
    Q, K, V, mask = _problem(8, 1, 2, 128, N, 64, "bf16", [0, N], pad=0)
    Y, Z, L = _call(flare.flare_fwd, Q, K, V, None, [0, N], kernel=kernel)
    Zo, Lo, Yo = oracle.flare_fwd(Q, K, V, None)
    assert_close("Z", Z, Zo, "bf16")
    assert_L_close("L", L, Lo)
    assert_close("Y", Y, Yo, "bf16")


def test_no_tokens(cuda_device):
    Q, K, V, _ = _problem(9, 2, 2, 16, 0, 32, "f32", [0, 0], pad=0)
    O_r, L_r, Z, L = flare.flare_encoder_fwd(Q, K, V, None, [0, 0, 0], shard_outputs=True)
    assert torch.all(L == -math.inf) and torch.all(Z == 0)
    assert torch.all(L_r == -math.inf) and torch.all(O_r == 0)
    Y = flare.flare_decode_fwd(Q, Z, K)
    assert Y.numel() == 0


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("M,D", [(128, 64), (256, 64), (64, 128), (128, 128)])
@pytest.mark.parametrize("N", [1, 127, 129])
def test_mixer_bwd_tiny_token_counts(cuda_device, kernel, N, M, D):
    """FLARE and FLARE++ backward with a single tile that is partly or almost
    entirely past N (tokens past N are neither read nor written), for every
    tensor-core backward shape family (two latent passes at M = 256, two
    column passes at D = 128). With one
    token every latent output equals that token's value, so Y does not depend
    on the queries or keys and no gradient reaches the query-synthesis
    encoder: dQ, dK, dQseed, dK~, dV~ are exactly zero. A bound relative to a
    zero reference means nothing, so those are held to the absolute bf16
    bound alone (the device's values are rounding noise: dZ enters dP as a
    bf16 operand while c = <dZ, Z> is fp32)."""
    def check(name, dev, r):
        if N == 1 and name in ("dQ", "dK", "dQseed", "dKt", "dVt"):
            assert np.abs(r).max() < 1e-12
            assert dev.abs().max().item() <= 2e-2, name
        else:
            assert_close(name, dev, r, "bf16")

    Q, K, V, _ = _problem(11, 1, 2, M, N, D, "bf16", [0, N], pad=0, q_std=1.0)
    g = torch.Generator().manual_seed(12)
    dY = torch.randn(K.shape, generator=g).to(K.dtype).cuda()
    Zo, Lo = oracle.encode(Q, K, V, None)
    Zf, Lf = torch.from_numpy(Zo).float().cuda(), torch.from_numpy(Lo).float().cuda()
    dQ, dK, dV = _call(flare.flare_bwd, Q, K, V, None, [0, N], Zf, Lf, dY, kernel=kernel)
    flare.flare_device_status()
    ref = oracle.flare_bwd(Q, K, V, None, Zf, Lf, dY)
    for name, dev, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), ref):
        check(name, dev, r)
    Kt, Vt = (torch.randn(K.shape, generator=g).to(K.dtype).cuda() for _ in range(2))
    Qs = (0.5 * torch.randn(Q.shape, generator=g)).to(Q.dtype).cuda()
    Qdo, L1o, Zpo, L2o, _ = oracle.flare_pp_fwd(Qs, Kt, Vt, K, V, None)
    Qd, L1, Zp, L2 = (torch.from_numpy(x).float().cuda() for x in (Qdo, L1o, Zpo, L2o))
    out = _call(flare.flare_pp_bwd, Qs, Kt, Vt, K, V, None, [0, N], Qd, L1, Zp, L2, dY, kernel=kernel)
    flare.flare_device_status()
    refp = oracle.flare_pp_bwd(Qs, Kt, Vt, K, V, None, Qd.to(K.dtype).float(), L1, Zp, L2, dY)
    ref1 = oracle.encode_bwd(Qs, Kt, Vt, None, Qd, L1, refp[5])
    for name, dev, r in zip(("dQseed", "dKt", "dVt", "dK", "dV"), out[:5],
                            (ref1[0], ref1[1], ref1[2], refp[3], refp[4])):
        check(name, dev, r)


def test_mixer_bwd_no_tokens(cuda_device):
    """N = 0: no token gradient, and every latent gradient is zero."""
    Q, K, V, _ = _problem(13, 2, 2, 16, 0, 32, "f32", [0, 0], pad=0)
    Z = torch.zeros((2, 2, 16, 32), device="cuda")
    L = torch.full((2, 2, 16), -math.inf, device="cuda")
    dQ, dK, dV = flare.flare_bwd(Q, K, V, None, [0, 0], Z, L, torch.empty_like(K))
    flare.flare_device_status()
    assert dK.numel() == 0 and dV.numel() == 0 and torch.all(dQ == 0)


@pytest.mark.parametrize("kernel", KERNELS)
def test_flare_pp_shared_projection(cuda_device, kernel):
    """The shared-projection FLARE++ variant (K~ = K, V~ = V; the FLARE++
    page's closing remark): the same tensors passed as K~, V~ and K, V. The
    gradient of each shared projection is the sum of its two shares."""
    B, H, M, N, D = 2, 2, 128, 3000, 64
    off = [0, 1000, 3000]
    g = torch.Generator().manual_seed(33)
    Qs = (torch.randn((H, M, D), generator=g) * 0.5).bfloat16().cuda()
    K, V, dY = (torch.randn((B, N, H, D), generator=g).bfloat16().cuda() for _ in range(3))
    mask = (torch.rand((B, N), generator=g) > 0.1).to(torch.uint8).cuda()
    Y, Qd, L1, Z, L2 = _call(flare.flare_pp_fwd, Qs, K, V, K, V, mask, off, kernel=kernel)
    Qdo, L1o, Zo, L2o, Yo = oracle.flare_pp_fwd(Qs, K, V, K, V, mask)
    assert_close("Y", Y, Yo, "bf16")
    out = _call(flare.flare_pp_bwd, Qs, K, V, K, V, mask, off, Qd, L1, Z, L2, dY, kernel=kernel)
    flare.flare_device_status()
    ref = oracle.flare_pp_bwd(Qs, K, V, K, V, mask, Qd.bfloat16().float(), L1, Z, L2, dY)
    ref1 = oracle.encode_bwd(Qs, K, V, mask, Qd, L1, ref[5])
    assert_close("dQseed", out[0], ref1[0], "bf16")
    assert_close("dK + dK~", out[1].float() + out[3].float(), ref1[1] + ref[3], "bf16")
    assert_close("dV + dV~", out[2].float() + out[4].float(), ref1[2] + ref[4], "bf16")


def test_max_shards_and_single_token_shards(cuda_device):
    N = 300
    off = list(range(0, 256)) + [N]              # 255 one-token shards + one long shard
    Q, K, V, mask = _problem(10, 1, 1, 16, N, 32, "f32", off)
    O_r, L_r, Z, L = flare.flare_encoder_fwd(Q, K, V, mask, off, shard_outputs=True)
    Zo, Lo = oracle.encode(Q, K, V, mask)
    assert_close("Z", Z, Zo, "f32")
    assert_L_close("L", L, Lo)
    Oo, Lro = oracle.encode_shards(Q, K, V, mask, off)
    assert_close("O_r", O_r, Oo, "f32")
    assert_L_close("L_r", L_r, Lro)


@pytest.mark.parametrize("kernel", KERNELS)
def test_max_shards_bf16(cuda_device, kernel):
    """FLARE_MAX_SHARDS ragged shards (some empty) on the bf16 path."""
    N = 40000
    rng = np.random.default_rng(14)
    cuts = np.sort(rng.integers(0, N + 1, size=255))
    off = [0] + [int(c) for c in cuts] + [N]
    Q, K, V, mask = _problem(15, 1, 2, 128, N, 64, "bf16", off)
    O_r, L_r, Z, L = _call(flare.flare_encoder_fwd, Q, K, V, mask, off, shard_outputs=True,
                           kernel=kernel)
    Zo, Lo = oracle.encode(Q, K, V, mask)
    assert_close("Z", Z, Zo, "bf16")
    assert_L_close("L", L, Lo)
    Oo, Lro = oracle.encode_shards(Q, K, V, mask, off)
    assert_close("O_r", O_r, Oo, "bf16")
    assert_L_close("L_r", L_r, Lro)


def test_minimal_sizes(cuda_device):
    Q, K, V, _ = _problem(11, 1, 1, 1, 5, 1, "f32", [0, 5], pad=0)
    Y, Z, L = flare.flare_fwd(Q, K, V)
    Zo, Lo, Yo = oracle.flare_fwd(Q, K, V)
    assert_close("Z", Z, Zo, "f32")
    assert_close("Y", Y, Yo, "f32")


def test_merge_all_empty_rows_and_shard_order(cuda_device):
    g = torch.Generator().manual_seed(12)
    R, B, H, M, D = 5, 2, 2, 40, 24
    O_r = torch.randn((R, B, H, M, D), generator=g)
    L_r = torch.randn((R, B, H, M), generator=g) * 5
    L_r[1] = -math.inf
    O_r[1] = 0
    L_r[:, 0, 0, :3] = -math.inf
    O_r[:, 0, 0, :3] = 0
    Z, L = flare.flare_lse_merge(O_r.cuda(), L_r.cuda())
    Zo, Lo = oracle.lse_merge(O_r, L_r)
    assert_close("Z", Z, Zo, "f32", atol=1e-5, rel=1e-5)
    assert_L_close("L", L, Lo)
    assert torch.all(Z[0, 0, :3] == 0) and torch.all(L[0, 0, :3] == -math.inf)
    perm = torch.randperm(R, generator=g)
    Zp, Lp = flare.flare_lse_merge(O_r[perm].contiguous().cuda(), L_r[perm].contiguous().cuda())
    assert (Zp - Z).abs().max().item() <= 4 * R * 1.2e-7 * Z.abs().max().item()


@pytest.mark.parametrize("kernel", KERNELS)
def test_repeated_runs_are_bit_identical(cuda_device, kernel):
    Q, K, V, mask = _problem(13, 2, 2, 128, 4000, 64, "bf16", [0, 1000, 4000])
    off = [0, 1000, 4000]
    a = _call(flare.flare_fwd, Q, K, V, mask, off, kernel=kernel)
    b = _call(flare.flare_fwd, Q, K, V, mask, off, kernel=kernel)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
