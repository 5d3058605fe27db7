"""Every output and workspace of every entry point between canary regions.

Small problems that still span several tiles, a ragged tail, empty and
padded shards, the largest shard count, one token and no token; after each
call the device status must be clear and every guard intact (a kernel that
writes outside its tensors fails here). Run under the FLARE_DEBUG build too
(test_gpu_zdebug_build.py), where every TMA tile's place and workspace index
is also checked on the device.
"""
import pytest
import torch

from guards import guarded
from latent_query_split_gb300 import flare

pytestmark = pytest.mark.gpu

# B, H, M, N, D, dtype, offsets
CASES = [
    (2, 2, 128, 3001, 64, "bf16", [0, 700, 700, 2000, 3001]),
    (1, 2, 256, 2600, 64, "bf16", [0, 1000, 2600]),
    (1, 2, 64, 2100, 128, "bf16", [0, 129, 2100]),
    (2, 2, 16, 1000, 32, "f32", [0, 250, 500, 750, 1000]),
    (1, 1, 64, 1000, 64, "bf16", [min(4 * i, 1000) for i in range(257)]),   # 256 shards
    (1, 2, 128, 1, 64, "bf16", [0, 0, 1]),                                   # one token
]
IDS = ["m128", "m256", "d128", "f32", "max_shards", "tiny"]


def _inputs(case, seed=3):
    B, H, M, N, D, dt, off = case
    g = torch.Generator().manual_seed(seed)
    dtype = torch.float32 if dt == "f32" else torch.bfloat16
    Q = (torch.randn((H, M, D), generator=g) * 0.5).to(dtype).cuda()
    K = torch.randn((B, N, H, D), generator=g).to(dtype).cuda()
    V = torch.randn((B, N, H, D), generator=g).to(dtype).cuda()
    mask = (torch.rand((B, N), generator=g) > 0.1).to(torch.uint8).cuda()
    return Q, K, V, mask, off


def _ws(op, Q, K, off):
    n = flare.flare_workspace_bytes(op, flare.make_dims(Q, K), off)
    return guarded((max(n, 1),), torch.uint8)


def _check(*gs):
    flare.flare_device_status()
    for name, g in gs:
        g.check(name)


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_forward_entry_points_stay_inside_their_buffers(cuda_device, case):
    Q, K, V, mask, off = _inputs(case)
    B, H, M, N, D, dt, _ = case
    R = len(off) - 1
    f32 = torch.float32
    O_r, gO = guarded((R, B, H, M, D), f32)
    L_r, gLr = guarded((R, B, H, M), f32)
    Z, gZ = guarded((B, H, M, D), f32)
    L, gL = guarded((B, H, M), f32)
    ws, gw = _ws(flare.FLARE_OP_ENCODER_FWD, Q, K, off)
    flare.flare_encoder_fwd(Q, K, V, mask, off, O_r=O_r, L_r=L_r, Z=Z, L=L, workspace=ws)
    _check(("O_r", gO), ("L_r", gLr), ("Z", gZ), ("L", gL), ("workspace", gw))
    Zm, gZm = guarded((B, H, M, D), f32)
    Lm, gLm = guarded((B, H, M), f32)
    flare.flare_lse_merge(O_r, L_r, Z=Zm, L=Lm)
    _check(("merge Z", gZm), ("merge L", gLm))
    Y, gY = guarded(tuple(K.shape), K.dtype)
    flare.flare_decode_fwd(Q, Z, K, Y=Y)
    _check(("Y", gY))
    Y2, gY2 = guarded(tuple(K.shape), K.dtype)
    Z2, gZ2 = guarded((B, H, M, D), f32)
    L2, gL2 = guarded((B, H, M), f32)
    ws2, gw2 = _ws(flare.FLARE_OP_FWD, Q, K, off)
    flare.flare_fwd(Q, K, V, mask, off, Y=Y2, Z=Z2, L=L2, workspace=ws2)
    _check(("fwd Y", gY2), ("fwd Z", gZ2), ("fwd L", gL2), ("fwd workspace", gw2))
    # FLARE++: the seeds are the query, the projected tokens the same K, V
    Yp, gYp = guarded(tuple(K.shape), K.dtype)
    Qd, gQd = guarded((B, H, M, D), f32)
    L1, gL1 = guarded((B, H, M), f32)
    Zp, gZp = guarded((B, H, M, D), f32)
    L2p, gL2p = guarded((B, H, M), f32)
    ws3, gw3 = _ws(flare.FLARE_OP_PP_FWD, Q, K, off)
    flare.flare_pp_fwd(Q, K, V, K, V, mask, off, Y=Yp, Qdyn=Qd, L1=L1, Z=Zp, L2=L2p, workspace=ws3)
    _check(("pp Y", gYp), ("pp Qdyn", gQd), ("pp L1", gL1), ("pp Z", gZp), ("pp L2", gL2p),
           ("pp workspace", gw3))


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_backward_entry_points_stay_inside_their_buffers(cuda_device, case):
    Q, K, V, mask, off = _inputs(case, seed=4)
    B, H, M, N, D, dt, _ = case
    f32 = torch.float32
    _, _, Z, L = flare.flare_encoder_fwd(Q, K, V, mask, off)
    g = torch.Generator(device="cuda").manual_seed(9)
    dZ = torch.randn((B, H, M, D), generator=g, device="cuda")
    dY = torch.randn(K.shape, generator=g, device="cuda").to(K.dtype)
    dQ, gdQ = guarded((B, H, M, D), f32)
    dK, gdK = guarded(tuple(K.shape), K.dtype)
    dV, gdV = guarded(tuple(V.shape), V.dtype)
    ws, gw = _ws(flare.FLARE_OP_ENCODER_BWD, Q, K, off)
    flare.flare_encoder_bwd(Q, K, V, mask, off, Z, L, dZ, dQ=dQ, dK=dK, dV=dV, workspace=ws)
    _check(("dQ", gdQ), ("dK", gdK), ("dV", gdV), ("bwd workspace", gw))
    flare.flare_encoder_bwd_accumulate(Q, K, V, mask, off, Z, L, dZ, dQ, dK, dV=dV, workspace=ws)
    _check(("acc dQ", gdQ), ("acc dK", gdK), ("acc dV", gdV), ("acc workspace", gw))
    dQd, gdQd = guarded((B, H, M, D), f32)
    dZd, gdZd = guarded((B, H, M, D), f32)
    dKd, gdKd = guarded(tuple(K.shape), K.dtype)
    n = flare.flare_workspace_bytes(flare.FLARE_OP_DECODE_BWD, flare.make_dims(Q, K))
    wsd, gwd = guarded((max(n, 1),), torch.uint8)
    flare.flare_decode_bwd(Q, Z, K, dY, dQ=dQd, dZ=dZd, dK=dKd, workspace=wsd)
    _check(("dec dQ", gdQd), ("dec dZ", gdZd), ("dec dK", gdKd), ("dec workspace", gwd))
    mQ, gmQ = guarded((B, H, M, D), f32)
    mK, gmK = guarded(tuple(K.shape), K.dtype)
    mV, gmV = guarded(tuple(V.shape), V.dtype)
    wsm, gwm = _ws(flare.FLARE_OP_BWD, Q, K, off)
    flare.flare_bwd(Q, K, V, mask, off, Z, L, dY, dQ=mQ, dK=mK, dV=mV, workspace=wsm)
    _check(("mix dQ", gmQ), ("mix dK", gmK), ("mix dV", gmV), ("mix workspace", gwm))
    _, Qd, L1, Zp, L2 = flare.flare_pp_fwd(Q, K, V, K, V, mask, off)
    outs = [guarded((B, H, M, D), f32), guarded(tuple(K.shape), K.dtype), guarded(tuple(V.shape), V.dtype),
            guarded(tuple(K.shape), K.dtype), guarded(tuple(V.shape), V.dtype), guarded((B, H, M, D), f32)]
    wsp, gwp = _ws(flare.FLARE_OP_PP_BWD, Q, K, off)
    flare.flare_pp_bwd(Q, K, V, K, V, mask, off, Qd, L1, Zp, L2, dY, dQseed=outs[0][0], dKt=outs[1][0],
                       dVt=outs[2][0], dK=outs[3][0], dV=outs[4][0], dQdyn=outs[5][0], workspace=wsp)
    _check(*[(f"pp out {i}", o[1]) for i, o in enumerate(outs)], ("pp workspace", gwp))


def test_empty_problem_writes_only_its_outputs(cuda_device):
    Q, K, V, mask, _ = _inputs((1, 2, 128, 0, 64, "bf16", [0, 0]))
    Z, gZ = guarded((1, 2, 128, 64), torch.float32)
    L, gL = guarded((1, 2, 128), torch.float32)
    flare.flare_encoder_fwd(Q, K, V, None, [0, 0], Z=Z, L=L)
    _check(("Z", gZ), ("L", gL))
    assert torch.isneginf(L).all() and (Z == 0).all()
