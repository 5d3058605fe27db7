"""The allocation-free encoder entry point (flare_encoder_fwd_noalloc).

Some callers cannot allocate device memory (plugins of host frameworks that
own all device memory, code paths where cudaMalloc is not allowed); this entry
point runs the split-KV encoder on the library's static device scratch
instead of a caller workspace. These tests call it through the C ABI and
compare it with flare_encoder_fwd (which takes a workspace) on two calls in a
row, since every call reuses the same static scratch.

This file sorts last on purpose, so a run that stops at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

from latent_query_split_gb300 import flare
from parity import assert_L_close, assert_close


def _inputs(seed, B, H, M, N, D, dtype, off):
    g = torch.Generator().manual_seed(seed)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    Q = (torch.randn((H, M, D), generator=g) * 0.5).to(dt).cuda()
    K = torch.randn((B, N, H, D), generator=g).to(dt).cuda()
    V = torch.randn((B, N, H, D), generator=g).to(dt).cuda()
    mask = (torch.rand((B, N), generator=g) > 0.05).to(torch.uint8).cuda()
    return Q, K, V, mask


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,M,D", [("bf16", 128, 64), ("f32", 16, 32)])
def test_noalloc_matches_workspace_entry_point_twice(cuda_device, dtype, M, D):
    B, H, N = 2, 4, 20000
    off = [0, 3000, 3000, 9000, 14500, N]
    Q, K, V, mask = _inputs(31, B, H, M, N, D, dtype, off)
    O_w, L_rw, Z_w, L_w = flare.flare_encoder_fwd(Q, K, V, mask, off, shard_outputs=True)
    for _ in range(2):     # the static scratch keeps the previous call's contents
        O_n, L_rn, Z_n, L_n = flare.flare_encoder_fwd_noalloc(Q, K, V, mask, off,
                                                              shard_outputs=True)
        flare.flare_device_status()
        assert_close("Z", Z_n, Z_w, dtype)
        assert_L_close("L", L_n, L_w)
        assert_close("O_r", O_n, O_w, dtype)
        assert_L_close("L_r", L_rn, L_rw)


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_its_scratch(cuda_device):
    lib = flare.load_library()
    # 2^31 token-heads of partials cannot fit in the static scratch
    dims = flare.FlareDims(B=64, H=16, M=256, N=1 << 20, D=64, scale=0.0,
                           dtype=flare.FLARE_BF16, q_batch_stride=0, kernel=0)
    arr = (ctypes.c_int64 * 3)(0, 1 << 19, 1 << 20)
    st = lib.flare_encoder_fwd_noalloc(ctypes.byref(dims), 1 << 12, 1 << 13, 1 << 14, None, arr, 2,
                                       None, None, 1 << 15, 1 << 16, None)
    assert st == flare.FLARE_ERR_WORKSPACE
    assert b"static scratch" in lib.flare_last_error_string()
