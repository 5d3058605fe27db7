"""The allocation-free encoder entry point (flare_encoder_fwd_noalloc).

Some callers cannot allocate device memory (plugins of host frameworks that
own all device memory, code paths where cudaMalloc is not allowed); this entry
point runs the split-KV encoder on the library's static device scratch
instead of a caller workspace. It runs the same kernels in the same fold
order as flare_encoder_fwd, so the two must agree bit for bit. These tests
call it through the C ABI on two calls in a row with different inputs, shard
splits and masks, so a piece of scratch left over from the first call that
the second failed to overwrite (or a merge that read stale partials) shows up
as a mismatch.

This file sorts last on purpose, so a run that stops at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

from latent_query_split_gb300 import flare


def _inputs(seed, B, H, M, N, D, dtype, pad):
    g = torch.Generator().manual_seed(seed)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    Q = (torch.randn((H, M, D), generator=g) * 0.5).to(dt).cuda()
    K = torch.randn((B, N, H, D), generator=g).to(dt).cuda()
    V = torch.randn((B, N, H, D), generator=g).to(dt).cuda()
    mask = (torch.rand((B, N), generator=g) > pad).to(torch.uint8).cuda()
    return Q, K, V, mask


# two calls in a row: other seeds, other shard splits, other padding
CALLS = [(31, [0, 3000, 3000, 9000, 14500, 20000], 0.05),
         (57, [0, 7000, 7100, 12000, 20000], 0.30)]


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,M,D", [("bf16", 128, 64), ("f32", 16, 32)])
def test_noalloc_matches_workspace_entry_point_twice(cuda_device, dtype, M, D):
    B, H, N = 2, 4, 20000
    for seed, off, pad in CALLS:
        Q, K, V, mask = _inputs(seed, B, H, M, N, D, dtype, pad)
        O_w, L_rw, Z_w, L_w = flare.flare_encoder_fwd(Q, K, V, mask, off, shard_outputs=True)
        O_n, L_rn, Z_n, L_n = flare.flare_encoder_fwd_noalloc(Q, K, V, mask, off,
                                                              shard_outputs=True)
        flare.flare_device_status()     # raises if a kernel gave up a bounded wait
        for name, a, b in (("Z", Z_n, Z_w), ("L", L_n, L_w), ("O_r", O_n, O_w),
                           ("L_r", L_rn, L_rw)):
            assert torch.equal(a, b), f"{name} differs from flare_encoder_fwd (seed {seed})"


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_its_scratch(cuda_device):
    lib = flare.load_library()
    # 2^31 token-heads of partials cannot fit in the static scratch. No device
    # pointer is passed: the size check answers first, and were it ever to
    # pass, the argument check would reject the missing inputs before any
    # launch.
    dims = flare.FlareDims(B=64, H=16, M=256, N=1 << 20, D=64, scale=0.0,
                           dtype=flare.FLARE_BF16, q_batch_stride=0, kernel=0)
    arr = (ctypes.c_int64 * 3)(0, 1 << 19, 1 << 20)
    st = lib.flare_encoder_fwd_noalloc(ctypes.byref(dims), None, None, None, None, arr, 2,
                                       None, None, None, None, None)
    assert st == flare.FLARE_ERR_WORKSPACE
    assert b"static scratch" in lib.flare_last_error_string()
