"""The C-ABI library builds, loads and exports every declared entry point; host-side
argument validation rejects bad calls before anything reaches a GPU (CPU only)."""
import ctypes
import os
import re

import pytest
import torch

from latent_query_split_gb300 import build, flare

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "flare.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FLARE_API\s+[\w\s\*]+?\b(flare_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return flare.load_library()


def test_header_declares_the_binding_exports():
    assert _declared() == sorted(flare.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert lib.flare_version() >= 10000


def test_dims_struct_layout_matches_header():
    # int B,H,M,N,D; float scale; enum dtype; int64 q_batch_stride; enum kernel
    assert ctypes.sizeof(flare.FlareDims) == 48
    assert flare.FlareDims.q_batch_stride.offset == 32


def _dims(**kw):
    d = dict(B=1, H=2, M=16, N=100, D=32, scale=0.0, dtype=flare.FLARE_F32, q_batch_stride=0,
             kernel=0)
    d.update(kw)
    return flare.FlareDims(**d)


def _ws(lib, dims, offs):
    arr = (ctypes.c_int64 * len(offs))(*offs)
    return lib.flare_workspace_bytes(flare.FLARE_OP_ENCODER_FWD, ctypes.byref(dims), arr,
                                     len(offs) - 1)


BAD = ctypes.c_size_t(-1).value


def test_workspace_query_validates(lib):
    assert _ws(lib, _dims(), [0, 50, 100]) > 0
    assert _ws(lib, _dims(), [0, 50, 99]) == BAD          # offsets[R] != N
    assert _ws(lib, _dims(), [1, 50, 100]) == BAD         # offsets[0] != 0
    assert _ws(lib, _dims(), [0, 60, 50, 100]) == BAD     # decreasing
    assert _ws(lib, _dims(D=129), [0, 100]) == BAD        # D > 128
    assert _ws(lib, _dims(M=0), [0, 100]) == BAD
    assert _ws(lib, _dims(q_batch_stride=7), [0, 100]) == BAD
    assert lib.flare_workspace_bytes(flare.FLARE_OP_DECODE_FWD, ctypes.byref(_dims()), None, 0) == 0
    # empty shards are fine; the workspace does not depend on the stream or pointers
    assert _ws(lib, _dims(), [0, 0, 100, 100]) > 0


def _enc(lib, dims, offs, Z=1 << 20, L=1 << 21, ws=1 << 22, wsb=1 << 30, Or=None, Lr=None):
    arr = (ctypes.c_int64 * len(offs))(*offs)
    # fake, aligned non-null device addresses: validation fails before any use
    return lib.flare_encoder_fwd(ctypes.byref(dims), 1 << 12, 1 << 13, 1 << 14, None, arr,
                                 len(offs) - 1, Or, Lr, Z, L, ws, wsb, None)


def test_encoder_rejects_bad_arguments_before_launch(lib):
    assert _enc(lib, _dims(), [0, 40, 99]) == flare.FLARE_ERR_INVALID_ARG
    assert b"shard_offsets" in lib.flare_last_error_string()
    assert _enc(lib, _dims(), [0, 100], Z=None, L=None) == flare.FLARE_ERR_INVALID_ARG
    assert _enc(lib, _dims(), [0, 100], L=None) == flare.FLARE_ERR_INVALID_ARG
    assert _enc(lib, _dims(), [0, 100], Or=1 << 15) == flare.FLARE_ERR_INVALID_ARG
    assert _enc(lib, _dims(D=200), [0, 100]) == flare.FLARE_ERR_UNSUPPORTED
    assert _enc(lib, _dims(dtype=7), [0, 100]) == flare.FLARE_ERR_INVALID_ARG
    assert _enc(lib, _dims(), [0] * 258 + [100]) == flare.FLARE_ERR_INVALID_ARG   # R > 256


def test_tensor_kernel_request_for_fp32_is_unsupported(lib):
    assert _enc(lib, _dims(kernel=2), [0, 100]) == flare.FLARE_ERR_UNSUPPORTED


def test_merge_rejects_bad_sizes(lib):
    assert lib.flare_lse_merge(1 << 12, 1 << 13, 0, 1, 1, 1, 1, 1 << 14, 1 << 15, None) == \
        flare.FLARE_ERR_INVALID_ARG


def test_binding_refuses_host_tensors(lib):
    with pytest.raises(ValueError):
        flare._ptr(torch.zeros(3))


# The composite calls check the arguments of every stage before the first
# launch: a bad argument of a later stage is reported as such, with nothing
# launched (here, without a GPU, a launch attempt would fail as FLARE_ERR_CUDA).
_A = [1 << (12 + i) for i in range(24)]      # fake, aligned, distinct device addresses


def _bigws(lib, op, dims, offs):
    arr = (ctypes.c_int64 * len(offs))(*offs) if offs is not None else None
    n = lib.flare_workspace_bytes(op, ctypes.byref(dims), arr, len(offs) - 1 if offs else 0)
    assert n != BAD
    return 1 << 40, max(n, 1)


def _offs(offs):
    return (ctypes.c_int64 * len(offs))(*offs)


@pytest.mark.parametrize("dtype", [flare.FLARE_F32, flare.FLARE_BF16])
def test_flare_fwd_checks_the_decode_before_launching(lib, dtype):
    d = _dims(dtype=dtype, M=64, D=64, N=256)
    offs = [0, 100, 256]
    ws, nb = _bigws(lib, flare.FLARE_OP_FWD, d, offs)
    before = lib.flare_launch_count()
    s = lib.flare_fwd(ctypes.byref(d), _A[0], _A[1], _A[2], None, _offs(offs), 2,
                      None, _A[3], _A[4], ws, nb, None)       # Y missing
    assert s == flare.FLARE_ERR_INVALID_ARG
    assert b"NULL" in lib.flare_last_error_string()
    assert lib.flare_launch_count() == before


@pytest.mark.parametrize("dtype", [flare.FLARE_F32, flare.FLARE_BF16])
def test_flare_pp_fwd_checks_every_stage_before_launching(lib, dtype):
    d = _dims(dtype=dtype, M=64, D=64, N=256)
    offs = [0, 100, 256]
    ws, nb = _bigws(lib, flare.FLARE_OP_PP_FWD, d, offs)
    before = lib.flare_launch_count()
    # K missing: the first encoder (over K~, V~) is fine, the second is not
    s = lib.flare_pp_fwd(ctypes.byref(d), _A[0], _A[1], _A[2], None, _A[3], None, _offs(offs), 2,
                         _A[4], _A[5], _A[6], _A[7], _A[8], ws, nb, None)
    assert s == flare.FLARE_ERR_INVALID_ARG
    # Y missing: only the decode stage sees it
    s = lib.flare_pp_fwd(ctypes.byref(d), _A[0], _A[1], _A[2], _A[9], _A[3], None, _offs(offs), 2,
                         None, _A[5], _A[6], _A[7], _A[8], ws, nb, None)
    assert s == flare.FLARE_ERR_INVALID_ARG
    assert lib.flare_launch_count() == before


@pytest.mark.parametrize("dtype", [flare.FLARE_F32, flare.FLARE_BF16])
def test_flare_bwd_checks_the_encoder_stage_before_launching(lib, dtype):
    d = _dims(dtype=dtype, M=64, D=64, N=256)
    offs = [0, 100, 256]
    ws, nb = _bigws(lib, flare.FLARE_OP_BWD, d, offs)
    before = lib.flare_launch_count()
    # dV missing: the decode backward (first stage) needs no V or dV
    s = lib.flare_bwd(ctypes.byref(d), _A[0], _A[1], _A[2], None, _offs(offs), 2, _A[3], _A[4],
                      _A[5], _A[6], _A[7], None, ws, nb, None)
    assert s == flare.FLARE_ERR_INVALID_ARG
    # a workspace that is too small is reported before anything runs
    s = lib.flare_bwd(ctypes.byref(d), _A[0], _A[1], _A[2], None, _offs(offs), 2, _A[3], _A[4],
                      _A[5], _A[6], _A[7], _A[8], ws, 1024, None)
    assert s == flare.FLARE_ERR_WORKSPACE
    assert lib.flare_launch_count() == before


@pytest.mark.parametrize("dtype", [flare.FLARE_F32, flare.FLARE_BF16])
def test_flare_pp_bwd_checks_every_stage_before_launching(lib, dtype):
    d = _dims(dtype=dtype, M=64, D=64, N=256)
    offs = [0, 100, 256]
    ws, nb = _bigws(lib, flare.FLARE_OP_PP_BWD, d, offs)
    before = lib.flare_launch_count()

    def call(dKt=_A[15], dV=_A[18], Vt=_A[2]):
        return lib.flare_pp_bwd(ctypes.byref(d), _A[0], _A[1], Vt, _A[3], _A[4], None, _offs(offs), 2,
                                _A[5], _A[6], _A[7], _A[8], _A[9], _A[10], dKt, _A[16], _A[17], dV,
                                None, ws, nb, None)
    assert call(dV=None) == flare.FLARE_ERR_INVALID_ARG     # second stage
    assert call(dKt=None) == flare.FLARE_ERR_INVALID_ARG    # third stage
    assert call(Vt=None) == flare.FLARE_ERR_INVALID_ARG     # third stage's input
    assert lib.flare_launch_count() == before


def test_bounded_wait_check_rejects_limits_out_of_range(lib):
    for limit in (0, 1000001):
        assert lib.flare_check_bounded_wait(limit, None) == flare.FLARE_ERR_INVALID_ARG
        assert b"limit_us" in lib.flare_last_error_string()


def test_accumulating_encoder_bwd_validates_before_launch(lib):
    dims = _dims()
    arr = (ctypes.c_int64 * 3)(0, 50, 100)
    # NULL tensors are rejected before anything is launched
    assert lib.flare_encoder_bwd_accumulate(ctypes.byref(dims), None, None, None, None, arr, 2,
                                            None, None, None, None, None, None, None, 0,
                                            None) == flare.FLARE_ERR_INVALID_ARG
    bad = (ctypes.c_int64 * 3)(0, 50, 99)
    assert lib.flare_encoder_bwd_accumulate(ctypes.byref(dims), None, None, None, None, bad, 2,
                                            None, None, None, None, None, None, None, 0,
                                            None) == flare.FLARE_ERR_INVALID_ARG


def test_backward_workspaces_cover_the_tensor_core_layouts(lib):
    """The tensor-core backward workspaces hold what their passes use: the
    bf16 copy of Z (or dZ) with all D columns, one dQ (and dZ) piece array per
    64-column half of D, and at M = 256 the decode backward's per-token
    statistics, 8 bytes per (b, h, token)."""
    B, H, N = 2, 4, 5000

    def ws(op, M, D, kernel=2):
        d = _dims(B=B, H=H, M=M, N=N, D=D, dtype=flare.FLARE_BF16, kernel=kernel)
        offs = (ctypes.c_int64 * 2)(0, N)     # the encoder backward takes the shard split
        return lib.flare_workspace_bytes(op, ctypes.byref(d), offs, 1)

    dec, enc = flare.FLARE_OP_DECODE_BWD, flare.FLARE_OP_ENCODER_BWD
    for op in (dec, enc):
        for M, D in ((64, 64), (128, 64), (256, 64), (64, 128), (128, 128)):
            assert 0 < ws(op, M, D) != BAD, (op, M, D)
        # two column halves: twice the pieces and twice Z's (dZ's) bf16 copy
        # (the encoder's per-row constants, 8 bytes per latent row, do not
        # grow with D)
        slack = 8 * B * H * 128 + 4096
        assert ws(op, 64, 128) >= 2 * ws(op, 64, 64) - slack
        assert ws(op, 128, 128) >= 2 * ws(op, 128, 64) - slack
    assert ws(dec, 256, 64) >= 2 * ws(dec, 128, 64) + 8 * B * H * N - 4096
    assert ws(enc, 256, 64) >= 2 * ws(enc, 128, 64) - 4096
