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
