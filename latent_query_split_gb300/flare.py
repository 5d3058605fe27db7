"""Python binding of the C ABI in include/flare.h (ctypes; marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it derives the size struct from tensor shapes, takes
device pointers from torch tensors, allocates outputs and workspaces with
torch when the caller passes none, and raises FlareError on a non-zero
status. torch provides device memory and streams; every step of the mixer
runs in the library's CUDA kernels. There is no CPU fallback: without the
compiled library (or without a GPU) these calls fail.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import build as _build

FLARE_OK, FLARE_ERR_INVALID_ARG, FLARE_ERR_UNSUPPORTED = 0, 1, 2
FLARE_ERR_WORKSPACE, FLARE_ERR_CUDA, FLARE_ERR_TIMEOUT = 3, 4, 5
FLARE_ERR_DEVICE_CHECK = 6
FLARE_F32, FLARE_BF16 = 0, 1
KERNELS = {"auto": 0, "simt": 1, "tensor": 2}
(FLARE_OP_ENCODER_FWD, FLARE_OP_LSE_MERGE, FLARE_OP_DECODE_FWD, FLARE_OP_FWD,
 FLARE_OP_PP_FWD, FLARE_OP_ENCODER_BWD, FLARE_OP_DECODE_BWD, FLARE_OP_BWD,
 FLARE_OP_PP_BWD) = range(9)
FLARE_MAX_SHARDS = 256

# Every symbol the header declares (checked by the test-suite).
EXPORTS = ("flare_workspace_bytes", "flare_encoder_fwd", "flare_lse_merge", "flare_decode_fwd",
           "flare_fwd", "flare_pp_fwd", "flare_encoder_bwd", "flare_decode_bwd",
           "flare_bwd", "flare_pp_bwd", "flare_encoder_fwd_noalloc",
           "flare_encoder_bwd_accumulate", "flare_check_bounded_wait",
           "flare_device_status", "flare_last_error_string", "flare_version",
           "flare_launch_count")


class FlareError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"flare status {status}: {message}")
        self.status = status


class FlareDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("M", ctypes.c_int),
                ("N", ctypes.c_int), ("D", ctypes.c_int), ("scale", ctypes.c_float),
                ("dtype", ctypes.c_int), ("q_batch_stride", ctypes.c_int64),
                ("kernel", ctypes.c_int)]


_lib = None


def _debug_variant() -> bool:
    """FLARE_LIBRARY_VARIANT=debug selects the checking build (FLARE_DEBUG)."""
    return os.environ.get("FLARE_LIBRARY_VARIANT", "release") == "debug"


def library_path() -> str:
    return _build.lib_path(_debug_variant())


def load_library(build_if_missing: bool = True):
    """Load libflare.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    debug = _debug_variant()
    path = _build.lib_path(debug)
    if build_if_missing and not _build.up_to_date(debug):
        _build.build(debug=debug)
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run latent_query_split_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    D = ctypes.POINTER(FlareDims)
    lib.flare_workspace_bytes.argtypes = [I, D, P, I]
    lib.flare_workspace_bytes.restype = Z
    lib.flare_encoder_fwd.argtypes = [D, P, P, P, P, P, I, P, P, P, P, P, Z, P]
    lib.flare_lse_merge.argtypes = [P, P, I, I, I, I, I, P, P, P]
    lib.flare_decode_fwd.argtypes = [D, P, P, P, P, P]
    lib.flare_fwd.argtypes = [D, P, P, P, P, P, I, P, P, P, P, Z, P]
    lib.flare_pp_fwd.argtypes = [D, P, P, P, P, P, P, P, I, P, P, P, P, P, P, Z, P]
    lib.flare_encoder_bwd.argtypes = [D, P, P, P, P, P, I, P, P, P, P, P, P, P, Z, P]
    lib.flare_encoder_bwd_accumulate.argtypes = [D, P, P, P, P, P, I, P, P, P, P, P, P, P, Z, P]
    lib.flare_decode_bwd.argtypes = [D, P, P, P, P, P, P, P, P, Z, P]
    lib.flare_bwd.argtypes = [D, P, P, P, P, P, I, P, P, P, P, P, P, P, Z, P]
    lib.flare_pp_bwd.argtypes = [D, P, P, P, P, P, P, P, I, P, P, P, P, P, P, P, P, P, P, P, P, Z, P]
    lib.flare_encoder_fwd_noalloc.argtypes = [D, P, P, P, P, P, I, P, P, P, P, P]
    lib.flare_check_bounded_wait.argtypes = [ctypes.c_uint, P]
    lib.flare_device_status.argtypes = [P]
    lib.flare_last_error_string.restype = ctypes.c_char_p
    lib.flare_version.restype = I
    lib.flare_launch_count.restype = ctypes.c_ulonglong
    _lib = lib
    return lib


def _check(status: int):
    if status != FLARE_OK:
        msg = load_library().flare_last_error_string().decode(errors="replace")
        raise FlareError(status, msg)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _offsets(shard_offsets: Sequence[int]):
    arr = (ctypes.c_int64 * len(shard_offsets))(*[int(x) for x in shard_offsets])
    return arr, len(shard_offsets) - 1


def make_dims(Q: torch.Tensor, K: torch.Tensor, scale: Optional[float] = None,
              kernel: str = "auto") -> FlareDims:
    """Size struct for a query Q ([H,M,D] or [B,H,M,D]) and tokens K [B,N,H,D]."""
    B, N, H, D = K.shape
    M = Q.shape[-2]
    if K.dtype == torch.bfloat16:
        dt = FLARE_BF16
    elif K.dtype == torch.float32:
        dt = FLARE_F32
    else:
        raise TypeError(f"unsupported token dtype {K.dtype}")
    qbs = 0 if Q.dim() == 3 else H * M * D
    return FlareDims(B, H, M, N, D, 0.0 if scale is None else float(scale), dt, qbs,
                     KERNELS[kernel])


def flare_version() -> int:
    return load_library().flare_version()


def flare_workspace_bytes(op: int, dims: FlareDims, shard_offsets=None) -> int:
    lib = load_library()
    if shard_offsets is None:
        n = lib.flare_workspace_bytes(op, ctypes.byref(dims), None, 0)
    else:
        arr, R = _offsets(shard_offsets)
        n = lib.flare_workspace_bytes(op, ctypes.byref(dims), arr, R)
    if n == ctypes.c_size_t(-1).value:
        _check(FLARE_ERR_INVALID_ARG)
    return int(n)


def _workspace(op, dims, shard_offsets, workspace, device):
    need = flare_workspace_bytes(op, dims, shard_offsets)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def flare_encoder_fwd(Q, K, V, mask=None, shard_offsets=None, *, O_r=None, L_r=None, Z=None,
                      L=None, shard_outputs=False, global_outputs=True, workspace=None,
                      scale=None, kernel="auto", stream=None):
    """Split-KV encoder; returns (O_r, L_r, Z, L) with None for pairs not requested."""
    lib = load_library()
    dims = make_dims(Q, K, scale, kernel)
    B, N, H, D = K.shape
    M = Q.shape[-2]
    shard_offsets = [0, N] if shard_offsets is None else list(shard_offsets)
    R = len(shard_offsets) - 1
    f32 = dict(dtype=torch.float32, device=K.device)
    if shard_outputs and O_r is None:
        O_r, L_r = torch.empty((R, B, H, M, D), **f32), torch.empty((R, B, H, M), **f32)
    if global_outputs and Z is None:
        Z, L = torch.empty((B, H, M, D), **f32), torch.empty((B, H, M), **f32)
    ws, nbytes = _workspace(FLARE_OP_ENCODER_FWD, dims, shard_offsets, workspace, K.device)
    arr, R = _offsets(shard_offsets)
    _check(lib.flare_encoder_fwd(ctypes.byref(dims), _ptr(Q), _ptr(K), _ptr(V), _ptr(mask), arr, R,
                                 _ptr(O_r), _ptr(L_r), _ptr(Z), _ptr(L), _ptr(ws), nbytes,
                                 _stream(stream)))
    return O_r, L_r, Z, L


def flare_lse_merge(O_r, L_r, *, Z=None, L=None, stream=None):
    """Log-sum-exp merge of per-shard results O_r [R,B,H,M,D], L_r [R,B,H,M]."""
    lib = load_library()
    R, B, H, M, D = O_r.shape
    if Z is None:
        Z = torch.empty((B, H, M, D), dtype=torch.float32, device=O_r.device)
        L = torch.empty((B, H, M), dtype=torch.float32, device=O_r.device)
    _check(lib.flare_lse_merge(_ptr(O_r), _ptr(L_r), R, B, H, M, D, _ptr(Z), _ptr(L),
                               _stream(stream)))
    return Z, L


def flare_decode_fwd(Q, Z, K, *, Y=None, scale=None, kernel="auto", stream=None):
    """Local decode of every token slot; returns Y [B,N,H,D] (dtype of K)."""
    lib = load_library()
    dims = make_dims(Q, K, scale, kernel)
    if Y is None:
        Y = torch.empty_like(K)
    _check(lib.flare_decode_fwd(ctypes.byref(dims), _ptr(Q), _ptr(Z), _ptr(K), _ptr(Y),
                                _stream(stream)))
    return Y


def flare_fwd(Q, K, V, mask=None, shard_offsets=None, *, Y=None, Z=None, L=None, workspace=None,
              scale=None, kernel="auto", stream=None):
    """FLARE forward (encoder + fused merge + decode); returns (Y, Z, L)."""
    lib = load_library()
    dims = make_dims(Q, K, scale, kernel)
    B, N, H, D = K.shape
    M = Q.shape[-2]
    shard_offsets = [0, N] if shard_offsets is None else list(shard_offsets)
    if Y is None:
        Y = torch.empty_like(K)
    if Z is None:
        Z = torch.empty((B, H, M, D), dtype=torch.float32, device=K.device)
        L = torch.empty((B, H, M), dtype=torch.float32, device=K.device)
    ws, nbytes = _workspace(FLARE_OP_FWD, dims, shard_offsets, workspace, K.device)
    arr, R = _offsets(shard_offsets)
    _check(lib.flare_fwd(ctypes.byref(dims), _ptr(Q), _ptr(K), _ptr(V), _ptr(mask), arr, R,
                         _ptr(Y), _ptr(Z), _ptr(L), _ptr(ws), nbytes, _stream(stream)))
    return Y, Z, L


def flare_pp_fwd(Qseed, Kt, Vt, K, V, mask=None, shard_offsets=None, *, Y=None, Qdyn=None,
                 L1=None, Z=None, L2=None, workspace=None, scale=None, kernel="auto",
                 stream=None):
    """FLARE++ forward; returns (Y, Qdyn, L1, Z, L2)."""
    lib = load_library()
    dims = make_dims(Qseed, K, scale, kernel)
    B, N, H, D = K.shape
    M = Qseed.shape[-2]
    shard_offsets = [0, N] if shard_offsets is None else list(shard_offsets)
    f32 = dict(dtype=torch.float32, device=K.device)
    if Y is None:
        Y = torch.empty_like(K)
    if Qdyn is None:
        Qdyn, L1 = torch.empty((B, H, M, D), **f32), torch.empty((B, H, M), **f32)
    if Z is None:
        Z, L2 = torch.empty((B, H, M, D), **f32), torch.empty((B, H, M), **f32)
    ws, nbytes = _workspace(FLARE_OP_PP_FWD, dims, shard_offsets, workspace, K.device)
    arr, R = _offsets(shard_offsets)
    _check(lib.flare_pp_fwd(ctypes.byref(dims), _ptr(Qseed), _ptr(Kt), _ptr(Vt), _ptr(K), _ptr(V),
                            _ptr(mask), arr, R, _ptr(Y), _ptr(Qdyn), _ptr(L1), _ptr(Z), _ptr(L2),
                            _ptr(ws), nbytes, _stream(stream)))
    return Y, Qdyn, L1, Z, L2


def flare_encoder_bwd(Q, K, V, mask, shard_offsets, Z, L, dZ, *, dQ=None, dK=None, dV=None,
                      workspace=None, scale=None, kernel="auto", stream=None):
    """Global-normaliser encoder backward; returns (dQ [B,H,M,D] fp32, dK, dV)."""
    lib = load_library()
    dims = make_dims(Q, K, scale, kernel)
    B, N, H, D = K.shape
    M = Q.shape[-2]
    shard_offsets = [0, N] if shard_offsets is None else list(shard_offsets)
    if dQ is None:
        dQ = torch.empty((B, H, M, D), dtype=torch.float32, device=K.device)
    if dK is None:
        dK, dV = torch.empty_like(K), torch.empty_like(V)
    ws, nbytes = _workspace(FLARE_OP_ENCODER_BWD, dims, shard_offsets, workspace, K.device)
    arr, R = _offsets(shard_offsets)
    _check(lib.flare_encoder_bwd(ctypes.byref(dims), _ptr(Q), _ptr(K), _ptr(V), _ptr(mask), arr,
                                 R, _ptr(Z), _ptr(L), _ptr(dZ), _ptr(dQ), _ptr(dK), _ptr(dV),
                                 _ptr(ws), nbytes, _stream(stream)))
    return dQ, dK, dV


def flare_encoder_bwd_accumulate(Q, K, V, mask, shard_offsets, Z, L, dZ, dQ, dK, *, dV=None,
                                 workspace=None, scale=None, kernel="auto", stream=None):
    """Encoder backward adding its shares to the given dQ (fp32) and dK (K's
    dtype), which hold another consumer's shares; dV is written. Returns
    (dQ, dK, dV)."""
    lib = load_library()
    dims = make_dims(Q, K, scale, kernel)
    N = K.shape[1]
    shard_offsets = [0, N] if shard_offsets is None else list(shard_offsets)
    if dV is None:
        dV = torch.empty_like(V)
    ws, nbytes = _workspace(FLARE_OP_ENCODER_BWD, dims, shard_offsets, workspace, K.device)
    arr, R = _offsets(shard_offsets)
    _check(lib.flare_encoder_bwd_accumulate(ctypes.byref(dims), _ptr(Q), _ptr(K), _ptr(V),
                                            _ptr(mask), arr, R, _ptr(Z), _ptr(L), _ptr(dZ),
                                            _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws), nbytes,
                                            _stream(stream)))
    return dQ, dK, dV


def flare_decode_bwd(Q, Z, K, dY, *, dQ=None, dZ=None, dK=None, workspace=None, scale=None,
                     kernel="auto", stream=None):
    """Decode backward for the output gradient dY; returns (dQ [B,H,M,D] fp32,
    dZ [B,H,M,D] fp32, dK [B,N,H,D] in K's dtype)."""
    lib = load_library()
    dims = make_dims(Q, K, scale, kernel)
    B, N, H, D = K.shape
    M = Q.shape[-2]
    f32 = dict(dtype=torch.float32, device=K.device)
    if dQ is None:
        dQ = torch.empty((B, H, M, D), **f32)
    if dZ is None:
        dZ = torch.empty((B, H, M, D), **f32)
    if dK is None:
        dK = torch.empty_like(K)
    ws, nbytes = _workspace(FLARE_OP_DECODE_BWD, dims, None, workspace, K.device)
    _check(lib.flare_decode_bwd(ctypes.byref(dims), _ptr(Q), _ptr(Z), _ptr(K), _ptr(dY), _ptr(dQ),
                                _ptr(dZ), _ptr(dK), _ptr(ws), nbytes, _stream(stream)))
    return dQ, dZ, dK


def flare_bwd(Q, K, V, mask, shard_offsets, Z, L, dY, *, dQ=None, dK=None, dV=None,
              workspace=None, scale=None, kernel="auto", stream=None):
    """FLARE mixer backward from the forward's (Z, L) and the output gradient
    dY; returns (dQ [B,H,M,D] fp32, dK, dV in K's dtype)."""
    lib = load_library()
    dims = make_dims(Q, K, scale, kernel)
    B, N, H, D = K.shape
    M = Q.shape[-2]
    shard_offsets = [0, N] if shard_offsets is None else list(shard_offsets)
    if dQ is None:
        dQ = torch.empty((B, H, M, D), dtype=torch.float32, device=K.device)
    if dK is None:
        dK, dV = torch.empty_like(K), torch.empty_like(V)
    ws, nbytes = _workspace(FLARE_OP_BWD, dims, shard_offsets, workspace, K.device)
    arr, R = _offsets(shard_offsets)
    _check(lib.flare_bwd(ctypes.byref(dims), _ptr(Q), _ptr(K), _ptr(V), _ptr(mask), arr, R,
                         _ptr(Z), _ptr(L), _ptr(dY), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws),
                         nbytes, _stream(stream)))
    return dQ, dK, dV


def flare_pp_bwd(Qseed, Kt, Vt, K, V, mask, shard_offsets, Qdyn, L1, Z, L2, dY, *, dQseed=None,
                 dKt=None, dVt=None, dK=None, dV=None, dQdyn=None, want_dQdyn=False,
                 workspace=None, scale=None, kernel="auto", stream=None):
    """FLARE++ mixer backward from the forward's (Qdyn, L1, Z, L2) and dY;
    returns (dQseed [B,H,M,D] fp32, dKt, dVt, dK, dV, dQdyn or None)."""
    lib = load_library()
    dims = make_dims(Qseed, K, scale, kernel)
    B, N, H, D = K.shape
    M = Qseed.shape[-2]
    shard_offsets = [0, N] if shard_offsets is None else list(shard_offsets)
    f32 = dict(dtype=torch.float32, device=K.device)
    if dQseed is None:
        dQseed = torch.empty((B, H, M, D), **f32)
    if dKt is None:
        dKt, dVt = torch.empty_like(Kt), torch.empty_like(Vt)
    if dK is None:
        dK, dV = torch.empty_like(K), torch.empty_like(V)
    if dQdyn is None and want_dQdyn:
        dQdyn = torch.empty((B, H, M, D), **f32)
    ws, nbytes = _workspace(FLARE_OP_PP_BWD, dims, shard_offsets, workspace, K.device)
    arr, R = _offsets(shard_offsets)
    _check(lib.flare_pp_bwd(ctypes.byref(dims), _ptr(Qseed), _ptr(Kt), _ptr(Vt), _ptr(K), _ptr(V),
                            _ptr(mask), arr, R, _ptr(Qdyn), _ptr(L1), _ptr(Z), _ptr(L2), _ptr(dY),
                            _ptr(dQseed), _ptr(dKt), _ptr(dVt), _ptr(dK), _ptr(dV), _ptr(dQdyn),
                            _ptr(ws), nbytes, _stream(stream)))
    return dQseed, dKt, dVt, dK, dV, dQdyn


def flare_encoder_fwd_noalloc(Q, K, V, mask=None, shard_offsets=None, *, O_r=None, L_r=None,
                              Z=None, L=None, shard_outputs=False, global_outputs=True,
                              scale=None, kernel="auto", stream=None):
    """flare_encoder_fwd without a workspace: the library's static device
    scratch is used instead (see include/flare.h for its size and rules).
    Returns (O_r, L_r, Z, L) with None for pairs not requested."""
    lib = load_library()
    dims = make_dims(Q, K, scale, kernel)
    B, N, H, D = K.shape
    M = Q.shape[-2]
    shard_offsets = [0, N] if shard_offsets is None else list(shard_offsets)
    R = len(shard_offsets) - 1
    f32 = dict(dtype=torch.float32, device=K.device)
    if shard_outputs and O_r is None:
        O_r, L_r = torch.empty((R, B, H, M, D), **f32), torch.empty((R, B, H, M), **f32)
    if global_outputs and Z is None:
        Z, L = torch.empty((B, H, M, D), **f32), torch.empty((B, H, M), **f32)
    arr, R = _offsets(shard_offsets)
    _check(lib.flare_encoder_fwd_noalloc(ctypes.byref(dims), _ptr(Q), _ptr(K), _ptr(V), _ptr(mask),
                                         arr, R, _ptr(O_r), _ptr(L_r), _ptr(Z), _ptr(L),
                                         _stream(stream)))
    return O_r, L_r, Z, L


def flare_check_bounded_wait(limit_us: int, stream=None):
    """Launch the bounded-wait check kernel (see include/flare.h): it gives
    up a wait that never completes after limit_us and records
    FLARE_ERR_TIMEOUT for flare_device_status."""
    _check(load_library().flare_check_bounded_wait(int(limit_us), _stream(stream)))


def flare_device_status(stream=None):
    """Synchronise the stream and raise FlareError if a kernel gave up a bounded wait."""
    _check(load_library().flare_device_status(_stream(stream)))


def flare_launch_count() -> int:
    """Kernels the library has launched in this process (see include/flare.h)."""
    return int(load_library().flare_launch_count())
