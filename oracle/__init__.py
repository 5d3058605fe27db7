"""fp64 CPU oracle for the FLARE / FLARE++ token mixer -- test infrastructure.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA library:
the arithmetic lives in ``flare_oracle.c`` (plain double-precision loops, each
function citing the passage of "FLARE++: Low-rank attention with dynamic
attention routing", context-parallel appendix, that it writes out), compiled
here with gcc and called through ctypes. This module only marshals arrays.

Every function takes numpy arrays or CPU/CUDA torch tensors. Floating inputs
may be float64, float32 or bfloat16 (torch bf16, or a numpy uint16 array of
bf16 bit patterns); conversion to double is exact. Results are float64 numpy.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(brute force, closed forms, library routines, invariants, finite differences).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "flare_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

T_F64, T_F32, T_BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile flare_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
    os.close(fd)
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)   # serial build
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I, L, Dbl = ctypes.c_int, ctypes.c_long, ctypes.c_double
        lib.oracle_encode.argtypes = [I, I, I, I, I, Dbl, L, P, I, P, P, I, P, L, L,
                                      P, L, P, P]
        lib.oracle_lse_merge.argtypes = [I, L, I, P, P, P, P]
        lib.oracle_decode.argtypes = [I, I, I, I, I, Dbl, L, P, I, P, P, I, P, L, P]
        lib.oracle_encode_bwd.argtypes = [I, I, I, I, I, Dbl, L, P, I, P, P, I, P,
                                          P, P, P, P, P, P]
        lib.oracle_decode_bwd.argtypes = [I, I, I, I, I, Dbl, L, P, I, P, P, I, P, I,
                                          P, P, P]
        lib.oracle_num_threads.restype = I
        _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().oracle_num_threads())


def _as_input(x):
    """Return (contiguous numpy array, element code) without changing values."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), T_BF16
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float64:
        return x, T_F64
    if x.dtype == np.float32:
        return x, T_F32
    if x.dtype == np.uint16:
        return x, T_BF16
    raise TypeError(f"unsupported oracle input dtype {x.dtype}")


def _f64(x):
    a, t = _as_input(x)
    if t == T_BF16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.ascontiguousarray(a, dtype=np.float64)


def _mask(mask):
    if mask is None:
        return None
    try:
        import torch
        if isinstance(mask, torch.Tensor):
            mask = mask.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(mask, dtype=np.uint8)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _query_layout(Q, B, H, M, D):
    if Q.ndim == 3:
        assert Q.shape == (H, M, D), Q.shape
        return 0
    assert Q.shape == (B, H, M, D), Q.shape
    return H * M * D


def encode(Q, K, V, mask=None, scale=None, n_range=None, rows=None):
    """Encoder, eq. 18 (or one shard's O_r, L_r when n_range = (n0, n1)).

    Q [H,M,D] (replicated) or [B,H,M,D]; K, V [B,N,H,D]; mask [B,N] uint8.
    rows: optional flat row indices (b*H+h)*M+m to evaluate (others are NaN).
    Returns Z [B,H,M,D], L [B,H,M] (float64).
    """
    q, qt = _as_input(Q)
    k, kt = _as_input(K)
    v, vt = _as_input(V)
    assert kt == vt, "K and V must share an element type"
    B, N, H, D = k.shape
    M = q.shape[-2]
    qbs = _query_layout(q, B, H, M, D)
    s = 1.0 / math.sqrt(D) if scale is None else float(scale)
    mk = _mask(mask)
    n0, n1 = (0, N) if n_range is None else (int(n_range[0]), int(n_range[1]))
    Z = np.full((B, H, M, D), np.nan)
    L = np.full((B, H, M), np.nan)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    _load().oracle_encode(B, H, M, N, D, s, qbs, _ptr(q), qt, _ptr(k), _ptr(v), kt,
                          _ptr(mk), n0, n1, _ptr(r), 0 if r is None else len(r),
                          _ptr(Z), _ptr(L))
    return Z, L


def encode_shards(Q, K, V, mask, offsets, scale=None):
    """Per-shard encoder outputs (O_r [R,B,H,M,D], L_r [R,B,H,M])."""
    R = len(offsets) - 1
    outs = [encode(Q, K, V, mask, scale, (offsets[r], offsets[r + 1])) for r in range(R)]
    return np.stack([o[0] for o in outs]), np.stack([o[1] for o in outs])


def lse_merge(O_r, L_r):
    """Log-sum-exp merge, eq. 23: O_r [R,...,D], L_r [R,...] -> Z [...,D], L [...]."""
    O = _f64(O_r)
    Lr = _f64(L_r)
    R, D = O.shape[0], O.shape[-1]
    rows = int(np.prod(O.shape[1:-1]))
    Z = np.empty(O.shape[1:])
    L = np.empty(Lr.shape[1:])
    _load().oracle_lse_merge(R, rows, D, _ptr(O), _ptr(Lr), _ptr(Z), _ptr(L))
    return Z, L


def decode(Q, Z, K, scale=None, tokens=None):
    """Local decode: Y_n = softmax_m(s K_n . Q_m) Z over the M latents.

    tokens: optional flat slot indices b*N+n; then Y is [len(tokens), H, D],
    otherwise [B,N,H,D].
    """
    q, qt = _as_input(Q)
    k, kt = _as_input(K)
    z = _f64(Z)
    B, N, H, D = k.shape
    M = q.shape[-2]
    qbs = _query_layout(q, B, H, M, D)
    assert z.shape == (B, H, M, D), z.shape
    s = 1.0 / math.sqrt(D) if scale is None else float(scale)
    t = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    Y = np.empty((B, N, H, D) if t is None else (len(t), H, D))
    _load().oracle_decode(B, H, M, N, D, s, qbs, _ptr(q), qt, _ptr(z), _ptr(k), kt,
                          _ptr(t), 0 if t is None else len(t), _ptr(Y))
    return Y


def flare_fwd(Q, K, V, mask=None, scale=None, tokens=None):
    """FLARE mixer forward: encoder (eq. 18) then the local decode."""
    Z, L = encode(Q, K, V, mask, scale)
    return Z, L, decode(Q, Z, K, scale, tokens)


def flare_pp_fwd(Qseed, Kt, Vt, K, V, mask=None, scale=None, tokens=None):
    """FLARE++ forward: Q(X) = encode(seeds, K~, V~); Z = encode(Q(X), K, V);
    Y = decode with (Q(X), Z). Returns Qdyn, L1, Z, L2, Y."""
    Qd, L1 = encode(Qseed, Kt, Vt, mask, scale)
    Z, L2 = encode(Qd, K, V, mask, scale)
    return Qd, L1, Z, L2, decode(Qd, Z, K, scale, tokens)


def encode_bwd(Q, K, V, mask, Z, L, dZ, scale=None):
    """Global-normaliser encoder backward. Returns dQ [B,H,M,D] (per batch
    element), dK, dV [B,N,H,D]."""
    q, qt = _as_input(Q)
    k, kt = _as_input(K)
    v, vt = _as_input(V)
    assert kt == vt
    B, N, H, D = k.shape
    M = q.shape[-2]
    qbs = _query_layout(q, B, H, M, D)
    s = 1.0 / math.sqrt(D) if scale is None else float(scale)
    z, l, dz = _f64(Z), _f64(L), _f64(dZ)
    mk = _mask(mask)
    dQ = np.empty((B, H, M, D))
    dK = np.empty((B, N, H, D))
    dV = np.empty((B, N, H, D))
    _load().oracle_encode_bwd(B, H, M, N, D, s, qbs, _ptr(q), qt, _ptr(k), _ptr(v), kt,
                              _ptr(mk), _ptr(z), _ptr(l), _ptr(dz), _ptr(dQ), _ptr(dK),
                              _ptr(dV))
    return dQ, dK, dV


def decode_bwd(Q, Z, K, dY, scale=None):
    """Decode backward for the output gradient dY [B,N,H,D]. Returns dQ
    [B,H,M,D] (per batch element), dZ [B,H,M,D] and dK [B,N,H,D]."""
    q, qt = _as_input(Q)
    k, kt = _as_input(K)
    y, yt = _as_input(dY)
    z = _f64(Z)
    B, N, H, D = k.shape
    M = q.shape[-2]
    qbs = _query_layout(q, B, H, M, D)
    assert z.shape == (B, H, M, D) and y.shape == k.shape
    s = 1.0 / math.sqrt(D) if scale is None else float(scale)
    dQ = np.empty((B, H, M, D))
    dZ = np.empty((B, H, M, D))
    dK = np.empty((B, N, H, D))
    _load().oracle_decode_bwd(B, H, M, N, D, s, qbs, _ptr(q), qt, _ptr(z), _ptr(k), kt,
                              _ptr(y), yt, _ptr(dQ), _ptr(dZ), _ptr(dK))
    return dQ, dZ, dK


def flare_bwd(Q, K, V, mask, Z, L, dY, scale=None):
    """FLARE mixer backward (backward paragraphs of the appendix): the
    gradient of the replicated Z is first summed over its consumers -- in the
    mixer only the decode -- and then the encoder is differentiated with the
    forward's global (Z, L). Q is both the encoder's latent query and the
    decode's latent key, K both the encoder's key and the decode's token
    query, so their gradients add. Returns dQ [B,H,M,D] (per batch element),
    dK, dV [B,N,H,D]."""
    dQ_dec, dZ, dK_dec = decode_bwd(Q, Z, K, dY, scale)
    dQ_enc, dK_enc, dV = encode_bwd(Q, K, V, mask, Z, L, dZ, scale)
    return dQ_dec + dQ_enc, dK_dec + dK_enc, dV


def flare_pp_bwd(Qseed, Kt, Vt, K, V, mask, Qdyn, L1, Z, L2, dY, scale=None):
    """FLARE++ mixer backward (FLARE++ backward paragraph of the appendix):
    the decode with Q(X) gives its shares of dQ(X), dZ and dK; the
    physical-value encoder (saved Z, L2) adds its shares of dQ(X) and dK and
    gives dV; the summed dQ(X) is the output gradient of the query-synthesis
    encoder, differentiated with its own saved output Q(X) and L1. Returns
    dQseed [B,H,M,D] (per batch element), dKt, dVt, dK, dV, dQdyn."""
    dQX_dec, dZ, dK_dec = decode_bwd(Qdyn, Z, K, dY, scale)
    dQX_enc, dK_enc, dV = encode_bwd(Qdyn, K, V, mask, Z, L2, dZ, scale)
    dQX = dQX_dec + dQX_enc
    dQs, dKt, dVt = encode_bwd(Qseed, Kt, Vt, mask, Qdyn, L1, dQX, scale)
    return dQs, dKt, dVt, dK_dec + dK_enc, dV, dQX
