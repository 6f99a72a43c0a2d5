"""ORACLE: test infrastructure, not part of the library.

Python access to the fp64 C oracle in ``oracle.c`` (a plain m/n/k loop over
bf16 inputs decoded exactly, from "How I made Muse's GPU projections 1.32×
faster in the Open Kernel Challenge", section "The full equation, now with the
letters explained").  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  It never imports the CUDA library
and the CUDA library never imports it.

All array arguments are numpy uint16 bf16 bit patterns; results are float64.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import tempfile
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = None

W_NK, W_KN = 0, 1


def lib_path() -> str:
    # ORACLE_LIB lets the mutation test load a deliberately broken build.
    return os.environ.get("ORACLE_LIB") or os.path.join(
        _HERE, f"_oracle.{platform.machine()}.so")


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, OpenMP, no fast-math) next to this file."""
    out = lib_path()
    if os.environ.get("ORACLE_LIB"):
        return out
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    # -ffp-contract=off: each product and each sum is its own rounded fp64 op,
    # exactly as the loop is written (no fused multiply-add reassociation).
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(build())
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_project.argtypes = [i64, i64, i64, vp, vp, ctypes.c_int, vp, vp]
        lib.oracle_project.restype = None
        lib.oracle_project_cells.argtypes = [i64, i64, i64, vp, vp, ctypes.c_int, vp,
                                             i64, vp, vp, vp]
        lib.oracle_project_cells.restype = None
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_split_hilo.argtypes = [i64, vp, vp, vp]
        lib.oracle_split_hilo.restype = None
        lib.oracle_project_f32w.argtypes = [i64, i64, i64, vp, vp, ctypes.c_int, vp, vp]
        lib.oracle_project_f32w.restype = None
        lib.oracle_gelu.argtypes = [ctypes.c_double]
        lib.oracle_gelu.restype = ctypes.c_double
        lib.oracle_apply_activation.argtypes = [i64, ctypes.c_int, vp]
        lib.oracle_apply_activation.restype = None
        lib.oracle_silu.argtypes = [ctypes.c_double]
        lib.oracle_silu.restype = ctypes.c_double
        lib.oracle_swiglu.argtypes = [i64, vp, vp, vp]
        lib.oracle_swiglu.restype = None
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        _LIB = lib
    return _LIB


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return a


def _shapes(X, W, w_layout):
    M, K = X.shape
    if w_layout == W_NK:
        N, K2 = W.shape
    elif w_layout == W_KN:
        K2, N = W.shape
    else:
        raise ValueError("w_layout must be 0 ([N,K]) or 1 ([K,N])")
    if K2 != K:
        raise ValueError(f"K mismatch: X has {K}, W has {K2}")
    return M, N, K


def bf16_to_double(bits) -> np.ndarray:
    """Decode bf16 bit patterns one by one through the oracle's own decoder."""
    lib = _lib()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_bf16_to_double(int(b)) for b in flat],
                    dtype=np.float64).reshape(np.shape(bits))


def project(X, W, w_layout: int = W_NK, bias=None) -> np.ndarray:
    """fp64 ``Y[m,n] = Σ_k X[m,k]·W(n,k) (+ bias[n])`` for the whole problem."""
    X, W = _u16(X), _u16(W)
    M, N, K = _shapes(X, W, w_layout)
    b = None if bias is None else _u16(bias)
    if b is not None and b.shape != (N,):
        raise ValueError("bias must have shape [N]")
    Y = np.empty((M, N), dtype=np.float64)
    if M and N:
        _lib().oracle_project(M, N, K, X.ctypes.data, W.ctypes.data, int(w_layout),
                              None if b is None else b.ctypes.data, Y.ctypes.data)
    return Y


def project_cells(X, W, w_layout: int, bias, ms, ns) -> np.ndarray:
    """fp64 output cells at coordinates ``(ms[i], ns[i])``."""
    X, W = _u16(X), _u16(W)
    M, N, K = _shapes(X, W, w_layout)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    if ms.shape != ns.shape or ms.ndim != 1:
        raise ValueError("ms and ns must be equal-length 1-D arrays")
    if ms.size and (ms.min() < 0 or ms.max() >= M or ns.min() < 0 or ns.max() >= N):
        raise IndexError("cell coordinate out of range")
    b = None if bias is None else _u16(bias)
    out = np.empty(ms.size, dtype=np.float64)
    if ms.size:
        _lib().oracle_project_cells(M, N, K, X.ctypes.data, W.ctypes.data,
                                    int(w_layout), None if b is None else b.ctypes.data,
                                    ms.size, ms.ctypes.data, ns.ctypes.data,
                                    out.ctypes.data)
    return out


def f32_to_bf16(values) -> np.ndarray:
    """bf16 bit patterns of fp32 values, through the oracle's own rounding (RNE)."""
    lib = _lib()
    flat = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib.oracle_f32_to_bf16(float(v)) for v in flat],
                    dtype=np.uint16).reshape(np.shape(values))


def split_hilo(W) -> tuple:
    """The router's high and low bf16 parts of fp32 weights (any shape):
    H = roundBF16(W), L = roundBF16(W − FP32(H)), as uint16 bit patterns."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    H = np.empty(W.shape, dtype=np.uint16)
    L = np.empty(W.shape, dtype=np.uint16)
    if W.size:
        _lib().oracle_split_hilo(W.size, W.ctypes.data, H.ctypes.data, L.ctypes.data)
    return H, L


def project_f32w(X, W, w_layout: int = W_NK, bias=None) -> np.ndarray:
    """fp64 ``Y = X·Wᵀ (+ bias)`` with fp32 weights ``W`` (the router's reference)."""
    X = _u16(X)
    W = np.ascontiguousarray(W, dtype=np.float32)
    M, K = X.shape
    if w_layout == W_NK:
        N, K2 = W.shape
    else:
        K2, N = W.shape
    if K2 != K:
        raise ValueError(f"K mismatch: X has {K}, W has {K2}")
    b = None if bias is None else _u16(bias)
    Y = np.empty((M, N), dtype=np.float64)
    if M and N:
        _lib().oracle_project_f32w(M, N, K, X.ctypes.data, W.ctypes.data, int(w_layout),
                                   None if b is None else b.ctypes.data, Y.ctypes.data)
    return Y


def project_hilo(X, W, w_layout: int = W_NK, bias=None) -> np.ndarray:
    """The router method itself in fp64: X·Hᵀ + X·Lᵀ (+ bias)."""
    H, L = split_hilo(W)
    return project(X, H, w_layout, bias) + project(X, L, w_layout, None)


ACT_NONE, ACT_GELU, ACT_SWIGLU = 0, 1, 2


def gelu(x) -> np.ndarray:
    """GELU(x) = x/2 · (1 + erf(x/√2)) of fp64 values, one by one."""
    lib = _lib()
    flat = np.asarray(x, dtype=np.float64).ravel()
    return np.array([lib.oracle_gelu(float(v)) for v in flat]).reshape(np.shape(x))


def project_fused(X, W, w_layout: int = W_NK, bias=None, act: int = ACT_NONE,
                  residual=None) -> np.ndarray:
    """The fused epilogue: act(X·Wᵀ + bias) + residual, all in fp64.  ``residual``
    is [M,N] fp64 (the decoded residual input) or None."""
    Y = np.ascontiguousarray(project(X, W, w_layout, bias))
    if act not in (ACT_NONE, ACT_GELU):
        raise ValueError("act must be ACT_NONE or ACT_GELU")
    if Y.size:
        _lib().oracle_apply_activation(Y.size, int(act), Y.ctypes.data)
    if residual is not None:
        Y = Y + np.asarray(residual, dtype=np.float64)
    return Y


def silu(x) -> np.ndarray:
    """SiLU(x) = x·σ(x) of fp64 values, one by one."""
    lib = _lib()
    flat = np.asarray(x, dtype=np.float64).ravel()
    return np.array([lib.oracle_silu(float(v)) for v in flat]).reshape(np.shape(x))


def project_swiglu(X, W, w_layout: int = W_NK, residual=None) -> np.ndarray:
    """SwiGLU of the stacked projection: W holds the gate rows then the up rows
    ([2F,K] for W_NK, [K,2F] for W_KN); Y[m,f] = SiLU(G[m,f])·U[m,f] (+ residual),
    with G = X·W_gateᵀ and U = X·W_upᵀ in fp64."""
    GU = np.ascontiguousarray(project(X, W, w_layout, None))
    M, N2 = GU.shape
    if N2 % 2:
        raise ValueError("SwiGLU weights stack 2F rows")
    F = N2 // 2
    G = np.ascontiguousarray(GU[:, :F])
    U = np.ascontiguousarray(GU[:, F:])
    Y = np.empty((M, F), dtype=np.float64)
    if Y.size:
        _lib().oracle_swiglu(Y.size, G.ctypes.data, U.ctypes.data, Y.ctypes.data)
    if residual is not None:
        Y = Y + np.asarray(residual, dtype=np.float64)
    return Y


def max_threads() -> int:
    return int(_lib().oracle_max_threads())


def set_threads(n: int) -> None:
    _lib().oracle_set_threads(int(n))
