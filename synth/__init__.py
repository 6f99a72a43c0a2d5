"""Seeded synthetic inputs for the dense projection ``Y = X·Wᵀ (+ bias)``.

This module draws the test and benchmark operands and nothing else: it holds no
step of the projection itself (no products, no sums, no output rounding).  Both
the fp64 oracle and the CUDA path are fed from here, so that neither needs the
other.

Workload shapes follow the decode/prefill projection family of "How I made
Muse's GPU projections 1.32× faster in the Open Kernel Challenge"
(bishal.us worklog, section "The same calculation shows up in different sizes":
K = 8,192 input features, thousands of outputs, a few to a few hundred token
rows, bf16 weights).  The model's real weights and activations are not used;
every value below is synthetic.

Generator
---------
* Uniform bits: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014), in its counter form:
  output ``j`` of a stream seeded with ``s`` is ``mix(s + (j+1)·γ)`` with
  ``γ = 0x9E3779B97F4A7C15`` and ``mix`` the published 64-bit finaliser
  (xor-shift 30, ×0xBF58476D1CE4E5B9, xor-shift 27, ×0x94D049BB133111EB,
  xor-shift 31).
* Uniform doubles on (0, 1]: ``((bits >> 11) + 1) · 2⁻⁵³``.
* Normal deviates: Box–Muller.  Element ``j`` uses the uniform pair
  ``(u₁, u₂) = (U[2⌊j/2⌋], U[2⌊j/2⌋+1])`` and takes
  ``√(−2 ln u₁)·cos(2πu₂)`` for even ``j`` and ``…·sin(2πu₂)`` for odd ``j``,
  so any element can be drawn on its own (sampled checks need this).
* Storage: the double is rounded to fp32 (round-to-nearest-even) and the fp32
  to bf16 (round-to-nearest-even on the upper 16 bits).  This double rounding
  is part of how inputs are *made*, not part of the method under test.
* Streams: X, W and the bias each draw from their own stream, whose seed is
  ``mix(seed·256 + t)`` with ``t`` = 1 (X), 2 (W), 3 (bias).  W is drawn in its
  *storage* order (``[N,K]`` or ``[K,N]``); because the draws are iid this is
  the same distribution as drawing ``[N,K]`` and transposing.  Separate streams
  keep W identical across the token-count sweep, where only M changes.
"""
from __future__ import annotations

import ctypes
import math
import os
import platform
import subprocess
import tempfile
from dataclasses import dataclass
from typing import Optional

import numpy as np

__all__ = [
    "GAMMA", "mix64", "splitmix64", "uniform01", "normal", "to_bf16_bits",
    "normal_bf16", "normal_bf16_numpy", "sample_normal_bf16", "build",
    "Workload", "WORKLOADS", "FFN_SWEEP_M", "workload", "make_inputs",
]

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # elements per vectorised block (keeps temporaries ~100 MB)

STREAM_X, STREAM_W, STREAM_BIAS = 1, 2, 3


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output finaliser on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_seed(seed: int, tensor: int) -> np.uint64:
    """Seed of the per-tensor stream: ``mix(seed·256 + tensor)``."""
    base = np.uint64((int(seed) * 256 + int(tensor)) & 0xFFFFFFFFFFFFFFFF)
    return mix64(np.array([base], dtype=np.uint64))[0]


def splitmix64(s: np.uint64, idx: np.ndarray) -> np.ndarray:
    """Outputs ``idx`` (0-based) of the SplitMix64 stream seeded with ``s``."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(s) + (idx + np.uint64(1)) * GAMMA
    return mix64(state)


def uniform01(s: np.uint64, idx: np.ndarray) -> np.ndarray:
    """Uniform doubles on (0, 1] from outputs ``idx`` of stream ``s``."""
    bits = splitmix64(s, idx) >> np.uint64(11)
    return (bits.astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(s: np.uint64, idx: np.ndarray) -> np.ndarray:
    """Standard normal deviates for element indices ``idx`` of stream ``s``."""
    idx = np.asarray(idx, dtype=np.uint64)
    pair = (idx >> np.uint64(1)) << np.uint64(1)
    u1 = uniform01(s, pair)
    u2 = uniform01(s, pair + np.uint64(1))
    r = np.sqrt(-2.0 * np.log(u1))
    theta = 2.0 * math.pi * u2
    odd = (idx & np.uint64(1)).astype(bool)
    return np.where(odd, r * np.sin(theta), r * np.cos(theta))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round doubles to fp32 then to bf16 (both round-to-nearest-even).

    Returns the bf16 bit patterns as uint16.  Inputs here are finite, so the
    NaN/Inf special cases of the rounding never arise.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def normal_bf16_numpy(seed: int, tensor: int, count: int, std: float,
                      first: int = 0) -> np.ndarray:
    """Elements ``first … first+count-1`` of one tensor stream, in numpy."""
    s = stream_seed(seed, tensor)
    out = np.empty(count, dtype=np.uint16)
    for lo in range(0, count, _CHUNK):
        hi = min(count, lo + _CHUNK)
        idx = np.arange(first + lo, first + hi, dtype=np.uint64)
        out[lo:hi] = to_bf16_bits(normal(s, idx) * std)
    return out


_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = None


def lib_path() -> str:
    return os.path.join(_HERE, f"_synth.{platform.machine()}.so")


def build(force: bool = False) -> str:
    """Compile synth.c with gcc (OpenMP) next to this file; return the path."""
    out = lib_path()
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)  # atomic: concurrent builders never see a partial file
    return out


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(build())
        lib.synth_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_double, ctypes.c_void_p]
        lib.synth_normal_bf16.restype = None
        lib.synth_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_double, ctypes.c_void_p]
        lib.synth_normal_f32.restype = None
        lib.synth_stream_seed.argtypes = [ctypes.c_uint64, ctypes.c_int]
        lib.synth_stream_seed.restype = ctypes.c_uint64
        _LIB = lib
    return _LIB


def normal_bf16(seed: int, tensor: int, count: int, std: float,
                first: int = 0) -> np.ndarray:
    """``count`` bf16 bit patterns of N(0, std²) from one tensor stream (C)."""
    out = np.empty(count, dtype=np.uint16)
    if count:
        _lib().synth_normal_bf16(int(seed), int(tensor), int(first), int(count),
                                 float(std), out.ctypes.data)
    return out


def normal_f32(seed: int, tensor: int, count: int, std: float, first: int = 0) -> np.ndarray:
    """``count`` fp32 values of N(0, std²) from one tensor stream (C): the same
    normals as :func:`normal_bf16`, rounded to fp32 instead of bf16."""
    out = np.empty(count, dtype=np.float32)
    if count:
        _lib().synth_normal_f32(int(seed), int(tensor), int(first), int(count),
                                float(std), out.ctypes.data)
    return out


def sample_normal_bf16(seed: int, tensor: int, idx: np.ndarray, std: float) -> np.ndarray:
    """The same values as :func:`normal_bf16` at flat storage indices ``idx``."""
    s = stream_seed(seed, tensor)
    return to_bf16_bits(normal(s, np.asarray(idx, dtype=np.uint64)) * std)


W_NK, W_KN = 0, 1  # weight storage: [N,K] (K contiguous) or [K,N] (N contiguous)


@dataclass(frozen=True)
class Workload:
    """One projection problem: shapes, layouts, dtypes and the seed."""
    name: str
    M: int
    N: int
    K: int
    w_layout: int = W_NK
    has_bias: bool = False
    y_dtype: str = "bf16"  # "bf16" or "f32"
    seed: int = 0
    x_std: float = 1.0
    bias_std: float = 0.02
    w_dtype: str = "bf16"  # "bf16", or "f32" (router weights: the high/low bf16 split)

    @property
    def w_std(self) -> float:
        # W ~ N(0, 1/K): variance 1/K, so each output has unit variance.
        return 1.0 / math.sqrt(self.K)

    def with_m(self, M: int) -> "Workload":
        return Workload(self.name, M, self.N, self.K, self.w_layout, self.has_bias,
                        self.y_dtype, self.seed, self.x_std, self.bias_std, self.w_dtype)

    # ---- byte / flop accounting (the pages' roofline model: F = 2MNK) ----
    @property
    def weight_bytes(self) -> int:
        # fp32 router weights stream as two bf16 parts: 4 bytes a weight either way.
        return (4 if self.w_dtype == "f32" else 2) * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        yb = 4 if self.y_dtype == "f32" else 2
        return (self.weight_bytes + 2 * self.M * self.K
                + (2 * self.N if self.has_bias else 0) + yb * self.M * self.N)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# The five workloads this library is measured and checked on.
WORKLOADS = {
    "decode_f32out": Workload("decode_f32out", 16, 2048, 8192, W_NK, False, "f32", 0),
    "decode_bias": Workload("decode_bias", 16, 8192, 8192, W_NK, True, "bf16", 1),
    "ffn_up_sweep": Workload("ffn_up_sweep", 16, 28672, 8192, W_NK, False, "bf16", 2),
    "qkv_kn_bias": Workload("qkv_kn_bias", 256, 12288, 4096, W_KN, True, "bf16", 3),
    "prefill": Workload("prefill", 4096, 8192, 8192, W_NK, False, "bf16", 4),
    # The worklog's fp32-weight router (N = 256, K = 8192) through the high/low
    # bf16 split, fp32 output; a §8(f) extension, not one of the five configs.
    "router_f32w": Workload("router_f32w", 16, 256, 8192, W_NK, False, "f32", 5, w_dtype="f32"),
}
FFN_SWEEP_M = (1, 2, 4, 8, 16, 32, 64)


def workload(name: str, M: Optional[int] = None) -> Workload:
    w = WORKLOADS[name]
    return w if M is None else w.with_m(M)


def make_inputs(w: Workload) -> dict:
    """Draw X ``[M,K]``, W in storage order and (optionally) the bias.

    All arrays are uint16 bf16 bit patterns, except W of an fp32-weight
    workload (float32); W is ``[N,K]`` for ``W_NK`` and ``[K,N]`` for ``W_KN``.
    """
    X = normal_bf16(w.seed, STREAM_X, w.M * w.K, w.x_std).reshape(w.M, w.K)
    gen = normal_f32 if w.w_dtype == "f32" else normal_bf16
    Wf = gen(w.seed, STREAM_W, w.N * w.K, w.w_std)
    Wm = Wf.reshape(w.N, w.K) if w.w_layout == W_NK else Wf.reshape(w.K, w.N)
    b = normal_bf16(w.seed, STREAM_BIAS, w.N, w.bias_std) if w.has_bias else None
    return {"X": X, "W": Wm, "bias": b}
