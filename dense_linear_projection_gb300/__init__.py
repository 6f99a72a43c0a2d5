"""GB300-native dense projection ``Y = X·Wᵀ (+ bias)``: Python binding.

A thin ctypes layer over the C ABI in ``include/proj.h`` (libproj_gb300): the
functions here carry the same names and only marshal arguments.  Every step of
the projection runs in the library's sm_103a kernels.  There is no fallback: if
the library is missing or cannot load, every call raises.

``Projection`` is a convenience wrapper that takes PyTorch tensors (PyTorch only
provides device memory and streams) and returns ``Y``.
"""
from __future__ import annotations

import ctypes
import json
import os
from typing import Optional

from ._build import build, library_path

__all__ = [
    "PROJ_OK", "PROJ_ERR_INVALID_ARG", "PROJ_ERR_UNSUPPORTED", "PROJ_ERR_MISALIGNED",
    "PROJ_ERR_OUT_OF_MEMORY", "PROJ_ERR_CUDA", "PROJ_ERR_DEVICE_TIMEOUT",
    "PROJ_BF16", "PROJ_F32", "PROJ_W_NK", "PROJ_W_KN",
    "PROJ_KERNEL_NONE", "PROJ_KERNEL_FILL", "PROJ_KERNEL_TC",
    "ProjError", "lib", "build", "library_path", "EXPORTED_SYMBOLS",
    "proj_plan_compute", "proj_plan_segments", "proj_plan_reduction_order", "proj_create",
    "proj_run", "proj_run_host", "proj_device_status",
    "proj_get_plan", "proj_plan_info", "proj_destroy", "proj_status_string",
    "proj_selftest_wait_timeout", "proj_set_trace", "proj_set_overlap", "TRACE_FIELDS",
    "PROJ_OVERLAP_NONE", "PROJ_OVERLAP_PROLOGUE", "PROJ_OVERLAP_WEIGHTS", "proj_run_noalloc",
    "proj_noalloc_device_status", "proj_noalloc_selftest_wait_timeout",
    "proj_packed_weight_bytes", "proj_pack_weights", "proj_run_packed", "proj_run_host_packed",
    "proj_set_activation", "proj_run_fused", "PROJ_ACT_NONE", "PROJ_ACT_GELU", "PROJ_ACT_SWIGLU",
    "Projection",
]

PROJ_OK, PROJ_ERR_INVALID_ARG, PROJ_ERR_UNSUPPORTED, PROJ_ERR_MISALIGNED = 0, 1, 2, 3
PROJ_ERR_OUT_OF_MEMORY, PROJ_ERR_CUDA, PROJ_ERR_DEVICE_TIMEOUT = 4, 5, 6
PROJ_BF16, PROJ_F32 = 0, 1
PROJ_W_NK, PROJ_W_KN = 0, 1
PROJ_KERNEL_NONE, PROJ_KERNEL_FILL, PROJ_KERNEL_TC = 0, 1, 2
PROJ_OVERLAP_NONE, PROJ_OVERLAP_PROLOGUE, PROJ_OVERLAP_WEIGHTS = 0, 1, 2
PROJ_ACT_NONE, PROJ_ACT_GELU, PROJ_ACT_SWIGLU = 0, 1, 2

EXPORTED_SYMBOLS = (
    "proj_plan_compute", "proj_plan_segments", "proj_plan_reduction_order", "proj_create", "proj_run", "proj_run_host", "proj_device_status",
    "proj_get_plan", "proj_plan_info", "proj_destroy", "proj_status_string",
    "proj_selftest_wait_timeout", "proj_set_trace", "proj_set_overlap", "proj_run_noalloc",
    "proj_packed_weight_bytes", "proj_pack_weights", "proj_run_packed", "proj_run_host_packed",
    "proj_set_activation", "proj_run_fused", "proj_noalloc_device_status",
    "proj_noalloc_selftest_wait_timeout",
)


class ProjError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {proj_status_string(status)} ({status})")


class DeviceDesc(ctypes.Structure):
    _fields_ = [("sm_count", ctypes.c_int32), ("smem_optin_bytes", ctypes.c_int32)]


class PlanDesc(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in (
        "kernel", "block_n", "block_t", "block_k", "stages", "grid", "threads", "smem_bytes",
        "tmem_cols", "raster_group", "swap_ab", "cluster_split", "cta_pair")] + [(name, ctypes.c_int64) for name in (
        "tiles_m", "tiles_n", "k_blocks", "tiles_dp", "tiles_sk", "units_sk", "scratch_bytes")] + [
        ("cluster_groups", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class Segment(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in (
        "tile", "tile_m", "tile_n", "k_block_begin", "k_block_end", "slot", "split", "reserved")]

    def as_tuple(self):
        return (self.tile, self.tile_m, self.tile_n, self.k_block_begin, self.k_block_end,
                self.slot, self.split)


def _plan_struct(plan: dict) -> PlanDesc:
    p = PlanDesc()
    for name, _ in PlanDesc._fields_:
        setattr(p, name, int(plan.get(name, 0)))
    return p


_LIB = None


def lib() -> ctypes.CDLL:
    """Load libproj_gb300 (building it first if the sources are newer)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        path = build()
    L = ctypes.CDLL(path)
    i64, i32, vp, st = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_int
    L.proj_plan_compute.argtypes = [i64, i64, i64, i32, i32, i32, ctypes.POINTER(DeviceDesc),
                                    ctypes.POINTER(PlanDesc)]
    L.proj_plan_segments.argtypes = [ctypes.POINTER(PlanDesc), ctypes.c_int32,
                                     ctypes.POINTER(Segment), i64, ctypes.POINTER(i64)]
    L.proj_plan_reduction_order.argtypes = [ctypes.POINTER(PlanDesc), i64,
                                            ctypes.POINTER(ctypes.c_int32),
                                            ctypes.POINTER(ctypes.c_int32), i64, ctypes.POINTER(i64)]
    L.proj_create.argtypes = [ctypes.POINTER(vp), i64, i64, i64, i32, i32, i32, i32, i32, i32, vp]
    L.proj_run.argtypes = [vp, vp, vp, vp, vp, vp]
    L.proj_run_host.argtypes = [vp, vp, vp, vp, vp, vp]
    L.proj_device_status.argtypes = [vp, vp]
    L.proj_get_plan.argtypes = [vp, ctypes.POINTER(PlanDesc)]
    L.proj_plan_info.argtypes = [vp, ctypes.c_char_p, ctypes.c_size_t]
    L.proj_destroy.argtypes = [vp]
    L.proj_status_string.argtypes = [st]
    L.proj_status_string.restype = ctypes.c_char_p
    L.proj_selftest_wait_timeout.argtypes = [i64, vp]
    L.proj_set_trace.argtypes = [vp, vp, ctypes.c_size_t]
    L.proj_set_overlap.argtypes = [vp, i32]
    L.proj_run_noalloc.argtypes = [i64, i64, i64, i32, i32, vp, vp, vp, vp, vp]
    L.proj_noalloc_device_status.argtypes = [vp]
    L.proj_noalloc_selftest_wait_timeout.argtypes = [i64, vp]
    L.proj_packed_weight_bytes.argtypes = [vp, ctypes.POINTER(ctypes.c_size_t)]
    L.proj_pack_weights.argtypes = [vp, vp, vp, vp]
    L.proj_run_packed.argtypes = [vp, vp, vp, vp, vp, vp]
    L.proj_run_host_packed.argtypes = [vp, vp, vp, vp, vp, vp]
    L.proj_set_activation.argtypes = [vp, i32]
    L.proj_run_fused.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp]
    for name in EXPORTED_SYMBOLS:
        if name != "proj_status_string":
            getattr(L, name).restype = st
    _LIB = L
    return L


def _check(status: int, what: str) -> int:
    if status != PROJ_OK:
        raise ProjError(status, what)
    return status


def _ptr(x) -> Optional[int]:
    """Device/host address of a tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)  # torch.cuda.Stream


# ---------------------------------------------------------------- the C ABI
def proj_status_string(status: int) -> str:
    return lib().proj_status_string(int(status)).decode()


def proj_plan_compute(M: int, N: int, K: int, w_layout: int = PROJ_W_NK,
                      y_dtype: int = PROJ_BF16, has_bias: bool = False,
                      sm_count: int = 152, smem_optin_bytes: int = 232448) -> dict:
    dev = DeviceDesc(sm_count, smem_optin_bytes)
    out = PlanDesc()
    _check(lib().proj_plan_compute(M, N, K, w_layout, y_dtype, int(bool(has_bias)),
                                   ctypes.byref(dev), ctypes.byref(out)), "proj_plan_compute")
    return out.as_dict()


def proj_plan_segments(plan: dict, cta: int) -> list:
    """Segments (tile, tile_m, tile_n, kb_begin, kb_end, slot, split) of one CTA."""
    p = _plan_struct(plan)
    n = ctypes.c_int64()
    _check(lib().proj_plan_segments(ctypes.byref(p), cta, None, 0, ctypes.byref(n)),
           "proj_plan_segments")
    buf = (Segment * max(1, n.value))()
    _check(lib().proj_plan_segments(ctypes.byref(p), cta, buf, n.value, ctypes.byref(n)),
           "proj_plan_segments")
    return [buf[i].as_tuple() for i in range(n.value)]


def proj_plan_reduction_order(plan: dict, split_tile: int) -> list:
    """[(cta, slot), ...] in the order split tile `split_tile`'s partials are added."""
    p = _plan_struct(plan)
    n = ctypes.c_int64()
    _check(lib().proj_plan_reduction_order(ctypes.byref(p), split_tile, None, None, 0,
                                           ctypes.byref(n)), "proj_plan_reduction_order")
    cap = max(1, n.value)
    ctas = (ctypes.c_int32 * cap)()
    slots = (ctypes.c_int32 * cap)()
    _check(lib().proj_plan_reduction_order(ctypes.byref(p), split_tile, ctas, slots, n.value,
                                           ctypes.byref(n)), "proj_plan_reduction_order")
    return [(ctas[i], slots[i]) for i in range(n.value)]


def proj_create(M: int, N: int, K: int, w_layout: int = PROJ_W_NK, x_dtype: int = PROJ_BF16,
                w_dtype: int = PROJ_BF16, y_dtype: int = PROJ_BF16, has_bias: bool = False,
                bias_dtype: int = PROJ_BF16, stream=None) -> int:
    h = ctypes.c_void_p()
    _check(lib().proj_create(ctypes.byref(h), M, N, K, w_layout, x_dtype, w_dtype, y_dtype,
                             int(bool(has_bias)), bias_dtype, _stream(stream)), "proj_create")
    return h.value


def proj_run(h: int, X, W, bias, Y, stream=None) -> None:
    _check(lib().proj_run(h, _ptr(X), _ptr(W), _ptr(bias), _ptr(Y), _stream(stream)), "proj_run")


def proj_run_host(h: int, X_host, W, bias, Y_host, stream=None) -> None:
    _check(lib().proj_run_host(h, _ptr(X_host), _ptr(W), _ptr(bias), _ptr(Y_host),
                               _stream(stream)), "proj_run_host")


def proj_run_noalloc(M: int, N: int, K: int, w_layout: int, y_dtype: int, X, W, bias, Y,
                     stream=None) -> None:
    """proj_run without a handle or any allocation (fixed 8 MiB device scratch).

    For callers that cannot allocate device memory.  The first call on a device
    looks up the scratch address; calls that overlap on the GPU race.  A device
    wait that gave up is reported later, by proj_noalloc_device_status.
    """
    _check(lib().proj_run_noalloc(M, N, K, w_layout, y_dtype, _ptr(X), _ptr(W), _ptr(bias),
                                  _ptr(Y), _stream(stream)), "proj_run_noalloc")


def proj_noalloc_device_status(stream=None) -> int:
    """Raw status of the allocation-free path's status word (read and
    cleared; synchronises the stream); does not raise."""
    return int(lib().proj_noalloc_device_status(_stream(stream)))


def proj_noalloc_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Queue a bounded wait that gives up and records a timeout in the
    allocation-free path's status word."""
    _check(lib().proj_noalloc_selftest_wait_timeout(int(limit_ns), _stream(stream)),
           "proj_noalloc_selftest_wait_timeout")


def proj_packed_weight_bytes(h: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().proj_packed_weight_bytes(h, ctypes.byref(out)), "proj_packed_weight_bytes")
    return int(out.value)


def proj_pack_weights(h: int, W, W_packed, stream=None) -> None:
    _check(lib().proj_pack_weights(h, _ptr(W), _ptr(W_packed), _stream(stream)), "proj_pack_weights")


def proj_run_packed(h: int, X, W_packed, bias, Y, stream=None) -> None:
    _check(lib().proj_run_packed(h, _ptr(X), _ptr(W_packed), _ptr(bias), _ptr(Y), _stream(stream)),
           "proj_run_packed")


def proj_run_host_packed(h: int, X_host, W_packed, bias, Y_host, stream=None) -> None:
    _check(lib().proj_run_host_packed(h, _ptr(X_host), _ptr(W_packed), _ptr(bias), _ptr(Y_host),
                                      _stream(stream)), "proj_run_host_packed")


def proj_set_activation(h: int, act: int) -> None:
    _check(lib().proj_set_activation(h, int(act)), "proj_set_activation")


def proj_run_fused(h: int, X, W, packed: bool, bias, residual, Y, stream=None) -> None:
    _check(lib().proj_run_fused(h, _ptr(X), _ptr(W), int(bool(packed)), _ptr(bias), _ptr(residual),
                                _ptr(Y), _stream(stream)), "proj_run_fused")


def proj_device_status(h: int, stream=None) -> int:
    """Raw status (PROJ_OK or an error code); does not raise."""
    return int(lib().proj_device_status(h, _stream(stream)))


def proj_get_plan(h: int) -> dict:
    out = PlanDesc()
    _check(lib().proj_get_plan(h, ctypes.byref(out)), "proj_get_plan")
    return out.as_dict()


def proj_plan_info(h: int) -> dict:
    buf = ctypes.create_string_buffer(2048)
    _check(lib().proj_plan_info(h, buf, len(buf)), "proj_plan_info")
    return json.loads(buf.value.decode())


def proj_destroy(h: Optional[int]) -> None:
    _check(lib().proj_destroy(h), "proj_destroy")


def proj_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    """Raw status; PROJ_ERR_DEVICE_TIMEOUT means the bounded wait gave up as designed."""
    return int(lib().proj_selftest_wait_timeout(int(limit_ns), _stream(stream)))


TRACE_FIELDS = ("entry", "setup", "first_load", "last_load", "first_data", "last_mma",
                "first_acc", "epilogue_done", "teardown", "smid", "reductions", "dep_wait",
                "epi_dep_wait", "split_partial", "split_ready", "split_stored")


def proj_set_overlap(h: int, mode: int) -> None:
    """Overlap with the preceding kernel: PROJ_OVERLAP_NONE / _PROLOGUE / _WEIGHTS."""
    _check(lib().proj_set_overlap(h, int(mode)), "proj_set_overlap")


def proj_set_trace(h: int, buf=None, nbytes: int = 0) -> None:
    """Point the handle's phase trace at a device buffer (None turns it off)."""
    _check(lib().proj_set_trace(h, _ptr(buf), int(nbytes)), "proj_set_trace")


# ---------------------------------------------------------------- convenience
class Projection:
    """A planned projection for one shape; call it with PyTorch tensors.

    ``X``: [M,K] bf16 CUDA tensor; ``W``: [N,K] (``PROJ_W_NK``) or [K,N]
    (``PROJ_W_KN``) bf16; ``bias``: [N] bf16 or None.  Returns ``Y`` [M,N] in
    ``y_dtype`` (allocated with torch unless ``out`` is given).
    """

    def __init__(self, M: int, N: int, K: int, w_layout: int = PROJ_W_NK,
                 y_dtype: int = PROJ_BF16, has_bias: bool = False, stream=None,
                 overlap: Optional[int] = None, w_dtype: int = PROJ_BF16):
        import torch  # noqa: F401  (PyTorch provides memory and streams only)
        self.M, self.N, self.K = M, N, K
        self.w_layout, self.y_dtype, self.has_bias = w_layout, y_dtype, bool(has_bias)
        self.w_dtype = w_dtype
        self.act = PROJ_ACT_NONE
        self.handle = proj_create(M, N, K, w_layout, PROJ_BF16, w_dtype, y_dtype, has_bias,
                                  PROJ_BF16, stream)
        if overlap is not None:
            proj_set_overlap(self.handle, overlap)

    @property
    def plan(self) -> dict:
        return proj_plan_info(self.handle)

    def __call__(self, X, W, bias=None, out=None, stream=None, packed: bool = False, residual=None):
        """Y = act(X·Wᵀ + bias) + residual; ``packed=True`` takes weights from
        :meth:`pack`; the activation is set by :meth:`set_activation`."""
        import torch
        if out is None:
            dt = torch.float32 if self.y_dtype == PROJ_F32 else torch.bfloat16
            n_out = self.N // 2 if self.act == PROJ_ACT_SWIGLU else self.N
            out = torch.empty((self.M, n_out), dtype=dt, device=X.device)
        if stream is None:
            stream = torch.cuda.current_stream(X.device)
        if residual is not None:
            proj_run_fused(self.handle, X, W, packed, bias, residual, out, stream)
        else:
            (proj_run_packed if packed else proj_run)(self.handle, X, W, bias, out, stream)
        return out

    def set_activation(self, act: int) -> None:
        """PROJ_ACT_NONE, PROJ_ACT_GELU, or PROJ_ACT_SWIGLU (set it before
        :meth:`pack`; the output then has N / 2 columns)."""
        proj_set_activation(self.handle, act)
        self.act = act

    def pack(self, W, stream=None):
        """Repack weights into this handle's tile-contiguous layout (a preparation
        step; fp32 weights of a ``w_dtype=PROJ_F32`` handle are split into high
        and low bf16 parts here); returns a new bf16 CUDA tensor to pass with
        ``packed=True``."""
        import torch
        n = proj_packed_weight_bytes(self.handle)
        P = torch.empty(max(n // 2, 8), dtype=torch.bfloat16, device=W.device)
        if stream is None:
            stream = torch.cuda.current_stream(W.device)
        proj_pack_weights(self.handle, W, P, stream)
        return P

    def status(self, stream=None) -> int:
        return proj_device_status(self.handle, stream)

    def close(self) -> None:
        if self.handle:
            proj_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
