"""ctypes declarations of the libsarbp C-ABI (include/sarbp.h). Marshalling only."""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsarbp.so")

SARBP_OK = 0
SARBP_ERR_INVALID_ARG = 1
SARBP_ERR_PLAN_MISMATCH = 2
SARBP_ERR_CUDA = 3
SARBP_ERR_OOM = 4
SARBP_ERR_UNSUPPORTED_DEVICE = 5
SARBP_ERR_SCRATCH_TOO_SMALL = 6
SARBP_ACCUMULATE = 1
SARBP_SINC8 = 2
SARBP_NEAREST = 4

EXPORTS = (
    "sarbp_plan", "sarbp_backproject", "sarbp_backproject_host", "sarbp_destroy",
    "sarbp_status_string", "sarbp_last_error", "sarbp_plan_describe",
    "sarbp_set_timing", "sarbp_kernel_times", "sarbp_backproject_noalloc",
    "sarbp_host_transfer_bytes", "sarbp_rc_plan", "sarbp_range_compress", "sarbp_rc_destroy",
    "sarbp_plan_heights", "sarbp_backproject_heights", "sarbp_backproject_streamed",
    "sarbp_backproject_volume", "sarbp_debug_fail_alloc", "sarbp_debug_sinc_taps",
    "sarbp_backproject_raw",
)

SARBP_WINDOW_NONE = 0
SARBP_WINDOW_HAMMING = 1
SARBP_WINDOW_TAYLOR = 2


class Params(ctypes.Structure):
    _fields_ = [
        ("nx", ctypes.c_int32), ("ny", ctypes.c_int32),
        ("na", ctypes.c_int32), ("nr", ctypes.c_int32),
        ("x0", ctypes.c_double), ("y0", ctypes.c_double), ("z0", ctypes.c_double),
        ("dx", ctypes.c_double), ("dy", ctypes.c_double),
        ("r0", ctypes.c_double), ("dr", ctypes.c_double),
        ("wavelength", ctypes.c_double),
        ("flags", ctypes.c_uint32),
    ]

    @classmethod
    def from_dict(cls, d: dict, flags: int = 0) -> "Params":
        return cls(int(d["nx"]), int(d["ny"]), int(d["na"]), int(d["nr"]),
                   float(d["x0"]), float(d["y0"]), float(d["z0"]),
                   float(d["dx"]), float(d["dy"]), float(d["r0"]), float(d["dr"]),
                   float(d["wavelength"]), int(d.get("flags", flags)))


class RcParams(ctypes.Structure):
    _fields_ = [
        ("na", ctypes.c_int32), ("ns", ctypes.c_int32), ("nref", ctypes.c_int32),
        ("window", ctypes.c_uint32), ("band_fraction", ctypes.c_double),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("tile_x", ctypes.c_int32), ("tile_y", ctypes.c_int32), ("tiles", ctypes.c_int32),
        ("ctas", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32), ("sms", ctypes.c_int32),
        ("window", ctypes.c_int32), ("full_window", ctypes.c_int32),
        ("kernels_per_call", ctypes.c_int32), ("scratch_bytes", ctypes.c_size_t),
    ]


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.POINTER
    vp = ctypes.c_void_p
    st = ctypes.c_int
    lib.sarbp_plan.argtypes = [P(vp), P(Params)]
    lib.sarbp_plan.restype = st
    lib.sarbp_backproject.argtypes = [vp, vp, vp, vp, P(Params), vp]
    lib.sarbp_backproject.restype = st
    lib.sarbp_backproject_volume.argtypes = [vp, vp, vp, vp, P(Params), ctypes.c_int32,
                                             ctypes.c_double, vp]
    lib.sarbp_backproject_volume.restype = st
    lib.sarbp_plan_heights.argtypes = [P(vp), P(Params), ctypes.c_double, ctypes.c_double]
    lib.sarbp_plan_heights.restype = st
    lib.sarbp_backproject_heights.argtypes = [vp, vp, vp, vp, vp, P(Params), vp]
    lib.sarbp_backproject_heights.restype = st
    lib.sarbp_backproject_host.argtypes = [vp, vp, vp, vp, P(Params), vp]
    lib.sarbp_backproject_host.restype = st
    lib.sarbp_backproject_streamed.argtypes = [vp, vp, vp, vp, P(Params), ctypes.c_int32, vp]
    lib.sarbp_backproject_streamed.restype = st
    lib.sarbp_backproject_noalloc.argtypes = [vp, vp, vp, P(Params), vp]
    lib.sarbp_backproject_noalloc.restype = st
    lib.sarbp_host_transfer_bytes.argtypes = [vp, P(ctypes.c_uint64), P(ctypes.c_uint64)]
    lib.sarbp_host_transfer_bytes.restype = st
    lib.sarbp_rc_plan.argtypes = [P(vp), P(RcParams), vp, vp]
    lib.sarbp_rc_plan.restype = st
    lib.sarbp_range_compress.argtypes = [vp, vp, vp, vp]
    lib.sarbp_range_compress.restype = st
    lib.sarbp_rc_destroy.argtypes = [vp]
    lib.sarbp_rc_destroy.restype = st
    lib.sarbp_backproject_raw.argtypes = [vp, vp, vp, vp, vp, P(Params), vp]
    lib.sarbp_backproject_raw.restype = st
    lib.sarbp_debug_fail_alloc.argtypes = [ctypes.c_int32]
    lib.sarbp_debug_fail_alloc.restype = None
    lib.sarbp_debug_sinc_taps.argtypes = [ctypes.POINTER(ctypes.c_float)]
    lib.sarbp_debug_sinc_taps.restype = ctypes.c_int32
    lib.sarbp_destroy.argtypes = [vp]
    lib.sarbp_destroy.restype = st
    lib.sarbp_status_string.argtypes = [st]
    lib.sarbp_status_string.restype = ctypes.c_char_p
    lib.sarbp_last_error.argtypes = [vp]
    lib.sarbp_last_error.restype = ctypes.c_char_p
    lib.sarbp_plan_describe.argtypes = [vp, P(PlanInfo)]
    lib.sarbp_plan_describe.restype = st
    lib.sarbp_set_timing.argtypes = [vp, ctypes.c_int]
    lib.sarbp_set_timing.restype = st
    lib.sarbp_kernel_times.argtypes = [vp, P(ctypes.c_double), P(ctypes.c_int32)]
    lib.sarbp_kernel_times.restype = st
    return lib


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libsarbp. Raises if the CUDA library has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"libsarbp is not built ({LIB_PATH} missing); run "
                "domain_backprojection_sarbp_gb300.build.build() first")
        _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib
