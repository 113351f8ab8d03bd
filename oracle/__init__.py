"""Plain FP64 CPU oracle for time-domain SAR backprojection.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product path (the CUDA
library and its binding) never imports this package.

Pinned functions (each pinned by tests that do not re-type its formula):
``backproject`` (linear) - pinned by hand-computed single-pulse values, the
closed form at an isolated noiseless target, linearity, focusing, symmetry and
the range window rule (tests/test_oracle_pins.py), and by planted-mistake
checks that each such pin rejects a broken copy of the oracle
(tests/test_oracle_mutations.py).
``backproject(interp="sinc8")`` - pinned by on-sample and half-sample values
of the windowed-sinc kernel, reconstruction of a band-limited signal, the
stencil window rule, linearity, pulse-order invariance and focusing
(tests/test_oracle_sinc_pins.py), with its own planted mistakes.
``backproject_heights`` - pinned by reduction to ``backproject`` (zero and
constant heights), a hand-derived value on a raised pixel, and focusing of
targets on a rough surface (tests/test_oracle_heights_pins.py); its sinc and
nearest forms by the same reductions to the pinned planar variants.
``backproject_volume`` - a stack of ``backproject`` planes at z0 + iz dz; pinned by
three-dimensional focusing of targets seen from a multi-pass aperture
(tests/test_oracle_volume_pins.py).
``backproject(interp="nearest")`` - pinned by on-sample values, the rounding
boundary at half a bin, the window rule and the generic invariants
(tests/test_oracle_nearest_pins.py), with its own planted mistakes.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sarbp_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


class OracleGeometry(ctypes.Structure):
    _fields_ = [
        ("nx", ctypes.c_int64), ("ny", ctypes.c_int64),
        ("na", ctypes.c_int64), ("nr", ctypes.c_int64),
        ("x0", ctypes.c_double), ("y0", ctypes.c_double), ("z0", ctypes.c_double),
        ("dx", ctypes.c_double), ("dy", ctypes.c_double),
        ("r0", ctypes.c_double), ("dr", ctypes.c_double),
        ("wavelength", ctypes.c_double),
    ]


def compile_library(src: str = _SRC, out: str = _LIB) -> str:
    """Compile the C oracle with gcc (plain -O2, IEEE floating point)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", out, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    with _lock:
        stale = (not os.path.exists(_LIB)
                 or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
                 or os.path.getmtime(_LIB) < os.path.getmtime(os.path.join(_HERE, "sarbp_oracle.h")))
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            compile_library(out=tmp)
            os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    for name in ("oracle_backproject", "oracle_backproject_sinc8", "oracle_backproject_nearest"):
        fn = getattr(lib, name, None)
        if fn is None:
            continue
        fn.restype = ctypes.c_int
        fn.argtypes = [
            ctypes.POINTER(OracleGeometry), ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,
        ]
    for name in ("oracle_backproject_heights", "oracle_backproject_heights_sinc8",
                 "oracle_backproject_heights_nearest"):
        fn = getattr(lib, name, None)
        if fn is None:
            continue
        fn.restype = ctypes.c_int
        fn.argtypes = [
            ctypes.POINTER(OracleGeometry), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,
        ]
    return lib


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def geometry(params: dict) -> OracleGeometry:
    return OracleGeometry(
        int(params["nx"]), int(params["ny"]), int(params["na"]), int(params["nr"]),
        float(params["x0"]), float(params["y0"]), float(params["z0"]),
        float(params["dx"]), float(params["dy"]),
        float(params["r0"]), float(params["dr"]), float(params["wavelength"]))


def backproject(params: dict, echoes: np.ndarray, antenna_pos: np.ndarray,
                pixels: np.ndarray | None = None, threads: int = 0,
                library: ctypes.CDLL | None = None, return_info: bool = False,
                interp: str = "linear"):
    """FP64 image at ``pixels`` (linear iy*nx+ix); the full [ny, nx] image if None.

    ``echoes`` complex64 [na, nr]; ``antenna_pos`` float64 [na, 3].
    ``interp`` is "linear" (the page's kernel), "sinc8" (8-tap windowed sinc) or
    "nearest" (nearest sample).
    With ``return_info`` also returns (seconds, threads used).
    """
    library = library or lib()
    fn = {"linear": library.oracle_backproject,
          "sinc8": library.oracle_backproject_sinc8,
          "nearest": library.oracle_backproject_nearest}[interp]
    nx, ny, na, nr = (int(params[k]) for k in ("nx", "ny", "na", "nr"))
    echoes = np.ascontiguousarray(echoes, dtype=np.complex64).reshape(na, nr)
    pos = np.ascontiguousarray(antenna_pos, dtype=np.float64).reshape(na, 3)
    full = pixels is None
    pix = (np.arange(nx * ny, dtype=np.int64) if full
           else np.ascontiguousarray(pixels, dtype=np.int64).reshape(-1))
    out = np.zeros((pix.size, 2), dtype=np.float64)
    g = geometry(params)
    t0 = time.perf_counter()
    used = fn(
        ctypes.byref(g), echoes.ctypes.data if echoes.size else None,
        pos.ctypes.data if pos.size else None, pix.ctypes.data if pix.size else None,
        pix.size, out.ctypes.data if out.size else None, int(threads))
    secs = time.perf_counter() - t0
    if used < 0:
        raise ValueError("oracle_backproject rejected its arguments")
    img = out[:, 0] + 1j * out[:, 1]
    if full:
        img = img.reshape(ny, nx)
    return (img, secs, used) if return_info else img


def backproject_volume(params: dict, echoes: np.ndarray, antenna_pos: np.ndarray, nz: int,
                       dz: float, threads: int = 0, library: ctypes.CDLL | None = None,
                       interp: str = "linear") -> np.ndarray:
    """FP64 voxel grid [nz, ny, nx]: plane iz is the image at height z0 + iz * dz."""
    planes = [backproject(dict(params, z0=float(params["z0"]) + iz * float(dz)), echoes,
                          antenna_pos, threads=threads, library=library, interp=interp)
              for iz in range(int(nz))]
    nx, ny = int(params["nx"]), int(params["ny"])
    return np.stack(planes) if planes else np.zeros((0, ny, nx), dtype=np.complex128)


def backproject_heights(params: dict, echoes: np.ndarray, antenna_pos: np.ndarray,
                        heights: np.ndarray, pixels: np.ndarray | None = None, threads: int = 0,
                        library: ctypes.CDLL | None = None, interp: str = "linear"):
    """FP64 image over pixels raised to z0 + heights[iy, ix] (``heights`` float32
    [ny, nx]); ``interp`` as for :func:`backproject`."""
    library = library or lib()
    fn = {"linear": library.oracle_backproject_heights,
          "sinc8": library.oracle_backproject_heights_sinc8,
          "nearest": library.oracle_backproject_heights_nearest}[interp]
    nx, ny, na, nr = (int(params[k]) for k in ("nx", "ny", "na", "nr"))
    echoes = np.ascontiguousarray(echoes, dtype=np.complex64).reshape(na, nr)
    pos = np.ascontiguousarray(antenna_pos, dtype=np.float64).reshape(na, 3)
    hts = np.ascontiguousarray(heights, dtype=np.float32).reshape(ny, nx)
    full = pixels is None
    pix = (np.arange(nx * ny, dtype=np.int64) if full
           else np.ascontiguousarray(pixels, dtype=np.int64).reshape(-1))
    out = np.zeros((pix.size, 2), dtype=np.float64)
    g = geometry(params)
    used = fn(
        ctypes.byref(g), echoes.ctypes.data if echoes.size else None,
        pos.ctypes.data if pos.size else None, hts.ctypes.data,
        pix.ctypes.data if pix.size else None, pix.size, out.ctypes.data if out.size else None,
        int(threads))
    if used < 0:
        raise ValueError("oracle_backproject_heights rejected its arguments")
    img = out[:, 0] + 1j * out[:, 1]
    return img.reshape(ny, nx) if full else img
