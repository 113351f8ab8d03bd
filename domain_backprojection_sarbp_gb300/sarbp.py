"""Python binding of libsarbp: argument marshalling over the C-ABI.

Every step of the backprojection runs in the library's CUDA kernels; this
module only checks tensor dtypes, shapes and devices and passes pointers.
PyTorch provides device memory and streams. There is no CPU fallback: when
the library is missing, the call raises.
"""

from __future__ import annotations

import ctypes

import numpy as np

from . import _native
from ._native import Params, PlanInfo, SARBP_ACCUMULATE, SARBP_NEAREST, SARBP_SINC8


class SarbpError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        text = _native.lib().sarbp_status_string(status).decode()
        super().__init__(f"{where}: {text}" + (f" ({detail})" if detail else ""))


def _params(p, accumulate=False, interp="linear") -> Params:
    if isinstance(p, Params):
        out = Params.from_buffer_copy(p)
    else:
        out = Params.from_dict(p)
    if accumulate:
        out.flags |= SARBP_ACCUMULATE
    if interp == "sinc8":
        out.flags |= SARBP_SINC8
    elif interp == "nearest":
        out.flags |= SARBP_NEAREST
    elif interp != "linear":
        raise ValueError(f"interp must be 'linear', 'sinc8' or 'nearest', got {interp!r}")
    return out


def _stream_handle(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check_device_tensor(t, name, dtype, shape):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr() if t.numel() else None)


# torch's name for each numpy dtype the host calls take (np.dtype(...).name
# costs microseconds per call)
_TORCH_DTYPE_NAME = {np.complex64: "torch.complex64", np.float64: "torch.float64",
                     np.float32: "torch.float32"}


def _host_ptr(a, name, shape, np_dtype):
    if hasattr(a, "is_cuda"):
        if a.is_cuda or not a.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
        if tuple(a.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}")
        if str(a.dtype) != _TORCH_DTYPE_NAME[np_dtype]:
            raise ValueError(f"{name} must have dtype {np.dtype(np_dtype).name}")
        return ctypes.c_void_p(a.data_ptr() if a.numel() else None)
    if not (isinstance(a, np.ndarray) and a.dtype == np_dtype and a.flags.c_contiguous
            and a.shape == shape):
        raise ValueError(f"{name} must be a C-contiguous {np_dtype} array of shape {shape}")
    return ctypes.c_void_p(a.ctypes.data if a.size else None)


def _host_args(p, image, echoes, antenna_pos):
    return (_host_ptr(image, "image", (p.ny, p.nx), np.complex64),
            _host_ptr(echoes, "echoes", (p.na, p.nr), np.complex64),
            _host_ptr(antenna_pos, "antenna_pos", (p.na, 3), np.float64))


class Plan:
    """A libsarbp plan: fixed sizes, device scratch, repeated backprojections."""

    def __init__(self, params, height_range=None, interp="linear"):
        """``height_range`` = (h_min, h_max) makes a height-map plan (sarbp_plan_heights),
        used with :meth:`backproject_heights` only. ``interp="sinc8"`` allocates the
        windowed-sinc coefficient rows with the plan (otherwise the first sinc call
        does); each call still chooses its own interpolation."""
        self._lib = _native.lib()
        self.params = _params(params)
        made = _params(params, interp=interp)
        self.height_range = None if height_range is None else tuple(map(float, height_range))
        handle = ctypes.c_void_p()
        if self.height_range is None:
            st = self._lib.sarbp_plan(ctypes.byref(handle), ctypes.byref(made))
            where = "sarbp_plan"
        else:
            st = self._lib.sarbp_plan_heights(ctypes.byref(handle), ctypes.byref(made),
                                              *self.height_range)
            where = "sarbp_plan_heights"
        if st != _native.SARBP_OK:
            raise SarbpError(st, where)
        self._h = handle

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            self._lib.sarbp_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def _raise(self, st, where):
        detail = self._lib.sarbp_last_error(self._h).decode(errors="replace")
        raise SarbpError(st, where, detail)

    def backproject(self, image, echoes, antenna_pos, params=None, accumulate=False, stream=None,
                    interp="linear"):
        """Enqueue I(p) = sum_n w_n exp(+j 4 pi R_n / lambda) on ``stream`` (device tensors).

        image complex64 [ny, nx]; echoes complex64 [na, nr]; antenna_pos float64 [na, 3].
        ``interp``: "linear", "sinc8" (8-tap windowed sinc) or "nearest".
        """
        import torch
        p = _params(params if params is not None else self.params, accumulate, interp)
        img = _check_device_tensor(image, "image", torch.complex64, (p.ny, p.nx))
        ech = _check_device_tensor(echoes, "echoes", torch.complex64, (p.na, p.nr))
        pos = _check_device_tensor(antenna_pos, "antenna_pos", torch.float64, (p.na, 3))
        st = self._lib.sarbp_backproject(self._h, img, ech, pos, ctypes.byref(p),
                                         _stream_handle(stream))
        if st != _native.SARBP_OK:
            self._raise(st, "sarbp_backproject")
        return image

    def backproject_raw(self, image, raw, antenna_pos, rc, params=None, accumulate=False,
                        stream=None):
        """Raw echoes to image (sarbp_backproject_raw): range compression with the
        RangeCompressor ``rc`` fused with the echo table, then the linear
        backprojection. raw complex64 [na, nr] on the device."""
        import torch
        p = _params(params if params is not None else self.params, accumulate)
        img = _check_device_tensor(image, "image", torch.complex64, (p.ny, p.nx))
        r = _check_device_tensor(raw, "raw", torch.complex64, (p.na, p.nr))
        pos = _check_device_tensor(antenna_pos, "antenna_pos", torch.float64, (p.na, 3))
        st = self._lib.sarbp_backproject_raw(self._h, rc.handle, img, r, pos, ctypes.byref(p),
                                             _stream_handle(stream))
        if st != _native.SARBP_OK:
            self._raise(st, "sarbp_backproject_raw")
        return image

    def backproject_volume(self, volume, echoes, antenna_pos, dz, params=None, accumulate=False,
                           stream=None, interp="linear"):
        """Voxel grid: volume complex64 [nz, ny, nx] on the device, plane iz at z0 + iz * dz."""
        import torch
        p = _params(params if params is not None else self.params, accumulate, interp)
        if not isinstance(volume, torch.Tensor) or volume.dim() != 3:
            raise ValueError("volume must be a 3-D tensor [nz, ny, nx]")
        nz = int(volume.shape[0])
        vol = _check_device_tensor(volume, "volume", torch.complex64, (nz, p.ny, p.nx))
        ech = _check_device_tensor(echoes, "echoes", torch.complex64, (p.na, p.nr))
        pos = _check_device_tensor(antenna_pos, "antenna_pos", torch.float64, (p.na, 3))
        st = self._lib.sarbp_backproject_volume(self._h, vol, ech, pos, ctypes.byref(p), nz,
                                                float(dz), _stream_handle(stream))
        if st != _native.SARBP_OK:
            self._raise(st, "sarbp_backproject_volume")
        return volume

    def backproject_heights(self, image, echoes, antenna_pos, heights, params=None,
                            accumulate=False, stream=None, interp="linear"):
        """Backprojection of pixels raised to z0 + heights[iy, ix].

        heights float32 [ny, nx] on the device, clamped to the plan's height range;
        ``interp``: "linear", "sinc8" or "nearest".
        """
        import torch
        p = _params(params if params is not None else self.params, accumulate, interp)
        img = _check_device_tensor(image, "image", torch.complex64, (p.ny, p.nx))
        ech = _check_device_tensor(echoes, "echoes", torch.complex64, (p.na, p.nr))
        pos = _check_device_tensor(antenna_pos, "antenna_pos", torch.float64, (p.na, 3))
        hts = _check_device_tensor(heights, "heights", torch.float32, (p.ny, p.nx))
        st = self._lib.sarbp_backproject_heights(self._h, img, ech, pos, hts, ctypes.byref(p),
                                                 _stream_handle(stream))
        if st != _native.SARBP_OK:
            self._raise(st, "sarbp_backproject_heights")
        return image

    def backproject_host(self, image, echoes, antenna_pos, params=None, accumulate=False,
                         stream=None, interp="linear"):
        """Same operation on host arrays (numpy or CPU tensors); returns when the image is on the host."""
        p = _params(params if params is not None else self.params, accumulate, interp)
        img, ech, pos = _host_args(p, image, echoes, antenna_pos)
        stream_h = ctypes.c_void_p(None) if stream is None else _stream_handle(stream)
        st = self._lib.sarbp_backproject_host(self._h, img, ech, pos, ctypes.byref(p), stream_h)
        if st != _native.SARBP_OK:
            self._raise(st, "sarbp_backproject_host")
        return image

    def backproject_streamed(self, image, echoes, antenna_pos, chunk_pulses=1024, params=None,
                             accumulate=False, stream=None, interp="linear"):
        """Host arrays, pulses in chunks of ``chunk_pulses`` whose copies overlap the compute;
        returns when the image is on the host."""
        p = _params(params if params is not None else self.params, accumulate, interp)
        img, ech, pos = _host_args(p, image, echoes, antenna_pos)
        stream_h = ctypes.c_void_p(None) if stream is None else _stream_handle(stream)
        st = self._lib.sarbp_backproject_streamed(self._h, img, ech, pos, ctypes.byref(p),
                                                  int(chunk_pulses), stream_h)
        if st != _native.SARBP_OK:
            self._raise(st, "sarbp_backproject_streamed")
        return image

    def host_transfer_bytes(self):
        """(host-to-device, device-to-host) bytes of the last backproject_host call."""
        h2d = ctypes.c_uint64()
        d2h = ctypes.c_uint64()
        st = self._lib.sarbp_host_transfer_bytes(self._h, ctypes.byref(h2d), ctypes.byref(d2h))
        if st != _native.SARBP_OK:
            self._raise(st, "sarbp_host_transfer_bytes")
        return h2d.value, d2h.value

    def describe(self) -> dict:
        info = PlanInfo()
        st = self._lib.sarbp_plan_describe(self._h, ctypes.byref(info))
        if st != _native.SARBP_OK:
            self._raise(st, "sarbp_plan_describe")
        return {name: getattr(info, name) for name, _ in PlanInfo._fields_}

    def set_timing(self, enable: bool = True):
        self._lib.sarbp_set_timing(self._h, 1 if enable else 0)

    def kernel_times(self):
        """(summed milliseconds, launches) of the main kernel since the last query."""
        ms = ctypes.c_double()
        n = ctypes.c_int32()
        st = self._lib.sarbp_kernel_times(self._h, ctypes.byref(ms), ctypes.byref(n))
        if st != _native.SARBP_OK:
            self._raise(st, "sarbp_kernel_times")
        return ms.value, n.value


def backproject(image, echoes, antenna_pos, params, accumulate=False, stream=None):
    """One-shot convenience: plan, backproject, destroy (the plan is freed after a stream sync)."""
    import torch
    with Plan(params) as plan:
        plan.backproject(image, echoes, antenna_pos, accumulate=accumulate, stream=stream)
        torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
    return image


class RangeCompressor:
    """Matched filtering of raw pulses (libsarbp's sarbp_range_compress)."""

    def __init__(self, reference, na, ns, window="none", band_fraction=1.0, stream=None):
        import torch
        self._lib = _native.lib()
        ref = _check_device_tensor(reference, "reference", torch.complex64, (reference.shape[0],))
        win = {"none": _native.SARBP_WINDOW_NONE, "hamming": _native.SARBP_WINDOW_HAMMING,
               "taylor": _native.SARBP_WINDOW_TAYLOR}[window]
        self.params = _native.RcParams(int(na), int(ns), int(reference.shape[0]), win,
                                       float(band_fraction))
        handle = ctypes.c_void_p()
        st = self._lib.sarbp_rc_plan(ctypes.byref(handle), ctypes.byref(self.params), ref,
                                     _stream_handle(stream))
        if st != _native.SARBP_OK:
            raise SarbpError(st, "sarbp_rc_plan")
        self._h = handle

    def __call__(self, out, raw, stream=None):
        """Enqueue rc[n][k] = sum_l raw[n][k + l] conj(ref[l]) (device tensors [na, ns])."""
        import torch
        shape = (self.params.na, self.params.ns)
        o = _check_device_tensor(out, "out", torch.complex64, shape)
        r = _check_device_tensor(raw, "raw", torch.complex64, shape)
        st = self._lib.sarbp_range_compress(self._h, o, r, _stream_handle(stream))
        if st != _native.SARBP_OK:
            raise SarbpError(st, "sarbp_range_compress")
        return out

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            self._lib.sarbp_rc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
