"""GB300-native time-domain SAR backprojection (libsarbp + a thin binding)."""

from ._native import SARBP_ACCUMULATE, Params  # noqa: F401
from .sarbp import Plan, RangeCompressor, SarbpError, backproject  # noqa: F401

__all__ = ["Plan", "Params", "RangeCompressor", "SarbpError", "backproject", "SARBP_ACCUMULATE"]
