"""GB300-native time-domain SAR backprojection (libsarbp + a thin binding)."""

from ._native import SARBP_ACCUMULATE, Params  # noqa: F401
from .sarbp import Plan, SarbpError, backproject  # noqa: F401

__all__ = ["Plan", "Params", "SarbpError", "backproject", "SARBP_ACCUMULATE"]
