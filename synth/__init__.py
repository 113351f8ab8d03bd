"""Seeded synthetic SAR scenes: airborne spotlight geometry, point targets, clutter.

This package is input generation only. It simulates range-compressed echoes
(the forward model) and holds none of the backprojection arithmetic; both the
CUDA path's tests and the CPU oracle consume what it produces.
"""

from .scenes import (  # noqa: F401
    C_LIGHT,
    CONFIGS,
    FC,
    RHO,
    DR,
    Scene,
    SceneConfig,
    config_by_name,
    make_scene,
    simulate_echoes,
    straight_track,
    compared_pixels,
    terrain,
    multipass_track,
)
