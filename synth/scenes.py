"""Seeded synthetic airborne-spotlight scenes for time-domain SAR backprojection.

What the scenes follow (SARBP-GPU = the page "基于GPU的SAR后向投影成像优化与CUDA加速实践",
a GPU back-projection SAR imaging retrospective):

* SARBP-GPU §3.2 (imaging grid and observation geometry): the radar flies a straight
  line, the beam stays on one scene centre, the grid spacing is a fraction of the
  resolution.
* SARBP-GPU §4.2 (validation): small simulated point-target scenes whose echoes are
  known in closed form.
* SARBP-GPU §1.2 (workload): the page-sized scene has Na = 4096 pulses over a
  1024 x 1024 grid; the large scene Na = 16384 over 2048 x 2048.

The echo of a target of amplitude ``a`` at slant range ``R`` is the
range-compressed response ``a * sinc((r_k - R) / rho) * exp(-j 4 pi R / lambda)``
on the range bins ``r_k = r0 + k * dr``, kept where ``|r_k - R| <= 16 rho``
(normalised sinc, sin(pi x) / (pi x)). Complex Gaussian clutter of power
``sigma**2`` is added (each of Re and Im has variance ``sigma**2 / 2``).
Everything is computed in float64 and stored as complex64.

This module is input generation only: it never backprojects.
"""

from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

C_LIGHT = 299_792_458.0          # m/s
FC = 9.6e9                       # carrier, Hz
WAVELENGTH = C_LIGHT / FC        # carrier wavelength (not the bandwidth one)
RHO = 1.0                        # range resolution of the compressed pulse, m
DR = 0.8333                      # range-bin spacing, m
ALTITUDE = 5000.0                # m
GROUND_OFFSET = 7000.0           # track's ground distance from the scene centre, m
SINC_HALF_SUPPORT = 16.0         # in units of rho
TARGET_BORDER = 12               # pixels kept free at the image border
TARGET_SPACING = 24              # minimum Chebyshev distance between targets, pixels
NOISE_CHUNK = 512                # pulses per noise draw (fixes the random stream)
SEED_BASE = 20260


@dataclass(frozen=True)
class SceneConfig:
    index: int
    name: str
    na: int                 # pulses
    nr: int                 # range bins
    nx: int                 # image width (along track, x)
    ny: int                 # image height (cross track, y)
    spacing: float          # dx = dy, metres
    pulse_step: float       # along-track distance between pulses, metres
    n_targets: int
    amp_lo: float
    amp_hi: float
    noise_sigma: float
    motion: bool = False    # smooth seeded track deviations (+-0.5 m per axis)

    @property
    def updates(self) -> int:
        """Pixel-pulse backprojections in one image."""
        return self.na * self.nx * self.ny

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index


CONFIGS = (
    SceneConfig(1, "tiny_stripmap", 64, 256, 64, 64, 0.5, 0.1, 3, 1.0, 1.0, 0.01),
    SceneConfig(2, "small_spotlight", 1024, 2048, 512, 512, 0.25, 200.0 / 1024, 16, 0.5, 1.0, 0.05),
    SceneConfig(3, "page_spotlight", 4096, 4096, 1024, 1024, 0.15, 0.1, 64, 0.5, 1.0, 0.1),
    SceneConfig(4, "large_scene", 16384, 8192, 2048, 2048, 0.15, 0.1, 256, 0.5, 1.0, 0.1),
    SceneConfig(5, "nonideal_track", 8192, 8192, 4096, 4096, 0.2, 0.1, 512, 0.5, 1.0, 0.1,
                motion=True),
)


def config_by_name(name: str) -> SceneConfig:
    for c in CONFIGS:
        if c.name == name or str(c.index) == str(name):
            return c
    raise KeyError(name)


@dataclass
class Scene:
    cfg: SceneConfig
    params: dict                 # nx ny na nr x0 y0 z0 dx dy r0 dr wavelength
    echoes: np.ndarray           # complex64 [na, nr], pulse-major
    antenna_pos: np.ndarray      # float64 [na, 3]
    targets: np.ndarray          # int64 [T, 2] as (ix, iy), on pixel centres
    amps: np.ndarray             # float64 [T]
    heights: np.ndarray | None = None   # float32 [ny, nx] terrain above z0, or None (flat)


def straight_track(na: int, step: float, altitude: float = ALTITUDE,
                   ground_offset: float = GROUND_OFFSET) -> np.ndarray:
    """Antenna phase centres along x, centred on x = 0, at y = -ground_offset, z = altitude."""
    n = np.arange(na, dtype=np.float64)
    pos = np.empty((na, 3), dtype=np.float64)
    pos[:, 0] = (n - (na - 1) / 2.0) * step
    pos[:, 1] = -ground_offset
    pos[:, 2] = altitude
    return pos


def multipass_track(na_per_pass: int, passes: int, step: float, baseline: float,
                    altitude: float = ALTITUDE, ground_offset: float = GROUND_OFFSET) -> np.ndarray:
    """Several parallel straight passes stacked vertically, ``baseline`` metres
    apart and centred on ``altitude`` (a two-dimensional aperture, as used for
    three-dimensional imaging). Pulses of pass 0 first, float64 [passes * na_per_pass, 3]."""
    tracks = []
    for p in range(passes):
        alt = altitude + (p - (passes - 1) / 2.0) * baseline
        tracks.append(straight_track(na_per_pass, step, altitude=alt, ground_offset=ground_offset))
    return np.concatenate(tracks, axis=0)


def _motion(rng: np.random.Generator, na: int) -> np.ndarray:
    """Per-axis sum of three seeded sinusoids, |delta| <= 0.5 m."""
    n = np.arange(na, dtype=np.float64)
    out = np.zeros((na, 3), dtype=np.float64)
    for axis in range(3):
        amp = rng.uniform(0.0, 0.5 / 3.0, size=3)
        freq = rng.uniform(0.5, 4.0, size=3)
        phase = rng.uniform(0.0, 2.0 * np.pi, size=3)
        for m in range(3):
            out[:, axis] += amp[m] * np.sin(2.0 * np.pi * freq[m] * n / na + phase[m])
    return out


def _place_targets(rng: np.random.Generator, nx: int, ny: int, count: int) -> np.ndarray:
    """Seeded rejection sampling; starts over when an early choice leaves no room."""
    lo = TARGET_BORDER
    hix, hiy = nx - TARGET_BORDER, ny - TARGET_BORDER
    for _restart in range(1000):
        placed: list[tuple[int, int]] = []
        misses = 0
        while len(placed) < count and misses < 2000:
            ix = int(rng.integers(lo, hix))
            iy = int(rng.integers(lo, hiy))
            if all(max(abs(ix - px), abs(iy - py)) >= TARGET_SPACING for px, py in placed):
                placed.append((ix, iy))
                misses = 0
            else:
                misses += 1
        if len(placed) == count:
            return np.array(placed, dtype=np.int64).reshape(-1, 2)
    raise RuntimeError("cannot place targets with the requested spacing")


def image_geometry(nx: int, ny: int, spacing: float) -> dict:
    """Grid centred so that pixel (nx/2, ny/2) sits on the scene centre (0, 0, 0)."""
    return dict(x0=-(nx // 2) * spacing, y0=-(ny // 2) * spacing, z0=0.0,
                dx=spacing, dy=spacing)


def simulate_echoes(antenna_pos: np.ndarray, target_xyz: np.ndarray, amps: np.ndarray,
                    r0: float, dr: float, nr: int, wavelength: float = WAVELENGTH,
                    rho: float = RHO, half_support: float = SINC_HALF_SUPPORT,
                    out: np.ndarray | None = None) -> np.ndarray:
    """Noiseless range-compressed echoes (complex128 [na, nr]) of point targets."""
    na = antenna_pos.shape[0]
    if out is None:
        out = np.zeros((na, nr), dtype=np.complex128)
    span = int(np.ceil(2.0 * half_support * rho / dr)) + 2
    offs = np.arange(span, dtype=np.int64)
    rows = np.arange(na, dtype=np.int64)[:, None]
    for t in range(target_xyz.shape[0]):
        d = antenna_pos - target_xyz[t][None, :]
        rng_t = np.sqrt(np.sum(d * d, axis=1))                      # [na]
        kstart = np.ceil((rng_t - half_support * rho - r0) / dr).astype(np.int64)
        k = kstart[:, None] + offs[None, :]                          # [na, span]
        rk = r0 + k * dr
        x = (rk - rng_t[:, None]) / rho
        keep = (np.abs(x) <= half_support) & (k >= 0) & (k < nr)
        val = amps[t] * np.sinc(x) * np.exp(-1j * 4.0 * np.pi * rng_t[:, None] / wavelength)
        rr = np.broadcast_to(rows, k.shape)
        out[rr[keep], k[keep]] += val[keep]
    return out


def terrain(nx: int, ny: int, spacing: float, seed: int, relief: float = 40.0,
            mean: float = 20.0) -> np.ndarray:
    """Seeded smooth terrain, float32 [ny, nx] metres above z0.

    Four 2-D sinusoids (wavelengths 60 to 600 m, random directions, phases and
    amplitudes), shifted and scaled so that the heights span exactly
    ``relief`` metres peak to peak around ``mean``. The steepest slope is of
    order pi * relief / 60 m.
    """
    rng = np.random.default_rng(seed)
    yy, xx = np.mgrid[0:ny, 0:nx].astype(np.float64) * spacing
    h = np.zeros((ny, nx), dtype=np.float64)
    for _ in range(4):
        lam = rng.uniform(60.0, 600.0)
        ang = rng.uniform(0.0, np.pi)
        ph = rng.uniform(0.0, 2.0 * np.pi)
        amp = rng.uniform(0.5, 1.0)
        h += amp * np.sin(2.0 * np.pi * (xx * np.cos(ang) + yy * np.sin(ang)) / lam + ph)
    span = float(h.max() - h.min()) if h.size else 0.0
    if span > 0:
        h = (h - 0.5 * (h.max() + h.min())) * (relief / span)
    return (mean + h).astype(np.float32)


def make_scene(cfg: SceneConfig, noise: bool = True, seed: int | None = None,
               n_targets: int | None = None, heights: np.ndarray | None = None) -> Scene:
    """Build one seeded scene. The result is a pure function of (cfg, seed, noise, n_targets).

    With ``heights`` (float32 [ny, nx]) every target sits on that surface,
    at z0 + heights[iy, ix] above its pixel.
    """
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    count = cfg.n_targets if n_targets is None else n_targets
    targets = _place_targets(rng, cfg.nx, cfg.ny, count)
    if cfg.amp_lo == cfg.amp_hi:
        amps = np.full(count, cfg.amp_lo, dtype=np.float64)
    else:
        amps = rng.uniform(cfg.amp_lo, cfg.amp_hi, size=count)
    pos = straight_track(cfg.na, cfg.pulse_step)
    if cfg.motion:
        pos = pos + _motion(rng, cfg.na)

    geo = image_geometry(cfg.nx, cfg.ny, cfg.spacing)
    centre = np.zeros(3)
    r_mid = float(np.linalg.norm(centre - pos[cfg.na // 2]))
    r0 = r_mid - (cfg.nr // 2) * DR
    params = dict(nx=cfg.nx, ny=cfg.ny, na=cfg.na, nr=cfg.nr, r0=r0, dr=DR,
                  wavelength=WAVELENGTH, **geo)

    txyz = np.zeros((count, 3), dtype=np.float64)
    txyz[:, 0] = geo["x0"] + targets[:, 0] * geo["dx"]
    txyz[:, 1] = geo["y0"] + targets[:, 1] * geo["dy"]
    txyz[:, 2] = geo["z0"]
    if heights is not None:
        txyz[:, 2] += heights[targets[:, 1], targets[:, 0]].astype(np.float64)

    echoes = np.empty((cfg.na, cfg.nr), dtype=np.complex64)
    scale = cfg.noise_sigma / np.sqrt(2.0)
    # the noiseless blocks do not touch the random stream, so they are made on
    # worker threads while this thread draws the noise in block order
    chunks = [(n0, min(cfg.na, n0 + NOISE_CHUNK)) for n0 in range(0, cfg.na, NOISE_CHUNK)]
    workers = max(1, min(len(chunks), (os.cpu_count() or 1), 16))
    with ThreadPoolExecutor(max_workers=workers) as pool:
        def submit(i):
            n0, n1 = chunks[i]
            return pool.submit(simulate_echoes, pos[n0:n1], txyz, amps, r0, DR, cfg.nr)
        ahead = 2 * workers                     # blocks in flight (bounds host memory)
        blocks = [submit(i) for i in range(min(ahead, len(chunks)))]
        for i, (n0, n1) in enumerate(chunks):
            if i + ahead < len(chunks):
                blocks.append(submit(i + ahead))
            fut = blocks[i]
            blocks[i] = None
            g = None
            if noise and cfg.noise_sigma > 0:
                g = rng.standard_normal((n1 - n0, cfg.nr, 2))
            block = fut.result()
            if g is not None:
                block += scale * (g[..., 0] + 1j * g[..., 1])
            echoes[n0:n1] = block.astype(np.complex64)
    return Scene(cfg=cfg, params=params, echoes=echoes, antenna_pos=pos,
                 targets=targets, amps=amps, heights=heights)


def compared_pixels(scene: Scene, n_random: int = 4096, full_limit: int = 512 * 512,
                    halo: int = 4) -> np.ndarray:
    """Linear pixel indices (iy * nx + ix) compared against the oracle.

    Small images are compared in full; larger ones on ``n_random`` seeded random
    pixels plus the (2 halo + 1)^2 neighbourhood of every target.
    """
    nx, ny = scene.params["nx"], scene.params["ny"]
    if nx * ny <= full_limit:
        return np.arange(nx * ny, dtype=np.int64)
    rng = np.random.default_rng(scene.cfg.seed + 1000)
    rand = rng.choice(nx * ny, size=min(n_random, nx * ny), replace=False).astype(np.int64)
    d = np.arange(-halo, halo + 1)
    ix = (scene.targets[:, 0][:, None, None] + d[None, None, :]).clip(0, nx - 1)
    iy = (scene.targets[:, 1][:, None, None] + d[None, :, None]).clip(0, ny - 1)
    hood = (iy * nx + ix).reshape(-1)
    return np.unique(np.concatenate([rand, hood]))


def shrink(cfg: SceneConfig, **changes) -> SceneConfig:
    """A copy of ``cfg`` with some fields replaced (used for scaled-down test cases)."""
    return dataclasses.replace(cfg, **changes)
