// sarbp_device.cuh - device helpers shared by the echo-table kernels
// (sarbp_kernels.cu) and the fused range-compression table kernel
// (sarbp_rc.cu). Not part of the public C-ABI.
#pragma once

#include "sarbp_internal.h"

namespace sarbp {

// First bin (absolute) of pulse n's table row: the row covers the range
// extent of the tile-padded image box (a rectangle at z0, or the slab
// z0 + [h_min, h_max] for a height map) seen from antenna position a, from
// its nearest point less one tile reach and MARGIN bins. KLO_INVALID when
// the position is not finite. rmin receives the distance to the nearest point.
__device__ __forceinline__ int window_start(const BpConst& k, double ax, double ay, double az,
                                            double& rmin)
{
    rmin = 0.0;
    if (!(isfinite(ax) && isfinite(ay) && isfinite(az)))
        return KLO_INVALID;
    if (k.full_window)
        return -(MARGIN + 4);
    const double cx = fmin(fmax(ax, k.rect_x0), k.rect_x1);
    const double cy = fmin(fmax(ay, k.rect_y0), k.rect_y1);
    const double cz = k.heights_mode ? fmin(fmax(az, k.z_lo), k.z_hi) : k.z0;
    const double ddx = cx - ax, ddy = cy - ay, ddz = cz - az;
    rmin = sqrt(ddx * ddx + ddy * ddy + ddz * ddz);
    double u = (rmin - (k.heights_mode ? k.qmax3 : k.qmax) - k.r0) * k.inv_dr;
    u = fmin(fmax(u, -1.0e9), 1.0e9);
    return (int)floor(u) - MARGIN;
}

// psi_k = exp(j 2 pi frac(2 r_k / lambda)) of absolute bin kk, from the 64-bit
// fixed-point phase accumulator (exact up to the rounding of two constants).
__device__ __forceinline__ float2 bin_phasor(const BpConst& k, long long kk)
{
    const unsigned long long ph = k.beta_fx + k.alpha_fx * (unsigned long long)kk;
    const float turns = (float)(ph >> 40) * 0x1p-24f;
    float s, c;
    sincospif(2.0f * turns, &s, &c);
    return make_float2(c, s);
}

// Linear-interpolation table entry of bin kk from its samples e_kk, e_kk+1:
// (A_k, D_k / c) with A_k = e_k psi_k and D_k = (e_k+1 - e_k) psi_k.
__device__ __forceinline__ float4 linear_entry(const BpConst& k, long long kk, float2 e0, float2 e1)
{
    const float2 ps = bin_phasor(k, kk);
    const float dre = e1.x - e0.x;
    const float dim = e1.y - e0.y;
    return make_float4(e0.x * ps.x - e0.y * ps.y, e0.x * ps.y + e0.y * ps.x,
                       (dre * ps.x - dim * ps.y) * k.inv_c, (dre * ps.y + dim * ps.x) * k.inv_c);
}

}  // namespace sarbp
