// sarbp_kernels.cu - the device side of libsarbp (sm_103a).
//
// SARBP-GPU = the page "基于GPU的SAR后向投影成像优化与CUDA加速实践". The page's
// loop (§2.2 steps, §3.3 pseudo-code) spends, per pixel and pulse, a square
// root for the slant range, a floor and two complex gathers for the linear
// interpolation, and a sine and a cosine for exp(+j 4 pi R / lambda). Its
// design (one thread per pixel, §2.1; shared-memory echo tiles, §2.3; double
// precision phase or Kahan sums, §2.2 and §4.3) targets an sm_86 card. This file
// computes the same sum with less work per update:
//
// 1. Echo table (table_kernel). Writing u = (R - r0)/dr = k + f, the phase
//    4 pi R / lambda splits into 2 pi (2 r_k / lambda) + c f with
//    c = 2 pi (2 dr / lambda). So
//        w(f) exp(j 4 pi R / lambda) = exp(j c f) [A_k + f D_k],
//        A_k = e_k psi_k,  D_k = (e_{k+1} - e_k) psi_k,  psi_k = exp(j 2 pi 2 r_k / lambda).
//    One 16-byte row entry (A_k, D_k / c) then serves one update: one gather
//    instead of two, and a phase that depends on the in-bin fraction f only,
//    so it needs no reduction of a thousand-turn argument. psi_k comes from an
//    exact 64-bit fixed-point phase accumulator. Each row keeps only the bins
//    the image can reach (its window starts at klo[n]), zero outside the
//    recorded range 0 <= k <= nr - 2, so the window rule costs nothing per update.
//
// 2. Range without a square root (bp_kernel). For each (tile, pulse) the slant
//    range to the tile centre is computed in float64 and the range of every
//    pixel of the tile is a Taylor polynomial of |p - a_n| about it (complete
//    to third order, with the fourth-order terms in the row offset), in bins.
//    A thread owns 32 pixels of one row, so per pulse it reduces the
//    polynomial to a quadratic in its column offset (a split float for the
//    large linear term keeps 2^-22-bin accuracy), and each update costs two
//    FMAs for u. Pulses where the remainder bound exceeds 5e-5 rad of phase
//    (near field, very fine bins) take an exact path instead (float64 range
//    per row, float32 difference across the row).
//
// 3. Work split (stream-K). The (tile, pulse) units are cut into one equal,
//    contiguous range per resident CTA. A tile covered by one CTA is written
//    directly; the pieces of a shared tile go to partial buffers that
//    reduce_kernel sums in CTA order, so the result is deterministic.
//
// 4. Linear interpolation, two-entry form: when a thread's 32 pixels fall in
//    two range bins, the interpolated, phase-compensated samples are one line
//    plus a hinge in y = c (u - k0 - 1) (hinge_pulse): two table entries per
//    thread and pulse, no per-pixel gather; other threads gather per pixel.
//
// 5. Variants of the same kernel (template INTERP): the 8-tap windowed sinc
//    (one polynomial per thread and pulse, of degree 2 to 4 by the spread of
//    the thread's pixels up to 0.34 bin, and in a second instantiation for
//    wide geometries degree 5 or 6 up to 0.8 bin), the nearest
//    sample (one table entry per thread and pulse when its pixels round to
//    two bins), and pixels on a height map (a float-pair row reference and a
//    range series per pixel, with the two-entry form for rows in two bins).
#include "sarbp_device.cuh"
#include "sarbp_internal.h"

#include <cmath>
#include <cstdint>
#include <algorithm>

namespace sarbp {
namespace {

constexpr float MAGIC = 12582912.0f;   // 1.5 * 2^23: adding it leaves floor/round(x) in the mantissa
constexpr int MAGIC_BITS = 0x4B400000; // bit pattern of MAGIC

enum Interp : int { INTERP_LINEAR = 0, INTERP_SINC8 = 1, INTERP_NEAREST = 2, INTERP_HEIGHTS = 3,
                    INTERP_HEIGHTS_SINC8 = 4, INTERP_HEIGHTS_NEAREST = 5 };
// pixels on a height map, with the linear, windowed-sinc or nearest interpolation
__host__ __device__ constexpr bool on_heights(int interp)
{
    return interp >= INTERP_HEIGHTS && interp <= INTERP_HEIGHTS_NEAREST;
}
// the windowed sinc on the plane: INTERP_SINC8 for geometries where every
// thread's pixels span at most SINC_SPAN bins, INTERP_SINC8_WIDE (with the
// degree-5 and degree-6 polynomial modes, and more registers in use) for the others
constexpr int INTERP_SINC8_WIDE = 6;
__host__ __device__ constexpr bool is_sinc(int interp)
{
    return interp == INTERP_SINC8 || interp == INTERP_SINC8_WIDE;
}
// float4 from one pulse's table row to the next: the sinc kinds read the
// coefficient rows (four entries per bin)
template <int INTERP>
__device__ __forceinline__ int row_pitch(const BpConst& k)
{
    return (is_sinc(INTERP) || INTERP == INTERP_HEIGHTS_SINC8) ? k.tw : k.W;
}
constexpr float SINC_SPAN = 0.34f;          // widest spread of u (bins) for the sinc polynomial
constexpr float SINC_HALF_MIN = 1.0f / 64;  // narrowest half-width of its interval
constexpr float SINC_SPAN3 = 0.17f;         // widest spread for the cubic on four nodes
constexpr float SINC_SPAN2 = 0.05f;         // widest spread for the quadratic on three nodes
constexpr float SINC_SPAN5 = 0.56f;         // widest spread for degree 5 on six nodes (wide kernel)
constexpr float SINC_SPAN6 = 0.80f;         // widest spread for degree 6 on seven nodes (wide kernel)
constexpr int SINC_MAXC = 7;                // coefficients of the highest-degree thread polynomial
// float4 per row of a tile's height terms: the 16 pixel pairs' terms, then the
// row's statistics (HRow) in three; an odd count keeps a warp's 16-byte reads
// of its 32 rows conflict-free
constexpr int HROW_STATS = TILE_X / 2;
constexpr int HROW4 = TILE_X / 2 + 3;

struct __align__(16) Record {
    float4 a;  // c00 (fraction of the tile-centre bin), c01 hi, c01 lo, c02
    float4 b;  // c03, c04, c10, c11
    float4 c;  // c12, c13, c20, c21
    float4 d;  // c22, row index of bin 0 (int bits), kbase (int bits), kind (int bits)
};

// Monomial coefficients of the windowed-sinc tap weights on one bin: with
// u = k + 1/2 + s (s in [-1/2, 1/2]) the tap on sample k + d (d = -3 .. 4) has
// weight h(1/2 + s - d), h(t) = sinc(t) (1 + cos(pi t / 4)) / 2, and
// c[d + 3][n] are the coefficients of s^n of its degree-7 interpolant at the
// eight Chebyshev nodes s_i = cos((2i + 1) pi / 16) / 2. Measured on a fine
// grid in float64, each interpolant is within 7.7e-7 of its weight and the
// eight errors sum to 5.2e-6, so |G - sum_n P_n s^n| <= 5.2e-6 max|e_m|.
struct SincTaps {
    float c[8][8];
};

SincTaps fit_sinc_taps()
{
    constexpr double pi = 3.14159265358979323846;
    SincTaps t{};
    for (int d = -3; d <= 4; ++d) {
        // Vandermonde system V c = h at the nodes, Gaussian elimination with
        // partial pivoting in float64
        double a[8][9];
        for (int i = 0; i < 8; ++i) {
            const double sn = 0.5 * std::cos((2 * i + 1) * pi / 16.0);
            const double x = 0.5 + sn - d;            // never 0: the nodes are inside the bin
            const double h = std::sin(pi * x) / (pi * x) * 0.5 * (1.0 + std::cos(pi * x / 4.0));
            double pw = 1.0;
            for (int n = 0; n < 8; ++n) {
                a[i][n] = pw;
                pw *= sn;
            }
            a[i][8] = h;
        }
        for (int c = 0; c < 8; ++c) {
            int piv = c;
            for (int r = c + 1; r < 8; ++r)
                if (std::fabs(a[r][c]) > std::fabs(a[piv][c]))
                    piv = r;
            for (int n = 0; n < 9; ++n)
                std::swap(a[c][n], a[piv][n]);
            for (int r = 0; r < 8; ++r) {
                if (r == c)
                    continue;
                const double f = a[r][c] / a[c][c];
                for (int n = c; n < 9; ++n)
                    a[r][n] -= f * a[c][n];
            }
        }
        for (int n = 0; n < 8; ++n)
            t.c[d + 3][n] = (float)(a[n][8] / a[n][n]);
    }
    return t;
}

// ---------------------------------------------------------------------------
// Echo table: one block per pulse.
// ---------------------------------------------------------------------------
// Linear interpolation (TABLE_LINEAR): entries (A_k, D_k / c) as above.
// Nearest neighbour (TABLE_PAIRS): entries (N_k, M_k) with N_k = e_k psi_k h
// and M_k = (e_{k+1} - e_k) psi_k h, h = exp(j c / 2), a sample taken as zero
// where it lies outside 0 .. nr - 1: a pixel whose nearest sample is k has
// the compensated echo N_k exp(j c (u - k - 1/2)), and the two samples of
// bins k and k + 1 seen from the boundary between them are N_k and N_k + M_k
// (psi_k+1 = psi_k exp(j c)). Windowed sinc (TABLE_SINC): four
// entries per bin k, the complex coefficients P_0 .. P_7 of the interpolant on
// that bin, G(k + 1/2 + s) = sum_n P_n s^n for s in [-1/2, 1/2], with
// P_n = sum_d taps.c[d + 3][n] e_{k+d}; zero unless the whole stencil
// k - 3 .. k + 4 lies in 0 .. nr - 1. The phase of the last two kinds comes
// of the sinc kind comes from psi_k (psi_kernel). Rows are k.tw float4 apart.
enum TableKind : int { TABLE_LINEAR = 0, TABLE_PAIRS = 1, TABLE_SINC = 2 };

template <int KIND>
__global__ void __launch_bounds__(256) table_kernel(BpConst k, const float2* __restrict__ echo,
                                                    const double* __restrict__ pos,
                                                    float4* __restrict__ table,
                                                    int* __restrict__ klo,
                                                    int* __restrict__ sinc_wide, SincTaps taps)
{
    constexpr bool SINC = KIND == TABLE_SINC;
    const int n = blockIdx.x;
    __shared__ int s_lo;
    if (threadIdx.x == 0) {
        const double ax = pos[3 * (size_t)n + 0];
        const double ay = pos[3 * (size_t)n + 1];
        const double az = pos[3 * (size_t)n + 2];
        double rmin;
        const int lo = window_start(k, ax, ay, az, rmin);
        if (SINC && sinc_wide && lo != KLO_INVALID && !k.full_window) {
            // a thread's 32 pixels span about 31 dx |g_x| / dr bins, |g_x| at
            // most the largest x distance over the nearest range; above
            // SINC_SPAN (with a margin for the curvature) the wide kernel runs
            const double gx = fmax(fabs(k.rect_x0 - ax), fabs(k.rect_x1 - ax)) / fmax(rmin, 1.0);
            if ((TILE_X - 1) * k.dx * gx * k.inv_dr + 0.01 > (double)SINC_SPAN)
                atomicOr(sinc_wide, 1);
        }
        s_lo = lo;
        klo[n] = lo;
    }
    __syncthreads();
    const int lo = s_lo;
    float4* row = table + (size_t)n * k.tw;
    const float2* erow = echo + (size_t)n * (size_t)k.echo_stride;
    for (int w = threadIdx.x; w < k.W; w += blockDim.x) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        const long long kk = (long long)lo + w;
        if (SINC) {
            float2 pc[8];
#pragma unroll
            for (int m = 0; m < 8; ++m)
                pc[m] = make_float2(0.f, 0.f);
            if (lo != KLO_INVALID && kk >= 3 && kk <= (long long)k.nr - 5) {
#pragma unroll
                for (int d = 0; d < 8; ++d) {
                    const float2 e = erow[kk - 3 + d];
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        pc[m].x = fmaf(taps.c[d][m], e.x, pc[m].x);
                        pc[m].y = fmaf(taps.c[d][m], e.y, pc[m].y);
                    }
                }
            }
            float4* out = row + 4 * (size_t)w;
#pragma unroll
            for (int m = 0; m < 4; ++m)
                out[m] = make_float4(pc[2 * m].x, pc[2 * m].y, pc[2 * m + 1].x, pc[2 * m + 1].y);
            continue;
        }
        if (KIND == TABLE_PAIRS) {
            float2 e0 = make_float2(0.f, 0.f), e1 = make_float2(0.f, 0.f);
            if (lo != KLO_INVALID && kk >= 0 && kk <= (long long)k.nr - 1)
                e0 = erow[kk];
            if (lo != KLO_INVALID && kk + 1 >= 0 && kk + 1 <= (long long)k.nr - 1)
                e1 = erow[kk + 1];
            // psi_k h, h = exp(j c / 2)
            const float2 ps = bin_phasor(k, kk);
            const float c = ps.x * k.hrot_re - ps.y * k.hrot_im;
            const float s = ps.x * k.hrot_im + ps.y * k.hrot_re;
            const float dre = e1.x - e0.x, dim = e1.y - e0.y;
            v.x = e0.x * c - e0.y * s;
            v.y = e0.x * s + e0.y * c;
            v.z = dre * c - dim * s;
            v.w = dre * s + dim * c;
        } else if (lo != KLO_INVALID && kk >= 0 && kk <= (long long)k.nr - 2) {
            v = linear_entry(k, kk, erow[kk], erow[kk + 1]);
        }
        row[w] = v;
    }
}

// psi_k = exp(j 2 pi frac(2 r_k / lambda)) for every bin of the range axis.
__global__ void __launch_bounds__(256) psi_kernel(BpConst k, float2* __restrict__ psi)
{
    const long long kk = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (kk >= k.nr)
        return;
    psi[kk] = bin_phasor(k, kk);
}

// ---------------------------------------------------------------------------
// Per-(tile, pulse) record, float64.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float f32(double v) { return __double2float_rn(v); }

template <int INTERP>
__device__ __forceinline__ void make_record(const BpConst& k, const double* __restrict__ pos,
                            const int* __restrict__ klo, int n, double xc, double yc,
                            Record& out)
{
    const double ax = pos[3 * (size_t)n + 0];
    const double ay = pos[3 * (size_t)n + 1];
    const double az = pos[3 * (size_t)n + 2];
    const int lo = klo[n];
    // the height-map kernels (plans of sarbp_plan_heights only) build their
    // records about the mid height, the planar ones on the image plane. The
    // linear kernel keeps this a run-time test of the plan (always false
    // there): compiled that way its register allocation has no spills.
    const bool HM = on_heights(INTERP) || (INTERP == INTERP_LINEAR && k.heights_mode);
    const double vx = xc - ax, vy = yc - ay, vz = (HM ? k.z_mid : k.z0) - az;
    const double r2 = vx * vx + vy * vy + vz * vz;
    const double r = sqrt(r2);
    const double reach = HM ? k.qmax3 : k.qmax;
    int kind = REC_SKIP;
    Record rec;
    rec.a = rec.b = rec.c = rec.d = make_float4(0.f, 0.f, 0.f, 0.f);
    rec.d.y = __int_as_float(-lo);
    if (lo != KLO_INVALID && isfinite(r)) {
        const double u = (r - k.r0) * k.inv_dr;
        const double umin = (r - reach - k.r0) * k.inv_dr - 1e-6;
        const double umax = (r + reach - k.r0) * k.inv_dr + 1e-6;
        // every pixel of the tile has k <= -1 or k >= nr - 1: no recorded echo
        if (!(umax < 0.0 || umin >= (double)k.nr - 1.0)) {
            const double kt = floor(fmin(fmax(u, -1.0e9), 1.0e9));
            const double kb = fmin(fmax(kt - lo, -1.0e9), 1.0e9);
            const double kmin_rel = floor(umin) - lo;
            const double kmax_rel = floor(umax) - lo;
            const bool in_row = kmin_rel >= MARGIN && kmax_rel <= (double)(k.W - 1 - MARGIN);

            // Taylor coefficients of |p - a_n| about the tile centre, in bins
            // per power of the pixel offsets (i, j). With g = v / R, M = I - g g^T,
            // a = (g.q)/R and b = |q|^2/R^2, |v + q| = R sqrt(1 + 2a + b) gives
            //   order 2:  (q^T M q) / (2R)
            //   order 3:  -(g.q)(q^T M q) / (2R^2)
            //   order 4:  (-|q|^4/8 + 3 (g.q)^2 |q|^2 / 4 - 5 (g.q)^4 / 8) / R^3
            // Order-4 terms with j^2 or more are kept (they fold into the
            // per-thread coefficients for free); the others are bounded below.
            // float64 only where float32 would not hold: the reciprocal range (one
            // Newton step on a float seed), gy and c01 (c01 j reaches tens of
            // bins and is split below), c10 (rounded once); every other
            // coefficient multiplies offsets small enough for float32
            double ir = (double)(1.0f / (float)r);
            ir = ir * fma(-r, ir, 2.0);
            const double gy = vy * ir;
            const double c01 = gy * k.dy * k.inv_dr;
            const float irf = (float)ir, gx = (float)(vx * ir), gyf = (float)gy;
            const float mxx = 1.0f - gx * gx, mxy = -gx * gyf, myy = 1.0f - gyf * gyf;
            const float dx = k.dx_f, dy = k.dy_f, idr = k.inv_dr_f;
            const float ir3 = irf * irf * irf;
            const float h2 = 0.5f * irf, h3 = -0.5f * irf * irf;
            const float c10 = f32(vx * ir * k.dx * k.inv_dr);   // times i: keep one rounding
            const float c20 = mxx * h2 * dx * dx * idr;
            const float c11 = 2.0f * mxy * h2 * dx * dy * idr;
            const float c02 = myy * h2 * dy * dy * idr;
            const float c21 = h3 * (2.0f * gx * mxy + gyf * mxx) * dx * dx * dy * idr;
            const float c12 = h3 * (gx * myy + 2.0f * gyf * mxy) * dx * dy * dy * idr;
            const float c03 = h3 * gyf * myy * dy * dy * dy * idr;
            const float gx2 = gx * gx, gy2 = gyf * gyf;
            const float k40 = -0.125f + 0.75f * gx2 - 0.625f * gx2 * gx2;
            const float k31 = 1.5f * gx * gyf - 2.5f * gx2 * gx * gyf;
            const float k22 = -0.25f + 0.75f * (gx2 + gy2) - 3.75f * gx2 * gy2;
            const float k13 = 1.5f * gx * gyf - 2.5f * gx * gy2 * gyf;
            const float k04 = -0.125f + 0.75f * gy2 - 0.625f * gy2 * gy2;
            const float c22 = k22 * ir3 * dx * dx * dy * dy * idr;
            const float c13 = k13 * ir3 * dx * dy * dy * dy * idr;
            const float c04 = k04 * ir3 * dy * dy * dy * dy * idr;

            // dropped: c30 i^3, c31 i^3 j, c40 i^4 (metres), plus the order-5
            // remainder, at most |q|^5 / R^4 while |q| <= R / 8
            const float hx = 0.5f * (TILE_X - 1) * dx, hy = 0.5f * (TILE_Y - 1) * dy;
            const float hx3 = hx * hx * hx;
            const float qm = (float)k.qmax;
            const float q5 = qm * qm * qm * qm * qm;
            const float dropped = fabsf(gx * mxx) * 0.5f * irf * irf * hx3
                                + (fabsf(k31) * hx3 * hy + fabsf(k40) * hx3 * hx) * ir3
                                + q5 * ir3 * irf;
            const bool fast = in_row && r > 8.0 * k.qmax && dropped * idr <= (float)k.fast_tol_bins;
            kind = fast ? REC_FAST : REC_EXACT;

            const float c01h = f32(c01);
            rec.a = make_float4(f32(u - kt), c01h, f32(c01 - (double)c01h), c02);
            rec.b = make_float4(c03, c04, c10, c11);
            rec.c = make_float4(c12, c13, c20, c21);
            rec.d = make_float4(c22, __int_as_float(-lo), __int_as_float((int)kb), 0.f);
            if (HM) {
                // height map: a row's reference point is offset from the tile
                // centre (at the mid height) by q = (0, Y, Z), Y = j dy, Z its
                // height above the mid height. The record carries what its
                // range expansion to fourth order in |q| / R needs (see
                // heights_row_curvature): the tile-centre bin and fraction,
                // the linear terms gy dy / dr and gz / dr as float pairs, gy,
                // gz, 1 / R, and v_x, v_z and R for the per-pixel series. The
                // order-5 remainder is at most |q|^5 / R^4 (|q| <= qmax3);
                // where that exceeds the fast-path tolerance the row takes
                // the float64 path.
                const double gz = vz * ir;
                const double bz = gz * k.inv_dr;
                const float bzh = f32(bz);
                const double qr = k.qmax3 * ir;
                const double q5 = qr * qr * qr * qr * k.qmax3 * k.inv_dr;   // |q|^5 / R^4, bins
                const bool hfast = r > 8.0 * k.qmax3 && q5 <= k.fast_tol_bins;
                rec.a = make_float4(f32(u - kt), c01h, f32(c01 - (double)c01h), bzh);
                rec.b = make_float4(f32(bz - (double)bzh), gyf, f32(gz), irf);
                rec.c = make_float4(f32(vx), f32(vz), f32(r), 0.f);
                rec.d = make_float4(0.f, __int_as_float(-lo), __int_as_float((int)kb), 0.f);
                kind = hfast ? REC_FAST : REC_EXACT;
            }
        }
    }
    rec.d.w = __int_as_float(kind);
    out = rec;
}

// The record builder as a call of its own (one thread per pulse, once per
// chunk of 512 pulses) for the nearest and height-map kernels: their main
// loops' register allocation then does not have to make room for its float64
// work (fewer spilled bytes, and 1-2 % faster). The linear and sinc kernels
// inline it (as a call it cost the linear kernel 5 %).
template <int INTERP>
__device__ __noinline__ void make_record_call(const BpConst& k, const double* __restrict__ pos,
                                              const int* __restrict__ klo, int n, double xc,
                                              double yc, Record& out)
{
    make_record<INTERP>(k, pos, klo, n, xc, yc, out);
}

// ---------------------------------------------------------------------------
// Updates of one pulse for the TILE_X pixels a thread owns.
//
// Pixels are handled in pairs (q, q + NP), NP = TILE_X / 2, as float2 values so
// that the range polynomial, the floor, the fraction, the phase scaling and
// the complex multiply-accumulate issue as packed f32x2 instructions.
// ---------------------------------------------------------------------------
constexpr int NP = TILE_X / 2;

// What one pulse needs, built one pulse ahead of its use. Nothing here waits
// on the table loads; their values are consumed by the next pulse step.
enum PulseMode : int { MODE_SKIP = 0, MODE_HINGE = 1, MODE_GATHER = 2, MODE_EXACT = 3, MODE_POLY = 4,
                       MODE_PAIR = 5, MODE_POLY3 = 6, MODE_POLY5 = 7, MODE_POLY6 = 8,
                       MODE_POLY2 = 9 };

struct PulseState {
    float2 q0, q1, q2;            // hinge: c (e0 - k0 - 1), c e1, c e2; otherwise e0, e1, e2 (both lanes)
    float4 t0;                    // hinge: table entry k0 + 1; sinc polynomial: lo_u, hi_u, k0, bin k0;
                                  // nearest pair: table entry (N_kn, M_kn)
    float2 t1d;                   // hinge: D part of entry k0
    int kb;                       // row index the polynomial u is relative to
    int bin0;                     // row index of absolute bin 0
    int mode;
};

// The interval of a polynomial: [lo, hi] widened to a half-width of at least
// SINC_HALF_MIN, its first bin k0 (row units) and k0's absolute bin; true when
// it spans at most `span` bins (less than one: the interval then touches bins
// k0 and k0 + 1 only) and the stencils of both bins lie inside the recorded range.
__device__ __forceinline__ bool poly_interval(const BpConst& k, int kb, int bin0, float lo, float hi,
                                              float span, float& lo_e, float& hi_e, float& k0,
                                              int& kabs0)
{
    const float mid = 0.5f * (lo + hi);
    lo_e = fminf(lo, mid - SINC_HALF_MIN);
    hi_e = fmaxf(hi, mid + SINC_HALF_MIN);
    const float tke = __fadd_rd(lo_e, MAGIC);
    k0 = tke - MAGIC;
    kabs0 = kb + (__float_as_int(tke) - MAGIC_BITS) - bin0;
    return hi_e - lo_e <= span && kabs0 >= 3 && kabs0 + 5 <= k.nr - 1;
}

template <int INTERP>
__device__ __forceinline__ PulseState pulse_setup(const BpConst& k, const Record& rec,
                                                  const float4* row, float jf)
{
    if (on_heights(INTERP)) {
        // height map: the row's range expansion (MODE_GATHER) or the float64 path
        PulseState st;
        const int kind = __float_as_int(rec.d.w);
        st.mode = kind == REC_FAST ? MODE_GATHER : (kind == REC_EXACT ? MODE_EXACT : MODE_SKIP);
        return st;
    }
    // u(i) = E0 + i E1 + i^2 E2 for this thread's row j; the large c01 j term
    // is split into an integer (folded into the row index) and a fraction
    const float4 ra = rec.a, rb = rec.b, rc = rec.c, rd = rec.d;
    const float hi = ra.y * jf;
    float lo = fmaf(ra.y, jf, -hi);
    lo = fmaf(ra.z, jf, lo);
    // polynomials in the row offset jf by Horner's rule (only jf stays live)
    const float small = fmaf(jf * jf, fmaf(jf, fmaf(jf, rb.y, rb.x), ra.w), ra.x + lo);
    const float t = hi + MAGIC;
    const float hir = t - MAGIC;
    const float e0 = (hi - hir) + small;
    const float e1 = fmaf(jf, fmaf(jf, fmaf(jf, rc.y, rc.x), rb.w), rb.z);
    const float e2 = fmaf(jf, fmaf(jf, rd.x, rc.w), rc.z);
    const int kb = __float_as_int(rd.z) + (__float_as_int(t) - MAGIC_BITS);
    const int kind = __float_as_int(rd.w);

    // Bounds of u over the thread's pixels; when they span less than one bin,
    // every pixel lies in bin k0 or k0 + 1 and two table entries serve all.
    constexpr float half = 0.5f * (TILE_X - 1);
    const float lo_u = e0 - half * fabsf(e1) - half * half * fmaxf(-e2, 0.0f);
    const float hi_u = e0 + half * fabsf(e1) + half * half * fmaxf(e2, 0.0f);
    const float tk = __fadd_rd(lo_u, MAGIC);
    const float k0 = tk - MAGIC;
    const int idx0 = kb + (__float_as_int(tk) - MAGIC_BITS);
    const int bin0 = __float_as_int(rd.y);               // row index of absolute bin 0
    // both bins must hold recorded samples: the identity behind the hinge
    // form does not hold across the zero entries outside 0 <= k <= nr - 2
    const bool hinge = INTERP == INTERP_LINEAR && kind == REC_FAST && hi_u - k0 < 2.0f &&
                       (unsigned)(idx0 - bin0) <= (unsigned)(k.nr - 3);
    PulseState st;
    st.mode = kind == REC_FAST ? (hinge ? MODE_HINGE : MODE_GATHER)
                               : (kind == REC_EXACT ? MODE_EXACT : MODE_SKIP);
    if (is_sinc(INTERP) && kind == REC_FAST) {
        // windowed sinc: when the thread's pixels span at most SINC_SPAN bins
        // (SINC_SPAN6 in the wide kernel) and the stencils of bins k0 and k0 + 1
        // lie inside the recorded range, the interpolated echo is one polynomial
        // in u, of a degree chosen by the span
        constexpr float widest = INTERP == INTERP_SINC8_WIDE ? SINC_SPAN6 : SINC_SPAN;
        float lo_e, hi_e, k0e;
        int kabs0;
        if (poly_interval(k, kb, bin0, lo_u, hi_u, widest, lo_e, hi_e, k0e, kabs0)) {
            const float sp = hi_e - lo_e;
            st.mode = sp <= SINC_SPAN2 ? MODE_POLY2 : (sp <= SINC_SPAN3 ? MODE_POLY3 : MODE_POLY);
            if (INTERP == INTERP_SINC8_WIDE && sp > SINC_SPAN)
                st.mode = sp <= SINC_SPAN5 ? MODE_POLY5 : MODE_POLY6;
            st.t0 = make_float4(lo_e, hi_e, k0e, __int_as_float(kabs0));
        }
    }
    if (st.mode != MODE_POLY && st.mode != MODE_POLY3 && st.mode != MODE_POLY2 &&
        st.mode != MODE_POLY5 && st.mode != MODE_POLY6)
        st.t0 = make_float4(0.f, 0.f, 0.f, 0.f);
    st.t1d = make_float2(0.f, 0.f);
    float kn = 0.0f;
    if (INTERP == INTERP_NEAREST && kind == REC_FAST) {
        // nearest sample: when every pixel rounds to bin kn or kn + 1, one table
        // entry (N_kn, M_kn) serves the thread (the fast path's pixels lie
        // inside the row, so entry kn does too)
        const float tkn = __fadd_rd(lo_u + 0.5f, MAGIC);
        kn = tkn - MAGIC;
        const int idxn = kb + (__float_as_int(tkn) - MAGIC_BITS);
        if (hi_u + 0.5f - kn < 2.0f) {
            st.mode = MODE_PAIR;
            st.t0 = __ldg(row + idxn);
        }
    }
    if (hinge) {
        st.t0 = __ldg(row + idx0 + 1);
        st.t1d = __ldg(reinterpret_cast<const float2*>(row + idx0) + 1);
        const float c = k.c_phase;
        const float v0 = c * ((e0 - k0) - 1.0f), w1 = c * e1, w2 = c * e2;
        st.q0 = make_float2(v0, v0);
        st.q1 = make_float2(w1, w1);
        st.q2 = make_float2(w2, w2);
    } else if (INTERP == INTERP_NEAREST && st.mode == MODE_PAIR) {
        // phase from the bin boundary kn + 1/2: x = c (u - kn - 1/2)
        const float c = k.c_phase;
        const float v0 = c * ((e0 - kn) - 0.5f), w1 = c * e1, w2 = c * e2;
        st.q0 = make_float2(v0, v0);
        st.q1 = make_float2(w1, w1);
        st.q2 = make_float2(w2, w2);
    } else {
        st.q0 = make_float2(e0, e0);
        st.q1 = make_float2(e1, e1);
        st.q2 = make_float2(e2, e2);
    }
    st.kb = kb;
    st.bin0 = bin0;
    return st;
}

// All pixels in bins k0, k0 + 1. With y = c (u - k0 - 1) in [-c, c), a pixel in
// bin k0 + 1 contributes exp(j y) (A1 + y D1) (entry k0 + 1 = (A1, D1)), one in
// bin k0 contributes exp(j y) (A1 + y B), B = exp(j c) D0 (D0 from entry k0;
// the two lines meet at y = 0 since psi_k0+1 = psi_k0 exp(j c)). So the
// interpolated, phase-compensated sample is
//   exp(j y) [A1 + y (D1 + B) / 2 + |y| (D1 - B) / 2].
__device__ __forceinline__ void hinge_pulse(const BpConst& k, const PulseState& st,
                                            float2 (&accre)[NP], float2 (&accim)[NP])
{
    // B = conj(r) D0 with r = exp(-j c) (the hinge FMA form of the height-map
    // kernel schedules worse here)
    const float bre = k.rot_re * st.t1d.x + k.rot_im * st.t1d.y;
    const float bim = k.rot_re * st.t1d.y - k.rot_im * st.t1d.x;
    const float d_re = 0.5f * (st.t0.z + bre), d_im = 0.5f * (st.t0.w + bim);
    const float g_re = 0.5f * (st.t0.z - bre), g_im = 0.5f * (st.t0.w - bim);
    const float2 are = make_float2(st.t0.x, st.t0.x), aim = make_float2(st.t0.y, st.t0.y);
    const float2 dre = make_float2(d_re, d_re), dim = make_float2(d_im, d_im);
    const float2 gre = make_float2(g_re, g_re), gim = make_float2(g_im, g_im);
    const float2 one = make_float2(1.0f, 1.0f);
    float2 id = make_float2(k.i0, k.i0 + NP);    // pixel offsets of pair 0 (runtime: no constant pairs)
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        const float2 y = __ffma2_rn(id, __ffma2_rn(id, st.q2, st.q1), st.q0);
        id = __fadd2_rn(id, one);
        const float2 ay = make_float2(fabsf(y.x), fabsf(y.y));
        const float2 wr = __ffma2_rn(ay, gre, __ffma2_rn(y, dre, are));
        const float2 wi = __ffma2_rn(ay, gim, __ffma2_rn(y, dim, aim));
        float sa, ca, sb, cb;
        __sincosf(y.x, &sa, &ca);
        __sincosf(y.y, &sb, &cb);
        const float2 cs = make_float2(ca, cb);
        const float2 sn = make_float2(sa, sb);
        accre[q] = __ffma2_rn(wr, cs, accre[q]);
        accim[q] = __ffma2_rn(wr, sn, __ffma2_rn(wi, cs, accim[q]));
        accre[q] = __ffma2_rn(make_float2(-wi.x, -wi.y), sn, accre[q]);
    }
}

__device__ __forceinline__ float4 gather(unsigned long long base, float biased_index)
{
    return __ldg(reinterpret_cast<const float4*>(
        base + (unsigned long long)(unsigned)__float_as_int(biased_index) * 16ull));
}

// General case: one gather per pixel.
__device__ __forceinline__ void gather_pulse(const BpConst& k, const PulseState& st, const float4* row,
                                             float2 (&accre)[NP], float2 (&accim)[NP])
{
    // row pointer + (kb - magic bias) entries, in bytes: adding the biased
    // float bits of floor(u) + MAGIC gives the entry of bin kb + floor(u)
    const unsigned long long base = reinterpret_cast<unsigned long long>(row) +
                                    (unsigned long long)(long long)(st.kb - MAGIC_BITS) * 16ull;
    const float2 mm = make_float2(MAGIC, MAGIC);
    const float2 nmm = make_float2(-MAGIC, -MAGIC);
    const float2 neg1 = make_float2(-1.0f, -1.0f);
    const float2 cc = make_float2(k.c_phase, k.c_phase);
    const float2 one = make_float2(1.0f, 1.0f);
    float2 id = make_float2(k.i0, k.i0 + NP);
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        const float2 u = __ffma2_rn(id, __ffma2_rn(id, st.q2, st.q1), st.q0);
        id = __fadd2_rn(id, one);
        const float2 tt = __fadd2_rd(u, mm);        // floor(u) + MAGIC: the index in the mantissa
        const float2 fl = __fadd2_rn(tt, nmm);      // floor(u), exact
        const float2 f = __ffma2_rn(fl, neg1, u);   // u - floor(u), exact
        const float2 x = __fmul2_rn(f, cc);         // phase inside the bin, radians
        const float4 va = gather(base, tt.x);
        const float4 vb = gather(base, tt.y);
        float sa, ca, sb, cb;
        __sincosf(x.x, &sa, &ca);
        __sincosf(x.y, &sb, &cb);
        const float2 wr = make_float2(fmaf(x.x, va.z, va.x), fmaf(x.y, vb.z, vb.x));
        const float2 wi = make_float2(fmaf(x.x, va.w, va.y), fmaf(x.y, vb.w, vb.y));
        const float2 c = make_float2(ca, cb);
        const float2 s = make_float2(sa, sb);
        accre[q] = __ffma2_rn(wr, c, accre[q]);
        accim[q] = __ffma2_rn(wr, s, __ffma2_rn(wi, c, accim[q]));
        accre[q] = __ffma2_rn(make_float2(-wi.x, -wi.y), s, accre[q]);
    }
}

// Fallback when the tile polynomial is not accurate enough (near field, very
// fine range bins): a float64 range to the centre of the thread's own row,
// then R - R_row = s / (R_row + R), s = 2 v.q + |q|^2, in float32 over the
// row's +-15.5 pixels, with explicit bounds on every table index.
__device__ __forceinline__ void exact_pulse(const BpConst& k, const Record& rec, const float4* row,
                                            const double* __restrict__ a, double xc, double yrow,
                                            float2 (&accre)[NP], float2 (&accim)[NP])
{
    const double vx = xc - a[0], vy = yrow - a[1], vz = k.z0 - a[2];
    const double r2 = vx * vx + vy * vy + vz * vz;
    const double r = sqrt(r2);
    const double u = (r - k.r0) * k.inv_dr;
    if (!(fabs(u) < 1.0e9))
        return;
    const double ku = floor(u);
    const int kbase = (int)ku + __float_as_int(rec.d.y);  // row index of the bin below u(0)
    const float frac0 = (float)(u - ku);
    const float two_vx = (float)(2.0 * vx), rf = (float)r, r2f = (float)r2;
    const float c_phase = k.c_phase;
#pragma unroll
    for (int m = 0; m < TILE_X; ++m) {
        const float qx = ((float)m - 0.5f * (TILE_X - 1)) * k.dx_f;
        const float s = qx * (two_vx + qx);
        const float rp = sqrtf(fmaxf(r2f + s, 0.0f));
        const float den = rf + rp;
        const float dr_m = den > 0.0f ? s / den : 0.0f;
        const float ub = fmaf(dr_m, k.inv_dr_f, frac0);
        if (!(ub > -1.0e6f && ub < 1.0e6f))
            continue;
        const float kf = floorf(ub);
        const int kr = kbase + (int)kf;
        if (kr < 0 || kr > k.W - 1)
            continue;                       // outside the row: no recorded echo there
        const float x = (ub - kf) * c_phase;
        const float4 v = __ldg(row + kr);
        const float wr = fmaf(x, v.z, v.x);
        const float wi = fmaf(x, v.w, v.y);
        float sn, cs;
        __sincosf(x, &sn, &cs);
        float& re = (m < NP) ? accre[m % NP].x : accre[m % NP].y;
        float& im = (m < NP) ? accim[m % NP].x : accim[m % NP].y;
        re = fmaf(wr, cs, fmaf(-wi, sn, re));
        im = fmaf(wr, sn, fmaf(wi, cs, im));
    }
}

// ---------------------------------------------------------------------------
// Windowed-sinc interpolation (8 taps, k-3 .. k+4).
//
// The echo at range u = k + f is psi(u) G(u), G(u) = sum_m e_m h(u - m),
// psi(u) = psi_k exp(j c f). On each bin G is a fixed combination of the
// bin's eight samples with weights h(f - d), d = -3 .. 4; the table kernel
// stores it as a degree-7 polynomial in s = f - 1/2 (each weight interpolated
// at eight Chebyshev nodes of the bin, fit_sinc_taps), so a value of G costs
// four loads and seven packed FMAs.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// G at s = f - 1/2 from the four coefficient entries of its bin.
__device__ __forceinline__ float2 bin_poly(const float4* c, float s)
{
    const float4 c0 = __ldg(c), c1 = __ldg(c + 1), c2 = __ldg(c + 2), c3 = __ldg(c + 3);
    const float2 sv = make_float2(s, s);
    float2 g = __ffma2_rn(make_float2(c3.z, c3.w), sv, make_float2(c3.x, c3.y));
    g = __ffma2_rn(g, sv, make_float2(c2.z, c2.w));
    g = __ffma2_rn(g, sv, make_float2(c2.x, c2.y));
    g = __ffma2_rn(g, sv, make_float2(c1.z, c1.w));
    g = __ffma2_rn(g, sv, make_float2(c1.x, c1.y));
    g = __ffma2_rn(g, sv, make_float2(c0.z, c0.w));
    return __ffma2_rn(g, sv, make_float2(c0.x, c0.y));
}

// One pixel at row position ub (relative to row index kb). CHECK_ROW adds
// bounds on the table row for the exact path.
template <bool CHECK_ROW>
__device__ __forceinline__ void sinc_pixel(const BpConst& k, float ub, int kb, int bin0,
                                           const float4* row, const float2* __restrict__ psi,
                                           float& re, float& im)
{
    if (CHECK_ROW && !(ub > -1.0e6f && ub < 1.0e6f))
        return;
    const float tt = __fadd_rd(ub, MAGIC);
    const float f = ub - (tt - MAGIC);
    const int kr = kb + (__float_as_int(tt) - MAGIC_BITS);
    const int kabs = kr - bin0;
    if (kabs < 3 || kabs > k.nr - 5)
        return;                                 // stencil reaches outside the recorded range
    if (CHECK_ROW && (kr < 0 || kr > k.W - 1))
        return;
    const float2 ps = __ldg(psi + kabs);
    const float2 gsum = bin_poly(row + 4 * kr, f - 0.5f);
    float sn, cs;
    __sincosf(f * k.c_phase, &sn, &cs);
    const float zr = ps.x * cs - ps.y * sn;
    const float zi = ps.x * sn + ps.y * cs;
    re = fmaf(gsum.x, zr, fmaf(-gsum.y, zi, re));
    im = fmaf(gsum.x, zi, fmaf(gsum.y, zr, im));
}

// Windowed-sinc interpolant G(u) = sum_m e_m h(u - m) at one position ub
// (row units, relative to kb), no phase. Its bin must lie inside the row.
__device__ __forceinline__ float2 sinc_value(float ub, int kb, const float4* row)
{
    const float tt = __fadd_rd(ub, MAGIC);
    const float s = (ub - (tt - MAGIC)) - 0.5f;
    const int kr = kb + (__float_as_int(tt) - MAGIC_BITS);
    return bin_poly(row + 4 * kr, s);
}

// Complex a x + b y, with real weights a, b.
__device__ __forceinline__ float2 cmix3(float a, float2 x, float b, float2 y, float c, float2 z)
{
    return make_float2(fmaf(a, x.x, fmaf(b, y.x, c * z.x)), fmaf(a, x.y, fmaf(b, y.y, c * z.y)));
}
__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }

// Monomial coefficients p[n] (complex, in t = (u - mid) / half) of the
// interpolant of G on [mid - half, mid + half] at the NN Chebyshev nodes
// mid + half cos((2i + 1) pi / (2 NN)) (degree NN - 1, NN = 3 .. 7), by the
// inverse Vandermonde matrix. The nodes are symmetric about mid, so the even
// coefficients come from the sums g_i + g_(NN-1-i) and the odd ones from the
// differences; for NN = 6 and 7 the weights are the inverses of those
// halves' Vandermonde matrices, in float64 and rounded once.
template <int NN>
__device__ __forceinline__ void poly_coeffs(float mid, float half, int kb, const float4* row,
                                            float2 (&p)[SINC_MAXC])
{
    if (NN == 6) {
        constexpr float C1 = 0.965925826f, C2 = 0.707106781f, C3 = 0.258819045f;
        const float2 g0 = sinc_value(fmaf(half, C1, mid), kb, row);
        const float2 g5 = sinc_value(fmaf(half, -C1, mid), kb, row);
        const float2 g1 = sinc_value(fmaf(half, C2, mid), kb, row);
        const float2 g4 = sinc_value(fmaf(half, -C2, mid), kb, row);
        const float2 g2 = sinc_value(fmaf(half, C3, mid), kb, row);
        const float2 g3 = sinc_value(fmaf(half, -C3, mid), kb, row);
        const float2 s0 = cadd(g0, g5), s1 = cadd(g1, g4), s2 = cadd(g2, g3);
        const float2 d0 = csub(g0, g5), d1 = csub(g1, g4), d2 = csub(g2, g3);
        p[0] = cmix3(0.0446581987f, s0, -0.166666667f, s1, 0.622008468f, s2);
        p[2] = cmix3(-0.755983064f, s0, 2.66666667f, s1, -1.91068360f, s2);
        p[4] = cmix3(1.33333333f, s0, -2.66666667f, s1, 1.33333333f, s2);
        p[1] = cmix3(0.0462335694f, d0, -0.235702260f, d1, 2.40325617f, d2);
        p[3] = cmix3(-0.782651259f, d0, 3.77123617f, d1, -7.38231455f, d2);
        p[5] = cmix3(1.38036824f, d0, -3.77123617f, d1, 5.15160441f, d2);
        p[6] = make_float2(0.0f, 0.0f);
        return;
    }
    if (NN == 7) {
        constexpr float C1 = 0.974927912f, C2 = 0.781831482f, C3 = 0.433883739f;
        const float2 g0 = sinc_value(fmaf(half, C1, mid), kb, row);
        const float2 g6 = sinc_value(fmaf(half, -C1, mid), kb, row);
        const float2 g1 = sinc_value(fmaf(half, C2, mid), kb, row);
        const float2 g5 = sinc_value(fmaf(half, -C2, mid), kb, row);
        const float2 g2 = sinc_value(fmaf(half, C3, mid), kb, row);
        const float2 g4 = sinc_value(fmaf(half, -C3, mid), kb, row);
        const float2 g3 = sinc_value(mid, kb, row);
        // even part: (s_i / 2 - g3) against [t^2 t^4 t^6]; odd: d_i / 2 against [t t^3 t^5]
        const float2 s0 = make_float2(fmaf(0.5f, g0.x + g6.x, -g3.x), fmaf(0.5f, g0.y + g6.y, -g3.y));
        const float2 s1 = make_float2(fmaf(0.5f, g1.x + g5.x, -g3.x), fmaf(0.5f, g1.y + g5.y, -g3.y));
        const float2 s2 = make_float2(fmaf(0.5f, g2.x + g4.x, -g3.x), fmaf(0.5f, g2.y + g4.y, -g3.y));
        const float2 d0 = csub(g0, g6), d1 = csub(g1, g5), d2 = csub(g2, g4);
        p[0] = g3;
        p[2] = cmix3(0.468226361f, s0, -2.04001350f, s1, 9.57178714f, s2);
        p[4] = cmix3(-3.25319224f, s0, 12.9827197f, s1, -25.7295275f, s2);
        p[6] = cmix3(4.06895422f, s0, -11.4009564f, s1, 16.4748593f, s2);
        p[1] = cmix3(0.228243474f, d0, -0.797473389f, d1, 2.07652140f, d2);
        p[3] = cmix3(-1.58581396f, d0, 5.07514951f, d1, -5.58181180f, d2);
        p[5] = cmix3(1.98346852f, d0, -4.45681331f, d1, 3.57408678f, d2);
        return;
    }
    if (NN == 3) {
        constexpr float C1 = 0.866025404f;                       // cos(pi/6)
        const float2 g0 = sinc_value(fmaf(half, C1, mid), kb, row);
        const float2 g1 = sinc_value(mid, kb, row);
        const float2 g2 = sinc_value(fmaf(half, -C1, mid), kb, row);
        p[0] = g1;
        p[1] = make_float2(0.577350269f * (g0.x - g2.x), 0.577350269f * (g0.y - g2.y));
        p[2] = make_float2(0.666666667f * (g0.x + g2.x - 2.0f * g1.x),
                           0.666666667f * (g0.y + g2.y - 2.0f * g1.y));
        p[3] = p[4] = p[5] = p[6] = make_float2(0.0f, 0.0f);
        return;
    }
    if (NN == 4) {
        constexpr float C1 = 0.923879533f, C2 = 0.382683432f;   // cos(pi/8), cos(3 pi/8)
        const float2 g0 = sinc_value(fmaf(half, C1, mid), kb, row);
        const float2 g1 = sinc_value(fmaf(half, C2, mid), kb, row);
        const float2 g2 = sinc_value(fmaf(half, -C2, mid), kb, row);
        const float2 g3 = sinc_value(fmaf(half, -C1, mid), kb, row);
        const float2 s03 = make_float2(g0.x + g3.x, g0.y + g3.y), d03 = make_float2(g0.x - g3.x, g0.y - g3.y);
        const float2 s12 = make_float2(g1.x + g2.x, g1.y + g2.y), d12 = make_float2(g1.x - g2.x, g1.y - g2.y);
        p[0] = make_float2(fmaf(-0.103553391f, s03.x, 0.603553391f * s12.x),
                           fmaf(-0.103553391f, s03.y, 0.603553391f * s12.y));
        p[1] = make_float2(fmaf(-0.112085382f, d03.x, 1.577161015f * d12.x),
                           fmaf(-0.112085382f, d03.y, 1.577161015f * d12.y));
        p[2] = make_float2(0.707106781f * (s03.x - s12.x), 0.707106781f * (s03.y - s12.y));
        p[3] = make_float2(fmaf(0.765366865f, d03.x, -1.847759065f * d12.x),
                           fmaf(0.765366865f, d03.y, -1.847759065f * d12.y));
        p[4] = p[5] = p[6] = make_float2(0.0f, 0.0f);
        return;
    }
    constexpr float C1 = 0.951056516f, C2 = 0.587785252f;   // cos(pi/10), cos(3 pi/10)
    const float2 g0 = sinc_value(fmaf(half, C1, mid), kb, row);
    const float2 g1 = sinc_value(fmaf(half, C2, mid), kb, row);
    const float2 g2 = sinc_value(mid, kb, row);
    const float2 g3 = sinc_value(fmaf(half, -C2, mid), kb, row);
    const float2 g4 = sinc_value(fmaf(half, -C1, mid), kb, row);
    const float2 s04 = make_float2(g0.x + g4.x, g0.y + g4.y), d04 = make_float2(g0.x - g4.x, g0.y - g4.y);
    const float2 s13 = make_float2(g1.x + g3.x, g1.y + g3.y), d13 = make_float2(g1.x - g3.x, g1.y - g3.y);
    p[0] = g2;
    p[1] = make_float2(fmaf(1.376381920f, d13.x, -0.324919696f * d04.x),
                       fmaf(1.376381920f, d13.y, -0.324919696f * d04.y));
    p[2] = make_float2(fmaf(-0.341640786f, s04.x, fmaf(2.341640786f, s13.x, -4.0f * g2.x)),
                       fmaf(-0.341640786f, s04.y, fmaf(2.341640786f, s13.y, -4.0f * g2.y)));
    p[3] = make_float2(fmaf(0.940456404f, d04.x, -1.521690426f * d13.x),
                       fmaf(0.940456404f, d04.y, -1.521690426f * d13.y));
    p[4] = make_float2(fmaf(0.988854382f, s04.x, fmaf(-2.588854382f, s13.x, 3.2f * g2.x)),
                       fmaf(0.988854382f, s04.y, fmaf(-2.588854382f, s13.y, 3.2f * g2.y)));
    p[5] = p[6] = make_float2(0.0f, 0.0f);
}

// frac(2 r_k / lambda) of absolute bin k, in turns: the phase of psi_k from the
// same 64-bit fixed-point accumulator the table kernel uses.
__device__ __forceinline__ float bin_turns(const BpConst& k, int kabs)
{
    const unsigned long long ph = k.beta_fx + k.alpha_fx * (unsigned long long)(long long)kabs;
    return (float)(ph >> 40) * 0x1p-24f;
}

// The coefficients in s = u - mid, p[n] / half^n, in both lanes of the pairs pr
// (real parts) and pi (imaginary parts).
template <int ND>
__device__ __forceinline__ void poly_scale(const float2 (&p)[SINC_MAXC], float half,
                                           float2 (&pr)[SINC_MAXC], float2 (&pi)[SINC_MAXC])
{
    const float ih = rcp_approx(half);            // half >= SINC_HALF_MIN
    float sc = 1.0f;
#pragma unroll
    for (int n = 0; n < ND; ++n) {
        const float re = p[n].x * sc, im = p[n].y * sc;
        pr[n] = make_float2(re, re);
        pi[n] = make_float2(im, im);
        sc *= ih;
    }
}

// The per-pixel part of the polynomial modes: lane .x of every pixel pair
// (the left 16 pixels) evaluates the .x coefficients about midL, lane .y (the
// right 16) the .y coefficients about midR, each with the echo phase
// psi_k0 exp(j c (u - k0)) = exp(j (c (u - mid) + cm)) of its own k0, with
// cm = c (mid - k0) + arg psi_k0.
template <int ND, int Q0 = 0, int NQ = NP>
__device__ __forceinline__ void sinc_poly_apply(const BpConst& k, const PulseState& st,
                                                const float2 (&pr)[SINC_MAXC],
                                                const float2 (&pi)[SINC_MAXC],
                                                float midL, float midR, float cmL, float cmR,
                                                float2 (&accre)[NP], float2 (&accim)[NP])
{
    const float c = k.c_phase;
    const float2 c2 = make_float2(c, c);
    const float2 cm2 = make_float2(cmL, cmR);
    const float2 q0s = make_float2(st.q0.x - midL, st.q0.x - midR);
    const float2 one = make_float2(1.0f, 1.0f);
    float2 id = make_float2(k.i0 + Q0, k.i0 + (NP + Q0));
#pragma unroll
    for (int q = Q0; q < Q0 + NQ; ++q) {
        const float2 sv = __ffma2_rn(id, __ffma2_rn(id, st.q2, st.q1), q0s);
        id = __fadd2_rn(id, one);
        float2 gr = pr[ND - 1], gi = pi[ND - 1];
#pragma unroll
        for (int n = ND - 2; n >= 0; --n) {
            gr = __ffma2_rn(gr, sv, pr[n]);
            gi = __ffma2_rn(gi, sv, pi[n]);
        }
        const float2 x = __ffma2_rn(sv, c2, cm2);
        float sa, ca, sb, cb;
        __sincosf(x.x, &sa, &ca);
        __sincosf(x.y, &sb, &cb);
        const float2 cs = make_float2(ca, cb);
        const float2 sn = make_float2(sa, sb);
        accre[q] = __ffma2_rn(gr, cs, accre[q]);
        accim[q] = __ffma2_rn(gr, sn, __ffma2_rn(gi, cs, accim[q]));
        accre[q] = __ffma2_rn(make_float2(-gi.x, -gi.y), sn, accre[q]);
    }
}

// All of the thread's pixels within SINC_SPAN bins, every stencil inside the
// recorded range. Within a bin G(u) is smooth (a sum of eight windowed sincs);
// where a tap enters or leaves the stencil (a bin boundary) the Hann taper
// makes G twice continuously differentiable. Over the interval [lo_u, hi_u]
// (widened to a half-width of at least SINC_HALF_MIN) G is interpolated at the
// five Chebyshev nodes mid + half cos((2i+1) pi / 10) by a degree-4 polynomial
// in t = (u - mid) / half, evaluated per pixel as a polynomial in s = u - mid.
// Inside one bin the error is at most max|G^(5)| half^5 / (2^4 5!), and
// |G^(n)| <= max|e| max_f sum_d |h^(n)(f - d)|, which is 312 max|e| for n = 5
// and 98 max|e| for n = 4 with this window (against 8 pi^n for a bare bound);
// so half <= 0.17 gives at most 2.3e-5 max|e|. Spans of at most SINC_SPAN3
// take the cubic on the four nodes mid + half cos((2i+1) pi / 8) instead
// (NN = 4): error at most 98 max|e| half^4 / (2^3 4!) <= 2.7e-5 max|e| for
// half <= 0.085, one node evaluation and two packed FMAs per pixel pair fewer;
// spans of at most SINC_SPAN2 the quadratic on mid, mid +- half cos(pi / 6)
// (NN = 3): at most 31 max|e| half^3 / (2^2 3!) <= 2.0e-5 max|e| for
// half <= 0.025 (the third derivative is bounded on both sides of a bin
// boundary, so this bound also holds across one).
// Intervals across a bin boundary, where the bound does not apply, measure no
// worse on random samples (at most 3.3e-5 max|e| at these spans). The echo
// phase exp(j 4 pi R / lambda) = psi_k0 exp(j c (u - k0)) is applied per
// pixel as one angle, c (u - k0) + 2 pi frac(2 r_k0 / lambda).
template <int NN>
__device__ __forceinline__ void sinc_poly_pulse(const BpConst& k, const PulseState& st,
                                                const float4* row, const float2* __restrict__ psi,
                                                float2 (&accre)[NP], float2 (&accim)[NP])
{
    const float lo_u = st.t0.x, hi_u = st.t0.y, k0 = st.t0.z;
    const int kabs0 = __float_as_int(st.t0.w);
    const float mid = 0.5f * (lo_u + hi_u), half = 0.5f * (hi_u - lo_u);
    float2 p[SINC_MAXC], pr[SINC_MAXC], pi[SINC_MAXC];
    poly_coeffs<NN>(mid, half, st.kb, row, p);
    poly_scale<NN>(p, half, pr, pi);
    constexpr float TWO_PI = 6.283185307f;
    const float cm = fmaf(TWO_PI, bin_turns(k, kabs0), k.c_phase * (mid - k0));
    sinc_poly_apply<NN>(k, st, pr, pi, mid, mid, cm, cm, accre, accim);
}

// Any span: the 8 taps evaluated per pixel.
__device__ __forceinline__ void sinc_pulse(const BpConst& k, const PulseState& st, const float4* row,
                                           const float2* __restrict__ psi,
                                           float2 (&accre)[NP], float2 (&accim)[NP])
{
    const float e0 = st.q0.x, e1 = st.q1.x, e2 = st.q2.x;
#pragma unroll
    for (int m = 0; m < TILE_X; ++m) {
        const float i = k.i0 + (float)m;
        const float ub = fmaf(i, fmaf(i, e2, e1), e0);
        float& re = (m < NP) ? accre[m % NP].x : accre[m % NP].y;
        float& im = (m < NP) ? accim[m % NP].x : accim[m % NP].y;
        sinc_pixel<false>(k, ub, st.kb, st.bin0, row, psi, re, im);
    }
}

__device__ __forceinline__ void sinc_exact_pulse(const BpConst& k, const Record& rec, const float4* row,
                                                 const double* __restrict__ a, double xc,
                                                 double yrow, const float2* __restrict__ psi,
                                                 float2 (&accre)[NP], float2 (&accim)[NP])
{
    const double vx = xc - a[0], vy = yrow - a[1], vz = k.z0 - a[2];
    const double r2 = vx * vx + vy * vy + vz * vz;
    const double r = sqrt(r2);
    const double u = (r - k.r0) * k.inv_dr;
    if (!(fabs(u) < 1.0e9))
        return;
    const double ku = floor(u);
    const int bin0 = __float_as_int(rec.d.y);
    const int kbase = (int)ku + bin0;
    const float frac0 = (float)(u - ku);
    const float two_vx = (float)(2.0 * vx), rf = (float)r, r2f = (float)r2;
#pragma unroll
    for (int m = 0; m < TILE_X; ++m) {
        const float qx = ((float)m - 0.5f * (TILE_X - 1)) * k.dx_f;
        const float s = qx * (two_vx + qx);
        const float rp = sqrtf(fmaxf(r2f + s, 0.0f));
        const float den = rf + rp;
        const float dr_m = den > 0.0f ? s / den : 0.0f;
        const float ub = fmaf(dr_m, k.inv_dr_f, frac0);
        float& re = (m < NP) ? accre[m % NP].x : accre[m % NP].y;
        float& im = (m < NP) ? accim[m % NP].x : accim[m % NP].y;
        sinc_pixel<true>(k, ub, kbase, bin0, row, psi, re, im);
    }
}

// ---------------------------------------------------------------------------
// Nearest-neighbour interpolation: k = floor(u + 1/2), value e_k psi(u) with
// psi(u) = psi_k exp(j c (u - k)), u - k in [-1/2, 1/2).
// ---------------------------------------------------------------------------
template <bool CHECK_ROW>
__device__ __forceinline__ void nearest_pixel(const BpConst& k, float ub, int kb,
                                              const float4* row, float& re, float& im)
{
    if (CHECK_ROW && !(ub > -1.0e6f && ub < 1.0e6f))
        return;
    const float tt = __fadd_rd(ub + 0.5f, MAGIC);
    const float d = ub - (tt - MAGIC);                  // u - k in [-1/2, 1/2)
    const int kr = kb + (__float_as_int(tt) - MAGIC_BITS);
    if (CHECK_ROW && (kr < 0 || kr > k.W - 1))
        return;
    // N_k: zero where sample k was not recorded
    const float2 e = __ldg(reinterpret_cast<const float2*>(row) + 2 * (size_t)kr);
    float sn, cs;
    __sincosf(fmaf(d, k.c_phase, -0.5f * k.c_phase), &sn, &cs);
    re = fmaf(e.x, cs, fmaf(-e.y, sn, re));
    im = fmaf(e.x, sn, fmaf(e.y, cs, im));
}

// Every pixel rounds to bin kn or kn + 1: one table entry (N_kn, M_kn) serves
// all, since the echo phase psi_k exp(j c (u - k)) equals
// psi_kn exp(j c (u - kn)) for either k. Per pixel: the choice of sample
// (u + 1/2 >= kn + 1), the phase, the sum.
__device__ __forceinline__ void nearest_pair_pulse(const BpConst& k, const PulseState& st,
                                                   float2 (&accre)[NP], float2 (&accim)[NP])
{
    // With x = c (u - kn - 1/2) (the state's polynomial), a pixel takes sample
    // kn + 1 when x >= 0 (u + 1/2 >= kn + 1), else sample kn, and its echo is
    // (N_kn + h M_kn) exp(j x) with h = 1 or 0: one set and one packed FMA per
    // lane pair instead of compares and selects (N + M is the second sample to
    // one rounding)
    const float4 e = st.t0;
    const float w0r = e.x, w0i = e.y, w1r = e.z, w1i = e.w;
    const float2 w0r2 = make_float2(w0r, w0r), w0i2 = make_float2(w0i, w0i);
    const float2 dwr2 = make_float2(w1r, w1r), dwi2 = make_float2(w1i, w1i);
    const float2 one = make_float2(1.0f, 1.0f);
    float2 id = make_float2(k.i0, k.i0 + NP);
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        const float2 x = __ffma2_rn(id, __ffma2_rn(id, st.q2, st.q1), st.q0);
        id = __fadd2_rn(id, one);
        const float2 h = make_float2(x.x >= 0.0f ? 1.0f : 0.0f, x.y >= 0.0f ? 1.0f : 0.0f);
        const float2 wr = __ffma2_rn(h, dwr2, w0r2);
        const float2 wi = __ffma2_rn(h, dwi2, w0i2);
        float sa, ca, sb, cb;
        __sincosf(x.x, &sa, &ca);
        __sincosf(x.y, &sb, &cb);
        const float2 cs = make_float2(ca, cb);
        const float2 sn = make_float2(sa, sb);
        accre[q] = __ffma2_rn(wr, cs, accre[q]);
        accim[q] = __ffma2_rn(wr, sn, __ffma2_rn(wi, cs, accim[q]));
        accre[q] = __ffma2_rn(make_float2(-wi.x, -wi.y), sn, accre[q]);
    }
}

__device__ __forceinline__ void nearest_pulse(const BpConst& k, const PulseState& st, const float4* row,
                                              float2 (&accre)[NP], float2 (&accim)[NP])
{
    const float e0 = st.q0.x, e1 = st.q1.x, e2 = st.q2.x;
#pragma unroll
    for (int m = 0; m < TILE_X; ++m) {
        const float i = k.i0 + (float)m;
        const float ub = fmaf(i, fmaf(i, e2, e1), e0);
        float& re = (m < NP) ? accre[m % NP].x : accre[m % NP].y;
        float& im = (m < NP) ? accim[m % NP].x : accim[m % NP].y;
        nearest_pixel<false>(k, ub, st.kb, row, re, im);
    }
}

__device__ __forceinline__ void nearest_exact_pulse(const BpConst& k, const Record& rec,
                                                    const float4* row, const double* __restrict__ a,
                                                    double xc, double yrow,
                                                    float2 (&accre)[NP], float2 (&accim)[NP])
{
    const double vx = xc - a[0], vy = yrow - a[1], vz = k.z0 - a[2];
    const double r2 = vx * vx + vy * vy + vz * vz;
    const double r = sqrt(r2);
    const double u = (r - k.r0) * k.inv_dr;
    if (!(fabs(u) < 1.0e9))
        return;
    const double ku = floor(u);
    const int kbase = (int)ku + __float_as_int(rec.d.y);
    const float frac0 = (float)(u - ku);
    const float two_vx = (float)(2.0 * vx), rf = (float)r, r2f = (float)r2;
#pragma unroll
    for (int m = 0; m < TILE_X; ++m) {
        const float qx = ((float)m - 0.5f * (TILE_X - 1)) * k.dx_f;
        const float s = qx * (two_vx + qx);
        const float rp = sqrtf(fmaxf(r2f + s, 0.0f));
        const float den = rf + rp;
        const float dr_m = den > 0.0f ? s / den : 0.0f;
        const float ub = fmaf(dr_m, k.inv_dr_f, frac0);
        float& re = (m < NP) ? accre[m % NP].x : accre[m % NP].y;
        float& im = (m < NP) ? accim[m % NP].x : accim[m % NP].y;
        nearest_pixel<true>(k, ub, kbase, row, re, im);
    }
}

// ---------------------------------------------------------------------------
// Pixels on a height map.
//
// Each thread's row has a reference point: the tile-centre column of its row
// at the row's mean height h_row. Its range R_row is found in float-pair
// arithmetic (about 44 bits: error-free sums and products, Knuth and
// Dekker), so u_row = (R_row - r0) / dr is exact to ~1e-9 bins. A pixel is
// offset from it by q = (q_x, 0, h - h_row); with s = 2 v.q + |q|^2 and
// t = s / R_row^2,
//   R - R_row = (s / (2 R_row)) (1 - t/4 + t^2/8 - 5 t^3/64 + ...),
// which is used when |t| <= 0.01 for every pixel of the row (the next term
// is then below 6e-10 of the offset). Otherwise the row falls back to the
// float64 reference and an exact float32 difference per pixel.
// ---------------------------------------------------------------------------
struct HRow {
    float hrow;    // the row's reference height (mean of its pixels)
    float qm;      // largest |q| over the row's pixels
    float jy;      // row offset from the tile centre, in pixels
    float zh, zl;  // Z = hrow - mid height as a float pair
    float qq;      // Y^2 + Z^2, Y = jy dy: squared offset of the row's reference point
    float dz_lo, dz_hi;   // range of h - hrow over the row's pixels
    float p_lo, p_hi;     // range of (i dx)^2 + (h - hrow)^2
};

// The row statistics as the prologue left them in shared memory, read where
// a pulse needs them (volatile, so that they are not held in registers across
// the pulse loop).
__device__ __forceinline__ float4 lds_volatile(const float4* p)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"((unsigned)__cvta_generic_to_shared(p)));
    return v;
}
__device__ __forceinline__ HRow load_hrow(const float4* s_row)
{
    const float4 a = lds_volatile(s_row + HROW_STATS);
    const float4 b = lds_volatile(s_row + HROW_STATS + 1);
    const float4 c = lds_volatile(s_row + HROW_STATS + 2);
    return HRow{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y};
}

struct F2 {
    float hi, lo;
};

__device__ __forceinline__ F2 two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

// Returns false (and leaves the sums untouched) when the series does not apply.
// One pulse of the range series over the thread's pixels (see
// heights_series_pulse); DEG4 keeps the s^4 term.
template <int INTERP, bool DEG4>
__device__ __forceinline__ void heights_series_loop(const BpConst& k, const float4* row,
                                                    const float4* s_hp,
                                                    const float2* __restrict__ psi, int kbase,
                                                    int bin0, float frac, float ax, float two_vz, float hb,
                                                    float g, float2 (&accre)[NP],
                                                    float2 (&accim)[NP])
{
    const float2 ax2 = make_float2(ax, ax), tvz2 = make_float2(two_vz, two_vz);
    const float a1 = hb, a2 = -0.25f * hb * g, a3 = 0.125f * hb * g * g,
                a4 = -0.078125f * hb * g * g * g;
    const float2 a12 = make_float2(a1, a1), a22 = make_float2(a2, a2);
    const float2 a32 = make_float2(a3, a3), a42 = make_float2(a4, a4);
    const float2 one = make_float2(1.0f, 1.0f), neg1 = make_float2(-1.0f, -1.0f);
    const float2 f0 = make_float2(frac, frac);
    const float2 mm = make_float2(MAGIC, MAGIC), nmm = make_float2(-MAGIC, -MAGIC);
    const float2 cc = make_float2(k.c_phase, k.c_phase);
    float2 id = make_float2(k.i0, k.i0 + NP);
    const int wmax = k.W - 1;
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        const float4 hp = s_hp[q];
        const float2 s = __ffma2_rn(id, ax2, __ffma2_rn(make_float2(hp.x, hp.y), tvz2,
                                                        make_float2(hp.z, hp.w)));
        id = __fadd2_rn(id, one);
        const float2 poly = DEG4 ? __ffma2_rn(__ffma2_rn(__ffma2_rn(a42, s, a32), s, a22), s, a12)
                                 : __ffma2_rn(__ffma2_rn(a32, s, a22), s, a12);
        const float2 ub = __ffma2_rn(s, poly, f0);
        if (INTERP != INTERP_HEIGHTS) {
            // windowed sinc or nearest sample at this range, bounds checked
            if (INTERP == INTERP_HEIGHTS_SINC8) {
                sinc_pixel<true>(k, ub.x, kbase, bin0, row, psi, accre[q].x, accim[q].x);
                sinc_pixel<true>(k, ub.y, kbase, bin0, row, psi, accre[q].y, accim[q].y);
            } else {
                nearest_pixel<true>(k, ub.x, kbase, row, accre[q].x, accim[q].x);
                nearest_pixel<true>(k, ub.y, kbase, row, accre[q].y, accim[q].y);
            }
            // keep the next pair's table loads from being hoisted above this
            // pair's arithmetic: bounds the registers held in flight
            asm volatile("" ::: "memory");
            continue;
        }
        const float2 tt = __fadd2_rd(ub, mm);
        const float2 f = __ffma2_rn(__fadd2_rn(tt, nmm), neg1, ub);
        const float2 x = __fmul2_rn(f, cc);
        const int ka = min(max(kbase + (__float_as_int(tt.x) - MAGIC_BITS), 0), wmax);
        const int kb = min(max(kbase + (__float_as_int(tt.y) - MAGIC_BITS), 0), wmax);
        const float4 va = __ldg(row + ka);
        const float4 vb = __ldg(row + kb);
        float sa, ca, sb, cb;
        __sincosf(x.x, &sa, &ca);
        __sincosf(x.y, &sb, &cb);
        const float2 wr = make_float2(fmaf(x.x, va.z, va.x), fmaf(x.y, vb.z, vb.x));
        const float2 wi = make_float2(fmaf(x.x, va.w, va.y), fmaf(x.y, vb.w, vb.y));
        const float2 c = make_float2(ca, cb);
        const float2 sn = make_float2(sa, sb);
        accre[q] = __ffma2_rn(wr, c, accre[q]);
        accim[q] = __ffma2_rn(wr, sn, __ffma2_rn(wi, c, accim[q]));
        accre[q] = __ffma2_rn(make_float2(-wi.x, -wi.y), sn, accre[q]);
    }
}

// Linear interpolation when every pixel of the row lies in bins k0 and k0 + 1:
// the two-entry form of hinge_pulse with y = c (u - k0 - 1) from the range
// series (u - k0 - 1 = frac - k0 - 1 + s poly(s), folded so that y comes out
// of one FFMA). t0, t1: table entries k0, k0 + 1; y0 = c (frac - k0 - 1).
template <bool DEG4>
__device__ __forceinline__ void heights_hinge_loop(const BpConst& k, const float4* s_hp, float4 t0,
                                                   float4 t1, float y0, float ax, float two_vz,
                                                   float hb, float g, float2 (&accre)[NP],
                                                   float2 (&accim)[NP])
{
    const float c = k.c_phase;
    const float2 ax2 = make_float2(ax, ax), tvz2 = make_float2(two_vz, two_vz);
    const float a1 = c * hb, a2 = -0.25f * a1 * g, a3 = 0.125f * a1 * g * g,
                a4 = -0.078125f * a1 * g * g * g;
    const float2 a12 = make_float2(a1, a1), a22 = make_float2(a2, a2);
    const float2 a32 = make_float2(a3, a3), a42 = make_float2(a4, a4);
    const float2 y02 = make_float2(y0, y0);
    // B / 2 = exp(j c) D0 / 2 (half the rotation from the constants), then the
    // line and hinge slopes (D1 +- B) / 2 in one FMA each: the same bits as
    // halving the sums
    const float bre = k.hrt_re * t0.z + k.hrt_im * t0.w;
    const float bim = k.hrt_re * t0.w - k.hrt_im * t0.z;
    const float d_re = fmaf(0.5f, t1.z, bre), d_im = fmaf(0.5f, t1.w, bim);
    const float gre = fmaf(0.5f, t1.z, -bre), gim = fmaf(0.5f, t1.w, -bim);
    const float2 are = make_float2(t1.x, t1.x), aim = make_float2(t1.y, t1.y);
    const float2 dre = make_float2(d_re, d_re), dim = make_float2(d_im, d_im);
    const float2 g_re = make_float2(gre, gre), g_im = make_float2(gim, gim);
    const float2 one = make_float2(1.0f, 1.0f);
    float2 id = make_float2(k.i0, k.i0 + NP);
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        const float4 hp = s_hp[q];
        const float2 s = __ffma2_rn(id, ax2, __ffma2_rn(make_float2(hp.x, hp.y), tvz2,
                                                        make_float2(hp.z, hp.w)));
        id = __fadd2_rn(id, one);
        const float2 poly = DEG4 ? __ffma2_rn(__ffma2_rn(__ffma2_rn(a42, s, a32), s, a22), s, a12)
                                 : __ffma2_rn(__ffma2_rn(a32, s, a22), s, a12);
        const float2 y = __ffma2_rn(s, poly, y02);
        const float2 ay = make_float2(fabsf(y.x), fabsf(y.y));
        const float2 wr = __ffma2_rn(ay, g_re, __ffma2_rn(y, dre, are));
        const float2 wi = __ffma2_rn(ay, g_im, __ffma2_rn(y, dim, aim));
        float sa, ca, sb, cb;
        __sincosf(y.x, &sa, &ca);
        __sincosf(y.y, &sb, &cb);
        const float2 cs = make_float2(ca, cb);
        const float2 sn = make_float2(sa, sb);
        accre[q] = __ffma2_rn(wr, cs, accre[q]);
        accim[q] = __ffma2_rn(wr, sn, __ffma2_rn(wi, cs, accim[q]));
        accre[q] = __ffma2_rn(make_float2(-wi.x, -wi.y), sn, accre[q]);
    }
}

// Windowed sinc on a height map when the row's pixels span at most SINC_SPAN6
// bins: G is interpolated over [lo, hi] (row units, relative to kb) at NN
// Chebyshev nodes as in the planar polynomial modes (same degrees, spans and
// error bounds), and each pixel evaluates it at s_v = u - mid from the range
// series; the echo phase is psi_k0 exp(j c (u - k0)), one angle per pixel.
// a4 is the series' s^4 coefficient, or 0 where that term is left out.
template <int NN>
__device__ __forceinline__ void heights_sinc_poly(const BpConst& k, const float4* s_hp,
                                                  const float4* row, int kb, float lo, float hi,
                                                  float k0, int kabs0, float frac, float ax,
                                                  float two_vz, float hb, float g, float a4,
                                                  float2 (&accre)[NP], float2 (&accim)[NP])
{
    const float mid = 0.5f * (lo + hi), half = 0.5f * (hi - lo);
    float2 p[SINC_MAXC], pr[SINC_MAXC], pi[SINC_MAXC];
    poly_coeffs<NN>(mid, half, kb, row, p);
    poly_scale<NN>(p, half, pr, pi);
    constexpr float TWO_PI = 6.283185307f;
    const float cm = fmaf(TWO_PI, bin_turns(k, kabs0), k.c_phase * (mid - k0));
    const float2 c2 = make_float2(k.c_phase, k.c_phase), cm2 = make_float2(cm, cm);
    const float2 ax2 = make_float2(ax, ax), tvz2 = make_float2(two_vz, two_vz);
    const float a2 = -0.25f * hb * g, a3 = 0.125f * hb * g * g;
    const float2 a12 = make_float2(hb, hb), a22 = make_float2(a2, a2);
    const float2 a32 = make_float2(a3, a3), a42 = make_float2(a4, a4);
    const float2 f0 = make_float2(frac - mid, frac - mid);
    const float2 one = make_float2(1.0f, 1.0f);
    float2 id = make_float2(k.i0, k.i0 + NP);
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        const float4 hp = s_hp[q];
        const float2 s = __ffma2_rn(id, ax2, __ffma2_rn(make_float2(hp.x, hp.y), tvz2,
                                                        make_float2(hp.z, hp.w)));
        id = __fadd2_rn(id, one);
        const float2 poly = __ffma2_rn(__ffma2_rn(__ffma2_rn(a42, s, a32), s, a22), s, a12);
        const float2 sv = __ffma2_rn(s, poly, f0);
        float2 gr = pr[NN - 1], gi = pi[NN - 1];
#pragma unroll
        for (int n = NN - 2; n >= 0; --n) {
            gr = __ffma2_rn(gr, sv, pr[n]);
            gi = __ffma2_rn(gi, sv, pi[n]);
        }
        const float2 x = __ffma2_rn(sv, c2, cm2);
        float sa, ca, sb, cb;
        __sincosf(x.x, &sa, &ca);
        __sincosf(x.y, &sb, &cb);
        const float2 cs = make_float2(ca, cb);
        const float2 sn = make_float2(sa, sb);
        accre[q] = __ffma2_rn(gr, cs, accre[q]);
        accim[q] = __ffma2_rn(gr, sn, __ffma2_rn(gi, cs, accim[q]));
        accre[q] = __ffma2_rn(make_float2(-gi.x, -gi.y), sn, accre[q]);
    }
}

// Nearest sample on a height map when every pixel of the row rounds to bin kn
// or kn + 1: the two-sample form of nearest_pair_pulse with
// x = c (u - kn - 1/2) from the range series (c folded into its
// coefficients, y0 = c (frac - kn - 1/2)); e is table entry (N_kn, M_kn).
__device__ __forceinline__ void heights_nearest_pair(const BpConst& k, const float4* s_hp, float4 e,
                                                     float y0, float ax, float two_vz, float hb,
                                                     float g, float a4, float2 (&accre)[NP],
                                                     float2 (&accim)[NP])
{
    const float c = k.c_phase;
    const float2 ax2 = make_float2(ax, ax), tvz2 = make_float2(two_vz, two_vz);
    const float a1 = c * hb, a2 = -0.25f * a1 * g, a3 = 0.125f * a1 * g * g, a4c = c * a4;
    const float2 a12 = make_float2(a1, a1), a22 = make_float2(a2, a2);
    const float2 a32 = make_float2(a3, a3), a42 = make_float2(a4c, a4c);
    const float2 y02 = make_float2(y0, y0);
    const float2 w0r2 = make_float2(e.x, e.x), w0i2 = make_float2(e.y, e.y);
    const float2 dwr2 = make_float2(e.z, e.z), dwi2 = make_float2(e.w, e.w);
    const float2 one = make_float2(1.0f, 1.0f);
    float2 id = make_float2(k.i0, k.i0 + NP);
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        const float4 hp = s_hp[q];
        const float2 s = __ffma2_rn(id, ax2, __ffma2_rn(make_float2(hp.x, hp.y), tvz2,
                                                        make_float2(hp.z, hp.w)));
        id = __fadd2_rn(id, one);
        const float2 poly = __ffma2_rn(__ffma2_rn(__ffma2_rn(a42, s, a32), s, a22), s, a12);
        const float2 x = __ffma2_rn(s, poly, y02);
        const float2 h = make_float2(x.x >= 0.0f ? 1.0f : 0.0f, x.y >= 0.0f ? 1.0f : 0.0f);
        const float2 wr = __ffma2_rn(h, dwr2, w0r2);
        const float2 wi = __ffma2_rn(h, dwi2, w0i2);
        float sa, ca, sb, cb;
        __sincosf(x.x, &sa, &ca);
        __sincosf(x.y, &sb, &cb);
        const float2 cs = make_float2(ca, cb);
        const float2 sn = make_float2(sa, sb);
        accre[q] = __ffma2_rn(wr, cs, accre[q]);
        accim[q] = __ffma2_rn(wr, sn, __ffma2_rn(wi, cs, accim[q]));
        accre[q] = __ffma2_rn(make_float2(-wi.x, -wi.y), sn, accre[q]);
    }
}

// Range from the tile centre (at the mid height) to a row's reference point,
// offset by q = (0, Y, Z), Y = jy dy: with g = v / R, L = g.q = gy Y + gz Z and
// Q = |q|^2, |v + q| - R = L + (Q - L^2) / (2R) - L (Q - L^2) / (2R^2)
//   + (-Q^2 / 8 + 3 L^2 Q / 4 - 5 L^4 / 8) / R^3 + O(|q|^5 / R^4).
// This is the part beyond the linear term L, in metres (small enough for
// float32; the linear term is taken in split precision by the caller).
__device__ __forceinline__ float heights_row_curvature(const Record& rec, const HRow& hr, float dy)
{
    const float L = fmaf(rec.b.y, hr.jy * dy, rec.b.z * hr.zh);
    const float ir = rec.b.w;
    const float L2 = L * L;
    const float P = hr.qq - L2;                            // |q|^2 - (g.q)^2 >= 0
    const float o4 = fmaf(hr.qq, fmaf(-0.125f, hr.qq, 0.75f * L2), -0.625f * L2 * L2);
    // ((o4 / R - L P / 2) / R + P / 2) / R
    return fmaf(fmaf(o4, ir, -0.5f * L * P), ir, 0.5f * P) * ir;
}

template <int INTERP>
__device__ __forceinline__ bool heights_series_pulse(const BpConst& k, const Record& rec,
                                                     const float4* row, const HRow& hr,
                                                     const float4* s_hp,
                                                     const float2* __restrict__ psi,
                                                     float2 (&accre)[NP], float2 (&accim)[NP])
{
    // the row's reference point, by the range expansion about the tile centre
    const float curv = heights_row_curvature(rec, hr, k.dy_f);
    const float R = rec.c.z + fmaf(rec.b.y, hr.jy * k.dy_f, fmaf(rec.b.z, hr.zh, curv));
    // u_row = kb + (c01 j + bz Z) + c00 + curv / dr, the linear terms as float
    // pairs with their integer part kept apart
    const float jf = hr.jy;
    const float h1 = rec.a.y * jf;
    const float l1 = fmaf(rec.a.z, jf, fmaf(rec.a.y, jf, -h1));
    const float h2 = rec.a.w * hr.zh;
    const float l2 = fmaf(rec.a.w, hr.zl, fmaf(rec.b.x, hr.zh, fmaf(rec.a.w, hr.zh, -h2)));
    const F2 sl = two_sum(h1, h2);
    const float tr = sl.hi + MAGIC;
    const float ki = tr - MAGIC;
    float frac = (((sl.hi - ki) + sl.lo) + (l1 + l2)) + fmaf(curv, k.inv_dr_f, rec.a.x);
    const float kf = floorf(frac);
    frac -= kf;
    // 1 / R to float precision: the SFU reciprocal and one Newton step
    const float r0i = rcp_approx(R);
    const float inv_r = fmaf(r0i, fmaf(-R, r0i, 1.0f), r0i);
    const float t_bound = hr.qm * (2.0f * R + hr.qm) * (inv_r * inv_r);
    if (!(t_bound <= 0.01f))
        return false;
    const int bin0 = __float_as_int(rec.d.y);
    const int kbase = __float_as_int(rec.d.z) + (__float_as_int(tr) - MAGIC_BITS) + (int)kf;
    const float g = inv_r * inv_r;                // 1 / R^2
    const float hb = 0.5f * inv_r * k.inv_dr_f;   // bins per metre of s, first order

    // s = q_x (2 v_x + q_x) + dz (2 v_z + dz) with q_x = i dx, i.e.
    // i (2 v_x dx) + dz (2 v_z) + P with the pulse-independent P = (i dx)^2 + dz^2
    // held per pixel beside dz; the series times hb is the polynomial
    // a1 s + a2 s^2 + a3 s^3 + a4 s^4 with a_n = hb g^(n-1) c_n. Its s^4 term
    // adds at most (4 pi R / lambda) (5/128) t^4 radians of phase; pulses where
    // that is below 1e-5 rad leave it out.
    const float vzr = rec.c.y + hr.zh;              // v_z at the row's height
    const float ax = 2.0f * rec.c.x * k.dx_f;
    const float tb2 = t_bound * t_bound;
    const bool deg4 = k.c_phase * R * k.inv_dr_f * 0.0390625f * tb2 * tb2 > 1.0e-5f;
    {
        // bounds of s over the row from the row's ranges of dz and P; u grows
        // with s (s poly(s) is increasing for |s| / R^2 <= 0.01)
        const float tvz = 2.0f * vzr;
        const float sx = -k.i0 * fabsf(ax);
        const float s_lo = -sx + fminf(tvz * hr.dz_lo, tvz * hr.dz_hi) + hr.p_lo;
        const float s_hi = sx + fmaxf(tvz * hr.dz_lo, tvz * hr.dz_hi) + hr.p_hi;
        const float a2 = -0.25f * hb * g, a3 = 0.125f * hb * g * g;
        const float lo_u = fmaf(s_lo, fmaf(fmaf(a3, s_lo, a2), s_lo, hb), frac) - 1.0e-5f;
        const float hi_u = fmaf(s_hi, fmaf(fmaf(a3, s_hi, a2), s_hi, hb), frac) + 1.0e-5f;
        const float k0 = floorf(lo_u);
        const int idx0 = kbase + (int)k0;
        // both bins recorded (0 <= k <= nr - 2) and inside the row
        if (INTERP == INTERP_HEIGHTS && hi_u - k0 < 2.0f && idx0 >= bin0 &&
            idx0 + 1 <= bin0 + k.nr - 2 && idx0 >= 0 && idx0 + 1 <= k.W - 1) {
            const float4 t0 = __ldg(row + idx0);
            const float4 t1 = __ldg(row + idx0 + 1);
            const float y0 = k.c_phase * ((frac - k0) - 1.0f);
            if (deg4)
                heights_hinge_loop<true>(k, s_hp, t0, t1, y0, ax, tvz, hb, g, accre, accim);
            else
                heights_hinge_loop<false>(k, s_hp, t0, t1, y0, ax, tvz, hb, g, accre, accim);
            return true;
        }
        if (INTERP == INTERP_HEIGHTS_SINC8) {
            // the row within SINC_SPAN6 bins, the stencils of its two bins
            // recorded and both bins inside the row: one polynomial in u, of
            // degree 2 to 6 by the span (the planar kernels' degrees and
            // spans). The warp takes one path: the polynomial when all its
            // rows here can, at the highest degree any of them needs (on a
            // narrower interval a higher degree is as accurate), else the
            // per-pixel taps for all of them, so that it never runs two paths
            // one after the other.
            float lo_e, hi_e, k0e;
            int kabs0;
            const bool poly = poly_interval(k, kbase, bin0, lo_u, hi_u, SINC_SPAN6, lo_e, hi_e, k0e, kabs0) &&
                              kabs0 + bin0 >= 0 && kabs0 + bin0 + 1 <= k.W - 1;
            const float sp = hi_e - lo_e;
            const int nn = !poly ? 0 : (sp <= SINC_SPAN2 ? 3 : sp <= SINC_SPAN3 ? 4 : sp <= SINC_SPAN ? 5 :
                                       sp <= SINC_SPAN5 ? 6 : 7);
            const unsigned lanes = __activemask();
            const int wn = __reduce_max_sync(lanes, nn);
            if (__all_sync(lanes, poly)) {
                const float a4 = deg4 ? -0.078125f * hb * g * g * g : 0.0f;
                if (wn <= 3)
                    heights_sinc_poly<3>(k, s_hp, row, kbase, lo_e, hi_e, k0e, kabs0, frac, ax, tvz,
                                         hb, g, a4, accre, accim);
                else if (wn == 4)
                    heights_sinc_poly<4>(k, s_hp, row, kbase, lo_e, hi_e, k0e, kabs0, frac, ax, tvz,
                                         hb, g, a4, accre, accim);
                else if (wn == 5)
                    heights_sinc_poly<5>(k, s_hp, row, kbase, lo_e, hi_e, k0e, kabs0, frac, ax, tvz,
                                         hb, g, a4, accre, accim);
                else if (wn == 6)
                    heights_sinc_poly<6>(k, s_hp, row, kbase, lo_e, hi_e, k0e, kabs0, frac, ax, tvz,
                                         hb, g, a4, accre, accim);
                else
                    heights_sinc_poly<7>(k, s_hp, row, kbase, lo_e, hi_e, k0e, kabs0, frac, ax, tvz,
                                         hb, g, a4, accre, accim);
                return true;
            }
        }
        if (INTERP == INTERP_HEIGHTS_NEAREST) {
            // every pixel rounds to bin kn or kn + 1, entry kn inside the row
            const float kn = floorf(lo_u + 0.5f);
            const int idxn = kbase + (int)kn;
            if (hi_u + 0.5f - kn < 2.0f && idxn >= 0 && idxn <= k.W - 1) {
                const float4 e = __ldg(row + idxn);
                const float y0 = k.c_phase * ((frac - kn) - 0.5f);
                const float a4 = deg4 ? -0.078125f * hb * g * g * g : 0.0f;
                heights_nearest_pair(k, s_hp, e, y0, ax, tvz, hb, g, a4, accre, accim);
                return true;
            }
        }
    }
    if (deg4)
        heights_series_loop<INTERP, true>(k, row, s_hp, psi, kbase, bin0, frac, ax, 2.0f * vzr, hb, g,
                                          accre, accim);
    else
        heights_series_loop<INTERP, false>(k, row, s_hp, psi, kbase, bin0, frac, ax, 2.0f * vzr, hb, g,
                                           accre, accim);
    return true;
}

// The fallback: float64 range to the row's reference point, then
// R - R_row = s / (R_row + R) in float32, bounds on every table index.
template <int INTERP>
__device__ __forceinline__ void heights_exact_pulse(const BpConst& k, const Record& rec,
                                                    const float4* row, const double* __restrict__ a,
                                                    double xc, double yrow, const HRow& hr,
                                                    const float4* s_hp,
                                                    const float2* __restrict__ psi,
                                                    float2 (&accre)[NP], float2 (&accim)[NP])
{
    const double vx = xc - a[0], vy = yrow - a[1], vz = (k.z0 + (double)hr.hrow) - a[2];
    const double r2 = vx * vx + vy * vy + vz * vz;
    const double r = sqrt(r2);
    const double u = (r - k.r0) * k.inv_dr;
    if (!(fabs(u) < 1.0e9))
        return;
    const double ku = floor(u);
    const int kbase = (int)ku + __float_as_int(rec.d.y);
    const float frac0 = (float)(u - ku);
    const float two_vx = (float)(2.0 * vx), two_vz = (float)(2.0 * vz);
    const float rf = (float)r, r2f = (float)r2;
    const float c_phase = k.c_phase;
#pragma unroll
    for (int m = 0; m < TILE_X; ++m) {
        const float qx = ((float)m - 0.5f * (TILE_X - 1)) * k.dx_f;
        const float dz = (m < NP) ? s_hp[m % NP].x : s_hp[m % NP].y;   // h - hrow
        const float s = fmaf(qx, two_vx + qx, dz * (two_vz + dz));
        const float rp = sqrtf(fmaxf(r2f + s, 0.0f));
        const float den = rf + rp;
        const float dr_m = den > 0.0f ? s / den : 0.0f;
        const float ub = fmaf(dr_m, k.inv_dr_f, frac0);
        if (INTERP != INTERP_HEIGHTS) {
            float& re = (m < NP) ? accre[m % NP].x : accre[m % NP].y;
            float& im = (m < NP) ? accim[m % NP].x : accim[m % NP].y;
            if (INTERP == INTERP_HEIGHTS_SINC8)
                sinc_pixel<true>(k, ub, kbase, __float_as_int(rec.d.y), row, psi, re, im);
            else
                nearest_pixel<true>(k, ub, kbase, row, re, im);
            continue;
        }
        if (!(ub > -1.0e6f && ub < 1.0e6f))
            continue;
        const float kf = floorf(ub);
        const int kr = kbase + (int)kf;
        if (kr < 0 || kr > k.W - 1)
            continue;                       // outside the row: no recorded echo there
        const float x = (ub - kf) * c_phase;
        const float4 v = __ldg(row + kr);
        const float wr = fmaf(x, v.z, v.x);
        const float wi = fmaf(x, v.w, v.y);
        float sn, cs;
        __sincosf(x, &sn, &cs);
        float& re = (m < NP) ? accre[m % NP].x : accre[m % NP].y;
        float& im = (m < NP) ? accim[m % NP].x : accim[m % NP].y;
        re = fmaf(wr, cs, fmaf(-wi, sn, re));
        im = fmaf(wr, sn, fmaf(wi, cs, im));
    }
}

// x of a tile's centre column and y of an image row, float64 (recomputed where
// needed rather than held in registers across the pulse loop)
__device__ __forceinline__ double tile_xc(const BpConst& k, int col0)
{
    return k.x0 + ((double)col0 + 0.5 * (TILE_X - 1)) * k.dx;
}
__device__ __forceinline__ double row_y(const BpConst& k, int rowi)
{
    return k.y0 + (double)rowi * k.dy;
}

template <int INTERP>
__device__ __forceinline__ void apply_pulse(const BpConst& k, const PulseState& st, const Record& rec,
                                            const float4* row, const double* a, int col0,
                                            int rowi, const HRow& hr_reg, const float4* s_hp,
                                            const float2* __restrict__ psi,
                                            float2 (&accre)[NP], float2 (&accim)[NP])
{
    if (on_heights(INTERP)) {
        // the linear kernel holds the row statistics in registers (1.3 %
        // faster); the sinc and nearest kernels read them from shared memory
        // per pulse (sinc 5 % faster, with fewer registers held)
        const HRow hr = INTERP == INTERP_HEIGHTS ? hr_reg : load_hrow(s_hp);
        if (st.mode == MODE_EXACT ||
            (st.mode == MODE_GATHER &&
             !heights_series_pulse<INTERP>(k, rec, row, hr, s_hp, psi, accre, accim)))
            heights_exact_pulse<INTERP>(k, rec, row, a, tile_xc(k, col0), row_y(k, rowi), hr, s_hp,
                                        psi, accre, accim);
        return;
    }
    if (INTERP == INTERP_NEAREST) {
        if (st.mode == MODE_PAIR)
            nearest_pair_pulse(k, st, accre, accim);
        else if (st.mode == MODE_GATHER)
            nearest_pulse(k, st, row, accre, accim);
        else if (st.mode == MODE_EXACT)
            nearest_exact_pulse(k, rec, row, a, tile_xc(k, col0), row_y(k, rowi), accre, accim);
        return;
    }
    if (is_sinc(INTERP)) {
        if (st.mode == MODE_POLY2)
            sinc_poly_pulse<3>(k, st, row, psi, accre, accim);
        else if (st.mode == MODE_POLY3)
            sinc_poly_pulse<4>(k, st, row, psi, accre, accim);
        else if (st.mode == MODE_POLY)
            sinc_poly_pulse<5>(k, st, row, psi, accre, accim);
        else if (INTERP == INTERP_SINC8_WIDE && st.mode == MODE_POLY5)
            sinc_poly_pulse<6>(k, st, row, psi, accre, accim);
        else if (INTERP == INTERP_SINC8_WIDE && st.mode == MODE_POLY6)
            sinc_poly_pulse<7>(k, st, row, psi, accre, accim);
        else if (st.mode == MODE_GATHER)
            sinc_pulse(k, st, row, psi, accre, accim);
        else if (st.mode == MODE_EXACT)
            sinc_exact_pulse(k, rec, row, a, tile_xc(k, col0), row_y(k, rowi), psi, accre, accim);
        return;
    }
    if (st.mode == MODE_HINGE)
        hinge_pulse(k, st, accre, accim);
    else if (st.mode == MODE_GATHER)
        gather_pulse(k, st, row, accre, accim);
    else if (st.mode == MODE_EXACT)
        exact_pulse(k, rec, row, a, tile_xc(k, col0), row_y(k, rowi), accre, accim);
}

__device__ __forceinline__ long long cta_start(const BpConst& k, long long b)
{
    return k.starts ? k.starts[b] : b * k.units / k.ctas;
}

// ---------------------------------------------------------------------------
// Main kernel: persistent, one contiguous range of (tile, pulse) units per CTA.
// ---------------------------------------------------------------------------
template <int INTERP>
__global__ void __launch_bounds__(THREADS, MIN_BLOCKS) bp_kernel(BpConst k, const double* __restrict__ pos,
                                                        const float4* __restrict__ table,
                                                        const int* __restrict__ klo,
                                                        float2* __restrict__ image,
                                                        float4* __restrict__ partial,
                                                        const float2* __restrict__ psi,
                                                        const float* __restrict__ heights,
                                                        const int* __restrict__ sinc_wide)
{
    __shared__ Record s_rec[CHUNK];
    // heights mode: per row, HROW4 float4 (dz[q], dz[q + 16], P[q], P[q + 16]) with
    // dz = h - hrow and P = (i dx)^2 + dz^2 for the pixels at offsets i of q and q + 16
    extern __shared__ float4 s_hp[];
    const int tid = threadIdx.x;
    const int jr = tid;                                   // warp w, lane l -> row 32 w + l
    const float jf = (float)jr - 0.5f * (TILE_Y - 1);
    const long long b = blockIdx.x;
    const long long u0 = cta_start(k, b);
    const long long u1 = cta_start(k, b + 1);
    if (u0 >= u1)
        return;
    // the two sinc kernels are both launched; the flag the table kernel set
    // says which one does the work (tested after the CTA's range: the narrow
    // kernel's register allocation then spills nothing, and it runs 3 % faster)
    if (is_sinc(INTERP) && ((*sinc_wide != 0) != (INTERP == INTERP_SINC8_WIDE)))
        return;
    // The CTA's tiles and the pulse bounds in its first and last tile, as
    // 32-bit values (tile indices and pulse counts fit): fewer registers held
    // through the pulse loop than the 64-bit unit bounds (the wide sinc kernel
    // 2 % faster, fewer spilled bytes)
    const int t_first = (int)(u0 / k.na);
    const int t_last = (int)((u1 - 1) / k.na);
    const int n0_first = (int)(u0 - (long long)t_first * k.na);
    const int n1_last = (int)(u1 - (long long)t_last * k.na);

    for (int t = t_first; t <= t_last; ++t) {
        const int n0 = (t == t_first) ? n0_first : 0;
        const int n1 = (t == t_last) ? n1_last : k.na;
        const int col0 = (int)(t % k.tiles_x) * TILE_X;
        const int row0 = (int)(t / k.tiles_x) * TILE_Y;
        const int rowi = row0 + jr;
        HRow hr{0.0f, 0.0f, (float)jr - 0.5f * (TILE_Y - 1), 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        if (on_heights(INTERP)) {
            // the thread's own row of the tile, heights clamped to the plan's
            // bounds; pixels outside the image repeat the last row or column
            // (their results are never stored)
            const int rowi_h = min(row0 + jr, k.ny - 1);
            const float* hsrc = heights + (size_t)rowi_h * k.nx;
            float4* hp = s_hp + jr * HROW4;
            float sum = 0.0f;
#pragma unroll 4
            for (int q = 0; q < NP; ++q) {
                const float a = fminf(fmaxf(hsrc[min(col0 + q, k.nx - 1)], k.h_lo_f), k.h_hi_f);
                const float b = fminf(fmaxf(hsrc[min(col0 + q + NP, k.nx - 1)], k.h_lo_f), k.h_hi_f);
                hp[q] = make_float4(a, b, 0.0f, 0.0f);
                sum += a + b;
            }
            hr.hrow = sum * (1.0f / TILE_X);
            float dzm = 0.0f;
            hr.dz_lo = hr.p_lo = 3.0e38f;
            hr.dz_hi = hr.p_hi = -3.0e38f;
#pragma unroll 4
            for (int q = 0; q < NP; ++q) {
                const float4 h2 = hp[q];
                const float dza = h2.x - hr.hrow, dzb = h2.y - hr.hrow;
                const float qa = (k.i0 + (float)q) * k.dx_f, qb = (k.i0 + (float)(q + NP)) * k.dx_f;
                const float pa = fmaf(qa, qa, dza * dza), pb = fmaf(qb, qb, dzb * dzb);
                hp[q] = make_float4(dza, dzb, pa, pb);
                dzm = fmaxf(dzm, fmaxf(fabsf(dza), fabsf(dzb)));
                hr.dz_lo = fminf(hr.dz_lo, fminf(dza, dzb));
                hr.dz_hi = fmaxf(hr.dz_hi, fmaxf(dza, dzb));
                hr.p_lo = fminf(hr.p_lo, fminf(pa, pb));
                hr.p_hi = fmaxf(hr.p_hi, fmaxf(pa, pb));
            }
            const float hx = 0.5f * (TILE_X - 1) * k.dx_f;
            hr.qm = 1.0001f * sqrtf(hx * hx + dzm * dzm);
            const F2 zp = two_sum(hr.hrow, -k.h_mid_f);
            hr.zh = zp.hi;
            hr.zl = zp.lo - k.h_mid_lo;
            const float yy = hr.jy * k.dy_f;
            hr.qq = fmaf(yy, yy, hr.zh * hr.zh);
            if (INTERP != INTERP_HEIGHTS) {
                hp[HROW_STATS] = make_float4(hr.hrow, hr.qm, hr.jy, hr.zh);
                hp[HROW_STATS + 1] = make_float4(hr.zl, hr.qq, hr.dz_lo, hr.dz_hi);
                hp[HROW_STATS + 2] = make_float4(hr.p_lo, hr.p_hi, 0.0f, 0.0f);
            }
        }
        float2 accre[NP], accim[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            accre[q] = make_float2(0.f, 0.f);
            accim[q] = make_float2(0.f, 0.f);
        }

        for (int c0 = n0; c0 < n1; c0 += CHUNK) {
            const int cnt = min(CHUNK, n1 - c0);
            __syncthreads();
            if (tid < cnt)
            {
                const double xct = tile_xc(k, col0);
                const double yct = k.y0 + ((double)row0 + 0.5 * (TILE_Y - 1)) * k.dy;
                if (is_sinc(INTERP) || INTERP == INTERP_LINEAR)
                    make_record<INTERP>(k, pos, klo, c0 + tid, xct, yct, s_rec[tid]);
                else
                    make_record_call<INTERP>(k, pos, klo, c0 + tid, xct, yct, s_rec[tid]);
            }
            __syncthreads();
            const int tw = row_pitch<INTERP>(k);
            const float4* rows = table + (size_t)c0 * tw;
            if (is_sinc(INTERP) || INTERP == INTERP_NEAREST || INTERP == INTERP_HEIGHTS_SINC8) {
                // the sinc modes load their table entries inside the pulse step
                // (the polynomial's nodes), so nothing is gained by building the
                // next pulse's state early, and one state leaves registers free
                // (the height-map sinc kernel 9 % faster than with two); the
                // nearest kernel too runs faster with one state (3 %)
                // (the wide kernel forms the row pointer from the table per
                // pulse, and the nearest kernel unrolls this loop by two: their
                // register allocations then spill nothing)
                if constexpr (INTERP == INTERP_NEAREST) {
#pragma unroll 2
                    for (int p = 0; p < cnt; ++p) {
                        const PulseState st = pulse_setup<INTERP>(k, s_rec[p], rows + (size_t)p * tw, jf);
                        apply_pulse<INTERP>(k, st, s_rec[p], rows + (size_t)p * tw,
                                            pos + 3 * (size_t)(c0 + p), col0, rowi, hr,
                                            s_hp + jr * HROW4, psi, accre, accim);
                    }
                } else {
#pragma unroll 1
                    for (int p = 0; p < cnt; ++p) {
                        const float4* rowp = INTERP == INTERP_SINC8_WIDE ? table + (size_t)(c0 + p) * tw
                                                                         : rows + (size_t)p * tw;
                        const PulseState st = pulse_setup<INTERP>(k, s_rec[p], rowp, jf);
                        apply_pulse<INTERP>(k, st, s_rec[p], rowp,
                                            pos + 3 * (size_t)(c0 + p), col0, rowi, hr,
                                            s_hp + jr * HROW4, psi, accre, accim);
                    }
                }
                continue;
            }
            // Two pulse states in ping-pong: the state of pulse p + 1 is built
            // while pulse p is applied, with no copy between them.
            PulseState sa = pulse_setup<INTERP>(k, s_rec[0], rows, jf);
#pragma unroll 1
            for (int p = 0; p < cnt; p += 2) {
                const int p1 = min(p + 1, cnt - 1);
                const PulseState sb =
                    pulse_setup<INTERP>(k, s_rec[p1], rows + (size_t)p1 * tw, jf);
                // (the height-map nearest kernel forms this row pointer from the
                // table per pulse: its register allocation then spills nothing)
                apply_pulse<INTERP>(k, sa, s_rec[p],
                                    INTERP == INTERP_HEIGHTS_NEAREST ? table + (size_t)(c0 + p) * tw
                                                                     : rows + (size_t)p * tw,
                                    pos + 3 * (size_t)(c0 + p), col0, rowi, hr,
                                  s_hp + jr * HROW4, psi, accre, accim);
                if (p + 1 >= cnt)
                    break;
                const int p2 = min(p + 2, cnt - 1);
                sa = pulse_setup<INTERP>(k, s_rec[p2], rows + (size_t)p2 * tw, jf);
                apply_pulse<INTERP>(k, sb, s_rec[p + 1], rows + (size_t)(p + 1) * tw,
                                  pos + 3 * (size_t)(c0 + p + 1), col0, rowi, hr,
                                  s_hp + jr * HROW4, psi, accre, accim);
            }
        }

        if (n0 == 0 && n1 == k.na) {
            if (rowi < k.ny) {
                float2* dst = image + (size_t)rowi * k.nx;
                const bool acc = (k.flags & FLAG_ACCUMULATE) != 0;
#pragma unroll
                for (int m = 0; m < TILE_X; ++m) {
                    const int col = col0 + m;
                    if (col < k.nx) {
                        const int q = m % NP;
                        float2 v = (m < NP) ? make_float2(accre[q].x, accim[q].x)
                                            : make_float2(accre[q].y, accim[q].y);
                        if (acc) {
                            const float2 o = dst[col];
                            v.x += o.x;
                            v.y += o.y;
                        }
                        dst[col] = v;
                    }
                }
            }
        } else {
            const int slot = (t == t_first) ? 0 : 1;
            float4* dst = partial + ((size_t)(b * 2 + slot) * TILE_PIX + (size_t)jr * TILE_X) / 2;
#pragma unroll
            for (int m = 0; m < TILE_X; m += 2) {
                const int q0 = m % NP, q1 = (m + 1) % NP;
                const float2 v0 = (m < NP) ? make_float2(accre[q0].x, accim[q0].x)
                                           : make_float2(accre[q0].y, accim[q0].y);
                const float2 v1 = (m + 1 < NP) ? make_float2(accre[q1].x, accim[q1].x)
                                               : make_float2(accre[q1].y, accim[q1].y);
                dst[m / 2] = make_float4(v0.x, v0.y, v1.x, v1.y);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Sum the partial pieces of shared tiles in CTA order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ long long cta_of_unit(const BpConst& k, long long u)
{
    // largest b < ctas with cta_start(b) <= u
    if (!k.starts)
        return ((u + 1) * k.ctas - 1) / k.units;
    long long lo = 0, hi = k.ctas - 1;
    while (lo < hi) {
        const long long mid = (lo + hi + 1) / 2;
        if (k.starts[mid] <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

constexpr int REDUCE_THREADS = 256;
constexpr int REDUCE_VEC = 8;                                  // float4 (2 pixels) per thread
constexpr int REDUCE_PIX = REDUCE_THREADS * REDUCE_VEC * 2;    // pixels per block
constexpr int REDUCE_PARTS = (TILE_PIX + REDUCE_PIX - 1) / REDUCE_PIX;

// One block per (tile, part of the tile). The CTAs that share the tile are
// visited in ascending order, so the sum is the same on every run.
__global__ void __launch_bounds__(REDUCE_THREADS) reduce_kernel(BpConst k, const float4* __restrict__ partial,
                                                                float2* __restrict__ image)
{
    const long long t = blockIdx.x / REDUCE_PARTS;
    const int part = blockIdx.x % REDUCE_PARTS;
    const long long bf = cta_of_unit(k, t * k.na);
    const long long bl = cta_of_unit(k, (t + 1) * k.na - 1);
    if (bf == bl)
        return;                                    // written directly by one CTA
    const int col0 = (int)(t % k.tiles_x) * TILE_X;
    const int row0 = (int)(t / k.tiles_x) * TILE_Y;
    float4 sum[REDUCE_VEC];
#pragma unroll
    for (int r = 0; r < REDUCE_VEC; ++r)
        sum[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int f0 = part * (REDUCE_PIX / 2) + threadIdx.x;   // float4 index within the tile
    for (long long b = bf; b <= bl; ++b) {
        const long long s0 = cta_start(k, b);
        if (s0 >= cta_start(k, b + 1))
            continue;                              // CTA with no work
        const int slot = (s0 / k.na == t) ? 0 : 1;
        const float4* src = partial + (size_t)(b * 2 + slot) * (TILE_PIX / 2);
#pragma unroll
        for (int r = 0; r < REDUCE_VEC; ++r) {
            const int f = f0 + r * REDUCE_THREADS;
            if (f < TILE_PIX / 2) {
                const float4 v = src[f];
                sum[r].x += v.x;
                sum[r].y += v.y;
                sum[r].z += v.z;
                sum[r].w += v.w;
            }
        }
    }
    const bool acc = (k.flags & FLAG_ACCUMULATE) != 0;
#pragma unroll
    for (int r = 0; r < REDUCE_VEC; ++r) {
        const int f = f0 + r * REDUCE_THREADS;
        if (f >= TILE_PIX / 2)
            continue;
        {
            // both pixels of the float4 (adjacent in one image row) in one 16-byte
            // store where the row allows it: whole sectors, which matters when the
            // image is mapped host memory
            const int rowi = row0 + (2 * f) / TILE_X;
            const int col = col0 + (2 * f) % TILE_X;
            float4* dst4 = (rowi < k.ny && col + 1 < k.nx)
                               ? reinterpret_cast<float4*>(image + (size_t)rowi * k.nx + col)
                               : nullptr;
            if (dst4 && (reinterpret_cast<uintptr_t>(dst4) & 15) == 0) {
                float4 v = sum[r];
                if (acc) {
                    const float4 o = *dst4;
                    v.x += o.x;
                    v.y += o.y;
                    v.z += o.z;
                    v.w += o.w;
                }
                *dst4 = v;
                continue;
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int p = 2 * f + h;
            const int rowi = row0 + p / TILE_X;
            const int col = col0 + p % TILE_X;
            if (rowi < k.ny && col < k.nx) {
                float2 v = h ? make_float2(sum[r].z, sum[r].w) : make_float2(sum[r].x, sum[r].y);
                float2* dst = image + (size_t)rowi * k.nx + col;
                if (acc) {
                    const float2 o = *dst;
                    v.x += o.x;
                    v.y += o.y;
                }
                *dst = v;
            }
        }
    }
}

// Scratch of sarbp_backproject_noalloc: window starts and echo-table rows of
// one chunk of pulses. Every GPU that loads the library holds it until exit.
static __device__ __align__(256) unsigned char noalloc_scratch_array[NOALLOC_SCRATCH_BYTES];

}  // namespace

cudaError_t noalloc_scratch(void** ptr)
{
    // The symbol's name is only a host-side stand-in; kernels need the device
    // address. It is looked up on every call, in the context current on the
    // calling thread: the array lives in each context that loads this module,
    // and a reset device or another context gives it a new address. The
    // lookup allocates nothing; the first one in a context loads the array.
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, noalloc_scratch_array);
    if (e != cudaSuccess)
        return e;
    *ptr = p;
    return cudaSuccess;
}

cudaError_t launch_table(const BpConst& k, const float2* echo, const double* pos, float4* table,
                         int* klo, int* sinc_wide, cudaStream_t s)
{
    static const SincTaps taps = fit_sinc_taps();
    if (k.flags & FLAG_SINC8)
        table_kernel<TABLE_SINC><<<k.na, 256, 0, s>>>(k, echo, pos, table, klo, sinc_wide, taps);
    else if (k.flags & FLAG_NEAREST)
        table_kernel<TABLE_PAIRS><<<k.na, 256, 0, s>>>(k, echo, pos, table, klo, nullptr, taps);
    else
        table_kernel<TABLE_LINEAR><<<k.na, 256, 0, s>>>(k, echo, pos, table, klo, nullptr, taps);
    return cudaGetLastError();
}

cudaError_t launch_psi(const BpConst& k, float2* psi, cudaStream_t s)
{
    psi_kernel<<<(unsigned)((k.nr + 255) / 256), 256, 0, s>>>(k, psi);
    return cudaGetLastError();
}

constexpr size_t HEIGHTS_SMEM = (size_t)TILE_Y * HROW4 * sizeof(float4);

cudaError_t prepare_kernels()
{
    cudaError_t e = cudaFuncSetAttribute(bp_kernel<INTERP_HEIGHTS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)HEIGHTS_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bp_kernel<INTERP_HEIGHTS_SINC8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)HEIGHTS_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bp_kernel<INTERP_HEIGHTS_NEAREST>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)HEIGHTS_SMEM);
    return e;
}

cudaError_t launch_backproject(const BpConst& k, const double* pos, const float4* table,
                               const int* klo, float2* image, float4* partial,
                               const float2* psi, const float* heights, const int* sinc_wide,
                               cudaStream_t s)
{
    if (k.heights_mode && (k.flags & FLAG_SINC8))
        bp_kernel<INTERP_HEIGHTS_SINC8><<<k.ctas, THREADS, HEIGHTS_SMEM, s>>>(
            k, pos, table, klo, image, partial, psi, heights, nullptr);
    else if (k.heights_mode && (k.flags & FLAG_NEAREST))
        bp_kernel<INTERP_HEIGHTS_NEAREST><<<k.ctas, THREADS, HEIGHTS_SMEM, s>>>(
            k, pos, table, klo, image, partial, psi, heights, nullptr);
    else if (k.heights_mode)
        bp_kernel<INTERP_HEIGHTS><<<k.ctas, THREADS, HEIGHTS_SMEM, s>>>(k, pos, table, klo, image,
                                                                       partial, psi, heights, nullptr);
    else if (k.flags & FLAG_SINC8)
    {
        bp_kernel<INTERP_SINC8><<<k.ctas, THREADS, 0, s>>>(k, pos, table, klo, image, partial, psi,
                                                           nullptr, sinc_wide);
        bp_kernel<INTERP_SINC8_WIDE><<<k.ctas, THREADS, 0, s>>>(k, pos, table, klo, image,
                                                                        partial, psi, nullptr,
                                                                        sinc_wide);
    }
    else if (k.flags & FLAG_NEAREST)
        bp_kernel<INTERP_NEAREST><<<k.ctas, THREADS, 0, s>>>(k, pos, table, klo, image, partial,
                                                             psi, nullptr, nullptr);
    else
        bp_kernel<INTERP_LINEAR><<<k.ctas, THREADS, 0, s>>>(k, pos, table, klo, image, partial,
                                                            psi, nullptr, nullptr);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Cost-weighted work split for the windowed-sinc kernels on a plane. What a
// (tile, pulse) unit costs depends on how far a thread's 32 pixels spread in
// range (a polynomial of degree 2 to 6, or per-pixel taps), and
// that spread grows with the tile's x distance from the antenna, so equal unit
// counts leave the CTAs holding the image's far edges working after the others
// have finished. split_kernel estimates each tile's cost from SPLIT_SAMPLES
// evenly spaced pulses, in integer units (the sums are exact and the split is
// the same on every run), and places the CTA boundaries at equal shares of the
// total; within a tile the pulses count as equally costly.
// ---------------------------------------------------------------------------
constexpr int SPLIT_THREADS = 1024;
constexpr int SPLIT_SAMPLES = 64;

// Relative cost of one (thread, pulse) by the spread of its pixels' range, in
// bins, from the modes' instruction counts per thread and pulse.
__device__ __forceinline__ unsigned sinc_unit_cost(float span, bool wide)
{
    if (span <= SINC_SPAN2)
        return 89;
    if (span <= SINC_SPAN3)
        return 100;
    if (span <= SINC_SPAN)
        return 113;
    if (wide && span <= SINC_SPAN5)
        return 125;
    if (wide && span <= SINC_SPAN6)
        return 138;
    return 330;
}

// Relative cost of one (thread, pulse) of the height-map sinc kernel by the
// spread of the thread's row in bins, in SM cycles per (row, pulse) times ten,
// fitted to per-CTA cycle counts on terrain. The cost is the warp's, since the
// warp takes one path for all its rows: the polynomial at the highest degree
// among them (8.9, 10.6, 11.5, 13.2 and 14.8 for degrees 2 to 6) when every
// row allows one, else the per-pixel taps: 24.7 when no row allows a
// polynomial, 123 when some do, and 49 more when a row takes the float64
// path. The last class is the fit's proxy for the tiles where the terrain
// steepens (1.3 % of the warps on a 40 m terrain): timed per warp, their
// per-pixel path costs what other warps' does.
// Called by all 32 lanes of a warp together.
__device__ __forceinline__ float heights_sinc_row_cost(float span, bool exact)
{
    const float sp = fmaxf(span, 2.0f * SINC_HALF_MIN);
    const int nn = exact ? 0 : (sp <= SINC_SPAN2 ? 1 : sp <= SINC_SPAN3 ? 2 : sp <= SINC_SPAN ? 3 :
                                sp <= SINC_SPAN5 ? 4 : sp <= SINC_SPAN6 ? 5 : 0);
    const int wn = __reduce_max_sync(0xffffffffu, nn);
    const bool any_pixel = __any_sync(0xffffffffu, !exact && nn == 0);
    const bool any_exact = __any_sync(0xffffffffu, exact);
    const float poly = wn == 0 ? 0.0f : wn == 1 ? 89.0f : wn == 2 ? 106.0f : wn == 3 ? 115.0f :
                       wn == 4 ? 132.0f : 148.0f;
    return (any_pixel ? (wn > 0 ? 1230.0f : 247.0f) : poly) + (any_exact ? 490.0f : 0.0f);
}

// The cells of split_kernel for the height-map sinc kernel, whose cost follows
// the terrain: one block per tile and up to COST_SAMPLES pulse segments, one
// thread per row. Each row takes the main kernel's statistics of its heights
// (the range of h - hrow and of P = (i dx)^2 + (h - hrow)^2) and, at the
// middle pulse of each of the NS pulse segments, the spread of its range in
// bins from the bound the main kernel uses (s = i 2 v_x dx + dz 2 v_z + P over
// the row, times 1 / (2 R dr)), or the float64 path where the record builder's
// or the row's test sends the row there; cum[1 + t NS + i] receives the
// tile's summed row cost times the segment's pulse count.
constexpr int COST_SAMPLES = 16;           // pulse segments per block of heights_cost_kernel

__global__ void __launch_bounds__(THREADS) heights_cost_kernel(BpConst k, const double* __restrict__ pos,
                                                               const float* __restrict__ heights,
                                                               unsigned long long* __restrict__ cum)
{
    __shared__ float s_sum[COST_SAMPLES][WARPS];
    const int t = blockIdx.x;
    const int NS = max(1, min(SPLIT_SAMPLES, SPLIT_CELLS / max(k.tiles, 1)));
    const int i0 = blockIdx.y * COST_SAMPLES, i1 = min(NS, i0 + COST_SAMPLES);
    const int col0 = (t % k.tiles_x) * TILE_X;
    const int row0 = (t / k.tiles_x) * TILE_Y;
    const int rowi = min(row0 + (int)threadIdx.x, k.ny - 1);
    const float* hsrc = heights + (size_t)rowi * k.nx;
    float sum = 0.0f, hmin = 3.0e38f, hmax = -3.0e38f;
    for (int m = 0; m < TILE_X; ++m) {
        const float h = fminf(fmaxf(hsrc[min(col0 + m, k.nx - 1)], k.h_lo_f), k.h_hi_f);
        sum += h;
        hmin = fminf(hmin, h);
        hmax = fmaxf(hmax, h);
    }
    const float hrow = sum * (1.0f / TILE_X);
    const float dzm = fmaxf(hmax - hrow, hrow - hmin);
    const float hx = 0.5f * (TILE_X - 1) * k.dx_f;
    const float dp = hx * hx + dzm * dzm;              // bound on the spread of P
    const float qm = 1.0001f * sqrtf(hx * hx + dzm * dzm);
    const float xc = (float)(k.x0 + ((double)col0 + 0.5 * (TILE_X - 1)) * k.dx);
    const float yc = (float)(k.y0 + ((double)row0 + 0.5 * (TILE_Y - 1)) * k.dy);
    const float yr = (float)(k.y0 + (double)(row0 + (int)threadIdx.x) * k.dy);
    const float zr = (float)k.z0 + hrow;
    const float q3 = (float)k.qmax3, zm = (float)k.z_mid;
    for (int i = i0; i < i1; ++i) {
        const long long n_lo = (long long)i * k.na / NS, n_hi = (long long)(i + 1) * k.na / NS;
        float cost = 0.0f;
        if (n_hi > n_lo) {
            const long long n = (n_lo + n_hi) / 2;
            const float ax = (float)pos[3 * n], ay = (float)pos[3 * n + 1], az = (float)pos[3 * n + 2];
            if (isfinite(ax) && isfinite(ay) && isfinite(az)) {
                // the record's test at the tile centre (mid height) ...
                const float tx = xc - ax, ty = yc - ay, tz = zm - az;
                const float rt = sqrtf(fmaf(tx, tx, fmaf(ty, ty, tz * tz)));
                const float qr = q3 / rt;
                const bool fast = rt > 8.0f * q3 && qr * qr * qr * qr * q3 * k.inv_dr_f <= (float)k.fast_tol_bins;
                // ... and the row's
                const float vx = xc - ax, vy = yr - ay, vz = zr - az;
                const float r = sqrtf(fmaf(vx, vx, fmaf(vy, vy, vz * vz)));
                const bool series = qm * (2.0f * r + qm) <= 0.01f * r * r;
                const float ss = (TILE_X - 1) * fabsf(2.0f * vx * k.dx_f) +
                                 fabsf(2.0f * vz) * (hmax - hmin) + dp;
                cost = heights_sinc_row_cost(ss * 0.5f * k.inv_dr_f / fmaxf(r, 1.0f),
                                             !(fast && series));
            }
        }
        // the warp's sum over its rows
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            cost += __shfl_down_sync(0xffffffffu, cost, o);
        if ((threadIdx.x & 31) == 0)
            s_sum[i - i0][threadIdx.x >> 5] = cost;
    }
    __syncthreads();
    // the block's sums, one sample per thread
    const int i = i0 + (int)threadIdx.x;
    if (i < i1) {
        float tot = 0.0f;
        for (int w = 0; w < WARPS; ++w)
            tot += s_sum[threadIdx.x][w];
        const long long n_lo = (long long)i * k.na / NS, n_hi = (long long)(i + 1) * k.na / NS;
        cum[1 + (size_t)t * NS + i] = (unsigned long long)tot * (unsigned long long)(n_hi - n_lo);
    }
}

// One block. The units are cut into cells: tile t, pulse segment i of NS
// (NS = min(SPLIT_SAMPLES, SPLIT_CELLS / tiles), at least 1), so that the cost
// can follow the antenna along the track; a cell's cost is the unit cost at
// its middle pulse times its pulse count. With `costed` the cells' costs are
// already in cum[1 ..] (heights_cost_kernel, whole numbers summed exactly in
// float32) and only the scan and the cuts run. cum: SPLIT_CELLS + 1 words of
// scratch; starts: ctas + 1 unit offsets.
__global__ void __launch_bounds__(SPLIT_THREADS) split_kernel(BpConst k, const double* __restrict__ pos,
                                                              const int* __restrict__ sinc_wide,
                                                              bool costed,
                                                              unsigned long long* __restrict__ cum,
                                                              long long* __restrict__ starts)
{
    __shared__ unsigned long long s_part[SPLIT_THREADS];
    const bool wide = !costed && *sinc_wide != 0;
    const int T = k.tiles;
    const int NS = max(1, min(SPLIT_SAMPLES, SPLIT_CELLS / max(T, 1)));
    const int C = T * NS;
    const int per = (C + SPLIT_THREADS - 1) / SPLIT_THREADS;
    const int c0 = min((int)threadIdx.x * per, C), c1 = min(c0 + per, C);
    const float span_scale = (float)((TILE_X - 1) * k.dx * k.inv_dr);
    // per-cell costs (held in cum[c + 1] until the scan), and this thread's sum
    unsigned long long sum = 0;
    for (int c = c0; c < c1; ++c) {
        const int t = c / NS, i = c % NS;
        const long long n_lo = (long long)i * k.na / NS, n_hi = (long long)(i + 1) * k.na / NS;
        unsigned long long w = 0;
        if (costed) {
            w = cum[c + 1];                        // written by heights_cost_kernel
        } else if (n_hi > n_lo) {
            const long long n = (n_lo + n_hi) / 2;
            const float xc = (float)(k.x0 + ((double)((t % k.tiles_x) * TILE_X) + 0.5 * (TILE_X - 1)) * k.dx);
            const float yc = (float)(k.y0 + ((double)((t / k.tiles_x) * TILE_Y) + 0.5 * (TILE_Y - 1)) * k.dy);
            const float ax = (float)pos[3 * n], ay = (float)pos[3 * n + 1], az = (float)pos[3 * n + 2];
            if (isfinite(ax) && isfinite(ay) && isfinite(az)) {
                const float vx = xc - ax, vy = yc - ay, vz = (float)k.z0 - az;
                const float r = sqrtf(fmaf(vx, vx, fmaf(vy, vy, vz * vz)));
                w = (unsigned long long)sinc_unit_cost(span_scale * fabsf(vx) / fmaxf(r, 1.0f), wide) *
                    (unsigned long long)(n_hi - n_lo);
            }
        }
        cum[c + 1] = w;
        sum += w;
    }
    // inclusive scan of the per-thread sums
    s_part[threadIdx.x] = sum;
    __syncthreads();
    for (int off = 1; off < SPLIT_THREADS; off <<= 1) {
        const unsigned long long v = threadIdx.x >= off ? s_part[threadIdx.x - off] : 0ull;
        __syncthreads();
        s_part[threadIdx.x] += v;
        __syncthreads();
    }
    unsigned long long run = threadIdx.x ? s_part[threadIdx.x - 1] : 0ull;
    if (threadIdx.x == 0)
        cum[0] = 0;
    for (int c = c0; c < c1; ++c) {
        run += cum[c + 1];
        cum[c + 1] = run;                          // cost of cells 0 .. c
    }
    __syncthreads();
    const unsigned long long total = s_part[SPLIT_THREADS - 1];
    // CTA b starts where the cumulative cost reaches b / ctas of the total
    const unsigned long long ctas = (unsigned long long)k.ctas;
    for (int b = threadIdx.x; b <= k.ctas; b += SPLIT_THREADS) {
        long long u;
        if (b == k.ctas) {
            u = k.units;
        } else if (total == 0) {
            u = (long long)b * k.units / k.ctas;
        } else {
            const unsigned long long target =
                (total / ctas) * (unsigned long long)b + (total % ctas) * (unsigned long long)b / ctas;
            int lo = 0, hi = C - 1;                // largest c < C with cum[c] <= target
            while (lo < hi) {
                const int mid = (lo + hi + 1) / 2;
                if (cum[mid] <= target)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            const int t = lo / NS, i = lo % NS;
            const long long n_lo = (long long)i * k.na / NS, n_hi = (long long)(i + 1) * k.na / NS;
            const unsigned long long w = cum[lo + 1] - cum[lo];
            const unsigned long long unit = n_hi > n_lo ? w / (unsigned long long)(n_hi - n_lo) : 0ull;
            const long long into =
                unit ? (long long)min((target - cum[lo]) / unit, (unsigned long long)(n_hi - n_lo)) : 0;
            u = (long long)t * k.na + n_lo + into;
        }
        starts[b] = u;
    }
}

void sinc_taps_host(float* out)
{
    static const SincTaps taps = fit_sinc_taps();
    for (int d = 0; d < 8; ++d)
        for (int n = 0; n < 8; ++n)
            out[8 * d + n] = taps.c[d][n];
}

cudaError_t launch_split(const BpConst& k, const double* pos, const int* sinc_wide,
                         unsigned long long* cum, long long* starts, cudaStream_t s)
{
    split_kernel<<<1, SPLIT_THREADS, 0, s>>>(k, pos, sinc_wide, false, cum, starts);
    return cudaGetLastError();
}

cudaError_t launch_heights_split(const BpConst& k, const double* pos, const float* heights,
                                 unsigned long long* cum, long long* starts, cudaStream_t s)
{
    const int ns = std::max(1, std::min(SPLIT_SAMPLES, SPLIT_CELLS / std::max(k.tiles, 1)));
    const dim3 grid((unsigned)k.tiles, (unsigned)((ns + COST_SAMPLES - 1) / COST_SAMPLES));
    heights_cost_kernel<<<grid, THREADS, 0, s>>>(k, pos, heights, cum);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    split_kernel<<<1, SPLIT_THREADS, 0, s>>>(k, pos, nullptr, true, cum, starts);
    return cudaGetLastError();
}

cudaError_t launch_reduce(const BpConst& k, const float4* partial, float2* image, cudaStream_t s)
{
    reduce_kernel<<<(unsigned)k.tiles * REDUCE_PARTS, REDUCE_THREADS, 0, s>>>(k, partial, image);
    return cudaGetLastError();
}

cudaError_t backproject_occupancy(int* ctas_per_sm)
{
    int a = 0, b = 0, c = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, bp_kernel<INTERP_LINEAR>,
                                                                  THREADS, 0);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, bp_kernel<INTERP_SINC8>, THREADS, 0);
    if (e == cudaSuccess) {
        int w = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&w, bp_kernel<INTERP_SINC8_WIDE>, THREADS,
                                                          0);
        b = std::min(b, w);
    }
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, bp_kernel<INTERP_NEAREST>, THREADS, 0);
    *ctas_per_sm = std::min(a, std::min(b, c));
    return e;
}

}  // namespace sarbp
