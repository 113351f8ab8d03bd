// sarbp_internal.h - constants and launch helpers shared by the libsarbp host
// code and its kernels. Not part of the public C-ABI (include/sarbp.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

struct sarbp_rc_plan_s;

namespace sarbp {

// Work tile: one thread owns TILE_X consecutive pixels of one image row; the
// 32 lanes of a warp own 32 consecutive rows; WARPS warps stack vertically.
#ifndef SARBP_TILE_X
#define SARBP_TILE_X 32
#endif
#ifndef SARBP_WARPS
#define SARBP_WARPS 16
#endif
#ifndef SARBP_MIN_BLOCKS
#define SARBP_MIN_BLOCKS 1
#endif
constexpr int TILE_X = SARBP_TILE_X;
constexpr int WARPS = SARBP_WARPS;
constexpr int MIN_BLOCKS = SARBP_MIN_BLOCKS;   // resident CTAs per SM the register budget targets
constexpr int THREADS = 32 * WARPS;
constexpr int TILE_Y = 32 * WARPS;
constexpr int TILE_PIX = TILE_X * TILE_Y;
constexpr int CHUNK = THREADS;             // pulses whose records are built together
constexpr int MARGIN = 4;                  // spare table entries at each end of a row
constexpr int TABLE_PAD = 64;              // spare entries before/after the whole table
constexpr int MIN_PULSES_PER_CTA = 32;     // keeps tiny problems from over-splitting
constexpr int KLO_INVALID = INT32_MIN;     // pulse with a non-finite antenna position

enum RecordKind : int { REC_SKIP = 0, REC_FAST = 1, REC_EXACT = 2 };
constexpr unsigned FLAG_ACCUMULATE = 1u;   // same values as SARBP_ACCUMULATE / _SINC8 / _NEAREST
constexpr unsigned FLAG_SINC8 = 2u;
constexpr unsigned FLAG_NEAREST = 4u;

// Launch constants, computed on the host in float64 for every call.
struct BpConst {
    int nx, ny, na, nr;
    int W;                       // table bins per pulse
    int tw;                      // row pitch in float4: W, or 4 W for the sinc coefficient rows
    int tiles_x, tiles;
    int full_window;             // every row spans bins [-MARGIN-4, nr+...)
    int ctas;                    // persistent CTAs of the main kernel
    unsigned flags;
    long long units;             // tiles * na (tile-pulse work units)
    long long echo_stride;       // complex samples from one pulse's echo row to the next
    const long long* starts;     // first unit of each CTA (ctas + 1 entries, device), or
                                 // null: CTA b starts at b * units / ctas

    double x0, y0, z0, dx, dy, r0, dr, inv_dr;
    double rect_x0, rect_x1, rect_y0, rect_y1;  // tile-padded image rectangle
    double qmax;                 // largest distance from a tile centre to its pixels
    double fast_tol_bins;        // Taylor remainder allowed on the fast path, in bins

    unsigned long long alpha_fx; // frac(2 dr / lambda) * 2^64
    unsigned long long beta_fx;  // frac(2 r0 / lambda) * 2^64
    float c_phase;               // 2 pi * 2 dr / lambda: phase per bin, radians
    float inv_c;                 // 1 / c_phase
    float dx_f, dy_f, inv_dr_f;
    int heights_mode;            // pixels raised by a height map (exact path only)
    double z_lo, z_hi;           // z0 + height bounds given at plan time
    double qmax3;                // tile reach including height offsets from the mid height
    double z_mid;                // z0 + mid height: records are built on this plane
    float h_lo_f, h_hi_f;        // height bounds; the kernel clamps heights into them
    float h_mid_f, h_mid_lo;     // mid height (z_mid - z0) as a float pair (hi + lo)
    float dy_lo;                 // dy - dy_f
    float r0_hi, r0_lo;          // r0 as a float pair (hi + lo)
    float idr_hi, idr_lo;        // 1 / dr as a float pair
    float rot_re, rot_im;        // exp(-j c_phase): phase step from one bin to the next
    float hrt_re, hrt_im;        // rot_re / 2, rot_im / 2
    float hrot_re, hrot_im;      // exp(+j c_phase / 2): phase across half a bin
    float i0;                    // column offset of a thread's first pixel from the tile centre
};

// sinc_wide (sinc only, else null): set to 1 when a thread's pixels can span more
// range bins than the narrow sinc kernel's polynomial modes cover
cudaError_t launch_table(const BpConst& k, const float2* echo, const double* pos,
                         float4* table, int* klo, int* sinc_wide, cudaStream_t s);
cudaError_t launch_psi(const BpConst& k, float2* psi, cudaStream_t s);
cudaError_t launch_backproject(const BpConst& k, const double* pos, const float4* table,
                               const int* klo, float2* image, float4* partial,
                               const float2* psi, const float* heights, const int* sinc_wide,
                               cudaStream_t s);
// Dynamic shared-memory limits of the kernels that use more than the default.
cudaError_t prepare_kernels();
// Cost-weighted CTA boundaries for the windowed-sinc kernels on a plane (after
// the table kernel on the same stream, which sets sinc_wide): cum holds
// SPLIT_CELLS + 1 words of scratch, starts receives ctas + 1 unit offsets.
// Only for k.tiles <= SPLIT_CELLS (one cell per tile at least).
constexpr int SPLIT_CELLS = 65536;         // (tile, pulse segment) cells of the cost estimate
cudaError_t launch_split(const BpConst& k, const double* pos, const int* sinc_wide,
                         unsigned long long* cum, long long* starts, cudaStream_t s);
// The same for the height-map sinc kernel, whose cost follows the terrain:
// per-tile costs from the rows' height statistics, then the split.
cudaError_t launch_heights_split(const BpConst& k, const double* pos, const float* heights,
                                 unsigned long long* cum, long long* starts, cudaStream_t s);
// Range compression fused with the linear echo table (sarbp_rc.cu): for every
// pulse the compressed samples of the table row's window only, written as the
// row's entries, with klo as launch_table sets it. k describes the
// backprojection; the raw frame is [k.na][k.nr].
cudaError_t launch_rc_table(const sarbp_rc_plan_s* rc, const BpConst& k, const float2* raw,
                            const double* pos, float4* table, int* klo, cudaStream_t s);
// Pulses, samples per pulse and device of a range-compression plan.
bool rc_plan_shape(const sarbp_rc_plan_s* rc, int* na, int* ns, int* device);
// The 8 x 8 windowed-sinc tap polynomial coefficients (row d + 3, column n).
void sinc_taps_host(float* out);
cudaError_t launch_reduce(const BpConst& k, const float4* partial, float2* image,
                          cudaStream_t s);
cudaError_t backproject_occupancy(int* ctas_per_sm);

// Every device allocation of the library goes through here, so that tests can
// make one of them fail on the host (sarbp_debug_fail_alloc) without touching
// the GPU.
cudaError_t device_alloc(void** ptr, size_t bytes);

// Device address of the fixed scratch array used by sarbp_backproject_noalloc
// in the context current on the calling thread (looked up on every call).
constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(16) << 20;
cudaError_t noalloc_scratch(void** ptr);

}  // namespace sarbp
