/*
 * sarbp_oracle.h - plain FP64 CPU time-domain SAR backprojector.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load or call this code; the product path
 * (libsarbp) never does, and shares no code, header or constant with it.
 *
 * Source of the method (SARBP-GPU = the page "基于GPU的SAR后向投影成像优化与CUDA加速实践"):
 *   SARBP-GPU §1.1  every pixel sums, over all pulses, the echo found at its
 *                    range history after phase compensation;
 *   SARBP-GPU §1.2  the loop is O(Na * Nx * Ny);
 *   SARBP-GPU §2.2  steps: pixel coordinates, slant range per pulse, linear
 *                    interpolation of the range-compressed echo, phase
 *                    compensation, accumulation;
 *   SARBP-GPU §3.3  kernel pseudo-code: uniform range axis (first sample and
 *                    spacing), floor/fraction interpolation, phase 4*pi*R/lambda
 *                    applied as exp(+j*phase), planar real/imaginary output,
 *                    monostatic geometry.
 */
#ifndef SARBP_ORACLE_H
#define SARBP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int64_t nx, ny;        /* image width (x) and height (y), pixels              */
    int64_t na, nr;        /* pulses, range bins                                  */
    double x0, y0, z0;     /* position of pixel (0, 0)                            */
    double dx, dy;         /* pixel spacing; pixel (ix, iy) = (x0+ix*dx, y0+iy*dy, z0) */
    double r0, dr;         /* range of bin k = r0 + k * dr                        */
    double wavelength;     /* carrier wavelength                                  */
} oracle_geometry;

/*
 * Backproject the pixels listed in `pixels` (linear index iy * nx + ix).
 *   echo        complex64 as interleaved float pairs, [na][nr][2], pulse-major
 *   antenna_pos float64 [na][3], antenna phase centre of each pulse (x, y, z)
 *   out         float64 [npix][2], complex128 result per listed pixel
 *   nthreads    worker threads; <= 0 means all online CPUs
 * Returns the number of threads used, or -1 on a bad argument.
 */
int oracle_backproject(const oracle_geometry* g, const float* echo,
                       const double* antenna_pos, const int64_t* pixels,
                       int64_t npix, double* out, int nthreads);

/*
 * Same sum with truncated-sinc interpolation instead of linear (SARBP-GPU
 * §2.2 names sinc interpolation as the more accurate, costlier choice):
 *   w_n = sum_{m = k-3}^{k+4} e[n][m] * h(u - m),
 *   h(t) = sinc(t) * (1/2 + 1/2 cos(2 pi t / 8)),  sinc(t) = sin(pi t) / (pi t),
 * and w_n = 0 unless the whole stencil k-3 .. k+4 lies in 0 .. nr-1.
 */
int oracle_backproject_sinc8(const oracle_geometry* g, const float* echo,
                             const double* antenna_pos, const int64_t* pixels,
                             int64_t npix, double* out, int nthreads);

/*
 * Same sum with nearest-neighbour interpolation (SARBP-GPU §2.2: the fastest,
 * least accurate of the three choices): k = floor(u + 1/2), w_n = e[n][k],
 * and w_n = 0 unless 0 <= k <= nr - 1.
 */
int oracle_backproject_nearest(const oracle_geometry* g, const float* echo,
                               const double* antenna_pos, const int64_t* pixels,
                               int64_t npix, double* out, int nthreads);

/*
 * Linear interpolation over a non-planar grid (SARBP-GPU §3.3: the range
 * history may need terrain elevation): pixel (ix, iy) sits at
 * (x0 + ix*dx, y0 + iy*dy, z0 + heights[iy*nx + ix]), heights float32 [ny][nx].
 */
int oracle_backproject_heights(const oracle_geometry* g, const float* echo,
                               const double* antenna_pos, const float* heights,
                               const int64_t* pixels, int64_t npix, double* out, int nthreads);

/* The height map with the windowed-sinc or nearest-sample interpolation. */
int oracle_backproject_heights_sinc8(const oracle_geometry* g, const float* echo,
                                     const double* antenna_pos, const float* heights,
                                     const int64_t* pixels, int64_t npix, double* out,
                                     int nthreads);
int oracle_backproject_heights_nearest(const oracle_geometry* g, const float* echo,
                                       const double* antenna_pos, const float* heights,
                                       const int64_t* pixels, int64_t npix, double* out,
                                       int nthreads);

#ifdef __cplusplus
}
#endif

#endif /* SARBP_ORACLE_H */
