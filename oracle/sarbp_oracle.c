/*
 * sarbp_oracle.c - plain, slow, FP64 CPU time-domain SAR backprojector.
 *
 * TEST INFRASTRUCTURE ONLY (see sarbp_oracle.h). Nothing here is blocked,
 * fused or reordered: pixel outer loop, pulse inner loop in ascending order,
 * libm sqrt/floor/cos/sin, complex64 echo samples widened to double.
 *
 * Definition (SARBP-GPU = the page "基于GPU的SAR后向投影成像优化与CUDA加速实践"):
 *
 *   p          = (x0 + ix*dx, y0 + iy*dy, z0)                 [SARBP-GPU §2.2 step 1]
 *   R_n        = |p - a_n|                                     [§2.2 step 2, §3.3 monostatic]
 *   u          = (R_n - r0) / dr,  k = floor(u),  f = u - k    [§2.2 step 3, §3.3 range axis]
 *   w_n        = (1 - f) * e[n][k] + f * e[n][k+1]             [§2.2 linear interpolation]
 *                (zero when k < 0 or k + 1 > nr - 1: no echo was recorded there)
 *   I(p)       = sum_n w_n * exp(+j * 4*pi*R_n / lambda)       [§1.1, §2.2 step 4, §3.3]
 *
 * The range axis is uniform (first sample r0, spacing dr), as the page's
 * kernel reads only the first two range-axis entries. lambda is the carrier
 * wavelength (§4.2 lists the bandwidth wavelength as a defocus cause).
 */
#include "sarbp_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <unistd.h>

static const double ORACLE_PI = 3.14159265358979323846;

/* One pixel, all pulses. */
static void backproject_pixel(const oracle_geometry* g, const float* echo,
                              const double* antenna_pos, const float* heights, int64_t pixel, double* out)
{
    (void)heights;
    const int64_t ix = pixel % g->nx;
    const int64_t iy = pixel / g->nx;
    const double x = g->x0 + (double)ix * g->dx;
    const double y = g->y0 + (double)iy * g->dy;
    const double z = g->z0;
    double acc_re = 0.0;
    double acc_im = 0.0;

    for (int64_t n = 0; n < g->na; ++n) {
        const double* a = antenna_pos + 3 * n;
        const double ddx = x - a[0];
        const double ddy = y - a[1];
        const double ddz = z - a[2];
        const double range = sqrt(ddx * ddx + ddy * ddy + ddz * ddz);

        const double u = (range - g->r0) / g->dr;
        const double k = floor(u);
        if (!(k >= 0.0 && k + 1.0 <= (double)(g->nr - 1)))
            continue;                      /* outside the recorded range window */
        const double f = u - k;
        const int64_t kk = (int64_t)k;

        const float* e0 = echo + 2 * (n * g->nr + kk);
        const float* e1 = e0 + 2;
        const double w_re = (1.0 - f) * (double)e0[0] + f * (double)e1[0];
        const double w_im = (1.0 - f) * (double)e0[1] + f * (double)e1[1];

        const double phase = 4.0 * ORACLE_PI * range / g->wavelength;
        const double c = cos(phase);
        const double s = sin(phase);
        acc_re += w_re * c - w_im * s;
        acc_im += w_re * s + w_im * c;
    }
    out[0] = acc_re;
    out[1] = acc_im;
}

/* Windowed-sinc kernel: sinc(t) * Hann window of half-width 4 samples. */
static double sinc8_kernel(double t)
{
    const double window = 0.5 + 0.5 * cos(2.0 * ORACLE_PI * t / 8.0);
    if (t == 0.0)
        return window;
    return sin(ORACLE_PI * t) / (ORACLE_PI * t) * window;
}

/* One pixel, all pulses, 8-tap windowed-sinc interpolation. */
static void backproject_pixel_sinc8(const oracle_geometry* g, const float* echo,
                                    const double* antenna_pos, const float* heights, int64_t pixel, double* out)
{
    (void)heights;
    const int64_t ix = pixel % g->nx;
    const int64_t iy = pixel / g->nx;
    const double x = g->x0 + (double)ix * g->dx;
    const double y = g->y0 + (double)iy * g->dy;
    const double z = g->z0;
    double acc_re = 0.0;
    double acc_im = 0.0;

    for (int64_t n = 0; n < g->na; ++n) {
        const double* a = antenna_pos + 3 * n;
        const double ddx = x - a[0];
        const double ddy = y - a[1];
        const double ddz = z - a[2];
        const double range = sqrt(ddx * ddx + ddy * ddy + ddz * ddz);

        const double u = (range - g->r0) / g->dr;
        const double k = floor(u);
        if (!(k - 3.0 >= 0.0 && k + 4.0 <= (double)(g->nr - 1)))
            continue;                      /* stencil outside the recorded range window */
        const int64_t kk = (int64_t)k;

        double w_re = 0.0;
        double w_im = 0.0;
        for (int64_t m = kk - 3; m <= kk + 4; ++m) {
            const double h = sinc8_kernel(u - (double)m);
            const float* e = echo + 2 * (n * g->nr + m);
            w_re += h * (double)e[0];
            w_im += h * (double)e[1];
        }

        const double phase = 4.0 * ORACLE_PI * range / g->wavelength;
        const double c = cos(phase);
        const double s = sin(phase);
        acc_re += w_re * c - w_im * s;
        acc_im += w_re * s + w_im * c;
    }
    out[0] = acc_re;
    out[1] = acc_im;
}

/* One pixel, all pulses, nearest-neighbour interpolation. */
static void backproject_pixel_nearest(const oracle_geometry* g, const float* echo,
                                      const double* antenna_pos, const float* heights, int64_t pixel, double* out)
{
    (void)heights;
    const int64_t ix = pixel % g->nx;
    const int64_t iy = pixel / g->nx;
    const double x = g->x0 + (double)ix * g->dx;
    const double y = g->y0 + (double)iy * g->dy;
    const double z = g->z0;
    double acc_re = 0.0;
    double acc_im = 0.0;

    for (int64_t n = 0; n < g->na; ++n) {
        const double* a = antenna_pos + 3 * n;
        const double ddx = x - a[0];
        const double ddy = y - a[1];
        const double ddz = z - a[2];
        const double range = sqrt(ddx * ddx + ddy * ddy + ddz * ddz);

        const double u = (range - g->r0) / g->dr;
        const double k = floor(u + 0.5);
        if (!(k >= 0.0 && k <= (double)(g->nr - 1)))
            continue;                      /* nearest sample not recorded */
        const float* e = echo + 2 * (n * g->nr + (int64_t)k);

        const double phase = 4.0 * ORACLE_PI * range / g->wavelength;
        const double c = cos(phase);
        const double s = sin(phase);
        acc_re += (double)e[0] * c - (double)e[1] * s;
        acc_im += (double)e[0] * s + (double)e[1] * c;
    }
    out[0] = acc_re;
    out[1] = acc_im;
}

/* One pixel of a non-planar grid: the linear-interpolation steps above with
   the pixel raised to z0 + heights[pixel]. */
/* The geometry with the image plane moved to the height of one pixel. */
static oracle_geometry raise_to_pixel(const oracle_geometry* g, const float* heights, int64_t pixel)
{
    oracle_geometry raised = *g;
    raised.z0 = g->z0 + (double)heights[pixel];
    return raised;
}

static void backproject_pixel_heights(const oracle_geometry* g, const float* echo,
                                      const double* antenna_pos, const float* heights,
                                      int64_t pixel, double* out)
{
    const oracle_geometry raised = raise_to_pixel(g, heights, pixel);
    backproject_pixel(&raised, echo, antenna_pos, NULL, pixel, out);
}

/* The same raised pixel with the windowed-sinc or nearest-sample interpolation. */
static void backproject_pixel_heights_sinc8(const oracle_geometry* g, const float* echo,
                                            const double* antenna_pos, const float* heights,
                                            int64_t pixel, double* out)
{
    const oracle_geometry raised = raise_to_pixel(g, heights, pixel);
    backproject_pixel_sinc8(&raised, echo, antenna_pos, NULL, pixel, out);
}

static void backproject_pixel_heights_nearest(const oracle_geometry* g, const float* echo,
                                              const double* antenna_pos, const float* heights,
                                              int64_t pixel, double* out)
{
    const oracle_geometry raised = raise_to_pixel(g, heights, pixel);
    backproject_pixel_nearest(&raised, echo, antenna_pos, NULL, pixel, out);
}

typedef struct {
    const oracle_geometry* g;
    const float* echo;
    const double* antenna_pos;
    const int64_t* pixels;
    const float* heights;
    double* out;
    int64_t begin, end;
    void (*pixel_fn)(const oracle_geometry*, const float*, const double*, const float*, int64_t,
                     double*);
} oracle_job;

static void* oracle_worker(void* arg)
{
    const oracle_job* job = (const oracle_job*)arg;
    for (int64_t i = job->begin; i < job->end; ++i)
        job->pixel_fn(job->g, job->echo, job->antenna_pos, job->heights, job->pixels[i],
                      job->out + 2 * i);
    return NULL;
}

static int run_pixels(const oracle_geometry* g, const float* echo,
                      const double* antenna_pos, const float* heights, const int64_t* pixels,
                      int64_t npix, double* out, int nthreads,
                      void (*pixel_fn)(const oracle_geometry*, const float*, const double*,
                                       const float*, int64_t, double*))
{
    if (!g || npix < 0 || g->nx <= 0 || g->ny <= 0 || g->na < 0 || g->nr < 0)
        return -1;
    if (npix > 0 && (!pixels || !out))
        return -1;
    if (g->na > 0 && (!antenna_pos || (g->nr > 0 && !echo)))
        return -1;
    for (int64_t i = 0; i < npix; ++i)
        if (pixels[i] < 0 || pixels[i] >= g->nx * g->ny)
            return -1;

    if (nthreads <= 0) {
        long cpus = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = cpus > 0 ? (int)cpus : 1;
    }
    if ((int64_t)nthreads > npix)
        nthreads = npix > 0 ? (int)npix : 1;

    oracle_job* jobs = (oracle_job*)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t* threads = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    char* joinable = (char*)calloc((size_t)nthreads, 1);
    if (!jobs || !threads || !joinable) {
        free(jobs);
        free(threads);
        free(joinable);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].g = g;
        jobs[t].echo = echo;
        jobs[t].antenna_pos = antenna_pos;
        jobs[t].pixels = pixels;
        jobs[t].out = out;
        jobs[t].begin = npix * t / nthreads;
        jobs[t].end = npix * (t + 1) / nthreads;
        jobs[t].pixel_fn = pixel_fn;
        jobs[t].heights = heights;
        if (t == 0)
            continue;
        if (pthread_create(&threads[t], NULL, oracle_worker, &jobs[t]) == 0)
            joinable[t] = 1;
        else
            oracle_worker(&jobs[t]);       /* run inline if a thread cannot start */
    }
    oracle_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (joinable[t])
            pthread_join(threads[t], NULL);
    free(jobs);
    free(threads);
    free(joinable);
    return nthreads;
}

int oracle_backproject(const oracle_geometry* g, const float* echo,
                       const double* antenna_pos, const int64_t* pixels,
                       int64_t npix, double* out, int nthreads)
{
    return run_pixels(g, echo, antenna_pos, NULL, pixels, npix, out, nthreads, backproject_pixel);
}

int oracle_backproject_sinc8(const oracle_geometry* g, const float* echo,
                             const double* antenna_pos, const int64_t* pixels,
                             int64_t npix, double* out, int nthreads)
{
    return run_pixels(g, echo, antenna_pos, NULL, pixels, npix, out, nthreads,
                      backproject_pixel_sinc8);
}

int oracle_backproject_nearest(const oracle_geometry* g, const float* echo,
                               const double* antenna_pos, const int64_t* pixels,
                               int64_t npix, double* out, int nthreads)
{
    return run_pixels(g, echo, antenna_pos, NULL, pixels, npix, out, nthreads,
                      backproject_pixel_nearest);
}

int oracle_backproject_heights(const oracle_geometry* g, const float* echo,
                               const double* antenna_pos, const float* heights,
                               const int64_t* pixels, int64_t npix, double* out, int nthreads)
{
    if (g && g->nx > 0 && g->ny > 0 && !heights)
        return -1;
    return run_pixels(g, echo, antenna_pos, heights, pixels, npix, out, nthreads,
                      backproject_pixel_heights);
}

int oracle_backproject_heights_sinc8(const oracle_geometry* g, const float* echo,
                                     const double* antenna_pos, const float* heights,
                                     const int64_t* pixels, int64_t npix, double* out,
                                     int nthreads)
{
    if (g && g->nx > 0 && g->ny > 0 && !heights)
        return -1;
    return run_pixels(g, echo, antenna_pos, heights, pixels, npix, out, nthreads,
                      backproject_pixel_heights_sinc8);
}

int oracle_backproject_heights_nearest(const oracle_geometry* g, const float* echo,
                                       const double* antenna_pos, const float* heights,
                                       const int64_t* pixels, int64_t npix, double* out,
                                       int nthreads)
{
    if (g && g->nx > 0 && g->ny > 0 && !heights)
        return -1;
    return run_pixels(g, echo, antenna_pos, heights, pixels, npix, out, nthreads,
                      backproject_pixel_heights_nearest);
}
