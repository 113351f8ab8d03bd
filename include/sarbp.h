/*
 * sarbp.h - libsarbp: time-domain SAR backprojection on one GB300 GPU (sm_103a).
 *
 * SARBP-GPU = the page "基于GPU的SAR后向投影成像优化与CUDA加速实践" (a GPU
 * back-projection SAR imaging retrospective). The operation every entry point
 * computes is the one that page defines:
 *
 *   SARBP-GPU §1.1  for every image pixel, visit every pulse, take the echo at
 *                   that pixel's range history, compensate its phase and add
 *                   it coherently into the pixel;
 *   SARBP-GPU §2.2  the per-pulse steps: slant range from the antenna phase
 *                   centre, linear interpolation of the range-compressed echo,
 *                   multiplication by the phase term, accumulation;
 *   SARBP-GPU §3.3  the kernel pseudo-code: uniform range axis (first sample
 *                   and spacing), fraction = index - floor(index), phase
 *                   4*pi*R/lambda applied as exp(+j*phase), monostatic range.
 *
 * In formulas, for pixel p = (x0 + ix*dx, y0 + iy*dy, z0) and antenna
 * positions a_n (n = 0 .. na-1):
 *
 *   R_n  = |p - a_n|,  u = (R_n - r0) / dr,  k = floor(u),  f = u - k
 *   w_n  = (1 - f) e[n][k] + f e[n][k+1]     if 0 <= k and k + 1 <= nr - 1, else 0
 *   I(p) = sum_n w_n * exp(+j 4 pi R_n / lambda)
 *
 * The zero outside the recorded range window is this library's reading of
 * the page's index clamp (the page treats an index outside the echo as a bug).
 *
 * Data layout. All arrays are dense and row-major:
 *   image        complex64 (interleaved float re, im), [ny][nx], x fastest
 *   echoes       complex64, [na][nr], pulse-major, range fastest
 *   antenna_pos  float64, [na][3] = (x, y, z) in metres
 *
 * Threading. A plan may be used from one host thread and one stream at a
 * time. Different plans are independent.
 *
 * CUDA graphs. The device-buffer calls (sarbp_backproject,
 * sarbp_backproject_heights, sarbp_backproject_volume, sarbp_range_compress,
 * sarbp_backproject_raw)
 * only enqueue kernels and memsets on `stream`: they allocate nothing and do
 * not synchronise, so they may be captured into a CUDA graph once the plan
 * exists; each replay does the same work on the buffers given at capture.
 * One exception: on a plan made without SARBP_SINC8 in its flags, the first
 * SARBP_SINC8 call allocates the plan's windowed-sinc coefficient rows (see
 * sarbp_plan), so that call must not be the first one captured.
 * The host-buffer calls synchronise and cannot be captured.
 *
 * Errors. No call throws or aborts. Every call returns a status; argument
 * checks happen before any GPU work is queued, and a call that returns an
 * error other than SARBP_ERR_CUDA has queued nothing. Errors raised by the
 * GPU after a call returned surface on a later call or on stream
 * synchronisation, as usual for asynchronous CUDA work.
 */
#ifndef SARBP_H
#define SARBP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SARBP_VERSION_MAJOR 0
#define SARBP_VERSION_MINOR 1

typedef enum sarbp_status {
    SARBP_OK = 0,
    SARBP_ERR_INVALID_ARG = 1,        /* null/misaligned pointer, bad size or geometry   */
    SARBP_ERR_PLAN_MISMATCH = 2,      /* params disagree with the plan's fixed fields     */
    SARBP_ERR_CUDA = 3,               /* a CUDA call failed; see sarbp_last_error         */
    SARBP_ERR_OOM = 4,                /* device or host allocation failed                 */
    SARBP_ERR_UNSUPPORTED_DEVICE = 5, /* current device is not compute capability 10.3    */
    SARBP_ERR_SCRATCH_TOO_SMALL = 6   /* one pulse's table row exceeds the fixed scratch
                                         of sarbp_backproject_noalloc                    */
} sarbp_status;

/* params.flags */
#define SARBP_ACCUMULATE 1u  /* add into the image instead of overwriting it: lets a
                                caller backproject pulses in batches (SARBP-GPU §3.3
                                stream overlap of echo loading and computation)       */

#define SARBP_SINC8 2u       /* interpolate with an 8-tap windowed sinc instead of linearly
                                (SARBP-GPU §2.2: sinc interpolation, more accurate and
                                costlier): w = sum_{m=k-3}^{k+4} e[m] h(u - m),
                                h(t) = sinc(t) (1/2 + 1/2 cos(2 pi t / 8)), zero unless
                                the whole stencil lies in 0 .. nr-1                    */

#define SARBP_NEAREST 4u     /* nearest-neighbour interpolation (SARBP-GPU §2.2: fastest,
                                least accurate): w = e[k], k = floor(u + 1/2), zero
                                unless 0 <= k <= nr-1. Not combinable with SINC8.  */

typedef struct sarbp_params {
    int32_t nx, ny;       /* image width (x) and height (y), pixels, >= 0             */
    int32_t na, nr;       /* pulses and range bins, >= 0                              */
    double x0, y0, z0;    /* position of pixel (0, 0), metres                         */
    double dx, dy;        /* pixel spacing, metres, > 0                               */
    double r0, dr;        /* range of bin k is r0 + k*dr, metres; dr > 0              */
    double wavelength;    /* carrier wavelength lambda = c / fc, metres, > 0
                             (SARBP-GPU §4.2: the carrier, not the bandwidth one)     */
    uint32_t flags;       /* SARBP_ACCUMULATE with at most one of SARBP_SINC8,
                             SARBP_NEAREST (default: linear interpolation)          */
} sarbp_params;

typedef struct sarbp_plan_s* sarbp_plan_t;

/*
 * sarbp_plan - fix the problem sizes and allocate the plan's device scratch.
 *
 * out    receives the new plan (set to NULL on error).
 * p      host pointer. Fixed for the plan's lifetime: nx, ny, na, nr, dx, dy,
 *        dr. The other fields may change from call to call.
 *
 * Uses the CUDA device current on the calling thread; later calls must run
 * with that device current. Scratch owned by the plan: the pre-multiplied
 * echo table (na x W x 16 bytes, W <= nr + 24, where W covers the image's
 * range extent), one int per pulse, one complex64 per range bin, and the
 * partial-sum buffers of the work split (about 40 MB). With SARBP_SINC8 in
 * p->flags also the windowed-sinc coefficient rows (na x W x 64 bytes: the
 * degree-7 polynomial of the interpolant on each bin); without it the first
 * SARBP_SINC8 call allocates them. Each call passes its own flags; p->flags
 * only decides this allocation and what sarbp_plan_describe counts. Returns SARBP_ERR_INVALID_ARG for negative sizes,
 * non-finite or non-positive dx, dy, dr, wavelength, unknown flags, or image
 * sizes above 2^30 pixels; SARBP_ERR_UNSUPPORTED_DEVICE off compute
 * capability 10.3; SARBP_ERR_OOM if an allocation fails.
 */
sarbp_status sarbp_plan(sarbp_plan_t* out, const sarbp_params* p);

/*
 * sarbp_backproject - enqueue one backprojection on `stream` and return.
 *
 * image        device pointer, complex64 [ny][nx], caller-owned, 8-byte aligned.
 *              Overwritten, or added into when params->flags has SARBP_ACCUMULATE.
 *              With SARBP_SINC8 or SARBP_NEAREST the echo is interpolated with
 *              the windowed sinc or the nearest sample instead of linearly.
 * echoes       device pointer, complex64 [na][nr], caller-owned, 8-byte aligned.
 * antenna_pos  device pointer, float64 [na][3], caller-owned, 8-byte aligned.
 * params       host pointer; nx, ny, na, nr, dx, dy, dr must equal the plan's
 *              (else SARBP_ERR_PLAN_MISMATCH).
 * stream       a cudaStream_t of the plan's device (NULL = legacy default stream).
 *
 * The inputs must stay valid and unmodified until the work on `stream` has
 * finished. A pulse whose antenna position is not finite contributes nothing.
 * Echo samples should be finite: a non-finite sample makes non-finite every
 * pixel whose interpolation uses it, and may also reach the other pixels of
 * the same 32-pixel row segment that take their samples from the adjacent
 * bin in that pulse (the two-bin form combines both bins). Samples no pixel
 * can reach are never used.
 * Two calls with identical inputs give bitwise identical images (the pulse
 * sum has a fixed order). Null pointers are accepted only where the matching
 * array is empty.
 */
sarbp_status sarbp_backproject(sarbp_plan_t plan, void* image, const void* echoes,
                               const double* antenna_pos, const sarbp_params* params,
                               void* stream);

/*
 * sarbp_backproject_host - the same operation on HOST buffers.
 *
 * image, echoes, antenna_pos are host pointers with the layouts above. From
 * the antenna positions the call finds, in float64 on the host, the band of
 * range bins that any pixel can reach (nearest and farthest point of the image
 * for every pulse, plus six bins of margin each side); only that band of every
 * pulse crosses to the device. It backprojects the band on `stream` against
 * the same range axis and waits for the stream: when it returns SARBP_OK the
 * image is on the host. The result equals sarbp_backproject's to float32
 * rounding.
 *
 * Transport: an echo or image buffer that is pinned and mapped into the
 * device's address space (cudaHostAlloc, cudaHostRegister, or any pinned
 * allocation on a unified-addressing system) is read or written in place by
 * the kernels, without a staging copy; any other buffer (pageable memory) is
 * staged through device buffers owned by the plan (allocated on first use,
 * kept until sarbp_destroy). Both give the same image bit for bit. With
 * SARBP_ACCUMULATE the host image is read and added into.
 */
sarbp_status sarbp_backproject_host(sarbp_plan_t plan, void* image, const void* echoes,
                                    const double* antenna_pos, const sarbp_params* params,
                                    void* stream);

/*
 * sarbp_backproject_streamed - sarbp_backproject_host with the pulses taken
 * in chunks and the copies overlapped with the computation (SARBP-GPU §3.3:
 * pulses processed in batches, with transfers to the GPU overlapped with its
 * work on streams).
 *
 * image, echoes, antenna_pos: HOST pointers as for sarbp_backproject_host.
 * chunk_pulses: pulses per chunk, >= 1 (values above na mean one chunk).
 * params->flags: as for sarbp_backproject (any interpolation).
 *
 * For chunk c (pulses c*chunk_pulses ...) the call finds on the host the band
 * of range bins those pulses can reach from the image, copies that band into
 * one of two device staging buffers on the plan's own copy stream, and
 * backprojects it on `stream` into a device image, adding into the sum of the
 * chunks before it; the copy of chunk c+1 runs while chunk c is computed.
 * Pinned host memory is needed for the copies to overlap. The call returns
 * when the image is on the host. With one chunk the result is bitwise that of
 * sarbp_backproject_host; with several, the pulse sum is grouped by chunk and
 * agrees to float32 rounding.
 *
 * Device memory owned by the plan, allocated on first use and kept until
 * sarbp_destroy: the image, the antenna positions and two staging buffers of
 * chunk_pulses x nr x 8 bytes. SARBP_ERR_INVALID_ARG for chunk_pulses < 1;
 * SARBP_ERR_PLAN_MISMATCH as for sarbp_backproject_host.
 */
sarbp_status sarbp_backproject_streamed(sarbp_plan_t plan, void* image, const void* echoes,
                                        const double* antenna_pos, const sarbp_params* params,
                                        int32_t chunk_pulses, void* stream);

/*
 * sarbp_backproject_volume - backprojection onto a voxel grid: nz planes at
 * heights z0 + iz * dz (iz = 0 .. nz-1), plane iz being the image
 * sarbp_backproject makes with params->z0 replaced by that height (SARBP-GPU
 * §3.3: the pixel grid may leave the ground plane; with a two-dimensional
 * aperture, e.g. several passes at different heights given as one pulse list,
 * the voxels resolve height).
 *
 * volume  device pointer, complex64 [nz][ny][nx], caller-owned, 8-byte aligned.
 *         Overwritten, or added into with SARBP_ACCUMULATE.
 * nz, dz  number of planes (>= 0) and their spacing in metres (finite).
 * echoes, antenna_pos, params, stream, the plan and the interpolation flags:
 *         as for sarbp_backproject. The planes are enqueued one after another
 *         on `stream`; each equals the corresponding sarbp_backproject call
 *         bit for bit.
 */
sarbp_status sarbp_backproject_volume(sarbp_plan_t plan, void* volume, const void* echoes,
                                      const double* antenna_pos, const sarbp_params* params,
                                      int32_t nz, double dz, void* stream);

/*
 * Pixels on a height map (SARBP-GPU §3.3 remarks that the range history may
 * have to take terrain elevation into account; the page gives no formula, so
 * this is the plain reading): pixel (ix, iy) sits at
 *   (x0 + ix*dx, y0 + iy*dy, z0 + heights[iy*nx + ix])
 * and the sum is otherwise that of sarbp_backproject.
 *
 * sarbp_plan_heights - as sarbp_plan, for heights within [h_min, h_max]
 * (metres, added to z0). The table rows cover the slab z0 + [h_min, h_max]
 * over the image, so W grows with h_max - h_min. SARBP_ERR_INVALID_ARG as for
 * sarbp_plan, and also for non-finite bounds or h_min > h_max.
 */
sarbp_status sarbp_plan_heights(sarbp_plan_t* out, const sarbp_params* p, double h_min,
                                double h_max);

/*
 * sarbp_backproject_heights - enqueue one backprojection over a height map.
 *
 * heights  device pointer, float32 [ny][nx], caller-owned, 4-byte aligned,
 *          read during the work on `stream`. Each value is clamped to the
 *          plan's [h_min, h_max] (a NaN height is taken as h_min).
 * image, echoes, antenna_pos, params, stream: as for sarbp_backproject
 * (SARBP_ACCUMULATE, SARBP_SINC8 and SARBP_NEAREST included). The plan must
 * come from sarbp_plan_heights, and
 * plans from sarbp_plan_heights are refused by sarbp_backproject and
 * sarbp_backproject_host (SARBP_ERR_PLAN_MISMATCH either way).
 *
 * Every pixel takes the float64 range to its row's centre at the row's mean
 * height and a float32 difference to the pixel, so this path runs slower than
 * the planar one; results are deterministic like sarbp_backproject's.
 */
sarbp_status sarbp_backproject_heights(sarbp_plan_t plan, void* image, const void* echoes,
                                       const double* antenna_pos, const float* heights,
                                       const sarbp_params* params, void* stream);

/* Bytes copied host-to-device and device-to-host by the plan's last
   sarbp_backproject_host call. */
sarbp_status sarbp_host_transfer_bytes(sarbp_plan_t plan, uint64_t* h2d, uint64_t* d2h);

/* sarbp_destroy - free the plan and its scratch. NULL is accepted. The caller
   must make sure no work that uses the plan is still running. */
sarbp_status sarbp_destroy(sarbp_plan_t plan);

/*
 * Testing aid (host-side failure injection): the countdown-th device
 * allocation the library makes from now on (plans, host-call staging,
 * range-compression plans) fails as if cudaMalloc had returned
 * cudaErrorMemoryAllocation, without touching the GPU; 0 disables. The call
 * that meets the failure returns SARBP_ERR_OOM and frees what it had
 * allocated. Process-wide, not meant for production use.
 */
void sarbp_debug_fail_alloc(int32_t countdown);

/*
 * Testing aid (host only, needs no GPU): the 64 coefficients of the
 * windowed-sinc tap polynomials the library's sinc table is built from.
 * out[8 * (d + 3) + n], d = -3 .. 4, n = 0 .. 7, is the coefficient of s^n in
 * the degree-7 interpolant (eight Chebyshev nodes of the bin) of the weight
 * h(1/2 + s - d), h(t) = sinc(t) (1 + cos(pi t / 4)) / 2, on s in [-1/2, 1/2]
 * (the interpolant of the 8-tap windowed sinc on bin k at u = k + 1/2 + s is
 * sum_n s^n sum_d out[8 (d + 3) + n] e_{k+d}). out: host pointer to 64 floats.
 * Returns SARBP_ERR_INVALID_ARG for a NULL pointer.
 */
sarbp_status sarbp_debug_sinc_taps(float* out);

/* Static, never-NULL description of a status code. */
const char* sarbp_status_string(sarbp_status status);

/* The message of the most recent CUDA failure seen by this plan ("" if none).
   The pointer stays valid until the plan's next call. */
const char* sarbp_last_error(sarbp_plan_t plan);

/* Plan facts, for tests and benchmarks. */
typedef struct sarbp_plan_info {
    int32_t tile_x, tile_y;       /* pixels per work tile                              */
    int32_t tiles;                /* work tiles covering the image                     */
    int32_t ctas;                 /* persistent CTAs of the main kernel                */
    int32_t ctas_per_sm, sms;     /* occupancy used to size the grid                   */
    int32_t window;               /* W: table entries per pulse                        */
    int32_t full_window;          /* 1 if every table row spans the whole range axis   */
    int32_t kernels_per_call;     /* kernel launches one sarbp_backproject enqueues
                                     with the plan's own params (flags included)      */
    size_t scratch_bytes;         /* device memory held by the plan                    */
} sarbp_plan_info;

sarbp_status sarbp_plan_describe(sarbp_plan_t plan, sarbp_plan_info* out);

/*
 * Kernel timing. When enabled, each sarbp_backproject records CUDA events
 * around its main backprojection kernel on the call's stream.
 * sarbp_kernel_times waits for the recorded events, returns the summed
 * milliseconds and the number of timed launches since the previous query,
 * and resets both. Timing adds two event records per call and no sync.
 */
sarbp_status sarbp_set_timing(sarbp_plan_t plan, int enable);
sarbp_status sarbp_kernel_times(sarbp_plan_t plan, double* main_ms, int32_t* launches);

/*
 * Range compression (matched filtering), the step that produces the echoes
 * backprojection consumes (SARBP-GPU §3.1: FFT every pulse along range,
 * multiply by the matched filter's frequency response, optionally weighted by
 * a Hamming window to lower the sidelobes, inverse FFT, all pulses as one
 * batch). For every pulse n and 0 <= k < ns:
 *
 *   rc[n][k] = sum_{l=0}^{nref-1} raw[n][k + l] * conj(ref[l])   (raw = 0 beyond ns)
 *
 * computed through FFTs of size N, the smallest power of two >= ns + nref - 1
 * (no circular wrap), N <= 16384. With a window the filter spectrum is
 * weighted over |f| <= b/2 and zeroed outside (f = signed frequency in cycles
 * per sample, b = band_fraction, the chirp bandwidth over the sampling rate):
 * SARBP_WINDOW_HAMMING by 0.54 + 0.46 cos(2 pi f / b); SARBP_WINDOW_TAYLOR by
 * Taylor's weighting 1 + 2 sum_{m=1}^{4} F_m cos(2 pi m f / b) with nbar = 5
 * and a 35 dB design sidelobe level (A = acosh(10^(35/20)) / pi,
 * sigma^2 = 25 / (A^2 + 4.5^2),
 * F_m = (-1)^(m+1) prod_i (1 - m^2 / (sigma^2 (A^2 + (i - 1/2)^2)))
 *       / (2 prod_{i != m} (1 - m^2 / i^2)), i = 1 .. 4).
 * SARBP_WINDOW_NONE is the plain matched filter.
 */
#define SARBP_WINDOW_NONE 0u
#define SARBP_WINDOW_HAMMING 1u
#define SARBP_WINDOW_TAYLOR 2u

typedef struct sarbp_rc_params {
    int32_t na;            /* pulses                                               */
    int32_t ns;            /* samples per pulse, input and output                  */
    int32_t nref;          /* samples of the reference (transmitted) pulse         */
    uint32_t window;       /* SARBP_WINDOW_NONE, _HAMMING or _TAYLOR              */
    double band_fraction;  /* b in (0, 1] for the Hamming and Taylor windows      */
} sarbp_rc_params;

typedef struct sarbp_rc_plan_s* sarbp_rc_plan_t;

/* Build the filter spectrum (N x 8 bytes of device memory, the plan's only
   allocation) from `ref` (device, complex64 [nref], read only during this
   call's work on `stream`). INVALID_ARG for bad sizes, N > 16384, an unknown
   window or b outside (0, 1]; SARBP_ERR_OOM if the allocation fails. */
sarbp_status sarbp_rc_plan(sarbp_rc_plan_t* out, const sarbp_rc_params* p, const void* ref,
                           void* stream);

/* Enqueue the compression of raw (device, complex64 [na][ns]) into out
   (device, complex64 [na][ns]); the two must not overlap. One CTA per pulse. */
sarbp_status sarbp_range_compress(sarbp_rc_plan_t plan, void* out, const void* raw, void* stream);

/* Free the plan. NULL is accepted. */
sarbp_status sarbp_rc_destroy(sarbp_rc_plan_t plan);

/*
 * sarbp_backproject_raw - raw echoes to image in one call: range compression
 * (SARBP-GPU §3.1, as sarbp_range_compress) feeding the backprojection
 * (SARBP-GPU §2.2, §3.3, as sarbp_backproject with linear interpolation).
 *
 * raw          device pointer, complex64 [na][nr] raw (uncompressed) echoes,
 *              caller-owned, 8-byte aligned; sample k of the compressed row
 *              is the echo from range r0 + k dr, as for sarbp_backproject.
 * rc           a range-compression plan with rc na == params->na and
 *              ns == params->nr, made on the plan's device (else
 *              SARBP_ERR_PLAN_MISMATCH).
 * plan, image, antenna_pos, params, stream: as for sarbp_backproject;
 *              params->flags may carry SARBP_ACCUMULATE only (SARBP_SINC8 or
 *              SARBP_NEAREST: SARBP_ERR_INVALID_ARG); height-map plans are
 *              refused (SARBP_ERR_PLAN_MISMATCH).
 *
 * Per pulse, one kernel compresses the raw row and keeps, in shared memory,
 * only the compressed samples of the band of range bins the image can reach
 * (the plan's table window), and writes the plan's echo-table entries from
 * them: the compressed frame is never written to global memory. The image
 * equals sarbp_range_compress followed by sarbp_backproject to float32
 * rounding (the same arithmetic in both; only where the samples live
 * differs). Enqueues on `stream` and returns; allocates nothing.
 */
sarbp_status sarbp_backproject_raw(sarbp_plan_t plan, sarbp_rc_plan_t rc, void* image,
                                   const void* raw, const double* antenna_pos,
                                   const sarbp_params* params, void* stream);

/*
 * sarbp_backproject_noalloc - the same backprojection without any device
 * memory allocation. The page has no counterpart: this is an interface for
 * callers that cannot allocate GPU memory themselves, for example a plug-in
 * that is only handed buffers by its host application, a framework whose
 * memory pool owns the whole device, or a real-time radar loop that forbids
 * cudaMalloc (it synchronises the device and has unbounded latency) once
 * processing has started. Such callers cannot create a plan either.
 *
 * image, echoes, antenna_pos, params, stream: as for sarbp_backproject. All
 * sizes come from params; no plan is involved. Linear interpolation only:
 * SARBP_SINC8 and SARBP_NEAREST are rejected with SARBP_ERR_INVALID_ARG.
 *
 * Scratch: a fixed, file-scope device array of SARBP_NOALLOC_SCRATCH_BYTES
 * (16 MiB) that every GPU loading the library holds until the process exits.
 * Pulses are processed in chunks whose echo-table rows fit in it, so the
 * pulse sum is grouped differently from sarbp_backproject and results agree
 * to float32 rounding, not bitwise. Problems where a single pulse's table row
 * (about (image range extent / dr) x 16 bytes) does not fit are rejected with
 * SARBP_ERR_SCRATCH_TOO_SMALL before any work is queued.
 *
 * Every call looks up the array's device address in the CUDA context current
 * on the calling thread (cudaGetSymbolAddress, which allocates nothing). The
 * array exists once per context that loads the library: after a
 * cudaDeviceReset, or in another context on the same device, it has a new
 * address and new, uninitialised contents, and the next call uses that one.
 * The first call in a context loads the array; make that first call before
 * any stream capture. The call allocates nothing: no cudaMalloc, no cudaFree,
 * no allocating library routine.
 *
 * All calls share the one array and it keeps the last call's contents; the
 * parts that must start at zero are cleared by each call. Calls whose work
 * overlaps on the GPU (for example on two streams, or from two threads) race
 * on the array: serialise them.
 */
#define SARBP_NOALLOC_SCRATCH_BYTES (16u << 20)
sarbp_status sarbp_backproject_noalloc(void* image, const void* echoes,
                                       const double* antenna_pos, const sarbp_params* params,
                                       void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SARBP_H */
