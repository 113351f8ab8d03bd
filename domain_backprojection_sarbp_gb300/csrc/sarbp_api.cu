// sarbp_api.cu - host side of libsarbp: argument checks, plans, launches.
//
// SARBP-GPU = the page "基于GPU的SAR后向投影成像优化与CUDA加速实践"; the operation
// and its parameters follow §2.2 and the kernel pseudo-code of §3.3 (range
// axis given by its first sample and spacing, carrier wavelength, pixel grid
// origin and spacing, antenna phase centre per pulse). The page has no
// library interface; this one fixes the sizes in a plan so that every call
// only enqueues kernels and never allocates.
#include "../../include/sarbp.h"
#include "sarbp_internal.h"

#include <cmath>
#include <cstdint>
#include <atomic>
#include <cstring>
#include <limits>
#include <new>
#include <string>
#include <utility>
#include <vector>

using namespace sarbp;

struct sarbp_plan_s {
    sarbp_params p{};
    int device = -1;
    int sms = 0, ctas_per_sm = 0;
    int tiles_x = 0, tiles_y = 0, tiles = 0;
    int W = 0, full_window = 0;
    int heights_mode = 0;            // plan made by sarbp_plan_heights
    double h_min = 0.0, h_max = 0.0; // its height bounds
    float4* table_alloc = nullptr;   // (na * W + 2 * TABLE_PAD) entries
    float4* sinc_alloc = nullptr;    // (4 na W + 8 TABLE_PAD) entries: windowed-sinc
                                     // coefficient rows, made by the plan when its flags
                                     // carry SARBP_SINC8, else by the first sinc call
    int* klo = nullptr;              // na
    float2* psi = nullptr;           // nr + 1: per-bin phasors (windowed-sinc interpolation),
                                     // then one word: the wide-sinc flag of the last call,
                                     // then the sinc work split: SPLIT_CELLS + 1 words of
                                     // cost scratch and max_ctas + 1 CTA start units
    float4* partial = nullptr;       // 2 * max_ctas * TILE_PIX / 2
    int max_ctas = 0;
    size_t scratch_bytes = 0;
    // host-buffer entry point staging (allocated on first use)
    void* d_image = nullptr;
    void* d_echo = nullptr;
    double* d_pos = nullptr;
    size_t last_h2d = 0, last_d2h = 0;   // bytes moved by the last host-buffer call
    // streamed entry point: two staging buffers, a copy stream, their events
    void* d_stage[2] = {nullptr, nullptr};
    size_t stage_bytes = 0;
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t copied[2] = {nullptr, nullptr}, consumed[2] = {nullptr, nullptr};
    cudaEvent_t call_start = nullptr;
    // kernel timing
    bool timing = false;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> events;
    size_t events_used = 0;
    std::string last_error;
};

namespace {

constexpr double PI = 3.14159265358979323846;

bool isfin(double v) { return std::isfinite(v); }

sarbp_status cuda_fail(sarbp_plan_s* plan, cudaError_t e, const char* what)
{
    if (plan) {
        plan->last_error = std::string(what) + ": " + cudaGetErrorString(e);
    }
    return e == cudaErrorMemoryAllocation ? SARBP_ERR_OOM : SARBP_ERR_CUDA;
}

sarbp_status check_sizes(const sarbp_params* p)
{
    if (!p)
        return SARBP_ERR_INVALID_ARG;
    if (p->nx < 0 || p->ny < 0 || p->na < 0 || p->nr < 0)
        return SARBP_ERR_INVALID_ARG;
    if ((int64_t)p->nx * (int64_t)p->ny > (int64_t(1) << 30))
        return SARBP_ERR_INVALID_ARG;
    if (!(isfin(p->dx) && p->dx > 0 && isfin(p->dy) && p->dy > 0))
        return SARBP_ERR_INVALID_ARG;
    if (!(isfin(p->dr) && p->dr > 0))
        return SARBP_ERR_INVALID_ARG;
    return SARBP_OK;
}

sarbp_status check_geometry(const sarbp_params* p)
{
    if (!(isfin(p->x0) && isfin(p->y0) && isfin(p->z0) && isfin(p->r0)))
        return SARBP_ERR_INVALID_ARG;
    if (!(isfin(p->wavelength) && p->wavelength > 0))
        return SARBP_ERR_INVALID_ARG;
    if (p->flags & ~(SARBP_ACCUMULATE | SARBP_SINC8 | SARBP_NEAREST))
        return SARBP_ERR_INVALID_ARG;
    if ((p->flags & SARBP_SINC8) && (p->flags & SARBP_NEAREST))
        return SARBP_ERR_INVALID_ARG;
    return SARBP_OK;
}

bool aligned8(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 7u) == 0; }

double tile_qmax(double dx, double dy)
{
    const double hx = 0.5 * (TILE_X - 1) * dx, hy = 0.5 * (TILE_Y - 1) * dy;
    return std::sqrt(hx * hx + hy * hy);
}

// Reach of a tile of a height-map plan: from the tile centre at the mid height
// to any pixel whose height lies in [h_min, h_max].
double tile_qmax3(double dx, double dy, double h_span)
{
    const double q = tile_qmax(dx, dy), hz = 0.5 * h_span;
    return std::sqrt(q * q + hz * hz);
}

unsigned long long frac_fixed64(double v)
{
    double f = v - std::floor(v);
    if (!(f >= 0.0 && f < 1.0))
        f = 0.0;
    const double scaled = std::ldexp(f, 64);
    if (scaled >= 18446744073709551615.0)
        return ~0ull;
    return (unsigned long long)scaled;
}

int ctas_for(const sarbp_plan_s* plan)
{
    const long long units = (long long)plan->tiles * plan->p.na;
    long long want = (units + MIN_PULSES_PER_CTA - 1) / MIN_PULSES_PER_CTA;
    if (want < 1)
        want = 1;
    return (int)std::min<long long>(plan->max_ctas, want);
}

BpConst make_const(const sarbp_plan_s* plan, const sarbp_params* p)
{
    BpConst k{};
    k.nx = p->nx;
    k.ny = p->ny;
    k.na = p->na;
    k.nr = p->nr;
    k.echo_stride = p->nr;
    k.W = plan->W;
    k.tiles_x = plan->tiles_x;
    k.tiles = plan->tiles;
    k.full_window = plan->full_window;
    k.ctas = ctas_for(plan);
    k.flags = p->flags;
    k.tw = (p->flags & SARBP_SINC8) ? 4 * plan->W : plan->W;
    k.units = (long long)plan->tiles * p->na;
    k.x0 = p->x0;
    k.y0 = p->y0;
    k.z0 = p->z0;
    k.dx = p->dx;
    k.dy = p->dy;
    k.r0 = p->r0;
    k.dr = p->dr;
    k.inv_dr = 1.0 / p->dr;
    k.rect_x0 = p->x0;
    k.rect_x1 = p->x0 + ((double)plan->tiles_x * TILE_X - 1.0) * p->dx;
    k.rect_y0 = p->y0;
    k.rect_y1 = p->y0 + ((double)plan->tiles_y * TILE_Y - 1.0) * p->dy;
    k.qmax = tile_qmax(p->dx, p->dy);
    // Taylor remainder allowed on the fast path: 5e-5 rad of phase
    k.fast_tol_bins = 5e-5 * p->wavelength / (4.0 * PI * p->dr);
    const double alpha = 2.0 * p->dr / p->wavelength;   // turns per bin
    const double beta = 2.0 * p->r0 / p->wavelength;    // turns at bin 0
    k.alpha_fx = frac_fixed64(alpha);
    k.beta_fx = frac_fixed64(beta);
    k.c_phase = (float)(2.0 * PI * alpha);
    k.inv_c = (float)(1.0 / (2.0 * PI * alpha));
    const double turns = alpha - std::floor(alpha);      // exp(-j c) = exp(-j 2 pi frac(alpha))
    k.rot_re = (float)std::cos(2.0 * PI * turns);
    k.rot_im = (float)-std::sin(2.0 * PI * turns);
    k.hrt_re = 0.5f * k.rot_re;                            // halving a float is exact
    k.hrt_im = 0.5f * k.rot_im;
    const double half_turns = 0.5 * alpha - std::floor(0.5 * alpha);   // exp(+j c / 2)
    k.hrot_re = (float)std::cos(2.0 * PI * half_turns);
    k.hrot_im = (float)std::sin(2.0 * PI * half_turns);
    k.i0 = -0.5f * (float)(TILE_X - 1);
    k.dx_f = (float)p->dx;
    k.dy_f = (float)p->dy;
    k.inv_dr_f = (float)(1.0 / p->dr);
    k.heights_mode = plan->heights_mode;
    k.z_lo = p->z0 + plan->h_min;
    k.z_hi = p->z0 + plan->h_max;
    k.z_mid = p->z0 + 0.5 * (plan->h_min + plan->h_max);
    k.qmax3 = tile_qmax3(p->dx, p->dy, plan->h_max - plan->h_min);
    k.h_lo_f = (float)plan->h_min;
    k.h_hi_f = (float)plan->h_max;
    const double h_mid = 0.5 * (plan->h_min + plan->h_max);
    k.h_mid_f = (float)h_mid;
    k.h_mid_lo = (float)(h_mid - (double)k.h_mid_f);
    k.dy_lo = (float)(p->dy - (double)k.dy_f);
    k.r0_hi = (float)p->r0;
    k.r0_lo = (float)(p->r0 - (double)k.r0_hi);
    k.idr_hi = (float)(1.0 / p->dr);
    k.idr_lo = (float)(1.0 / p->dr - (double)k.idr_hi);
    return k;
}

void free_plan(sarbp_plan_s* plan)
{
    if (!plan)
        return;
    cudaFree(plan->table_alloc);
    cudaFree(plan->sinc_alloc);
    cudaFree(plan->klo);
    cudaFree(plan->psi);
    cudaFree(plan->partial);
    cudaFree(plan->d_image);
    cudaFree(plan->d_echo);
    cudaFree(plan->d_pos);
    for (int b = 0; b < 2; ++b) {
        cudaFree(plan->d_stage[b]);
        if (plan->copied[b])
            cudaEventDestroy(plan->copied[b]);
        if (plan->consumed[b])
            cudaEventDestroy(plan->consumed[b]);
    }
    if (plan->call_start)
        cudaEventDestroy(plan->call_start);
    if (plan->copy_stream)
        cudaStreamDestroy(plan->copy_stream);
    for (auto& ev : plan->events) {
        cudaEventDestroy(ev.first);
        cudaEventDestroy(ev.second);
    }
    delete plan;
}

// Tiles whose units are split between CTAs need the reduce kernel.
bool any_split_tile(const BpConst& k)
{
    if (k.ctas <= 1)
        return false;
    for (long long b = 1; b < k.ctas; ++b) {
        const long long s = b * k.units / k.ctas;
        if (s % k.na != 0 && s < k.units)
            return true;                    // a CTA boundary inside a tile
    }
    return false;
}

}  // namespace

namespace {

// The device address of a pinned host buffer mapped into the device's
// address space, or null for any other buffer (pageable memory, device
// memory, a null pointer).
void* mapped_host(const void* p)
{
    if (!p)
        return nullptr;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// The band of range bins that pulses n0 .. n1-1 can reach from the image,
// found in float64 on the host from the antenna positions: for every pulse
// the nearest and farthest point of the image rectangle, plus margins (six
// bins below, seven above). Pulses with a non-finite position contribute
// nothing and are left out. Returns false when no pulse reaches the axis.
// The square root and the floor are monotone, so the band follows from the
// smallest and largest squared distances with two square roots in all.
bool host_band(const sarbp_params* params, const double* antenna_pos, int n0, int n1,
               long long* lo, long long* hi)
{
    const double xa = params->x0, xb = params->x0 + (params->nx - 1) * params->dx;
    const double ya = params->y0, yb = params->y0 + (params->ny - 1) * params->dy;
    double d2min = HUGE_VAL, d2max = -1.0;
    for (int n = n0; n < n1 && params->nr >= 2; ++n) {
        const double ax = antenna_pos[3 * (size_t)n], ay = antenna_pos[3 * (size_t)n + 1],
                     az = antenna_pos[3 * (size_t)n + 2];
        if (!(isfin(ax) && isfin(ay) && isfin(az)))
            continue;
        const double dz = params->z0 - az;
        const double nx_ = std::min(std::max(ax, xa), xb) - ax;
        const double ny_ = std::min(std::max(ay, ya), yb) - ay;
        const double fx = std::max(std::fabs(xa - ax), std::fabs(xb - ax));
        const double fy = std::max(std::fabs(ya - ay), std::fabs(yb - ay));
        d2min = std::min(d2min, nx_ * nx_ + ny_ * ny_ + dz * dz);
        d2max = std::max(d2max, fx * fx + fy * fy + dz * dz);
    }
    long long band_lo = params->nr, band_hi = -1;
    if (d2max >= 0.0) {
        const double ulo = std::floor((std::sqrt(d2min) - params->r0) / params->dr) - 6.0;
        const double uhi = std::floor((std::sqrt(d2max) - params->r0) / params->dr) + 7.0;
        band_lo = (long long)std::min(std::max(ulo, 0.0), (double)params->nr);
        band_hi = (long long)std::max(std::min(uhi, (double)params->nr - 1.0), -1.0);
    }
    *lo = band_lo;
    *hi = band_hi;
    return band_hi >= band_lo;
}

// The windowed-sinc coefficient rows: four float4 per table bin, zero pads of
// 4 TABLE_PAD entries at both ends.
cudaError_t ensure_sinc_table(sarbp_plan_s* plan)
{
    if (plan->sinc_alloc)
        return cudaSuccess;
    const size_t bytes = ((size_t)plan->p.na * 4 * plan->W + 8 * TABLE_PAD) * sizeof(float4);
    cudaError_t e = device_alloc(reinterpret_cast<void**>(&plan->sinc_alloc), bytes);
    if (e == cudaSuccess) {
        e = cudaMemset(plan->sinc_alloc, 0, bytes);
        if (e != cudaSuccess) {
            cudaFree(plan->sinc_alloc);
            plan->sinc_alloc = nullptr;
        }
    }
    if (e == cudaSuccess)
        plan->scratch_bytes += bytes;
    return e;
}

// Queue the three kernels of one backprojection. Arguments are already
// checked; params may describe a band of the plan's range axis (fewer bins,
// shifted r0), which the plan's table rows always cover. With a
// range-compression plan rc, `echoes` is the raw frame and the table rows
// come from the fused compression kernel (linear interpolation only).
sarbp_status enqueue_backprojection(sarbp_plan_s* plan, void* image, const void* echoes,
                                    const double* antenna_pos, const sarbp_params* params,
                                    cudaStream_t s, const float* heights = nullptr,
                                    long long echo_stride = 0,
                                    const sarbp_rc_plan_s* rc = nullptr)
{
    cudaError_t e = cudaSuccess;
    const long long pixels = (long long)params->nx * params->ny;
    if (pixels == 0)
        return SARBP_OK;
    if (params->na == 0 || params->nr < 2) {
        // no pulse can contribute: the image is the zero sum
        if (!(params->flags & SARBP_ACCUMULATE)) {
            e = cudaMemsetAsync(image, 0, (size_t)pixels * 8, s);
            if (e != cudaSuccess)
                return cuda_fail(plan, e, "cudaMemsetAsync");
        }
        return SARBP_OK;
    }

    BpConst k = make_const(plan, params);
    if (echo_stride > 0)
        k.echo_stride = echo_stride;
    float4* table = plan->table_alloc + TABLE_PAD;
    int* sinc_wide = reinterpret_cast<int*>(plan->psi + params->nr + 1);
    if (k.flags & SARBP_SINC8) {
        e = ensure_sinc_table(plan);
        if (e != cudaSuccess)
            return cuda_fail(plan, e, "cudaMalloc (sinc coefficient table)");
        table = plan->sinc_alloc + 4 * TABLE_PAD;
        e = cudaMemsetAsync(sinc_wide, 0, sizeof(int), s);
        if (e != cudaSuccess)
            return cuda_fail(plan, e, "cudaMemsetAsync");
    }
    if (rc)
        e = launch_rc_table(rc, k, static_cast<const float2*>(echoes), antenna_pos, table,
                            plan->klo, s);
    else
        e = launch_table(k, static_cast<const float2*>(echoes), antenna_pos, table, plan->klo,
                         sinc_wide, s);
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "table kernel launch");
    if (k.flags & SARBP_SINC8) {
        e = launch_psi(k, plan->psi, s);
        if (e != cudaSuccess)
            return cuda_fail(plan, e, "phasor kernel launch");
    }

    std::pair<cudaEvent_t, cudaEvent_t>* ev = nullptr;
    if (plan->timing) {
        if (plan->events_used == plan->events.size()) {
            cudaEvent_t a, b;
            e = cudaEventCreate(&a);
            if (e == cudaSuccess) {
                e = cudaEventCreate(&b);
                if (e != cudaSuccess)
                    cudaEventDestroy(a);
            }
            if (e != cudaSuccess)
                return cuda_fail(plan, e, "cudaEventCreate");
            plan->events.emplace_back(a, b);
        }
        ev = &plan->events[plan->events_used++];
        cudaEventRecord(ev->first, s);
    }
    // The cost-weighted split takes one cell per (tile, pulse segment), at
    // most SPLIT_CELLS of them; with more tiles than that (only narrow images
    // of over 33 million rows) every CTA covers many whole tiles, and the
    // even split serves.
    const bool costed = plan->tiles <= SPLIT_CELLS;
    if (costed && (k.flags & SARBP_SINC8) && !plan->heights_mode) {
        // the sinc kernels' cost varies across tiles: split the work by estimated cost
        auto* cum = reinterpret_cast<unsigned long long*>(plan->psi + plan->p.nr + 2);
        auto* starts = reinterpret_cast<long long*>(cum + SPLIT_CELLS + 1);
        e = launch_split(k, antenna_pos, sinc_wide, cum, starts, s);
        if (e != cudaSuccess)
            return cuda_fail(plan, e, "work-split kernel launch");
        k.starts = starts;
    } else if (costed && heights && (k.flags & SARBP_SINC8)) {
        // so does the height-map sinc kernel's, with the terrain (the nearest
        // kernel's rows cost the same on smooth terrain, where they all fall
        // in two bins, and it keeps the equal split)
        auto* cum = reinterpret_cast<unsigned long long*>(plan->psi + plan->p.nr + 2);
        auto* starts = reinterpret_cast<long long*>(cum + SPLIT_CELLS + 1);
        e = launch_heights_split(k, antenna_pos, heights, cum, starts, s);
        if (e != cudaSuccess)
            return cuda_fail(plan, e, "work-split kernel launch");
        k.starts = starts;
    }
    e = launch_backproject(k, antenna_pos, table, plan->klo, static_cast<float2*>(image),
                           plan->partial, plan->psi, heights, sinc_wide, s);
    if (ev)
        cudaEventRecord(ev->second, s);
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "backprojection kernel launch");
    if (k.starts || any_split_tile(k)) {
        e = launch_reduce(k, plan->partial, static_cast<float2*>(image), s);
        if (e != cudaSuccess)
            return cuda_fail(plan, e, "reduce kernel launch");
    }
    return SARBP_OK;
}


}  // namespace

namespace sarbp {

namespace {
std::atomic<int> g_fail_countdown{0};
}

cudaError_t device_alloc(void** ptr, size_t bytes)
{
    int c = g_fail_countdown.load();
    while (c > 0) {
        if (g_fail_countdown.compare_exchange_weak(c, c - 1)) {
            if (c == 1) {
                *ptr = nullptr;
                return cudaErrorMemoryAllocation;   // the injected failure
            }
            break;
        }
    }
    return cudaMalloc(ptr, bytes);
}

}  // namespace sarbp

extern "C" {

void sarbp_debug_fail_alloc(int32_t countdown)
{
    sarbp::g_fail_countdown.store(countdown > 0 ? countdown : 0);
}

sarbp_status sarbp_debug_sinc_taps(float* out)
{
    if (!out)
        return SARBP_ERR_INVALID_ARG;
    sarbp::sinc_taps_host(out);
    return SARBP_OK;
}

const char* sarbp_status_string(sarbp_status status)
{
    switch (status) {
    case SARBP_OK: return "ok";
    case SARBP_ERR_INVALID_ARG: return "invalid argument";
    case SARBP_ERR_PLAN_MISMATCH: return "parameters do not match the plan";
    case SARBP_ERR_CUDA: return "CUDA error";
    case SARBP_ERR_OOM: return "out of memory";
    case SARBP_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case SARBP_ERR_SCRATCH_TOO_SMALL:
        return "problem exceeds the 16 MiB fixed scratch of sarbp_backproject_noalloc";
    }
    return "unknown status";
}

const char* sarbp_last_error(sarbp_plan_t plan)
{
    return plan ? plan->last_error.c_str() : "";
}

}  // extern "C"

namespace {

sarbp_status plan_create(sarbp_plan_t* out, const sarbp_params* p, int heights_mode,
                         double h_min, double h_max)
{
    if (!out)
        return SARBP_ERR_INVALID_ARG;
    *out = nullptr;
    sarbp_status st = check_sizes(p);
    if (st != SARBP_OK)
        return st;
    if (p->flags & ~(SARBP_ACCUMULATE | SARBP_SINC8 | SARBP_NEAREST))
        return SARBP_ERR_INVALID_ARG;
    if ((p->flags & SARBP_SINC8) && (p->flags & SARBP_NEAREST))
        return SARBP_ERR_INVALID_ARG;
    if (!(isfin(p->wavelength) && p->wavelength > 0))
        return SARBP_ERR_INVALID_ARG;

    auto* plan = new (std::nothrow) sarbp_plan_s();
    if (!plan)
        return SARBP_ERR_OOM;
    plan->p = *p;
    plan->heights_mode = heights_mode;
    plan->h_min = h_min;
    plan->h_max = h_max;

    cudaError_t e = cudaGetDevice(&plan->device);
    if (e != cudaSuccess) {
        st = cuda_fail(plan, e, "cudaGetDevice");
        free_plan(plan);
        return st;
    }
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, plan->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, plan->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&plan->sms, cudaDevAttrMultiProcessorCount, plan->device);
    if (e != cudaSuccess) {
        st = cuda_fail(plan, e, "cudaDeviceGetAttribute");
        free_plan(plan);
        return st;
    }
    if (major != 10 || minor != 3) {
        free_plan(plan);
        return SARBP_ERR_UNSUPPORTED_DEVICE;
    }
    e = prepare_kernels();
    if (e == cudaSuccess)
        e = backproject_occupancy(&plan->ctas_per_sm);
    if (e != cudaSuccess || plan->ctas_per_sm < 1) {
        st = cuda_fail(plan, e == cudaSuccess ? cudaErrorInvalidConfiguration : e, "occupancy");
        free_plan(plan);
        return st;
    }
    plan->max_ctas = plan->sms * plan->ctas_per_sm;

    plan->tiles_x = (p->nx + TILE_X - 1) / TILE_X;
    plan->tiles_y = (p->ny + TILE_Y - 1) / TILE_Y;
    plan->tiles = plan->tiles_x * plan->tiles_y;

    // Table rows: the range extent of the tile-padded image plus a tile's reach
    const double ext_x = ((double)plan->tiles_x * TILE_X - 1.0) * p->dx;
    const double ext_y = ((double)plan->tiles_y * TILE_Y - 1.0) * p->dy;
    // (a height-map plan: the slab z0 + [h_min, h_max] over the padded image)
    const double h_span = h_max - h_min;
    const double diag = std::sqrt(ext_x * ext_x + ext_y * ext_y + h_span * h_span);
    const double w_geom =
        std::ceil((diag + 2.0 * tile_qmax3(p->dx, p->dy, h_span)) / p->dr) + 2 * MARGIN + 6;
    const long long w_full = (long long)p->nr + 2 * MARGIN + 8;
    if (w_geom < (double)w_full) {
        plan->W = (int)w_geom;
        plan->full_window = 0;
    } else {
        plan->W = (int)w_full;
        plan->full_window = 1;
    }
    plan->W = (plan->W + 3) & ~3;

    if (plan->tiles > 0 && p->na > 0) {
        const size_t table_entries = (size_t)p->na * plan->W + 2 * TABLE_PAD;
        const size_t sizes[4] = {table_entries * sizeof(float4), (size_t)p->na * sizeof(int),
                                 (size_t)plan->max_ctas * TILE_PIX * sizeof(float4),
                                 ((size_t)p->nr + 2 + (size_t)SPLIT_CELLS + 1 +
                                  (size_t)plan->max_ctas + 1) * sizeof(float2)};
        void** ptrs[4] = {reinterpret_cast<void**>(&plan->table_alloc),
                          reinterpret_cast<void**>(&plan->klo),
                          reinterpret_cast<void**>(&plan->partial),
                          reinterpret_cast<void**>(&plan->psi)};
        for (int i = 0; i < 4; ++i) {
            e = device_alloc(ptrs[i], sizes[i]);
            if (e != cudaSuccess) {
                st = cuda_fail(plan, e, "cudaMalloc");
                free_plan(plan);
                return st;
            }
            plan->scratch_bytes += sizes[i];
        }
        // the pads stay zero so that no read near the table's ends sees garbage
        e = cudaMemset(plan->table_alloc, 0, table_entries * sizeof(float4));
        if (e != cudaSuccess) {
            st = cuda_fail(plan, e, "cudaMemset");
            free_plan(plan);
            return st;
        }
        if (p->flags & SARBP_SINC8) {
            e = ensure_sinc_table(plan);
            if (e != cudaSuccess) {
                st = cuda_fail(plan, e, "cudaMalloc (sinc coefficient table)");
                free_plan(plan);
                return st;
            }
        }
    }
    *out = plan;
    return SARBP_OK;
}

}  // namespace

extern "C" {

sarbp_status sarbp_plan(sarbp_plan_t* out, const sarbp_params* p)
{
    return plan_create(out, p, 0, 0.0, 0.0);
}

sarbp_status sarbp_plan_heights(sarbp_plan_t* out, const sarbp_params* p, double h_min,
                                double h_max)
{
    if (!out)
        return SARBP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!p)
        return SARBP_ERR_INVALID_ARG;
    if (!(isfin(h_min) && isfin(h_max) && h_min <= h_max))
        return SARBP_ERR_INVALID_ARG;
    return plan_create(out, p, 1, h_min, h_max);
}

sarbp_status sarbp_destroy(sarbp_plan_t plan)
{
    free_plan(plan);
    return SARBP_OK;
}

sarbp_status sarbp_plan_describe(sarbp_plan_t plan, sarbp_plan_info* out)
{
    if (!plan || !out)
        return SARBP_ERR_INVALID_ARG;
    out->tile_x = TILE_X;
    out->tile_y = TILE_Y;
    out->tiles = plan->tiles;
    out->ctas = ctas_for(plan);
    out->ctas_per_sm = plan->ctas_per_sm;
    out->sms = plan->sms;
    out->window = plan->W;
    out->full_window = plan->full_window;
    out->kernels_per_call = 0;
    if (plan->tiles > 0 && plan->p.na > 0 && plan->p.nr >= 2)
        // table + main (+ reduce); the phasor kernel for sinc; sinc on a
        // plane also enqueues the work split, its wide-geometry kernel (one of the two
        // exits at once) and always the reduce
        out->kernels_per_call =
            ((plan->p.flags & SARBP_SINC8) && !plan->heights_mode)
                ? 6
                : (any_split_tile(make_const(plan, &plan->p)) ? 3 : 2) +
                      ((plan->p.flags & SARBP_SINC8) ? 1 : 0);
    else if (plan->tiles > 0)
        out->kernels_per_call = 0;   // a memset at most
    out->scratch_bytes = plan->scratch_bytes;
    return SARBP_OK;
}

sarbp_status sarbp_set_timing(sarbp_plan_t plan, int enable)
{
    if (!plan)
        return SARBP_ERR_INVALID_ARG;
    plan->timing = enable != 0;
    return SARBP_OK;
}

sarbp_status sarbp_kernel_times(sarbp_plan_t plan, double* main_ms, int32_t* launches)
{
    if (!plan || !main_ms || !launches)
        return SARBP_ERR_INVALID_ARG;
    double total = 0.0;
    for (size_t i = 0; i < plan->events_used; ++i) {
        cudaError_t e = cudaEventSynchronize(plan->events[i].second);
        float ms = 0.f;
        if (e == cudaSuccess)
            e = cudaEventElapsedTime(&ms, plan->events[i].first, plan->events[i].second);
        if (e != cudaSuccess)
            return cuda_fail(plan, e, "kernel timing");
        total += ms;
    }
    *main_ms = total;
    *launches = (int32_t)plan->events_used;
    plan->events_used = 0;
    return SARBP_OK;
}

sarbp_status sarbp_backproject(sarbp_plan_t plan, void* image, const void* echoes,
                               const double* antenna_pos, const sarbp_params* params,
                               void* stream)
{
    if (!plan || !params)
        return SARBP_ERR_INVALID_ARG;
    sarbp_status st = check_sizes(params);
    if (st != SARBP_OK)
        return st;
    st = check_geometry(params);
    if (st != SARBP_OK)
        return st;
    const sarbp_params& q = plan->p;
    if (params->nx != q.nx || params->ny != q.ny || params->na != q.na || params->nr != q.nr ||
        params->dx != q.dx || params->dy != q.dy || params->dr != q.dr || plan->heights_mode)
        return SARBP_ERR_PLAN_MISMATCH;
    const long long pixels = (long long)params->nx * params->ny;
    if (pixels > 0 && (!image || !aligned8(image)))
        return SARBP_ERR_INVALID_ARG;
    if (params->na > 0 && (!antenna_pos || !aligned8(antenna_pos)))
        return SARBP_ERR_INVALID_ARG;
    if (params->na > 0 && params->nr > 0 && (!echoes || !aligned8(echoes)))
        return SARBP_ERR_INVALID_ARG;
    plan->last_error.clear();

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "cudaGetDevice");
    if (dev != plan->device)
        return SARBP_ERR_INVALID_ARG;

    return enqueue_backprojection(plan, image, echoes, antenna_pos, params,
                                  static_cast<cudaStream_t>(stream));
}

sarbp_status sarbp_backproject_raw(sarbp_plan_t plan, sarbp_rc_plan_t rc, void* image,
                                   const void* raw, const double* antenna_pos,
                                   const sarbp_params* params, void* stream)
{
    if (!plan || !rc || !params)
        return SARBP_ERR_INVALID_ARG;
    sarbp_status st = check_sizes(params);
    if (st != SARBP_OK)
        return st;
    st = check_geometry(params);
    if (st != SARBP_OK)
        return st;
    if (params->flags & (SARBP_SINC8 | SARBP_NEAREST))
        return SARBP_ERR_INVALID_ARG;          // linear interpolation only
    const sarbp_params& q = plan->p;
    if (params->nx != q.nx || params->ny != q.ny || params->na != q.na || params->nr != q.nr ||
        params->dx != q.dx || params->dy != q.dy || params->dr != q.dr || plan->heights_mode)
        return SARBP_ERR_PLAN_MISMATCH;
    int rc_na = 0, rc_ns = 0, rc_dev = -1;
    rc_plan_shape(rc, &rc_na, &rc_ns, &rc_dev);
    if (rc_na != params->na || rc_ns != params->nr || rc_dev != plan->device)
        return SARBP_ERR_PLAN_MISMATCH;
    const long long pixels = (long long)params->nx * params->ny;
    if (pixels > 0 && (!image || !aligned8(image)))
        return SARBP_ERR_INVALID_ARG;
    if (params->na > 0 && (!antenna_pos || !aligned8(antenna_pos)))
        return SARBP_ERR_INVALID_ARG;
    if (params->na > 0 && params->nr > 0 && (!raw || !aligned8(raw)))
        return SARBP_ERR_INVALID_ARG;
    plan->last_error.clear();

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "cudaGetDevice");
    if (dev != plan->device)
        return SARBP_ERR_INVALID_ARG;
    return enqueue_backprojection(plan, image, raw, antenna_pos, params,
                                  static_cast<cudaStream_t>(stream), nullptr, 0, rc);
}

sarbp_status sarbp_backproject_volume(sarbp_plan_t plan, void* volume, const void* echoes,
                                      const double* antenna_pos, const sarbp_params* params,
                                      int32_t nz, double dz, void* stream)
{
    if (!plan || !params || nz < 0 || !isfin(dz))
        return SARBP_ERR_INVALID_ARG;
    sarbp_status st = check_sizes(params);
    if (st != SARBP_OK)
        return st;
    st = check_geometry(params);
    if (st != SARBP_OK)
        return st;
    const sarbp_params& q = plan->p;
    if (params->nx != q.nx || params->ny != q.ny || params->na != q.na || params->nr != q.nr ||
        params->dx != q.dx || params->dy != q.dy || params->dr != q.dr || plan->heights_mode)
        return SARBP_ERR_PLAN_MISMATCH;
    const long long pixels = (long long)params->nx * params->ny;
    if (pixels > 0 && nz > 0 && (!volume || !aligned8(volume)))
        return SARBP_ERR_INVALID_ARG;
    if (params->na > 0 && (!antenna_pos || !aligned8(antenna_pos)))
        return SARBP_ERR_INVALID_ARG;
    if (params->na > 0 && params->nr > 0 && (!echoes || !aligned8(echoes)))
        return SARBP_ERR_INVALID_ARG;
    for (int iz = 0; iz < nz; ++iz)
        if (!isfin(params->z0 + (double)iz * dz))
            return SARBP_ERR_INVALID_ARG;
    plan->last_error.clear();

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "cudaGetDevice");
    if (dev != plan->device)
        return SARBP_ERR_INVALID_ARG;

    for (int iz = 0; iz < nz; ++iz) {
        sarbp_params pz = *params;
        pz.z0 = params->z0 + (double)iz * dz;
        void* plane = static_cast<char*>(volume) + (size_t)iz * (size_t)pixels * 8;
        st = enqueue_backprojection(plan, plane, echoes, antenna_pos, &pz,
                                    static_cast<cudaStream_t>(stream));
        if (st != SARBP_OK)
            return st;
    }
    return SARBP_OK;
}

sarbp_status sarbp_backproject_heights(sarbp_plan_t plan, void* image, const void* echoes,
                                       const double* antenna_pos, const float* heights,
                                       const sarbp_params* params, void* stream)
{
    if (!plan || !params)
        return SARBP_ERR_INVALID_ARG;
    sarbp_status st = check_sizes(params);
    if (st != SARBP_OK)
        return st;
    st = check_geometry(params);
    if (st != SARBP_OK)
        return st;
    const sarbp_params& q = plan->p;
    if (params->nx != q.nx || params->ny != q.ny || params->na != q.na || params->nr != q.nr ||
        params->dx != q.dx || params->dy != q.dy || params->dr != q.dr || !plan->heights_mode)
        return SARBP_ERR_PLAN_MISMATCH;
    const long long pixels = (long long)params->nx * params->ny;
    if (pixels > 0 && (!image || !aligned8(image)))
        return SARBP_ERR_INVALID_ARG;
    if (pixels > 0 && (!heights || (reinterpret_cast<uintptr_t>(heights) & 3u) != 0))
        return SARBP_ERR_INVALID_ARG;
    if (params->na > 0 && (!antenna_pos || !aligned8(antenna_pos)))
        return SARBP_ERR_INVALID_ARG;
    if (params->na > 0 && params->nr > 0 && (!echoes || !aligned8(echoes)))
        return SARBP_ERR_INVALID_ARG;
    plan->last_error.clear();

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "cudaGetDevice");
    if (dev != plan->device)
        return SARBP_ERR_INVALID_ARG;

    return enqueue_backprojection(plan, image, echoes, antenna_pos, params,
                                  static_cast<cudaStream_t>(stream), heights);
}

sarbp_status sarbp_backproject_host(sarbp_plan_t plan, void* image, const void* echoes,
                                    const double* antenna_pos, const sarbp_params* params,
                                    void* stream)
{
    if (!plan || !params)
        return SARBP_ERR_INVALID_ARG;
    sarbp_status st = check_sizes(params);
    if (st != SARBP_OK)
        return st;
    st = check_geometry(params);
    if (st != SARBP_OK)
        return st;
    const sarbp_params& q = plan->p;
    if (params->nx != q.nx || params->ny != q.ny || params->na != q.na || params->nr != q.nr ||
        params->dx != q.dx || params->dy != q.dy || params->dr != q.dr || plan->heights_mode)
        return SARBP_ERR_PLAN_MISMATCH;
    const long long pixels = (long long)params->nx * params->ny;
    const size_t img_bytes = (size_t)pixels * 8;
    if (pixels > 0 && !image)
        return SARBP_ERR_INVALID_ARG;
    if (params->na > 0 && !antenna_pos)
        return SARBP_ERR_INVALID_ARG;
    if ((size_t)params->na * params->nr > 0 && !echoes)
        return SARBP_ERR_INVALID_ARG;
    plan->last_error.clear();
    plan->last_h2d = plan->last_d2h = 0;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "cudaGetDevice");
    if (dev != plan->device)
        return SARBP_ERR_INVALID_ARG;
    if (pixels == 0)
        return SARBP_OK;

    // Only the band of range bins the image can reach crosses to the device.
    long long band_lo = 0, band_hi = -1;
    host_band(params, antenna_pos, 0, params->na, &band_lo, &band_hi);
    const bool runs = band_hi - band_lo >= 1 && params->na > 0;   // the kernels will run

    // Pinned host buffers the device can address are read and written in
    // place by the kernels (the echo band through a row stride); other
    // buffers go through device staging copies.
    const void* const echo_map = runs ? mapped_host(echoes) : nullptr;
    void* const img_map = runs ? mapped_host(image) : nullptr;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (img_bytes && !img_map && !plan->d_image)
        e = device_alloc(&plan->d_image, img_bytes);
    if (e == cudaSuccess && params->na > 0 && !plan->d_pos)
        e = device_alloc(reinterpret_cast<void**>(&plan->d_pos), (size_t)params->na * 3 * sizeof(double));
    if (e == cudaSuccess && band_hi >= band_lo && !echo_map && !plan->d_echo)
        e = device_alloc(&plan->d_echo, (size_t)params->na * params->nr * 8);
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "cudaMalloc (host staging)");

    sarbp_params band = *params;
    const void* echo_src = plan->d_echo;
    long long echo_stride = 0;
    if (band_hi >= band_lo) {
        const size_t width = (size_t)(band_hi - band_lo + 1);
        band.nr = (int32_t)width;
        band.r0 = params->r0 + (double)band_lo * params->dr;
        if (echo_map) {
            echo_src = static_cast<const char*>(echo_map) + (size_t)band_lo * 8;
            echo_stride = params->nr;
        } else {
            e = cudaMemcpy2DAsync(plan->d_echo, width * 8,
                                  static_cast<const char*>(echoes) + (size_t)band_lo * 8,
                                  (size_t)params->nr * 8, width * 8, (size_t)params->na,
                                  cudaMemcpyHostToDevice, s);
        }
        plan->last_h2d += width * 8 * (size_t)params->na;
    } else {
        band.nr = 0;                         // no pulse reaches the range axis
    }
    if (e == cudaSuccess && params->na > 0) {
        e = cudaMemcpyAsync(plan->d_pos, antenna_pos, (size_t)params->na * 3 * sizeof(double),
                            cudaMemcpyHostToDevice, s);
        plan->last_h2d += (size_t)params->na * 3 * sizeof(double);
    }
    if (e == cudaSuccess && (params->flags & SARBP_ACCUMULATE)) {
        if (!img_map)
            e = cudaMemcpyAsync(plan->d_image, image, img_bytes, cudaMemcpyHostToDevice, s);
        plan->last_h2d += img_bytes;
    }
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "cudaMemcpyAsync (to device)");
    st = enqueue_backprojection(plan, img_map ? img_map : plan->d_image, echo_src, plan->d_pos,
                                &band, s, nullptr, echo_stride);
    if (st != SARBP_OK)
        return st;
    if (!img_map)
        e = cudaMemcpyAsync(image, plan->d_image, img_bytes, cudaMemcpyDeviceToHost, s);
    plan->last_d2h = img_bytes;
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "cudaMemcpyAsync (to host)");
    return SARBP_OK;
}

sarbp_status sarbp_backproject_streamed(sarbp_plan_t plan, void* image, const void* echoes,
                                        const double* antenna_pos, const sarbp_params* params,
                                        int32_t chunk_pulses, void* stream)
{
    if (!plan || !params || chunk_pulses < 1)
        return SARBP_ERR_INVALID_ARG;
    sarbp_status st = check_sizes(params);
    if (st != SARBP_OK)
        return st;
    st = check_geometry(params);
    if (st != SARBP_OK)
        return st;
    const sarbp_params& q = plan->p;
    if (params->nx != q.nx || params->ny != q.ny || params->na != q.na || params->nr != q.nr ||
        params->dx != q.dx || params->dy != q.dy || params->dr != q.dr || plan->heights_mode)
        return SARBP_ERR_PLAN_MISMATCH;
    const long long pixels = (long long)params->nx * params->ny;
    const size_t img_bytes = (size_t)pixels * 8;
    if (pixels > 0 && !image)
        return SARBP_ERR_INVALID_ARG;
    if (params->na > 0 && !antenna_pos)
        return SARBP_ERR_INVALID_ARG;
    if ((size_t)params->na * params->nr > 0 && !echoes)
        return SARBP_ERR_INVALID_ARG;
    plan->last_error.clear();
    plan->last_h2d = plan->last_d2h = 0;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "cudaGetDevice");
    if (dev != plan->device)
        return SARBP_ERR_INVALID_ARG;
    if (pixels == 0)
        return SARBP_OK;

    const int chunk = std::max(1, std::min(chunk_pulses, std::max(params->na, 1)));
    const size_t stage_need = (size_t)chunk * (size_t)params->nr * 8;
    if (img_bytes && !plan->d_image)
        e = device_alloc(&plan->d_image, img_bytes);
    if (e == cudaSuccess && params->na > 0 && !plan->d_pos)
        e = device_alloc(reinterpret_cast<void**>(&plan->d_pos), (size_t)params->na * 3 * sizeof(double));
    if (e == cudaSuccess && stage_need > plan->stage_bytes) {
        for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
            cudaFree(plan->d_stage[b]);
            plan->d_stage[b] = nullptr;
            e = device_alloc(&plan->d_stage[b], stage_need);
        }
        plan->stage_bytes = e == cudaSuccess ? stage_need : 0;
    }
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "cudaMalloc (streaming buffers)");
    if (!plan->copy_stream) {
        e = cudaStreamCreateWithFlags(&plan->copy_stream, cudaStreamNonBlocking);
        for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
            e = cudaEventCreateWithFlags(&plan->copied[b], cudaEventDisableTiming);
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(&plan->consumed[b], cudaEventDisableTiming);
        }
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&plan->call_start, cudaEventDisableTiming);
        if (e != cudaSuccess)
            return cuda_fail(plan, e, "stream/event creation");
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStream_t cs = plan->copy_stream;
    // the copy stream starts after all earlier work on `stream` (which may
    // still read the staging buffers of a previous call)
    e = cudaEventRecord(plan->call_start, s);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(cs, plan->call_start, 0);
    if (e == cudaSuccess && params->na > 0) {
        e = cudaMemcpyAsync(plan->d_pos, antenna_pos, (size_t)params->na * 3 * sizeof(double),
                            cudaMemcpyHostToDevice, cs);
        plan->last_h2d += (size_t)params->na * 3 * sizeof(double);
    }
    if (e == cudaSuccess && (params->flags & SARBP_ACCUMULATE)) {
        e = cudaMemcpyAsync(plan->d_image, image, img_bytes, cudaMemcpyHostToDevice, s);
        plan->last_h2d += img_bytes;
    }
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "cudaMemcpyAsync (to device)");

    if (params->na == 0 || params->nr < 2) {
        sarbp_params none = *params;
        st = enqueue_backprojection(plan, plan->d_image, nullptr, plan->d_pos, &none, s);
        if (st != SARBP_OK)
            return st;
    }
    for (int c0 = 0, i = 0; c0 < params->na && params->nr >= 2; c0 += chunk, ++i) {
        const int b = i & 1;
        const int cn = std::min(chunk, params->na - c0);
        long long lo = 0, hi = -1;
        const bool any = host_band(params, antenna_pos, c0, c0 + cn, &lo, &hi);
        sarbp_params sub = *params;
        sub.na = cn;
        if (c0 > 0)
            sub.flags |= SARBP_ACCUMULATE;
        // staging buffer b was last read by chunk i - 2
        if (i >= 2)
            e = cudaStreamWaitEvent(cs, plan->consumed[b], 0);
        if (e == cudaSuccess && any) {
            const size_t width = (size_t)(hi - lo + 1);
            sub.nr = (int32_t)width;
            sub.r0 = params->r0 + (double)lo * params->dr;
            e = cudaMemcpy2DAsync(plan->d_stage[b], width * 8,
                                  static_cast<const char*>(echoes) +
                                      ((size_t)c0 * params->nr + (size_t)lo) * 8,
                                  (size_t)params->nr * 8, width * 8, (size_t)cn,
                                  cudaMemcpyHostToDevice, cs);
            plan->last_h2d += width * 8 * (size_t)cn;
        } else {
            sub.nr = 0;                      // no pulse of the chunk reaches the axis
        }
        if (e == cudaSuccess)
            e = cudaEventRecord(plan->copied[b], cs);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(s, plan->copied[b], 0);
        if (e != cudaSuccess)
            return cuda_fail(plan, e, "chunk copy");
        st = enqueue_backprojection(plan, plan->d_image, plan->d_stage[b], plan->d_pos + 3 * (size_t)c0,
                                    &sub, s);
        if (st != SARBP_OK)
            return st;
        e = cudaEventRecord(plan->consumed[b], s);
        if (e != cudaSuccess)
            return cuda_fail(plan, e, "cudaEventRecord");
    }
    e = cudaMemcpyAsync(image, plan->d_image, img_bytes, cudaMemcpyDeviceToHost, s);
    plan->last_d2h = img_bytes;
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(plan, e, "cudaMemcpyAsync (to host)");
    return SARBP_OK;
}

sarbp_status sarbp_host_transfer_bytes(sarbp_plan_t plan, uint64_t* h2d, uint64_t* d2h)
{
    if (!plan || !h2d || !d2h)
        return SARBP_ERR_INVALID_ARG;
    *h2d = plan->last_h2d;
    *d2h = plan->last_d2h;
    return SARBP_OK;
}

// No-allocation variant: the table and window starts of one chunk of pulses
// live in a fixed device array; every CTA owns whole tiles, so no partial-sum
// buffer is needed.
sarbp_status sarbp_backproject_noalloc(void* image, const void* echoes,
                                       const double* antenna_pos, const sarbp_params* params,
                                       void* stream)
{
    if (!params)
        return SARBP_ERR_INVALID_ARG;
    sarbp_status st = check_sizes(params);
    if (st != SARBP_OK)
        return st;
    st = check_geometry(params);
    if (st != SARBP_OK)
        return st;
    if (params->flags & (SARBP_SINC8 | SARBP_NEAREST))
        return SARBP_ERR_INVALID_ARG;          // linear interpolation only
    const long long pixels = (long long)params->nx * params->ny;
    if (pixels > 0 && (!image || !aligned8(image)))
        return SARBP_ERR_INVALID_ARG;
    if (params->na > 0 && (!antenna_pos || !aligned8(antenna_pos)))
        return SARBP_ERR_INVALID_ARG;
    if (params->na > 0 && params->nr > 0 && (!echoes || !aligned8(echoes)))
        return SARBP_ERR_INVALID_ARG;

    // the geometry a plan would fix, computed locally (nothing is stored)
    sarbp_plan_s geo;
    geo.p = *params;
    geo.tiles_x = (params->nx + TILE_X - 1) / TILE_X;
    geo.tiles_y = (params->ny + TILE_Y - 1) / TILE_Y;
    geo.tiles = geo.tiles_x * geo.tiles_y;
    const double ext_x = ((double)geo.tiles_x * TILE_X - 1.0) * params->dx;
    const double ext_y = ((double)geo.tiles_y * TILE_Y - 1.0) * params->dy;
    const double diag = std::sqrt(ext_x * ext_x + ext_y * ext_y);
    const double w_geom =
        std::ceil((diag + 2.0 * tile_qmax(params->dx, params->dy)) / params->dr) + 2 * MARGIN + 6;
    const long long w_full = (long long)params->nr + 2 * MARGIN + 8;
    geo.full_window = w_geom < (double)w_full ? 0 : 1;
    const double w_any = geo.full_window ? (double)w_full : w_geom;
    // rows are (W x 16 B); the window starts take 4 B per pulse
    const double pad_bytes = 2.0 * TABLE_PAD * sizeof(float4) + 256.0;
    const double row_bytes = (std::ceil(w_any / 4.0) * 4.0) * sizeof(float4) + sizeof(int);
    if (pixels > 0 && params->na > 0 && params->nr >= 2 &&
        row_bytes + pad_bytes > (double)NOALLOC_SCRATCH_BYTES)
        return SARBP_ERR_SCRATCH_TOO_SMALL;
    geo.W = ((int)w_any + 3) & ~3;

    int dev = -1, major = 0, minor = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess)
        return SARBP_ERR_CUDA;
    if (major != 10 || minor != 3)
        return SARBP_ERR_UNSUPPORTED_DEVICE;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pixels == 0)
        return SARBP_OK;
    if (params->na == 0 || params->nr < 2) {
        if (!(params->flags & SARBP_ACCUMULATE) &&
            cudaMemsetAsync(image, 0, (size_t)pixels * 8, s) != cudaSuccess)
            return SARBP_ERR_CUDA;
        return SARBP_OK;
    }

    void* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess)
        return SARBP_ERR_CUDA;
    const size_t entry_bytes = (size_t)geo.W * sizeof(float4) + sizeof(int);
    const size_t usable = NOALLOC_SCRATCH_BYTES - (size_t)pad_bytes;
    const int chunk = (int)std::min<size_t>((size_t)params->na, usable / entry_bytes);
    // layout: [window starts, 256-B aligned][pad][chunk rows][pad]
    const size_t klo_bytes = (((size_t)chunk * sizeof(int)) + 255) & ~size_t(255);
    int* klo = static_cast<int*>(scratch);
    float4* table_alloc = reinterpret_cast<float4*>(static_cast<unsigned char*>(scratch) + klo_bytes);
    float4* table = table_alloc + TABLE_PAD;
    // the pads are never written by the kernels and must read as zero
    if (cudaMemsetAsync(table_alloc, 0, TABLE_PAD * sizeof(float4), s) != cudaSuccess ||
        cudaMemsetAsync(table + (size_t)chunk * geo.W, 0, TABLE_PAD * sizeof(float4), s) !=
            cudaSuccess)
        return SARBP_ERR_CUDA;

    const float2* ech = static_cast<const float2*>(echoes);
    for (int c0 = 0; c0 < params->na; c0 += chunk) {
        const int cn = std::min(chunk, params->na - c0);
        sarbp_params pc = *params;
        pc.na = cn;
        if (c0 > 0)
            pc.flags |= SARBP_ACCUMULATE;
        geo.p = pc;
        // a short last chunk: the zero pad the kernels may read past the last
        // row goes straight after row cn - 1, as in a plan's table (rows cn ..
        // chunk - 1 still hold the previous chunk's entries)
        if (cn < chunk &&
            cudaMemsetAsync(table + (size_t)cn * geo.W, 0, TABLE_PAD * sizeof(float4), s) !=
                cudaSuccess)
            return SARBP_ERR_CUDA;
        BpConst k = make_const(&geo, &pc);
        k.ctas = geo.tiles;                     // one whole tile per CTA: direct writes only
        k.units = (long long)geo.tiles * cn;
        e = launch_table(k, ech + (size_t)c0 * params->nr, antenna_pos + 3 * (size_t)c0, table,
                         klo, nullptr, s);
        if (e == cudaSuccess)
            e = launch_backproject(k, antenna_pos + 3 * (size_t)c0, table, klo,
                                   static_cast<float2*>(image), nullptr, nullptr, nullptr, nullptr,
                                   s);
        if (e != cudaSuccess)
            return SARBP_ERR_CUDA;
    }
    return SARBP_OK;
}

}  // extern "C"
