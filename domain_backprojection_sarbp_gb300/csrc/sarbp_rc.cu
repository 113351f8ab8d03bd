// sarbp_rc.cu - range compression (matched filtering) for libsarbp, sm_103a.
//
// SARBP-GPU = the page "基于GPU的SAR后向投影成像优化与CUDA加速实践". Its §3.1
// produces the backprojection input by range compression: FFT every pulse
// along range, multiply by the matched filter's frequency response (with a
// Hamming or Taylor window to lower the sidelobes), inverse FFT; all pulses
// form one batch. Here:
//
//   rc[n][k] = sum_{l<L} raw[n][k + l] conj(ref[l]),  0 <= k < ns,
//
// the linear correlation, through FFTs of size N = 2^m >= ns + L - 1, with an
// optional Hamming weighting 0.54 + 0.46 cos(2 pi f / b) over the centred band
// |f| <= b/2 (f in cycles per sample), zero outside it.
//
// One CTA per pulse holds its zero-padded row in shared memory. The forward
// transform is an in-place radix-4 decimation in frequency (natural order in,
// digit-reversed out); the filter spectrum H is stored in that same order, so
// the product needs no reordering; the inverse mirrors the forward passes
// (digit-reversed in, natural out). The plan builds H with the same forward
// transform on the zero-padded reference.
#include "../../include/sarbp.h"
#include "sarbp_internal.h"

#include <cmath>
#include <cstdint>
#include <new>
#include <vector>

namespace {

constexpr int RC_THREADS = 512;
constexpr int RC_MAX_LOG2 = 14;            // N <= 16384: 128 KB of shared memory per row

__device__ __forceinline__ float2 cmul(float2 a, float2 b)
{
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}

// Forward transform, in place: radix-4 decimation-in-frequency passes over
// spans N, N/4, ..., then one radix-2 pass of span 2 when log2 N is odd. The
// result at position p is X[sigma(p)], sigma the mixed digit reversal below.
// tw[t] = exp(-j 2 pi t / N), t < N.
__device__ void dif_forward(float2* x, int n, int log2n, const float2* __restrict__ tw)
{
    const int n4 = log2n / 2;
    for (int lvl = 0; lvl < n4; ++lvl) {
        const int lq = log2n - 2 * lvl - 2;          // q = span / 4 = 2^lq
        const int q = 1 << lq;
        const int tstep = 1 << (2 * lvl);            // N / span
        for (int b = threadIdx.x; b < n / 4; b += blockDim.x) {
            const int j = b & (q - 1);
            const int base = ((b >> lq) << (lq + 2)) + j;
            const float2 x0 = x[base], x1 = x[base + q], x2 = x[base + 2 * q], x3 = x[base + 3 * q];
            const float2 a0 = make_float2(x0.x + x2.x, x0.y + x2.y);
            const float2 a1 = make_float2(x0.x - x2.x, x0.y - x2.y);
            const float2 a2 = make_float2(x1.x + x3.x, x1.y + x3.y);
            const float2 a3 = make_float2(x1.y - x3.y, x3.x - x1.x);      // -j (x1 - x3)
            x[base] = make_float2(a0.x + a2.x, a0.y + a2.y);
            const int t = j * tstep;
            x[base + q] = cmul(make_float2(a1.x + a3.x, a1.y + a3.y), __ldg(tw + t));
            x[base + 2 * q] = cmul(make_float2(a0.x - a2.x, a0.y - a2.y), __ldg(tw + 2 * t));
            x[base + 3 * q] = cmul(make_float2(a1.x - a3.x, a1.y - a3.y), __ldg(tw + 3 * t));
        }
        __syncthreads();
    }
    if (log2n & 1) {                                 // span 2: no twiddle
        for (int b = threadIdx.x; b < n / 2; b += blockDim.x) {
            const float2 a = x[2 * b], c = x[2 * b + 1];
            x[2 * b] = make_float2(a.x + c.x, a.y + c.y);
            x[2 * b + 1] = make_float2(a.x - c.x, a.y - c.y);
        }
        __syncthreads();
    }
}

// Inverse of dif_forward up to the factor N: the same passes mirrored
// (conjugate twiddles first, then the inverse 4-point transform).
__device__ void dit_inverse(float2* x, int n, int log2n, const float2* __restrict__ tw)
{
    const int n4 = log2n / 2;
    if (log2n & 1) {
        for (int b = threadIdx.x; b < n / 2; b += blockDim.x) {
            const float2 a = x[2 * b], c = x[2 * b + 1];
            x[2 * b] = make_float2(a.x + c.x, a.y + c.y);
            x[2 * b + 1] = make_float2(a.x - c.x, a.y - c.y);
        }
        __syncthreads();
    }
    for (int lvl = n4 - 1; lvl >= 0; --lvl) {
        const int lq = log2n - 2 * lvl - 2;
        const int q = 1 << lq;
        const int tstep = 1 << (2 * lvl);
        for (int b = threadIdx.x; b < n / 4; b += blockDim.x) {
            const int j = b & (q - 1);
            const int base = ((b >> lq) << (lq + 2)) + j;
            const int t = j * tstep;
            const float2 w1 = __ldg(tw + t), w2 = __ldg(tw + 2 * t), w3 = __ldg(tw + 3 * t);
            const float2 z0 = x[base];
            const float2 z1 = cmul(x[base + q], make_float2(w1.x, -w1.y));
            const float2 z2 = cmul(x[base + 2 * q], make_float2(w2.x, -w2.y));
            const float2 z3 = cmul(x[base + 3 * q], make_float2(w3.x, -w3.y));
            const float2 b0 = make_float2(z0.x + z2.x, z0.y + z2.y);
            const float2 b1 = make_float2(z0.x - z2.x, z0.y - z2.y);
            const float2 b2 = make_float2(z1.x + z3.x, z1.y + z3.y);
            const float2 b3 = make_float2(z3.y - z1.y, z1.x - z3.x);     // +j (z1 - z3)
            x[base] = make_float2(b0.x + b2.x, b0.y + b2.y);
            x[base + q] = make_float2(b1.x + b3.x, b1.y + b3.y);
            x[base + 2 * q] = make_float2(b0.x - b2.x, b0.y - b2.y);
            x[base + 3 * q] = make_float2(b1.x - b3.x, b1.y - b3.y);
        }
        __syncthreads();
    }
}

// Natural frequency index held at position p after dif_forward: the base-4
// digits of p (most significant first) become the least significant digits
// of the index, and the final base-2 digit, if any, the most significant.
__device__ __forceinline__ int natural_index(int p, int log2n)
{
    const int n4 = log2n / 2;
    int k = 0;
    for (int lvl = 0; lvl < n4; ++lvl)
        k |= ((p >> (log2n - 2 * lvl - 2)) & 3) << (2 * lvl);
    if (log2n & 1)
        k |= (p & 1) << (2 * n4);
    return k;
}

// The filter: H[p] = conj(FFT(ref)[k]) * W(k) at position p, k = natural_index(p).
__global__ void __launch_bounds__(RC_THREADS) rc_filter_kernel(const float2* __restrict__ ref, int nref,
                                                               int n, int log2n,
                                                               const float2* __restrict__ tw,
                                                               unsigned window, float band,
                                                               float2* __restrict__ h)
{
    extern __shared__ float2 row[];
    for (int i = threadIdx.x; i < n; i += blockDim.x)
        row[i] = i < nref ? ref[i] : make_float2(0.f, 0.f);
    __syncthreads();
    dif_forward(row, n, log2n, tw);
    for (int p = threadIdx.x; p < n; p += blockDim.x) {
        const int k = natural_index(p, log2n);
        float w = 1.0f;
        if (window == SARBP_WINDOW_HAMMING) {
            const float f = (float)(k < n / 2 ? k : k - n) / (float)n;
            w = fabsf(f) <= 0.5f * band ? 0.54f + 0.46f * cospif(2.0f * f / band) : 0.0f;
        }
        const float2 v = row[p];
        h[p] = make_float2(v.x * w, -v.y * w);
    }
}

__global__ void __launch_bounds__(RC_THREADS) rc_kernel(const float2* __restrict__ raw, int ns, int n,
                                                        int log2n, const float2* __restrict__ tw,
                                                        const float2* __restrict__ h,
                                                        float2* __restrict__ out)
{
    extern __shared__ float2 row[];
    const size_t base = (size_t)blockIdx.x * ns;
    for (int i = threadIdx.x; i < n; i += blockDim.x)
        row[i] = i < ns ? raw[base + i] : make_float2(0.f, 0.f);
    __syncthreads();
    dif_forward(row, n, log2n, tw);
    for (int p = threadIdx.x; p < n; p += blockDim.x)
        row[p] = cmul(row[p], __ldg(h + p));
    __syncthreads();
    dit_inverse(row, n, log2n, tw);
    const float scale = 1.0f / (float)n;
    for (int i = threadIdx.x; i < ns; i += blockDim.x) {
        const float2 v = row[i];
        out[base + i] = make_float2(v.x * scale, v.y * scale);
    }
}

}  // namespace

struct sarbp_rc_plan_s {
    sarbp_rc_params p{};
    int n = 0, log2n = 0;
    int device = -1;
    float2* tw = nullptr;      // N twiddles
    float2* h = nullptr;       // N filter coefficients, in the forward transform's order
};

extern "C" {

sarbp_status sarbp_rc_plan(sarbp_rc_plan_t* out, const sarbp_rc_params* p, const void* ref,
                           void* stream)
{
    if (!out)
        return SARBP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!p || p->na < 0 || p->ns < 1 || p->nref < 1 || !ref ||
        (reinterpret_cast<uintptr_t>(ref) & 7u))
        return SARBP_ERR_INVALID_ARG;
    if (p->window != SARBP_WINDOW_NONE && p->window != SARBP_WINDOW_HAMMING)
        return SARBP_ERR_INVALID_ARG;
    if (p->window == SARBP_WINDOW_HAMMING && !(p->band_fraction > 0.0 && p->band_fraction <= 1.0))
        return SARBP_ERR_INVALID_ARG;
    int log2n = 0;
    while ((1ll << log2n) < (long long)p->ns + p->nref - 1)
        ++log2n;
    if (log2n < 1)
        log2n = 1;
    if (log2n > RC_MAX_LOG2)
        return SARBP_ERR_INVALID_ARG;           // N above 16384 does not fit one row in shared memory

    auto* plan = new (std::nothrow) sarbp_rc_plan_s();
    if (!plan)
        return SARBP_ERR_OOM;
    plan->p = *p;
    plan->log2n = log2n;
    plan->n = 1 << log2n;
    cudaError_t e = cudaGetDevice(&plan->device);
    int major = 0, minor = 0;
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, plan->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, plan->device);
    if (e == cudaSuccess && (major != 10 || minor != 3)) {
        delete plan;
        return SARBP_ERR_UNSUPPORTED_DEVICE;
    }
    const size_t smem = (size_t)plan->n * sizeof(float2);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_filter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
    if (e == cudaSuccess)
        e = cudaMalloc(&plan->tw, (size_t)plan->n * sizeof(float2));
    if (e == cudaSuccess)
        e = cudaMalloc(&plan->h, (size_t)plan->n * sizeof(float2));
    if (e == cudaSuccess) {
        // twiddles in float64, rounded once
        std::vector<float2> tw((size_t)plan->n);
        const double pi = 3.14159265358979323846;
        for (int m = 0; m < plan->n; ++m) {
            const double a = -2.0 * pi * (double)m / (double)plan->n;
            tw[m] = make_float2((float)std::cos(a), (float)std::sin(a));
        }
        e = cudaMemcpy(plan->tw, tw.data(), tw.size() * sizeof(float2), cudaMemcpyHostToDevice);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (e == cudaSuccess) {
        rc_filter_kernel<<<1, RC_THREADS, smem, s>>>(static_cast<const float2*>(ref), p->nref,
                                                     plan->n, plan->log2n, plan->tw, p->window,
                                                     (float)p->band_fraction, plan->h);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        cudaFree(plan->tw);
        cudaFree(plan->h);
        delete plan;
        return e == cudaErrorMemoryAllocation ? SARBP_ERR_OOM : SARBP_ERR_CUDA;
    }
    *out = plan;
    return SARBP_OK;
}

sarbp_status sarbp_range_compress(sarbp_rc_plan_t plan, void* out, const void* raw, void* stream)
{
    if (!plan)
        return SARBP_ERR_INVALID_ARG;
    const sarbp_rc_params& p = plan->p;
    if (p.na == 0)
        return SARBP_OK;
    if (!out || !raw || (reinterpret_cast<uintptr_t>(out) & 7u) ||
        (reinterpret_cast<uintptr_t>(raw) & 7u))
        return SARBP_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device)
        return SARBP_ERR_INVALID_ARG;
    rc_kernel<<<p.na, RC_THREADS, (size_t)plan->n * sizeof(float2), static_cast<cudaStream_t>(stream)>>>(
        static_cast<const float2*>(raw), p.ns, plan->n, plan->log2n, plan->tw, plan->h,
        static_cast<float2*>(out));
    return cudaGetLastError() == cudaSuccess ? SARBP_OK : SARBP_ERR_CUDA;
}

sarbp_status sarbp_rc_destroy(sarbp_rc_plan_t plan)
{
    if (plan) {
        cudaFree(plan->tw);
        cudaFree(plan->h);
        delete plan;
    }
    return SARBP_OK;
}

}  // extern "C"
