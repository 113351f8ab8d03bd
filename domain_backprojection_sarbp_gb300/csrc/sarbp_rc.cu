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
// One CTA per pulse. The transforms are self-sorting (Stockham) passes of
// radix 16 held in registers, plus one pass of radix 2, 4, 8 or 32 when log2 N
// is not a multiple of 4. For N = 2 16^m (N = 8192 for 4096-sample rows) a
// thread holds 32 values: the radix-32 pass is one thread's own DFT (two
// radix-16 DFTs and a radix-2 step; when the second half of the zero-padded
// input is empty, just the two DFTs), and each thread takes two radix-16
// butterflies per pass after it. Shared memory only carries the data between
// passes, as float2 values padded by one slot every 16. The input twiddles of
// a pass, exp(-2 pi i t k / (NS R)), come from the SFU (whose sine and cosine
// units the transform leaves idle) for t = 1, 4, 8, 12 (and 16 for radix 32)
// and as products for the other powers. The forward transform takes the raw
// row straight from global memory (zero beyond ns, not kept in L1) and its
// last pass leaves each thread holding the spectrum at indices j + t N/16,
// which are exactly the inputs of the inverse transform's first pass: the
// filter multiply happens there in registers, with no trip through shared
// memory. The inverse's last pass writes natural-order samples straight to
// global memory, or, fused with a backprojection plan's echo table, keeps
// the band of samples the table row needs in shared memory. The filter
// spectrum H (conj FFT of the reference times the window, divided by N) is
// built once by the plan, in natural order.
#include "../../include/sarbp.h"
#include "sarbp_device.cuh"
#include "sarbp_internal.h"

#include <cmath>
#include <cstdint>
#include <new>

namespace {

constexpr int RC_MAX_LOG2 = 14;            // N <= 16384: 135 KB of shared memory per row

// complex sums as one packed f32x2 operation (a - b = b * -1 + a, rounded once)
__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 csub(float2 a, float2 b)
{
    return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
}
__device__ __forceinline__ float2 cmul(float2 a, float2 b)
{
    return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
__device__ __forceinline__ float2 conj_if(float2 a, bool c) { return c ? make_float2(a.x, -a.y) : a; }
// a times S i, S = -1 (forward) or +1 (inverse)
template <int S>
__device__ __forceinline__ float2 mul_si(float2 a)
{
    return S < 0 ? make_float2(a.y, -a.x) : make_float2(-a.y, a.x);
}

// In-register DFTs, natural order in and out: X[k] = sum_m x[m] exp(S 2 pi i m k / R).
// b and d take s1 +- S i (b - d) in scalar form, where the lane swap of the
// factor i costs nothing.
template <int S>
__device__ __forceinline__ void dft4(float2& a, float2& b, float2& c, float2& d)
{
    const float2 s0 = cadd(a, c), s1 = csub(a, c), s2 = cadd(b, d), dd = csub(b, d);
    a = cadd(s0, s2);
    c = csub(s0, s2);
    if (S < 0) {
        b = make_float2(s1.x + dd.y, s1.y - dd.x);
        d = make_float2(s1.x - dd.y, s1.y + dd.x);
    } else {
        b = make_float2(s1.x - dd.y, s1.y + dd.x);
        d = make_float2(s1.x + dd.y, s1.y - dd.x);
    }
}

template <int R, int S>
__device__ __forceinline__ void dft(float2* v);

// exp(S 2 pi i s / 32) for s = 0 .. 15 (compile-time s)
template <int S>
__device__ __forceinline__ float2 w32(int s)
{
    constexpr float C[16] = {1.0f, 0.980785280f, 0.923879533f, 0.831469612f, 0.707106781f,
                             0.555570233f, 0.382683432f, 0.195090322f, 0.0f, -0.195090322f,
                             -0.382683432f, -0.555570233f, -0.707106781f, -0.831469612f,
                             -0.923879533f, -0.980785280f};
    constexpr float SN[16] = {0.0f, 0.195090322f, 0.382683432f, 0.555570233f, 0.707106781f,
                              0.831469612f, 0.923879533f, 0.980785280f, 1.0f, 0.980785280f,
                              0.923879533f, 0.831469612f, 0.707106781f, 0.555570233f,
                              0.382683432f, 0.195090322f};
    return make_float2(C[s], S * SN[s]);
}

// 32 = 2 x 16: the DFTs of the even and the odd inputs, then X[k] = E[k] +
// W32^k O[k] and X[k + 16] = E[k] - W32^k O[k] (W32^8 = S i costs nothing).
template <int S>
__device__ __forceinline__ void dft32(float2* v)
{
    float2 e[16], o[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        e[m] = v[2 * m];
        o[m] = v[2 * m + 1];
    }
    dft<16, S>(e);
    dft<16, S>(o);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float2 t = k == 0 ? o[k] : (k == 8 ? mul_si<S>(o[k]) : cmul(o[k], w32<S>(k)));
        v[k] = cadd(e[k], t);
        v[k + 16] = csub(e[k], t);
    }
}

// 32-point DFT of inputs whose second half is zero: X[2k] = DFT16(x)[k] and
// X[2k + 1] = DFT16(x W32^(S m))[k] (no radix-2 sums).
template <int S>
__device__ __forceinline__ void dft32_half(float2* v)
{
    float2 o[16];
#pragma unroll
    for (int m = 0; m < 16; ++m)
        o[m] = m == 0 ? v[0] : (m == 8 ? mul_si<S>(v[8]) : cmul(v[m], w32<S>(m)));
    dft<16, S>(v);
    dft<16, S>(o);
#pragma unroll
    for (int k = 15; k >= 0; --k) {
        v[2 * k] = v[k];
        v[2 * k + 1] = o[k];
    }
}

template <int R, int S>
__device__ __forceinline__ void dft(float2* v)
{
    constexpr float H = 0.707106781186547524f;     // cos(pi/4)
    constexpr float C1 = 0.923879532511286756f;    // cos(pi/8)
    constexpr float S1 = 0.382683432365089772f;    // sin(pi/8)
    if (R == 2) {
        const float2 a = v[0], b = v[1];
        v[0] = cadd(a, b);
        v[1] = csub(a, b);
    } else if (R == 4) {
        dft4<S>(v[0], v[1], v[2], v[3]);
    } else if (R == 8) {
        float2 e0 = v[0], e1 = v[2], e2 = v[4], e3 = v[6];
        float2 o0 = v[1], o1 = v[3], o2 = v[5], o3 = v[7];
        dft4<S>(e0, e1, e2, e3);
        dft4<S>(o0, o1, o2, o3);
        o1 = cmul(o1, make_float2(H, S * H));           // W8^1
        o2 = mul_si<S>(o2);                             // W8^2
        o3 = cmul(o3, make_float2(-H, S * H));          // W8^3
        v[0] = cadd(e0, o0); v[4] = csub(e0, o0);
        v[1] = cadd(e1, o1); v[5] = csub(e1, o1);
        v[2] = cadd(e2, o2); v[6] = csub(e2, o2);
        v[3] = cadd(e3, o3); v[7] = csub(e3, o3);
    } else if (R == 32) {
        dft32<S>(v);
    } else {
        // 16 = 4 x 4: m = 4 m1 + m2, k = k1 + 4 k2
        float2 y[16];
#pragma unroll
        for (int m2 = 0; m2 < 4; ++m2) {
            float2 a = v[m2], b = v[m2 + 4], c = v[m2 + 8], d = v[m2 + 12];
            dft4<S>(a, b, c, d);
            y[m2] = a; y[m2 + 4] = b; y[m2 + 8] = c; y[m2 + 12] = d;   // y[m2 + 4 k1]
        }
        // twiddles W16^(m2 k1)
        y[5] = cmul(y[5], make_float2(C1, S * S1));      // m2 1, k1 1
        y[9] = cmul(y[9], make_float2(H, S * H));        // 1, 2
        y[13] = cmul(y[13], make_float2(S1, S * C1));    // 1, 3
        y[6] = cmul(y[6], make_float2(H, S * H));        // 2, 1
        y[10] = mul_si<S>(y[10]);                        // 2, 2
        y[14] = cmul(y[14], make_float2(-H, S * H));     // 2, 3
        y[7] = cmul(y[7], make_float2(S1, S * C1));      // 3, 1
        y[11] = cmul(y[11], make_float2(-H, S * H));     // 3, 2
        y[15] = cmul(y[15], make_float2(-C1, -S * S1));  // 3, 3: W16^9
#pragma unroll
        for (int k1 = 0; k1 < 4; ++k1) {
            float2 a = y[4 * k1], b = y[4 * k1 + 1], c = y[4 * k1 + 2], d = y[4 * k1 + 3];
            dft4<S>(a, b, c, d);
            v[k1] = a; v[k1 + 4] = b; v[k1 + 8] = c; v[k1 + 12] = d;     // X[k1 + 4 k2]
        }
    }
}

// exp(S 2 pi i (t k mod M) / M), M = 2^m <= 16384, from the SFU (the sine and
// cosine units sit idle in this kernel otherwise): the angle is reduced exactly,
// in integer turns, to [-pi, pi), where the SFU's absolute error is about
// 2^-21; that adds about 1e-6 of relative error to a transform, within the
// 1e-5 the range-compression tests hold the library to.
template <int S, int M>
__device__ __forceinline__ float2 tw_sfu(int t, int k)
{
    float turns = (float)((t * k) & (M - 1)) * (1.0f / (float)M);
    turns = turns >= 0.5f ? turns - 1.0f : turns;
    float sn, cs;
    __sincosf(6.28318530718f * turns, &sn, &cs);
    return make_float2(cs, S * sn);
}

// v[t] *= w^t for t = 1 .. R-1, where w = exp(S 2 pi i k / (NS R)) is the input
// twiddle of span NS at position k: w, w^4, w^8 and w^12 from the SFU, the
// other powers as products at most three roundings deep.
template <int R, int S, int NS>
__device__ __forceinline__ void twiddle_inputs(float2* v, int k)
{
    if (R == 32) {
        // span NS = N / 32: w = exp(-2 pi i k / N), the rows of the span-N/2
        // region (stride NSH = N / 2); w^(16 + t) = w^16 w^t
        constexpr int M = 32 * NS;
        const float2 w1 = tw_sfu<S, M>(1, k), w4 = tw_sfu<S, M>(4, k);
        const float2 w8 = tw_sfu<S, M>(8, k), w12 = tw_sfu<S, M>(12, k);
        const float2 w2 = cmul(w1, w1), w3 = cmul(w2, w1), w16 = cmul(w8, w8);
        v[16] = cmul(v[16], w16);
        // each power formed where it is applied (few live registers)
#pragma unroll
        for (int a = 0; a < 16; a += 4) {
            const float2 wa = a == 0 ? make_float2(1.f, 0.f) : (a == 4 ? w4 : (a == 8 ? w8 : w12));
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                if (a + b == 0)
                    continue;
                const float2 wb = b == 1 ? w1 : (b == 2 ? w2 : w3);
                const float2 w = b == 0 ? wa : (a == 0 ? wb : cmul(wa, wb));
                v[a + b] = cmul(v[a + b], w);
                v[16 + a + b] = cmul(v[16 + a + b], cmul(w16, w));
            }
        }
        return;
    }
    constexpr int M = NS * R;
    const float2 w1 = tw_sfu<S, M>(1, k);
    v[1] = cmul(v[1], w1);
    if (R >= 4) {
        const float2 w2 = cmul(w1, w1), w3 = cmul(w2, w1);
        v[2] = cmul(v[2], w2);
        v[3] = cmul(v[3], w3);
        if (R >= 8) {
            const float2 w4 = tw_sfu<S, M>(4, k);
            v[4] = cmul(v[4], w4);
            v[5] = cmul(v[5], cmul(w4, w1));
            v[6] = cmul(v[6], cmul(w4, w2));
            v[7] = cmul(v[7], cmul(w4, w3));
            if (R == 16) {
                const float2 w8 = tw_sfu<S, M>(8, k);
                const float2 w12 = tw_sfu<S, M>(12, k);
                v[8] = cmul(v[8], w8);
                v[9] = cmul(v[9], cmul(w8, w1));
                v[10] = cmul(v[10], cmul(w8, w2));
                v[11] = cmul(v[11], cmul(w8, w3));
                v[12] = cmul(v[12], w12);
                v[13] = cmul(v[13], cmul(w12, w1));
                v[14] = cmul(v[14], cmul(w12, w2));
                v[15] = cmul(v[15], cmul(w12, w3));
            }
        }
    }
}

__host__ __device__ constexpr int pad(int i) { return i + (i >> 4); }

// A raw sample: read once, so it is not kept in L1, where the filter and
// twiddle rows that every pulse reads should stay.
__device__ __forceinline__ float2 ld_stream(const float2* p)
{
    float2 v;
    asm("ld.global.nc.L1::no_allocate.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}

// Pass structure of an N = 2^L transform: a first pass of radix R0 (2, 4, 8,
// 16 or 32, so that the rest are radix 16), PASSES passes in all, T threads,
// EPT complex values per thread. When log2 N = 1 mod 4 (N = 2 16^m) the first
// pass is radix 32 on 32 values a thread holds, and every radix-16 pass gives
// each thread two butterflies (BF = 2): no radix-2 pass and no exchange for it.
template <int L>
struct Fft {
    static constexpr int N = 1 << L;
    static constexpr bool R32 = L % 4 == 1 && L >= 5;
    static constexpr int R0 = R32 ? 32 : (L < 4 ? N : ((L % 4) ? (1 << (L % 4)) : 16));
    static constexpr int EPT = R32 ? 32 : 16;
    static constexpr int BF = EPT / 16;                // radix-16 butterflies per thread
    static constexpr int PASSES = R32 ? 1 + (L - 5) / 4 : (L < 4 ? 1 : 1 + (L - (L % 4 ? L % 4 : 4)) / 4);
    static constexpr int T = N / EPT > 32 ? N / EPT : 32;
    // resident CTAs per SM the fused table kernel's registers are sized for
    // (three CTAs of 256 threads fit the registers and the shared rows of one SM)
    static constexpr int TABLE_MINB = T <= 256 ? 3 : 1;
    static constexpr int SLOTS = pad(N - 1) + 1;       // float2 slots of the padded row
};

// Shared row: complex values as float2, one spare slot after every 16 (a
// warp's 8-byte accesses are served 16 lanes at a time; with this padding
// the strides used hit 16 distinct bank pairs). Every access pattern below is
// base + t S with (base mod 16) + (t S mod 16) < 16, for which
// pad(base + t S) = pad(base) + pad(t S): one padded base per butterfly and
// compile-time offsets.
struct Row {
    float2* d;
    __device__ __forceinline__ float2 ld(int pi) const { return d[pi]; }
    __device__ __forceinline__ void st(int pi, float2 v) const { d[pi] = v; }
};

// Radix-R Stockham pass body from shared memory: inputs x[j + t N/R], twiddles
// of span NS, the DFT. Outputs belong at pad(base) + pad(t NS), base =
// (j / NS) NS R + j % NS.
template <int R, int S, int N, int NS>
__device__ __forceinline__ void pass_load(const Row& r, float2* v, int j)
{
    constexpr int STRIDE = N / R;
    const int pb = pad(j);
#pragma unroll
    for (int t = 0; t < R; ++t)
        v[t] = r.ld(pb + pad(t * STRIDE));
    if (NS > 1)
        twiddle_inputs<R, S, NS>(v, j & (NS - 1));
    dft<R, S>(v);
}

template <int R, int NS>
__device__ __forceinline__ void pass_store(const Row& r, const float2* v, int j)
{
    const int k = j & (NS - 1);
    const int pb = pad((j - k) * R + k);
#pragma unroll
    for (int t = 0; t < R; ++t)
        r.st(pb + pad(t * NS), v[t]);
}

// Radix-16 passes p = P0 .. P1-1 of one direction (span NS at pass P0),
// shared memory to shared memory, ending with a barrier. Unrolled at compile
// time so that every span and offset is a constant.
template <int L, int S, int P, int P1, int NS>
struct Middle {
    static __device__ __forceinline__ void run(const Row& r, float2* v, int tid)
    {
        if constexpr (P < P1) {
            using F = Fft<L>;
#pragma unroll
            for (int b = 0; b < F::BF; ++b) {
                const int j = tid + b * F::T;
                if (j < F::N / 16)
                    pass_load<16, S, F::N, NS>(r, v + 16 * b, j);
            }
            __syncthreads();
#pragma unroll
            for (int b = 0; b < F::BF; ++b) {
                const int j = tid + b * F::T;
                if (j < F::N / 16)
                    pass_store<16, NS>(r, v + 16 * b, j);
            }
            __syncthreads();
            Middle<L, S, P + 1, P1, NS * 16>::run(r, v, tid);
        }
    }
};

// Forward transform of one zero-padded row (src[0 .. len-1], 0 beyond) up
// to its last pass, which stays in registers: thread tid holds X[j + t N/RL]
// in v[b RL + t], j = tid + b T, RL = 16 when PASSES > 1, else R0. Ends after
// a barrier, so the shared row may be rewritten.
template <int L>
__device__ __forceinline__ void forward_to_registers(const float2* __restrict__ src, int len, const Row& r,
                                                     float2 (&v)[Fft<L>::EPT])
{
    using F = Fft<L>;
    constexpr int R0 = F::R0, B0 = F::EPT / R0, NB0 = F::N / R0;
    const int tid = threadIdx.x;
    if (F::R32 && len <= F::N / 2) {
        // zero padding fills the second half of the row: the radix-32 pass
        // reads and transforms 16 values (one butterfly per thread)
        const int j = tid;
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const int i = j + t * NB0;
            v[t] = (j < NB0 && i < len) ? ld_stream(src + i) : make_float2(0.f, 0.f);
        }
        dft32_half<-1>(v);
    } else {
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = tid + b * F::T;
#pragma unroll
            for (int t = 0; t < R0; ++t) {
                const int i = j + t * NB0;
                v[b * R0 + t] = (j < NB0 && i < len) ? ld_stream(src + i) : make_float2(0.f, 0.f);
            }
            dft<R0, -1>(v + b * R0);
        }
    }
    if constexpr (F::PASSES > 1) {
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = tid + b * F::T;
            if (j < NB0)
                pass_store<R0, 1>(r, v + b * R0, j);
        }
        __syncthreads();
        Middle<L, -1, 1, F::PASSES - 1, R0>::run(r, v, tid);
        constexpr int NSL = F::N / 16;             // span of the last pass
#pragma unroll
        for (int b = 0; b < F::BF; ++b) {
            const int j = tid + b * F::T;
            if (j < F::N / 16)
                pass_load<16, -1, F::N, NSL>(r, v + 16 * b, j);
        }
        __syncthreads();
    }
}

template <int L>
__global__ void __launch_bounds__(Fft<L>::T) rc_filter_kernel(const float2* __restrict__ ref, int nref,
                                                              unsigned window, float band,
                                                              float4 taylor,
                                                              float2* __restrict__ h)
{
    using F = Fft<L>;
    extern __shared__ float2 smem[];
    const Row r{smem};
    float2 v[F::EPT];
    forward_to_registers<L>(ref, nref, r, v);
    constexpr int RL = F::PASSES > 1 ? 16 : F::R0;
    constexpr int BL = F::EPT / RL, NBL = F::N / RL;
    const float inv_n = 1.0f / (float)F::N;
#pragma unroll
    for (int b = 0; b < BL; ++b) {
        const int j = threadIdx.x + b * F::T;
        if (j >= NBL)
            continue;
#pragma unroll
        for (int t = 0; t < RL; ++t) {
            const int m = j + t * NBL;                  // natural frequency index
            float w = 1.0f;
            if (window != SARBP_WINDOW_NONE) {
                const float f = (float)(m < F::N / 2 ? m : m - F::N) / (float)F::N;
                const float x = f / band;
                if (!(fabsf(f) <= 0.5f * band))
                    w = 0.0f;
                else if (window == SARBP_WINDOW_HAMMING)
                    w = 0.54f + 0.46f * cospif(2.0f * x);
                else   // Taylor: 1 + 2 sum F_m cos(2 pi m x)
                    w = 1.0f + 2.0f * (taylor.x * cospif(2.0f * x) + taylor.y * cospif(4.0f * x) +
                                       taylor.z * cospif(6.0f * x) + taylor.w * cospif(8.0f * x));
            }
            const float2 x = v[b * RL + t];
            h[m] = make_float2(x.x * w * inv_n, -x.y * w * inv_n);
        }
    }
}

// Where the inverse transform's outputs go. GlobalOut writes sample i of the
// row (i < ns) to global memory. BandOut writes the samples lo .. lo + nb - 1
// of the compressed row into shared memory (band[i - lo]); it takes the
// place of the transform's own row buffer, so the outputs are held in
// registers until every thread has read its last inputs (SHARED).
struct GlobalOut {
    static constexpr bool SHARED = false;
    float2* out;
    int ns;
    __device__ __forceinline__ void put(int i, float2 v) const
    {
        if (i < ns)
            out[i] = v;
    }
};
struct BandOut {
    static constexpr bool SHARED = true;
    float2* band;
    int lo, nb, ns;
    __device__ __forceinline__ void put(int i, float2 v) const
    {
        const int w = i - lo;
        if (i < ns && (unsigned)w < (unsigned)nb)
            band[w] = v;
    }
};

// The filter product on the spectrum the forward transform left in registers,
// then the inverse transform, its outputs handed to `out`.
template <int L, class Out>
__device__ __forceinline__ void filter_inverse(const Row& r, float2 (&v)[Fft<L>::EPT],
                                               const float2* __restrict__ h, const Out& out)
{
    using F = Fft<L>;
    constexpr int N = F::N, R0 = F::R0;
    const int tid = threadIdx.x;
    if constexpr (F::PASSES == 1) {
        // N = R0 <= 32: thread 0 holds the whole spectrum
        if (tid == 0) {
#pragma unroll
            for (int t = 0; t < R0; ++t)
                v[t] = cmul(v[t], __ldg(h + t));
            dft<R0, 1>(v);
        }
        if (Out::SHARED)
            __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int t = 0; t < R0; ++t)
                out.put(t, v[t]);
        }
    } else {
        // filter, then the inverse's first pass (radix 16, span 1) on the held values
        constexpr int Q = (F::N / 16);
#pragma unroll
        for (int b = 0; b < F::BF; ++b) {
            const int j = tid + b * F::T;
            if (j < Q) {
                float2* w = v + 16 * b;
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    w[t] = cmul(w[t], __ldg(h + j + t * Q));
                dft<16, 1>(w);
                pass_store<16, 1>(r, w, j);
            }
        }
        __syncthreads();
        Middle<L, 1, 1, F::PASSES - 1, 16>::run(r, v, tid);
        // last pass: radix R0, span N / R0; outputs go to j + t N/R0
        constexpr int B0 = F::EPT / R0, NB0 = N / R0;
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = tid + b * F::T;
            if (j < NB0)
                pass_load<R0, 1, N, NB0>(r, v + b * R0, j);
        }
        if (Out::SHARED)
            __syncthreads();
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = tid + b * F::T;
            if (j >= NB0)
                continue;
#pragma unroll
            for (int t = 0; t < R0; ++t)
                out.put(j + t * NB0, v[b * R0 + t]);
        }
    }
}

template <int L>
__global__ void __launch_bounds__(Fft<L>::T, Fft<L>::TABLE_MINB) rc_kernel(const float2* __restrict__ raw, int ns_in,
                                                       const float2* __restrict__ h,
                                                       float2* __restrict__ out)
{
    extern __shared__ float2 smem[];
    const Row r{smem};
    const size_t row0 = (size_t)blockIdx.x * ns_in;
    float2 v[Fft<L>::EPT];
    forward_to_registers<L>(raw + row0, ns_in, r, v);
    filter_inverse<L>(r, v, h, GlobalOut{out + row0, ns_in});
}

// Range compression fused with the linear echo table of a backprojection
// plan: for pulse n the window start lo = klo[n] (as the table kernel finds
// it), the compressed samples lo .. lo + W kept in shared memory, and the
// W table entries (A_k, D_k / c) of that row written from them. The
// compressed frame itself never reaches global memory.
template <int L>
__global__ void __launch_bounds__(Fft<L>::T, Fft<L>::TABLE_MINB) rc_table_kernel(sarbp::BpConst k,
                                                             const float2* __restrict__ raw,
                                                             const float2* __restrict__ h,
                                                             const double* __restrict__ pos,
                                                             float4* __restrict__ table,
                                                             int* __restrict__ klo)
{
    extern __shared__ float2 smem[];
    __shared__ int s_lo;
    const int n = blockIdx.x;
    const int tid = threadIdx.x;
    if (tid == 0) {
        double rmin;
        const int lo = sarbp::window_start(k, pos[3 * (size_t)n], pos[3 * (size_t)n + 1],
                                           pos[3 * (size_t)n + 2], rmin);
        s_lo = lo;
        klo[n] = lo;
    }
    __syncthreads();
    const int lo = s_lo;
    float4* row = table + (size_t)n * k.tw;
    if (lo == sarbp::KLO_INVALID) {
        // the pulse contributes nothing: a zero row
        for (int w = tid; w < k.W; w += blockDim.x)
            row[w] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    const Row r{smem};
    const size_t row0 = (size_t)n * k.nr;
    float2 v[Fft<L>::EPT];
    forward_to_registers<L>(raw + row0, k.nr, r, v);
    filter_inverse<L>(r, v, h, BandOut{smem, lo, k.W + 1, k.nr});
    __syncthreads();
    for (int w = tid; w < k.W; w += blockDim.x) {
        float4 e = make_float4(0.f, 0.f, 0.f, 0.f);
        const long long kk = (long long)lo + w;
        if (kk >= 0 && kk <= (long long)k.nr - 2)
            e = sarbp::linear_entry(k, kk, smem[w], smem[w + 1]);
        row[w] = e;
    }
}

// Shared memory of the fused table kernel: the transform's row, or the band
// of W + 1 samples if that is longer (W <= ns + 19 <= N + 19)
template <int L>
constexpr int table_slots() { return Fft<L>::SLOTS > Fft<L>::N + 20 ? Fft<L>::SLOTS : Fft<L>::N + 20; }

template <int L>
cudaError_t set_smem_l()
{
    const int bytes = Fft<L>::SLOTS * (int)sizeof(float2);
    cudaError_t e = cudaFuncSetAttribute(rc_kernel<L>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_filter_kernel<L>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_table_kernel<L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 table_slots<L>() * (int)sizeof(float2));
    return e;
}

template <int L>
cudaError_t launch_table_l(const sarbp::BpConst& k, const float2* raw,
                           const float2* h, const double* pos, float4* table, int* klo,
                           cudaStream_t s)
{
    const int slots = Fft<L>::SLOTS > k.W + 1 ? Fft<L>::SLOTS : k.W + 1;
    rc_table_kernel<L><<<k.na, Fft<L>::T, (size_t)slots * sizeof(float2), s>>>(k, raw, h, pos,
                                                                                table, klo);
    return cudaGetLastError();
}

template <int L>
cudaError_t launch_l(bool filter, int na, const float2* in, int len,
                     const float2* h_in, unsigned window, float band, float4 taylor, float2* out,
                     cudaStream_t s)
{
    const size_t bytes = (size_t)Fft<L>::SLOTS * sizeof(float2);
    if (filter)
        rc_filter_kernel<L><<<1, Fft<L>::T, bytes, s>>>(in, len, window, band, taylor, out);
    else
        rc_kernel<L><<<na, Fft<L>::T, bytes, s>>>(in, len, h_in, out);
    return cudaGetLastError();
}

// log2 N -> the instantiation for it
cudaError_t set_smem(int log2n)
{
    switch (log2n) {
    case 1: return set_smem_l<1>();
    case 2: return set_smem_l<2>();
    case 3: return set_smem_l<3>();
    case 4: return set_smem_l<4>();
    case 5: return set_smem_l<5>();
    case 6: return set_smem_l<6>();
    case 7: return set_smem_l<7>();
    case 8: return set_smem_l<8>();
    case 9: return set_smem_l<9>();
    case 10: return set_smem_l<10>();
    case 11: return set_smem_l<11>();
    case 12: return set_smem_l<12>();
    case 13: return set_smem_l<13>();
    case 14: return set_smem_l<14>();
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_table_any(int log2n, const sarbp::BpConst& k, const float2* raw,
                             const float2* h, const double* pos, float4* table,
                             int* klo, cudaStream_t s)
{
    switch (log2n) {
    case 1: return launch_table_l<1>(k, raw, h, pos, table, klo, s);
    case 2: return launch_table_l<2>(k, raw, h, pos, table, klo, s);
    case 3: return launch_table_l<3>(k, raw, h, pos, table, klo, s);
    case 4: return launch_table_l<4>(k, raw, h, pos, table, klo, s);
    case 5: return launch_table_l<5>(k, raw, h, pos, table, klo, s);
    case 6: return launch_table_l<6>(k, raw, h, pos, table, klo, s);
    case 7: return launch_table_l<7>(k, raw, h, pos, table, klo, s);
    case 8: return launch_table_l<8>(k, raw, h, pos, table, klo, s);
    case 9: return launch_table_l<9>(k, raw, h, pos, table, klo, s);
    case 10: return launch_table_l<10>(k, raw, h, pos, table, klo, s);
    case 11: return launch_table_l<11>(k, raw, h, pos, table, klo, s);
    case 12: return launch_table_l<12>(k, raw, h, pos, table, klo, s);
    case 13: return launch_table_l<13>(k, raw, h, pos, table, klo, s);
    case 14: return launch_table_l<14>(k, raw, h, pos, table, klo, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch(int log2n, bool filter, int na, const float2* in, int len,
                   const float2* h_in, unsigned window, float band, float4 taylor, float2* out,
                   cudaStream_t s)
{
    switch (log2n) {
    case 1: return launch_l<1>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 2: return launch_l<2>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 3: return launch_l<3>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 4: return launch_l<4>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 5: return launch_l<5>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 6: return launch_l<6>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 7: return launch_l<7>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 8: return launch_l<8>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 9: return launch_l<9>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 10: return launch_l<10>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 11: return launch_l<11>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 12: return launch_l<12>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 13: return launch_l<13>(filter, na, in, len, h_in, window, band, taylor, out, s);
    case 14: return launch_l<14>(filter, na, in, len, h_in, window, band, taylor, out, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

namespace {

// Taylor's weighting coefficients F_1 .. F_4 (nbar = 5, 35 dB), in float64.
float4 taylor_coefficients()
{
    constexpr int NBAR = 5;
    const double pi = 3.14159265358979323846;
    const double a = std::acosh(std::pow(10.0, 35.0 / 20.0)) / pi;
    const double sigma2 = (double)(NBAR * NBAR) / (a * a + (NBAR - 0.5) * (NBAR - 0.5));
    double f[NBAR - 1];
    for (int m = 1; m < NBAR; ++m) {
        double num = 1.0, den = 1.0;
        for (int i = 1; i < NBAR; ++i) {
            num *= 1.0 - (double)(m * m) / (sigma2 * (a * a + (i - 0.5) * (i - 0.5)));
            if (i != m)
                den *= 1.0 - (double)(m * m) / (double)(i * i);
        }
        f[m - 1] = ((m % 2) ? 1.0 : -1.0) * num / (2.0 * den);
    }
    return make_float4((float)f[0], (float)f[1], (float)f[2], (float)f[3]);
}

}  // namespace

struct sarbp_rc_plan_s {
    sarbp_rc_params p{};
    int n = 0, log2n = 0;
    int device = -1;
    float2* h = nullptr;       // N filter coefficients / N, natural order
};

namespace sarbp {

bool rc_plan_shape(const sarbp_rc_plan_s* rc, int* na, int* ns, int* device)
{
    if (!rc)
        return false;
    *na = rc->p.na;
    *ns = rc->p.ns;
    *device = rc->device;
    return true;
}

cudaError_t launch_rc_table(const sarbp_rc_plan_s* rc, const BpConst& k, const float2* raw,
                            const double* pos, float4* table, int* klo, cudaStream_t s)
{
    return launch_table_any(rc->log2n, k, raw, rc->h, pos, table, klo, s);
}

}  // namespace sarbp

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
    if (p->window != SARBP_WINDOW_NONE && p->window != SARBP_WINDOW_HAMMING &&
        p->window != SARBP_WINDOW_TAYLOR)
        return SARBP_ERR_INVALID_ARG;
    if (p->window != SARBP_WINDOW_NONE && !(p->band_fraction > 0.0 && p->band_fraction <= 1.0))
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
    if (e == cudaSuccess)
        e = set_smem(log2n);
    if (e == cudaSuccess)
        e = sarbp::device_alloc(reinterpret_cast<void**>(&plan->h), (size_t)plan->n * sizeof(float2));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (e == cudaSuccess)
        e = launch(log2n, true, 1, static_cast<const float2*>(ref), p->nref, nullptr,
                   p->window, (float)p->band_fraction, taylor_coefficients(), plan->h, s);
    if (e != cudaSuccess) {
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
    return launch(plan->log2n, false, p.na, static_cast<const float2*>(raw), p.ns, plan->h,
                  p.window, 0.0f, make_float4(0.f, 0.f, 0.f, 0.f), static_cast<float2*>(out),
                  static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? SARBP_OK
               : SARBP_ERR_CUDA;
}

sarbp_status sarbp_rc_destroy(sarbp_rc_plan_t plan)
{
    if (plan) {
        cudaFree(plan->h);
        delete plan;
    }
    return SARBP_OK;
}

}  // extern "C"
