// dyt.cu -- Dynamic Tanh (DyT) forward and backward.
//
//   y_ij = gamma_j * tanh(alpha * x_ij) + beta_j          (scalar alpha)
//   dx_ij = dy_ij * gamma_j * alpha * sech^2(alpha x_ij)
//   dgamma_j = sum_i dy_ij tanh(alpha x_ij),  dbeta_j = sum_i dy_ij,
//   dalpha = sum_ij dy_ij gamma_j x_ij sech^2(alpha x_ij)
//
// The fused DyT kernels of Liger-Kernel PR 1617 ("fix(dyt): use a 1D grid and
// tile small-width rows", Summary) fix four properties this file keeps:
//  * a 1D grid: rows are never mapped to grid dimension 1 (65,535 limit);
//    here a persistent 1D grid loops over row blocks with 64-bit indices;
//  * several rows per CTA iteration for narrow widths (here: row groups of
//    W <= 32 threads, U rows each, from the fixed schedule table);
//  * padded rows masked AFTER the arithmetic: a padded row computes on zero
//    inputs (tanh(inf * 0) = NaN when alpha = inf) and its terms are then
//    dropped by a select, never by multiplying with a 0/1 mask;
//  * parameter gradients in the parameters' dtype, y and dx in x's dtype.
// The backward writes one partial row per CTA ([dgamma | dbeta | dalpha],
// fp32, every row written each launch); colsum.cu reduces the rows.
#include "common.cuh"
#include "internal.h"

namespace gbn {
namespace {

__device__ __forceinline__ float ex2_approx(float v)
{
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float rcp_approx(float v)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// tanh and sech^2 in float32, from two identities:
//  * |z| >= 1/8: with e = exp(-2|z|) = 2^(-2 |z| log2(e)),
//      tanh|z| = (1 - e) / (1 + e),  sech^2 z = 4e / (1 + e)^2;
//    neither loses relative accuracy for large |z| (no 1 - tanh^2).
//  * |z| < 1/8: the Maclaurin series tanh z = z - z^3/3 + 2z^5/15 - 17z^7/315
//    (the next term is below 2e-10 relative), where (1 - e) would cancel;
//    there sech^2 = 1 - tanh^2 is at least 63/64 and exact enough.
// z = +-inf gives tanh = +-1 and sech^2 = 0; NaN propagates.
constexpr float kM2Log2e = -2.0f * 1.44269504088896340736f;
constexpr float kSmall = 0.125f;
constexpr float kT3 = -1.0f / 3.0f, kT5 = 2.0f / 15.0f, kT7 = -17.0f / 315.0f;

__device__ __forceinline__ float tanh_series(float z)
{
    const float z2 = z * z;
    return z * fmaf(z2, fmaf(z2, fmaf(z2, kT7, kT5), kT3), 1.0f);
}

__device__ __forceinline__ float dyt_tanh(float z)
{
    const float a = fabsf(z);
    const float e = ex2_approx(a * kM2Log2e);
    const float tb = (1.0f - e) * rcp_approx(1.0f + e);
    return a < kSmall ? tanh_series(z) : copysignf(tb, z);
}

__device__ __forceinline__ void dyt_tanh_sech2(float z, float& t, float& s)
{
    const float a = fabsf(z);
    const float e = ex2_approx(a * kM2Log2e);
    const float q = rcp_approx(1.0f + e);
    const float ts = tanh_series(z);
    const bool small = a < kSmall;
    t = small ? ts : copysignf((1.0f - e) * q, z);
    s = small ? fmaf(-ts, ts, 1.0f) : 4.0f * e * q * q;
}

// ------------------------------------------------------------ fast forward
template <typename TX, int S>
__global__ void __launch_bounds__(kSched[S].T, kSched[S].MINB)
    dyt_fwd_fast(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ alpha,
                 const void* __restrict__ gamma, const void* __restrict__ beta, int pt,
                 int64_t M, int N, int64_t nblocks)
{
    constexpr int W = kSched[S].W, KV = kSched[S].KV, U = kSched[S].UF, T = kSched[S].T;
    constexpr int VEC = Vec<TX>::kN;
    constexpr int G = T / W;
    const int g = threadIdx.x / W, l = threadIdx.x % W;
    const int nvec = N / VEC;

    const float a = ld_param(alpha, pt, 0);
    float gm[KV][VEC], bt[KV][VEC];
#pragma unroll
    for (int kv = 0; kv < KV; ++kv) {
        const int cv = kv * W + l;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const bool ok = cv < nvec;
            gm[kv][e] = ok ? ld_param(gamma, pt, cv * VEC + e) : 0.f;
            bt[kv][e] = ok ? ld_param(beta, pt, cv * VEC + e) : 0.f;
        }
    }

    for (int64_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
        uint4 r[U][KV];
        int64_t row[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            row[u] = b * (G * U) + u * G + g;
#pragma unroll
            for (int kv = 0; kv < KV; ++kv) {
                const int cv = kv * W + l;
                if (row[u] < M && cv < nvec)
                    r[u][kv] = ld_stream(x + row[u] * N + cv * VEC);
                else
                    r[u][kv] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int kv = 0; kv < KV; ++kv) {
                const int cv = kv * W + l;
                float f[VEC];
                unpack(r[u][kv], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) f[e] = fmaf(gm[kv][e], dyt_tanh(a * f[e]), bt[kv][e]);
                if (row[u] < M && cv < nvec) st_stream(y + row[u] * N + cv * VEC, pack(f));
            }
        }
    }
}

// ----------------------------------------------------------- fast backward
template <typename TX, int S>
__global__ void __launch_bounds__(kSched[S].T, kSched[S].MINB)
    dyt_bwd_fast(const TX* __restrict__ x, const TX* __restrict__ dy, TX* __restrict__ dx,
                 const void* __restrict__ alpha, const void* __restrict__ gamma, int pt,
                 float* __restrict__ ws, int64_t M, int N, int64_t nblocks)
{
    constexpr int W = kSched[S].W, KV = kSched[S].KV, U = kSched[S].UB, T = kSched[S].T;
    constexpr int VEC = Vec<TX>::kN;
    constexpr int G = T / W;
    __shared__ float colbuf[G > 1 ? T * KV * VEC : 1];
    __shared__ float red[T / 32];
    const int g = threadIdx.x / W, l = threadIdx.x % W;
    const int nvec = N / VEC;

    const float a = ld_param(alpha, pt, 0);
    float gm[KV][VEC], ga[KV][VEC];
#pragma unroll
    for (int kv = 0; kv < KV; ++kv) {
        const int cv = kv * W + l;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            gm[kv][e] = cv < nvec ? ld_param(gamma, pt, cv * VEC + e) : 0.f;
            ga[kv][e] = gm[kv][e] * a;
        }
    }
    // Per-column accumulators: sum dy*t, sum dy, sum dy*x*sech^2 (gamma is
    // applied to the last one once, at the end).
    float acc_g[KV][VEC], acc_b[KV][VEC], acc_a[KV][VEC];
#pragma unroll
    for (int kv = 0; kv < KV; ++kv)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc_g[kv][e] = acc_b[kv][e] = acc_a[kv][e] = 0.f;

    for (int64_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
        uint4 rx[U][KV], rd[U][KV];
        int64_t row[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            row[u] = b * (G * U) + u * G + g;
#pragma unroll
            for (int kv = 0; kv < KV; ++kv) {
                const int cv = kv * W + l;
                if (row[u] < M && cv < nvec) {
                    rx[u][kv] = ld_stream(x + row[u] * N + cv * VEC);
                    rd[u][kv] = ld_stream(dy + row[u] * N + cv * VEC);
                } else {
                    rx[u][kv] = rd[u][kv] = make_uint4(0, 0, 0, 0);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int kv = 0; kv < KV; ++kv) {
                const int cv = kv * W + l;
                const bool ok = row[u] < M && cv < nvec;
                float xf[VEC], df[VEC], o[VEC];
                unpack(rx[u][kv], xf);
                unpack(rd[u][kv], df);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    float t, s;
                    dyt_tanh_sech2(a * xf[e], t, s);
                    const float ds = df[e] * s;
                    o[e] = ds * ga[kv][e];
                    // mask after the arithmetic: select, never multiply by 0/1
                    acc_g[kv][e] += ok ? df[e] * t : 0.f;
                    acc_b[kv][e] += ok ? df[e] : 0.f;
                    acc_a[kv][e] += ok ? ds * xf[e] : 0.f;
                }
                if (ok) st_stream(dx + row[u] * N + cv * VEC, pack(o));
            }
        }
    }

    if (ws == nullptr) return;  // no parameter gradient requested (uniform)
    const int64_t L = 2 * (int64_t)N + 1;
    float* wrow = ws + blockIdx.x * L;
    cta_store_columns<W, KV, VEC, T>(acc_g, colbuf, wrow, N);
    cta_store_columns<W, KV, VEC, T>(acc_b, colbuf, wrow + N, N);
    float da = 0.f;
#pragma unroll
    for (int kv = 0; kv < KV; ++kv)
#pragma unroll
        for (int e = 0; e < VEC; ++e) da = fmaf(gm[kv][e], acc_a[kv][e], da);
    const float tot = cta_sum<T>(da, red);
    if (threadIdx.x == 0) wrow[2 * N] = tot;
}

// ------------------------------------------------------ general (any shape)
template <typename TX>
__global__ void __launch_bounds__(kGenThreads)
    dyt_fwd_general(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ alpha,
                    const void* __restrict__ gamma, const void* __restrict__ beta, int pt,
                    int64_t M, int N)
{
    const float a = ld_param(alpha, pt, 0);
    const int64_t E = M * (int64_t)N;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < E;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % N);
        st1(y, i, fmaf(ld_param(gamma, pt, c), dyt_tanh(a * ld1(x, i)), ld_param(beta, pt, c)));
    }
}

// One warp per row; warp w owns workspace row w and accumulates into it
// (read-modify-write by the lane that owns each column, rows in order).
template <typename TX>
__global__ void __launch_bounds__(kGenThreads)
    dyt_bwd_general(const TX* __restrict__ x, const TX* __restrict__ dy, TX* __restrict__ dx,
                    const void* __restrict__ alpha, const void* __restrict__ gamma, int pt,
                    float* __restrict__ ws, int64_t M, int N)
{
    const int lane = threadIdx.x & 31;
    const int64_t w = blockIdx.x * (int64_t)kGenWarps + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * kGenWarps;
    const int64_t L = 2 * (int64_t)N + 1;
    float* wrow = ws ? ws + w * L : nullptr;
    if (wrow)
        for (int c = lane; c < 2 * N; c += 32) wrow[c] = 0.f;
    const float a = ld_param(alpha, pt, 0);
    float da = 0.f;
    for (int64_t r = w; r < M; r += nw) {
        for (int c = lane; c < N; c += 32) {
            const int64_t i = r * N + c;
            const float xv = ld1(x, i), dv = ld1(dy, i), gmv = ld_param(gamma, pt, c);
            float t, s;
            dyt_tanh_sech2(a * xv, t, s);
            const float ds = dv * s;
            st1(dx, i, ds * (gmv * a));
            if (wrow) {
                wrow[c] += dv * t;
                wrow[N + c] += dv;
            }
            da = fmaf(gmv, ds * xv, da);
        }
    }
    float v[1] = {da};
    butterfly<32, 1>(v);
    if (wrow && lane == 0) wrow[2 * N] = v[0];
}

template <typename TX>
cudaError_t fwd_dispatch(const Launch& L, int pt, const void* x, const void* alpha,
                         const void* gamma, const void* beta, void* y, int64_t M, int N)
{
    const TX* xp = static_cast<const TX*>(x);
    TX* yp = static_cast<TX*>(y);
    if (!L.fast) {
        dyt_fwd_general<TX><<<L.grid, kGenThreads, 0, L.stream>>>(xp, yp, alpha, gamma, beta, pt,
                                                                  M, N);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE(S)                                                                      \
    case S:                                                                              \
        dyt_fwd_fast<TX, S><<<L.grid, kSched[S].T, 0, L.stream>>>(xp, yp, alpha, gamma, \
                                                                  beta, pt, M, N,       \
                                                                  L.nblocks);           \
        break;
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9) GBN_CASE(10)
#undef GBN_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename TX>
cudaError_t bwd_dispatch(const Launch& L, int pt, const void* x, const void* dy, const void* alpha,
                         const void* gamma, void* dx, float* ws, int64_t M, int N)
{
    const TX* xp = static_cast<const TX*>(x);
    const TX* dyp = static_cast<const TX*>(dy);
    TX* dxp = static_cast<TX*>(dx);
    if (!L.fast) {
        dyt_bwd_general<TX><<<L.grid, kGenThreads, 0, L.stream>>>(xp, dyp, dxp, alpha, gamma, pt,
                                                                  ws, M, N);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE(S)                                                                           \
    case S:                                                                                   \
        dyt_bwd_fast<TX, S><<<L.grid, kSched[S].T, 0, L.stream>>>(xp, dyp, dxp, alpha, gamma, \
                                                                  pt, ws, M, N, L.nblocks);  \
        break;
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9) GBN_CASE(10)
#undef GBN_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dyt_fwd(const Launch& L, int xt, int pt, const void* x, const void* alpha,
                           const void* gamma, const void* beta, void* y, int64_t M, int N)
{
    if (xt == kF32) return fwd_dispatch<float>(L, pt, x, alpha, gamma, beta, y, M, N);
    return fwd_dispatch<__nv_bfloat16>(L, pt, x, alpha, gamma, beta, y, M, N);
}

cudaError_t launch_dyt_bwd(const Launch& L, int xt, int pt, const void* x, const void* dy,
                           const void* alpha, const void* gamma, void* dx, float* ws, int64_t M,
                           int N)
{
    if (xt == kF32) return bwd_dispatch<float>(L, pt, x, dy, alpha, gamma, dx, ws, M, N);
    return bwd_dispatch<__nv_bfloat16>(L, pt, x, dy, alpha, gamma, dx, ws, M, N);
}

}  // namespace gbn
