// layernorm.cu -- LayerNorm forward and backward over the last dimension.
//
//   mu = mean_j x,  var = mean_j (x - mu)^2 (biased),  r = 1/sqrt(var + eps)
//   xhat = (x - mu) r,  y = xhat * gamma_j + beta_j   (gamma, beta nullable)
//   backward (saved mu, r):  g = dy * gamma_j,
//     dx = r (g - mean_j g - xhat * mean_j(g xhat)),
//     dgamma_j = sum_i dy xhat,  dbeta_j = sum_i dy
//
// The torch-xpu-ops page "Layernorm bwd OPT #1880" shows the gamma/beta
// column reduction starving the GPU when M >> N (one workgroup for the
// [25088*16, 24] backward) and replaces it with per-workgroup partials plus a
// second summation pass.  Here the column partials are accumulated in
// registers by the same persistent CTAs that compute dx (x and dy are read
// once), written as one fp32 row per CTA, and summed by colsum.cu.
#include "common.cuh"
#include "internal.h"

namespace gbn {
namespace {

// ------------------------------------------------------------ fast forward
template <typename TX, int S>
__global__ void __launch_bounds__(kSched[S].T, kSched[S].MINB)
    ln_fwd_fast(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ gamma,
                const void* __restrict__ beta, int pt, float* __restrict__ mean,
                float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n,
                int64_t nblocks)
{
    constexpr int W = kSched[S].W, KV = kSched[S].KV, U = kSched[S].UB, T = kSched[S].T;
    constexpr int VEC = Vec<TX>::kN;
    constexpr int G = T / W;
    __shared__ float red[GroupRed<W, T, U>::kFloats];
    int parity = 0;
    const int g = threadIdx.x / W, l = threadIdx.x % W;
    const int nvec = N / VEC;

    float gm[KV][VEC], bt[KV][VEC];
#pragma unroll
    for (int kv = 0; kv < KV; ++kv) {
        const int cv = kv * W + l;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const bool ok = cv < nvec;
            gm[kv][e] = (ok && gamma) ? ld_param(gamma, pt, cv * VEC + e) : 1.f;
            bt[kv][e] = (ok && beta) ? ld_param(beta, pt, cv * VEC + e) : 0.f;
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
        // pass 1: row sums (absent columns were loaded as zeros)
        float s[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            s[u] = 0.f;
#pragma unroll
            for (int kv = 0; kv < KV; ++kv) {
                float f[VEC];
                unpack(r[u][kv], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) s[u] += f[e];
            }
        }
        group_allreduce<W, T, U>(s, red, parity);
        float mu[U], q[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            mu[u] = s[u] * inv_n;
            q[u] = 0.f;
#pragma unroll
            for (int kv = 0; kv < KV; ++kv) {
                const bool okc = (kv * W + l) < nvec;
                float f[VEC];
                unpack(r[u][kv], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float d = f[e] - mu[u];
                    q[u] += okc ? d * d : 0.f;
                }
            }
        }
        // pass 2: centred sum of squares
        group_allreduce<W, T, U>(q, red, parity);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float rs = rsqrtf(fmaf(q[u], inv_n, eps));
#pragma unroll
            for (int kv = 0; kv < KV; ++kv) {
                const int cv = kv * W + l;
                float f[VEC];
                unpack(r[u][kv], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) f[e] = fmaf((f[e] - mu[u]) * rs, gm[kv][e], bt[kv][e]);
                if (row[u] < M && cv < nvec) st_stream(y + row[u] * N + cv * VEC, pack(f));
            }
            if (l == 0 && row[u] < M) {
                if (mean) mean[row[u]] = mu[u];
                if (rstd) rstd[row[u]] = rs;
            }
        }
    }
}

// ----------------------------------------------------------- fast backward
template <typename TX, int S>
__global__ void __launch_bounds__(kSched[S].T, kSched[S].MINB)
    ln_bwd_fast(const TX* __restrict__ x, const TX* __restrict__ dy,
                const float* __restrict__ mean, const float* __restrict__ rstd,
                const void* __restrict__ gamma, int pt, TX* __restrict__ dx,
                float* __restrict__ ws, int64_t M, int N, float inv_n, int64_t nblocks)
{
    constexpr int W = kSched[S].W, KV = kSched[S].KV, U = kSched[S].UB, T = kSched[S].T;
    constexpr int VEC = Vec<TX>::kN;
    constexpr int G = T / W;
    __shared__ float colbuf[G > 1 ? T * KV * VEC : 1];
    __shared__ float red[GroupRed<W, T, 2 * U>::kFloats];
    int parity = 0;
    const int g = threadIdx.x / W, l = threadIdx.x % W;
    const int nvec = N / VEC;

    float gm[KV][VEC];
#pragma unroll
    for (int kv = 0; kv < KV; ++kv) {
        const int cv = kv * W + l;
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            gm[kv][e] = (cv < nvec && gamma) ? ld_param(gamma, pt, cv * VEC + e) : 1.f;
    }
    float acc_g[KV][VEC], acc_b[KV][VEC];
#pragma unroll
    for (int kv = 0; kv < KV; ++kv)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc_g[kv][e] = acc_b[kv][e] = 0.f;

    for (int64_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
        uint4 rx[U][KV], rd[U][KV];
        int64_t row[U];
        float mu[U], rs[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            row[u] = b * (G * U) + u * G + g;
            const bool okr = row[u] < M;
            mu[u] = okr ? mean[row[u]] : 0.f;
            rs[u] = okr ? rstd[row[u]] : 0.f;
#pragma unroll
            for (int kv = 0; kv < KV; ++kv) {
                const int cv = kv * W + l;
                if (okr && cv < nvec) {
                    rx[u][kv] = ld_stream(x + row[u] * N + cv * VEC);
                    rd[u][kv] = ld_stream(dy + row[u] * N + cv * VEC);
                } else {
                    rx[u][kv] = rd[u][kv] = make_uint4(0, 0, 0, 0);
                }
            }
        }
        // one all-reduce of (sum g, sum g*xhat) per row
        float s[2 * U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            s[2 * u] = s[2 * u + 1] = 0.f;
#pragma unroll
            for (int kv = 0; kv < KV; ++kv) {
                const bool okc = (kv * W + l) < nvec;
                float xf[VEC], df[VEC];
                unpack(rx[u][kv], xf);
                unpack(rd[u][kv], df);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float xh = (xf[e] - mu[u]) * rs[u];
                    const float gg = df[e] * gm[kv][e];
                    s[2 * u] += gg;
                    s[2 * u + 1] += okc ? gg * xh : 0.f;
                }
            }
        }
        group_allreduce<W, T, 2 * U>(s, red, parity);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float ma = s[2 * u] * inv_n;
            const float mb = s[2 * u + 1] * inv_n;
            const bool okr = row[u] < M;
#pragma unroll
            for (int kv = 0; kv < KV; ++kv) {
                const int cv = kv * W + l;
                const bool ok = okr && cv < nvec;
                float xf[VEC], df[VEC], o[VEC];
                unpack(rx[u][kv], xf);
                unpack(rd[u][kv], df);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float xh = (xf[e] - mu[u]) * rs[u];
                    const float gg = df[e] * gm[kv][e];
                    o[e] = rs[u] * (gg - ma - xh * mb);
                    acc_g[kv][e] += ok ? df[e] * xh : 0.f;
                    acc_b[kv][e] += ok ? df[e] : 0.f;
                }
                if (ok) st_stream(dx + row[u] * N + cv * VEC, pack(o));
            }
        }
    }

    if (ws == nullptr) return;  // no parameter gradient requested (uniform)
    float* wrow = ws + blockIdx.x * (2 * (int64_t)N);
    cta_store_columns<W, KV, VEC, T>(acc_g, colbuf, wrow, N);
    cta_store_columns<W, KV, VEC, T>(acc_b, colbuf, wrow + N, N);
}

// ------------------------------------------------------ general (any shape)
// One warp per row, scalar loads, row re-read from cache per pass.
template <typename TX>
__global__ void __launch_bounds__(kGenThreads)
    ln_fwd_general(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ gamma,
                   const void* __restrict__ beta, int pt, float* __restrict__ mean,
                   float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n)
{
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kGenWarps;
    for (int64_t r = blockIdx.x * (int64_t)kGenWarps + (threadIdx.x >> 5); r < M; r += nw) {
        const TX* xr = x + r * N;
        float v[1] = {0.f};
        for (int c = lane; c < N; c += 32) v[0] += ld1(xr, c);
        butterfly<32, 1>(v);
        const float mu = v[0] * inv_n;
        float q[1] = {0.f};
        for (int c = lane; c < N; c += 32) {
            const float d = ld1(xr, c) - mu;
            q[0] += d * d;
        }
        butterfly<32, 1>(q);
        const float rs = rsqrtf(fmaf(q[0], inv_n, eps));
        for (int c = lane; c < N; c += 32) {
            const float gm = gamma ? ld_param(gamma, pt, c) : 1.f;
            const float bt = beta ? ld_param(beta, pt, c) : 0.f;
            st1(y, r * N + c, fmaf((ld1(xr, c) - mu) * rs, gm, bt));
        }
        if (lane == 0) {
            if (mean) mean[r] = mu;
            if (rstd) rstd[r] = rs;
        }
    }
}

template <typename TX>
__global__ void __launch_bounds__(kGenThreads)
    ln_bwd_general(const TX* __restrict__ x, const TX* __restrict__ dy,
                   const float* __restrict__ mean, const float* __restrict__ rstd,
                   const void* __restrict__ gamma, int pt, TX* __restrict__ dx,
                   float* __restrict__ ws, int64_t M, int N, float inv_n)
{
    const int lane = threadIdx.x & 31;
    const int64_t w = blockIdx.x * (int64_t)kGenWarps + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * kGenWarps;
    float* wrow = ws ? ws + w * (2 * (int64_t)N) : nullptr;
    if (wrow)
        for (int c = lane; c < 2 * N; c += 32) wrow[c] = 0.f;
    for (int64_t r = w; r < M; r += nw) {
        const TX* xr = x + r * N;
        const TX* dr = dy + r * N;
        const float mu = mean[r], rs = rstd[r];
        float s[2] = {0.f, 0.f};
        for (int c = lane; c < N; c += 32) {
            const float xh = (ld1(xr, c) - mu) * rs;
            const float gg = ld1(dr, c) * (gamma ? ld_param(gamma, pt, c) : 1.f);
            s[0] += gg;
            s[1] += gg * xh;
        }
        butterfly<32, 2>(s);
        const float ma = s[0] * inv_n, mb = s[1] * inv_n;
        for (int c = lane; c < N; c += 32) {
            const float xh = (ld1(xr, c) - mu) * rs;
            const float dv = ld1(dr, c);
            const float gg = dv * (gamma ? ld_param(gamma, pt, c) : 1.f);
            st1(dx, r * N + c, rs * (gg - ma - xh * mb));
            if (wrow) {
                wrow[c] += dv * xh;
                wrow[N + c] += dv;
            }
        }
    }
}

template <typename TX>
cudaError_t fwd_dispatch(const Launch& L, int pt, const void* x, const void* gamma,
                         const void* beta, void* y, float* mean, float* rstd, int64_t M, int N,
                         float eps)
{
    const TX* xp = static_cast<const TX*>(x);
    TX* yp = static_cast<TX*>(y);
    const float inv_n = (float)(1.0 / (double)N);
    if (!L.fast) {
        ln_fwd_general<TX><<<L.grid, kGenThreads, 0, L.stream>>>(xp, yp, gamma, beta, pt, mean,
                                                                 rstd, M, N, eps, inv_n);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE(S)                                                                            \
    case S:                                                                                    \
        ln_fwd_fast<TX, S><<<L.grid, kSched[S].T, 0, L.stream>>>(xp, yp, gamma, beta, pt, mean, \
                                                                 rstd, M, N, eps, inv_n,       \
                                                                 L.nblocks);                  \
        break;
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9) GBN_CASE(10)
#undef GBN_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename TX>
cudaError_t bwd_dispatch(const Launch& L, int pt, const void* x, const void* dy,
                         const float* mean, const float* rstd, const void* gamma, void* dx,
                         float* ws, int64_t M, int N)
{
    const TX* xp = static_cast<const TX*>(x);
    const TX* dyp = static_cast<const TX*>(dy);
    TX* dxp = static_cast<TX*>(dx);
    const float inv_n = (float)(1.0 / (double)N);
    if (!L.fast) {
        ln_bwd_general<TX><<<L.grid, kGenThreads, 0, L.stream>>>(xp, dyp, mean, rstd, gamma, pt,
                                                                 dxp, ws, M, N, inv_n);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE(S)                                                                       \
    case S:                                                                               \
        ln_bwd_fast<TX, S><<<L.grid, kSched[S].T, 0, L.stream>>>(xp, dyp, mean, rstd,     \
                                                                 gamma, pt, dxp, ws, M, N, \
                                                                 inv_n, L.nblocks);       \
        break;
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9) GBN_CASE(10)
#undef GBN_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ln_fwd(const Launch& L, int xt, int pt, const void* x, const void* gamma,
                          const void* beta, void* y, float* mean, float* rstd, int64_t M, int N,
                          float eps)
{
    if (xt == kF32) return fwd_dispatch<float>(L, pt, x, gamma, beta, y, mean, rstd, M, N, eps);
    return fwd_dispatch<__nv_bfloat16>(L, pt, x, gamma, beta, y, mean, rstd, M, N, eps);
}

cudaError_t launch_ln_bwd(const Launch& L, int xt, int pt, const void* x, const void* dy,
                          const float* mean, const float* rstd, const void* gamma, void* dx,
                          float* ws, int64_t M, int N)
{
    if (xt == kF32) return bwd_dispatch<float>(L, pt, x, dy, mean, rstd, gamma, dx, ws, M, N);
    return bwd_dispatch<__nv_bfloat16>(L, pt, x, dy, mean, rstd, gamma, dx, ws, M, N);
}

}  // namespace gbn
