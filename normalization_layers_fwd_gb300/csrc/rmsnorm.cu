// rmsnorm.cu -- Llama-style RMSNorm forward and backward.
//
//   weight * (x.float() * rsqrt(mean(x.float()^2) + eps)).to(x.dtype)
//
// Rounding points, as the fused-RMSNorm page fixes them (DeepSpeed PR 8645,
// quoted in PR 8664, section "Semantics"): variance and normalization in
// fp32, ONE rounding of the normalized value n to x's dtype, then the
// multiply by the weight (rounded to x's dtype on store).  In the backward,
// dy*w is rounded to x's dtype (dn), and when the weight has x's dtype each
// weight-gradient term dy*n is rounded to x's dtype before its fp32 column
// sum (with an fp32 weight the term stays fp32):
//   r = rsqrt(mean_j x^2 + eps),  xhat = x r (fp32),  n = round_x(xhat)
//   dn = round_x(dy w),  dx = round_x(r (dn - xhat mean_j(dn xhat)))
//   dw_j = sum_i term_ij
// The backward takes the forward's rstd when given; otherwise it recomputes
// r with the same code, the same row-group layout and therefore the same
// summation order as the forward, so both give identical bits.
// The PR 8664 narrow-row follow-up computes dx and the weight-gradient
// partials in one pass over x and dy; every width does that here.
#include "common.cuh"
#include "internal.h"

namespace gbn {
namespace {

// Sum of squares of one thread's slice of a row (absent columns are zeros).
template <typename TX, int KV, int VEC>
__device__ __forceinline__ float slice_sumsq(const uint4 (&r)[KV])
{
    float s = 0.f;
#pragma unroll
    for (int kv = 0; kv < KV; ++kv) {
        float f[VEC];
        unpack(r[kv], f);
#pragma unroll
        for (int e = 0; e < VEC; ++e) s = fmaf(f[e], f[e], s);
    }
    return s;
}

// ------------------------------------------------------------ fast forward
template <typename TX, int S>
__global__ void __launch_bounds__(kSched[S].T, kSched[S].MINB)
    rms_fwd_fast(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ w,
                 int pt, float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n,
                 int64_t nblocks)
{
    constexpr int W = kSched[S].W, KV = kSched[S].KV, U = kSched[S].UF, T = kSched[S].T;
    constexpr int VEC = Vec<TX>::kN;
    constexpr int G = T / W;
    __shared__ float red[GroupRed<W, T, U>::kFloats];
    int parity = 0;
    const int g = threadIdx.x / W, l = threadIdx.x % W;
    const int nvec = N / VEC;

    float wf[KV][VEC];
#pragma unroll
    for (int kv = 0; kv < KV; ++kv) {
        const int cv = kv * W + l;
#pragma unroll
        for (int e = 0; e < VEC; ++e) wf[kv][e] = cv < nvec ? ld_param(w, pt, cv * VEC + e) : 0.f;
    }

    for (int64_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
        uint4 r[U][KV];
        int64_t row[U];
        float s[U];
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
        for (int u = 0; u < U; ++u) s[u] = slice_sumsq<TX, KV, VEC>(r[u]);
        group_allreduce<W, T, U>(s, red, parity);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float rs = rsqrtf(fmaf(s[u], inv_n, eps));
#pragma unroll
            for (int kv = 0; kv < KV; ++kv) {
                const int cv = kv * W + l;
                float f[VEC];
                unpack(r[u][kv], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) f[e] = wf[kv][e] * round_x<TX>(f[e] * rs);
                if (row[u] < M && cv < nvec) st_stream(y + row[u] * N + cv * VEC, pack(f));
            }
            if (rstd && l == 0 && row[u] < M) rstd[row[u]] = rs;
        }
    }
}

// ----------------------------------------------------------- fast backward
template <typename TX, int S>
__global__ void __launch_bounds__(kSched[S].T, kSched[S].MINB)
    rms_bwd_fast(const TX* __restrict__ x, const TX* __restrict__ dy, const void* __restrict__ w,
                 int pt, const float* __restrict__ rstd, TX* __restrict__ dx,
                 float* __restrict__ ws, int64_t M, int N, float eps, float inv_n,
                 int64_t nblocks)
{
    constexpr int W = kSched[S].W, KV = kSched[S].KV, U = kSched[S].UB, T = kSched[S].T;
    constexpr int VEC = Vec<TX>::kN;
    constexpr int G = T / W;
    __shared__ float colbuf[G > 1 ? T * KV * VEC : 1];
    __shared__ float red[GroupRed<W, T, U>::kFloats];
    int parity = 0;
    const int g = threadIdx.x / W, l = threadIdx.x % W;
    const int nvec = N / VEC;
    const bool round_terms = (pt != kF32);  // weight in x's dtype: round dy*n

    float wf[KV][VEC], acc[KV][VEC];
#pragma unroll
    for (int kv = 0; kv < KV; ++kv) {
        const int cv = kv * W + l;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            wf[kv][e] = cv < nvec ? ld_param(w, pt, cv * VEC + e) : 0.f;
            acc[kv][e] = 0.f;
        }
    }

    for (int64_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
        uint4 rx[U][KV], rd[U][KV];
        int64_t row[U];
        float rs[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            row[u] = b * (G * U) + u * G + g;
            if (rstd) rs[u] = row[u] < M ? rstd[row[u]] : 0.f;
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
        if (!rstd) {  // uniform branch: recompute r exactly as the forward does
#pragma unroll
            for (int u = 0; u < U; ++u) rs[u] = slice_sumsq<TX, KV, VEC>(rx[u]);
            group_allreduce<W, T, U>(rs, red, parity);
#pragma unroll
            for (int u = 0; u < U; ++u) rs[u] = rsqrtf(fmaf(rs[u], inv_n, eps));
        }
        float s[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            s[u] = 0.f;
#pragma unroll
            for (int kv = 0; kv < KV; ++kv) {
                float xf[VEC], df[VEC];
                unpack(rx[u][kv], xf);
                unpack(rd[u][kv], df);
#pragma unroll
                for (int e = 0; e < VEC; ++e) s[u] = fmaf(round_x<TX>(df[e] * wf[kv][e]), xf[e] * rs[u], s[u]);
            }
        }
        group_allreduce<W, T, U>(s, red, parity);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float m = s[u] * inv_n;
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
                    const float xh = xf[e] * rs[u];
                    const float dn = round_x<TX>(df[e] * wf[kv][e]);
                    o[e] = rs[u] * (dn - xh * m);
                    float term = df[e] * round_x<TX>(xh);
                    if (round_terms) term = round_x<TX>(term);
                    acc[kv][e] += ok ? term : 0.f;
                }
                if (ok) st_stream(dx + row[u] * N + cv * VEC, pack(o));
            }
        }
    }

    if (ws == nullptr) return;  // no weight gradient requested (uniform)
    float* wrow = ws + blockIdx.x * (int64_t)N;
    cta_store_columns<W, KV, VEC, T>(acc, colbuf, wrow, N);
}

// ------------------------------------------------------ general (any shape)
template <typename TX>
__device__ __forceinline__ float warp_row_rstd(const TX* xr, int N, int lane, float eps,
                                               float inv_n)
{
    float v[1] = {0.f};
    for (int c = lane; c < N; c += 32) {
        const float f = ld1(xr, c);
        v[0] = fmaf(f, f, v[0]);
    }
    butterfly<32, 1>(v);
    return rsqrtf(fmaf(v[0], inv_n, eps));
}

template <typename TX>
__global__ void __launch_bounds__(kGenThreads)
    rms_fwd_general(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ w,
                    int pt, float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n)
{
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kGenWarps;
    for (int64_t r = blockIdx.x * (int64_t)kGenWarps + (threadIdx.x >> 5); r < M; r += nw) {
        const TX* xr = x + r * N;
        const float rs = warp_row_rstd(xr, N, lane, eps, inv_n);
        for (int c = lane; c < N; c += 32)
            st1(y, r * N + c, ld_param(w, pt, c) * round_x<TX>(ld1(xr, c) * rs));
        if (rstd && lane == 0) rstd[r] = rs;
    }
}

template <typename TX>
__global__ void __launch_bounds__(kGenThreads)
    rms_bwd_general(const TX* __restrict__ x, const TX* __restrict__ dy,
                    const void* __restrict__ w, int pt, const float* __restrict__ rstd,
                    TX* __restrict__ dx, float* __restrict__ ws, int64_t M, int N, float eps,
                    float inv_n)
{
    const int lane = threadIdx.x & 31;
    const int64_t wi = blockIdx.x * (int64_t)kGenWarps + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * kGenWarps;
    const bool round_terms = (pt != kF32);
    float* wrow = ws ? ws + wi * (int64_t)N : nullptr;
    if (wrow)
        for (int c = lane; c < N; c += 32) wrow[c] = 0.f;
    for (int64_t r = wi; r < M; r += nw) {
        const TX* xr = x + r * N;
        const TX* dr = dy + r * N;
        const float rs = rstd ? rstd[r] : warp_row_rstd(xr, N, lane, eps, inv_n);
        float s[1] = {0.f};
        for (int c = lane; c < N; c += 32) {
            const float dn = round_x<TX>(ld1(dr, c) * ld_param(w, pt, c));
            s[0] = fmaf(dn, ld1(xr, c) * rs, s[0]);
        }
        butterfly<32, 1>(s);
        const float m = s[0] * inv_n;
        for (int c = lane; c < N; c += 32) {
            const float dv = ld1(dr, c);
            const float xh = ld1(xr, c) * rs;
            const float dn = round_x<TX>(dv * ld_param(w, pt, c));
            st1(dx, r * N + c, rs * (dn - xh * m));
            float term = dv * round_x<TX>(xh);
            if (round_terms) term = round_x<TX>(term);
            if (wrow) wrow[c] += term;
        }
    }
}

template <typename TX>
cudaError_t fwd_dispatch(const Launch& L, int pt, const void* x, const void* w, void* y,
                         float* rstd, int64_t M, int N, float eps)
{
    const TX* xp = static_cast<const TX*>(x);
    TX* yp = static_cast<TX*>(y);
    const float inv_n = (float)(1.0 / (double)N);
    if (!L.fast) {
        rms_fwd_general<TX><<<L.grid, kGenThreads, 0, L.stream>>>(xp, yp, w, pt, rstd, M, N, eps,
                                                                  inv_n);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE(S)                                                                           \
    case S:                                                                                   \
        rms_fwd_fast<TX, S><<<L.grid, kSched[S].T, 0, L.stream>>>(xp, yp, w, pt, rstd, M, N, \
                                                                  eps, inv_n, L.nblocks);    \
        break;
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9) GBN_CASE(10)
#undef GBN_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename TX>
cudaError_t bwd_dispatch(const Launch& L, int pt, const void* x, const void* dy, const void* w,
                         const float* rstd, void* dx, float* ws, int64_t M, int N, float eps)
{
    const TX* xp = static_cast<const TX*>(x);
    const TX* dyp = static_cast<const TX*>(dy);
    TX* dxp = static_cast<TX*>(dx);
    const float inv_n = (float)(1.0 / (double)N);
    if (!L.fast) {
        rms_bwd_general<TX><<<L.grid, kGenThreads, 0, L.stream>>>(xp, dyp, w, pt, rstd, dxp, ws,
                                                                  M, N, eps, inv_n);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE(S)                                                                         \
    case S:                                                                                 \
        rms_bwd_fast<TX, S><<<L.grid, kSched[S].T, 0, L.stream>>>(xp, dyp, w, pt, rstd, dxp, \
                                                                  ws, M, N, eps, inv_n,    \
                                                                  L.nblocks);              \
        break;
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9) GBN_CASE(10)
#undef GBN_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rms_fwd(const Launch& L, int xt, int pt, const void* x, const void* w, void* y,
                           float* rstd, int64_t M, int N, float eps)
{
    if (xt == kF32) return fwd_dispatch<float>(L, pt, x, w, y, rstd, M, N, eps);
    return fwd_dispatch<__nv_bfloat16>(L, pt, x, w, y, rstd, M, N, eps);
}

cudaError_t launch_rms_bwd(const Launch& L, int xt, int pt, const void* x, const void* dy,
                           const void* w, const float* rstd, void* dx, float* ws, int64_t M,
                           int N, float eps)
{
    if (xt == kF32) return bwd_dispatch<float>(L, pt, x, dy, w, rstd, dx, ws, M, N, eps);
    return bwd_dispatch<__nv_bfloat16>(L, pt, x, dy, w, rstd, dx, ws, M, N, eps);
}

}  // namespace gbn
