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
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace gbn {
namespace {

// Sum of squares of one thread's vector of a row (absent vectors are zeros):
// pairwise fma into two lanes, then the lanes added.  The forward and the
// backward's recomputation share it, so with the same row-group width they
// reduce a row identically.
template <int P>
__device__ __forceinline__ float vec_sumsq2(const f2 (&v)[P])
{
    f2 s = splat2(0.f);
#pragma unroll
    for (int p = 0; p < P; ++p) s = fma2(v[p], v[p], s);
    return lo2(s) + hi2(s);
}

// ------------------------------------------------------------ fast forward
template <typename TX, int S>
__global__ void __launch_bounds__(kSched[S].T, kSched[S].MINBF)
    rms_fwd_fast(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ w,
                 int pt, float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n,
                 int64_t nblocks, unsigned* fault)
{
    constexpr int W = kSched[S].W, U = kSched[S].UF, T = kSched[S].T;
    constexpr int VEC = Vec<TX>::kN, P = Pairs<TX>::kP;
    constexpr int G = T / W;
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ float red[GroupRed<W, T, U>::kFloats];
    int parity = 0;
    const int g = threadIdx.x / W, l = threadIdx.x % W;
    const bool colok = l < N / VEC;
    const int64_t rb = (int64_t)N * sizeof(TX);

    f2 wf[P];
#pragma unroll
    for (int p = 0; p < P; ++p) wf[p] = colok ? ld_param2(w, pt, l * VEC + 2 * p) : splat2(0.f);

    Ring<1, kStagesF> rg;
    rg.src[0] = reinterpret_cast<const unsigned char*>(x);
    rg.row_bytes = rb;
    rg.R = G * U;
    rg.M = M;
    rg.nblocks = nblocks;
    rg.slot = slot_bytes(S, false);
    rg.fault = fault;
    ring_loop(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        const unsigned char* tx = rg.tile(k, 0);
        bool ok[U];
        f2 xv[U][P];
        float s[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int lr = u * G + g;
            ok[u] = alive && colok && b * (G * U) + lr < M;
            unpack2(lds128_if(ok[u], tx + lr * rb + l * 16), xv[u]);
            s[u] = vec_sumsq2<P>(xv[u]);
        }
        group_allreduce<W, T, U>(s, red, parity);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = b * (G * U) + u * G + g;
            const float rs = rsqrtf(fmaf(s[u], inv_n, eps));
            if (ok[u]) {
                const f2 r2 = splat2(rs);
                f2 o[P];
#pragma unroll
                for (int p = 0; p < P; ++p) o[p] = mul2(wf[p], round2<TX>(mul2(xv[u][p], r2)));
                st_stream(y + row * N + l * VEC, pack2(o));
            }
            if (rstd && alive && l == 0 && row < M) rstd[row] = rs;
        }
    });
}

// ----------------------------------------------------------- fast backward
// x and dy stream through the ring; a given rstd of the next row block is
// prefetched into registers, otherwise r is recomputed with the forward's
// code.  Full row blocks run without masking; the ragged last block masks its
// padded rows by a select after the arithmetic.
template <typename TX, int S>
__global__ void __launch_bounds__(kSched[S].T, kSched[S].MINBB)
    rms_bwd_fast(const TX* __restrict__ x, const TX* __restrict__ dy, const void* __restrict__ w,
                 int pt, const float* __restrict__ rstd, TX* __restrict__ dx,
                 float* __restrict__ ws, int64_t M, int N, float eps, float inv_n,
                 int64_t nblocks, unsigned* fault)
{
    constexpr int W = kSched[S].W, U = kSched[S].UB, T = kSched[S].T;
    constexpr int VEC = Vec<TX>::kN, P = Pairs<TX>::kP;
    constexpr int G = T / W;
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ float red[GroupRed<W, T, U>::kFloats];
    int parity = 0;
    const int g = threadIdx.x / W, l = threadIdx.x % W;
    const bool colok = l < N / VEC;
    const int64_t rb = (int64_t)N * sizeof(TX);
    const bool round_terms = (pt != kF32);  // weight in x's dtype: round dy*n

    f2 wf[P], acc[P];
#pragma unroll
    for (int p = 0; p < P; ++p) {
        wf[p] = colok ? ld_param2(w, pt, l * VEC + 2 * p) : splat2(0.f);
        acc[p] = splat2(0.f);
    }
    float rs_n[U];
    auto load_rstd = [&](int64_t b) {
        if (rstd) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t row = b * (G * U) + u * G + g;
                rs_n[u] = row < M ? __ldcs(rstd + row) : 0.f;
            }
        }
    };
    load_rstd(blockIdx.x);

    auto rows = [&](int64_t b, const unsigned char* tx, const unsigned char* td, bool alive,
                    auto masked) {
        constexpr bool kMask = decltype(masked)::value;
        float rs[U];
        bool ok[U];
        f2 xv[U][P], dv[U][P];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int lr = u * G + g;
            ok[u] = alive && colok && (!kMask || b * (G * U) + lr < M);
            unpack2(lds128_if(ok[u], tx + lr * rb + l * 16), xv[u]);
            unpack2(lds128_if(ok[u], td + lr * rb + l * 16), dv[u]);
            rs[u] = rs_n[u];
        }
        load_rstd(b + gridDim.x);
        if (!rstd) {  // uniform branch: recompute r exactly as the forward does
#pragma unroll
            for (int u = 0; u < U; ++u) rs[u] = vec_sumsq2<P>(xv[u]);
            group_allreduce<W, T, U>(rs, red, parity);
#pragma unroll
            for (int u = 0; u < U; ++u) rs[u] = rsqrtf(fmaf(rs[u], inv_n, eps));
        }
        float s[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const f2 r2 = splat2(rs[u]);
            f2 a2 = splat2(0.f);
#pragma unroll
            for (int p = 0; p < P; ++p)
                a2 = fma2(round2<TX>(mul2(dv[u][p], wf[p])), mul2(xv[u][p], r2), a2);
            s[u] = lo2(a2) + hi2(a2);
        }
        group_allreduce<W, T, U>(s, red, parity);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = b * (G * U) + u * G + g;
            const bool okr = !kMask || row < M;
            const f2 r2 = splat2(rs[u]), nm = splat2(-(s[u] * inv_n));
            f2 o[P];
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const f2 xh = mul2(xv[u][p], r2);
                const f2 dn = round2<TX>(mul2(dv[u][p], wf[p]));
                o[p] = mul2(r2, fma2(xh, nm, dn));
                f2 term = mul2(dv[u][p], round2<TX>(xh));
                if (round_terms) term = round2<TX>(term);
                if constexpr (kMask)
                    acc[p] = add2(acc[p], sel2(okr, term, splat2(0.f)));
                else
                    acc[p] = add2(acc[p], term);
            }
            if (ok[u]) st_stream(dx + row * N + l * VEC, pack2(o));
        }
    };

    Ring<2, kStagesB> rg;
    rg.src[0] = reinterpret_cast<const unsigned char*>(x);
    rg.src[1] = reinterpret_cast<const unsigned char*>(dy);
    rg.row_bytes = rb;
    rg.R = G * U;
    rg.M = M;
    rg.nblocks = nblocks;
    rg.slot = slot_bytes(S, true);
    rg.fault = fault;
    ring_loop(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        if ((b + 1) * (G * U) <= M)
            rows(b, rg.tile(k, 0), rg.tile(k, 1), alive, std::false_type{});
        else
            rows(b, rg.tile(k, 0), rg.tile(k, 1), alive, std::true_type{});
    });

    if (ws == nullptr) return;  // no weight gradient requested (uniform)
    float* wrow = ws + blockIdx.x * (int64_t)N;
    cta_store_columns2<W, P, T>(acc, reinterpret_cast<float*>(dsm + 128), wrow, N);  // drained ring slots
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
#define GBN_CASE(S)                                                                          \
    case S: {                                                                                \
        constexpr int smem = ring_smem_bytes(S, false, 1);                                  \
        auto kern = rms_fwd_fast<TX, S>;                                                     \
        if (smem > 48 * 1024)                                                                \
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);   \
        kern<<<L.grid, kSched[S].T, smem, L.stream>>>(xp, yp, w, pt, rstd, M, N, eps, inv_n, L.nblocks, L.fault);                              \
        break;                                                                               \
    }
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
#define GBN_CASE(S)                                                                          \
    case S: {                                                                                \
        constexpr int smem = ring_smem_bytes(S, true, 2);                                  \
        auto kern = rms_bwd_fast<TX, S>;                                                     \
        if (smem > 48 * 1024)                                                                \
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);   \
        kern<<<L.grid, kSched[S].T, smem, L.stream>>>(xp, dyp, w, pt, rstd, dxp, ws, M, N, eps, inv_n, L.nblocks, L.fault);                              \
        break;                                                                               \
    }
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
