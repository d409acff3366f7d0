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

// Words of one 16-byte vector (4 bf16 pairs, or 2 f32 pairs' worth).
__device__ __forceinline__ uint32_t word(const uint4& v, int p)
{
    return p == 0 ? v.x : p == 1 ? v.y : p == 2 ? v.z : v.w;
}

// With 16-bit activations and a weight of the same type, the products w*n
// (forward), dy*w and dy*n (backward) are products of two 16-bit values,
// exact in float32 and rounded once to the activation type by the rounding
// points above; mul.rn.bf16x2 / mul.rn.f16x2 compute exactly that on a
// packed pair.  Other dtype pairs take float32 pairs.

// ------------------------------------------------------------ fast forward
template <typename TX, int S, bool kWF>
__global__ void __launch_bounds__(kSched[S].T, kind_minb(S, kFwdNorm))
    rms_fwd_fast(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ w,
                 int pt, float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n,
                 int64_t nblocks, unsigned* fault, int gemma)
{
    constexpr int W = kSched[S].W, U = kind_U(S, kFwdNorm), T = kSched[S].T, KV = kSched[S].KV;
    constexpr int VEC = Vec<TX>::kN, P = Pairs<TX>::kP;
    constexpr int G = groups_per_cta(W, T);
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ float red[GroupRed<W, T, U>::kFloats];
    int parity = 0;
    const int g = grp<W>(), l = lan<W>();
    // vector j of a row is vector l + j*W: in shared memory at +j*W*16 bytes
    bool colok[KV];
#pragma unroll
    for (int j = 0; j < KV; ++j) colok[j] = in_group<W>() && l + j * W < N / VEC;
    const int rb = N * (int)sizeof(TX);
    const int soff = g * rb + l * 16, srow = G * rb, grow = G * N;
    // the Llama expression's packed 16-bit product (weight of x's dtype)
    const bool w16 = !kWF && is16<TX>() && pt == dtype_code<TX>();

    f2 wf[KV][P];
    uint32_t wpk[KV][P];  // the 16-bit weight pair, packed (used when w16)
#pragma unroll
    for (int j = 0; j < KV; ++j) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int c = (l + j * W) * VEC + 2 * p;
            wf[j][p] = colok[j] ? ld_param2(w, pt, c) : splat2(0.f);
            if (gemma) wf[j][p] = add2(splat2(1.f), wf[j][p]);  // 1 + w in float32
            wpk[j][p] = (w16 && colok[j]) ? static_cast<const uint32_t*>(w)[c / 2] : 0u;
        }
    }

    Ring<1, kind_stages(S, kFwdNorm)> rg;
    rg.src[0] = reinterpret_cast<const unsigned char*>(x);
    rg.row_bytes = rb;
    rg.R = G * U;
    rg.M = M;
    rg.nblocks = nblocks;
    rg.slot = slot_bytes(S, kFwdNorm);
    rg.fault = fault;
    const int64_t nfull = M / (G * U);  // blocks without padded rows
    const int64_t rstride = (int64_t)gridDim.x * (G * U);
    int64_t row0 = (int64_t)blockIdx.x * (G * U) + g;  // this thread's first row
    TX* yb = y + row0 * N + l * VEC;
    const bool lead = l == 0 && in_group<W>();  // stores rstd
    ring_loop(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        const unsigned char* xs = rg.tile(k, 0) + soff;
        const bool full = b < nfull;
        bool okr[U];
        f2 xv[U][KV][P];
        float s[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            okr[u] = alive && (full || row0 + u * G < M);
            s[u] = 0.f;
#pragma unroll
            for (int j = 0; j < KV; ++j) {
                unpack2<TX>(lds128_if(okr[u] && colok[j], xs + u * srow + j * W * 16), xv[u][j]);
                s[u] += vec_sumsq2<P>(xv[u][j]);
            }
        }
        group_allreduce<W, T, U>(s, red, parity);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float rs = rsqrtf(fmaf(s[u], inv_n, eps));
            const f2 r2 = splat2(rs);
#pragma unroll
            for (int j = 0; j < KV; ++j) {
                uint4 out;
                if constexpr (is16<TX>() && !kWF) {
                    uint32_t o[4];
#pragma unroll
                    for (int p = 0; p < P; ++p) {
                        // n = round_x(x r)
                        const uint32_t npk = P16<TX>::from_f2(mul2(xv[u][j][p], r2));
                        o[p] = w16 ? P16<TX>::mul(wpk[j][p], npk)
                                   : P16<TX>::from_f2(mul2(wf[j][p], P16<TX>::to_f2(npk)));
                    }
                    out = make_uint4(o[0], o[1], o[2], o[3]);
                } else {
                    f2 o[P];
#pragma unroll
                    for (int p = 0; p < P; ++p) o[p] = mul2(wf[j][p], mul2(xv[u][j][p], r2));
                    out = pack2<TX>(o);
                }
                st_stream_if(okr[u] && colok[j], yb + u * grow + j * W * VEC, out);
            }
            if (rstd) st_f32_if(lead && okr[u], rstd + (row0 + u * G), rs);
        }
        row0 += rstride;
        yb += rstride * N;
    });
}

// ----------------------------------------------------------- fast backward
// x and dy stream through the ring; a given rstd of the next row block is
// prefetched into registers, otherwise r is recomputed with the forward's
// code.  Full row blocks run without masking; the ragged last block masks its
// padded rows by a select after the arithmetic.
template <typename TX, int S, bool kWF>
__global__ void __launch_bounds__(kSched[S].T, kind_minb(S, kBwdRms))
    rms_bwd_fast(const TX* __restrict__ x, const TX* __restrict__ dy, const void* __restrict__ w,
                 int pt, const float* __restrict__ rstd, TX* __restrict__ dx,
                 float* __restrict__ ws, int64_t M, int N, float eps, float inv_n,
                 int64_t nblocks, unsigned* fault, int gemma)
{
    constexpr int W = kSched[S].W, U = kind_U(S, kBwdRms), T = kSched[S].T, KV = kSched[S].KV;
    constexpr int VEC = Vec<TX>::kN, P = Pairs<TX>::kP;
    constexpr int G = groups_per_cta(W, T);
    static_assert(KV <= 2, "the RMSNorm backward takes at most 2 vectors per thread");
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ float red[GroupRed<W, T, U>::kFloats];
    int parity = 0;
    const int g = grp<W>(), l = lan<W>();
    // vector j of a row is vector l + j*W: in shared memory at +j*W*16 bytes
    bool colok[KV];
#pragma unroll
    for (int j = 0; j < KV; ++j) colok[j] = in_group<W>() && l + j * W < N / VEC;
    const int rb = N * (int)sizeof(TX);
    const int soff = g * rb + l * 16, srow = G * rb, grow = G * N;
    // a weight in x's dtype: each dy*n is rounded to x's dtype (bf16 pairs
    // then multiply in bf16); a float32 weight keeps the float32 product
    const bool w16 = !kWF && is16<TX>() && pt == dtype_code<TX>();

    f2 wf[KV][P], acc[KV][P];
    uint32_t wpk[KV][P];
#pragma unroll
    for (int j = 0; j < KV; ++j) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int c = (l + j * W) * VEC + 2 * p;
            wf[j][p] = colok[j] ? ld_param2(w, pt, c) : splat2(0.f);
            if (gemma) wf[j][p] = add2(splat2(1.f), wf[j][p]);  // 1 + w in float32
            wpk[j][p] = (w16 && colok[j]) ? static_cast<const uint32_t*>(w)[c / 2] : 0u;
            acc[j][p] = splat2(0.f);
        }
    }
    float rs_n[U];
    auto load_rstd = [&](int64_t row0) {
        if (rstd) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t row = row0 + u * G;
                rs_n[u] = row < M ? __ldcs(rstd + row) : 0.f;
            }
        }
    };
    load_rstd((int64_t)blockIdx.x * (G * U) + g);

    // Pass 1 (after r is known) computes dn and xhat, the reduction term and
    // the weight-gradient term (independent of the row reduction); pass 2
    // keeps only xhat and dn.
    auto rows = [&](const unsigned char* xs, const unsigned char* ds, TX* dxb, int64_t row0,
                    bool alive, auto masked) {
        constexpr bool kMask = decltype(masked)::value;
        float rs[U];
        bool okr[U];
        f2 xh[U][KV][P], dn[U][KV][P];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            okr[u] = !kMask || row0 + u * G < M;
#pragma unroll
            for (int j = 0; j < KV; ++j)  // x, scaled by r below
                unpack2<TX>(lds128_if(alive && okr[u] && colok[j], xs + u * srow + j * W * 16),
                        xh[u][j]);
            rs[u] = rs_n[u];
        }
        load_rstd(row0 + (int64_t)gridDim.x * (G * U));
        if (!rstd) {  // uniform branch: recompute r exactly as the forward does
#pragma unroll
            for (int u = 0; u < U; ++u) {
                rs[u] = 0.f;
#pragma unroll
                for (int j = 0; j < KV; ++j) rs[u] += vec_sumsq2<P>(xh[u][j]);
            }
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
            for (int j = 0; j < KV; ++j) {
                const uint4 dr = lds128_if(alive && okr[u] && colok[j], ds + u * srow + j * W * 16);
                f2 dv[P];
                unpack2<TX>(dr, dv);
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    xh[u][j][p] = mul2(xh[u][j][p], r2);
                    f2 nxt;  // the accumulator with this row's dw term added
                    if constexpr (is16<TX>() && !kWF) {
                        const uint32_t npk = P16<TX>::from_f2(xh[u][j][p]);  // n = round_x(xhat)
                        if (w16) {
                            dn[u][j][p] = P16<TX>::to_f2(P16<TX>::mul(word(dr, p), wpk[j][p]));
                            nxt = add2(acc[j][p], P16<TX>::to_f2(P16<TX>::mul(word(dr, p), npk)));
                        } else {
                            // float32 weight: dy*n unrounded, exact product of two 16-bit values
                            dn[u][j][p] = round2<TX>(mul2(dv[p], wf[j][p]));
                            nxt = mk2(P16<TX>::fma_lo(word(dr, p), npk, lo2(acc[j][p])),
                                      P16<TX>::fma_hi(word(dr, p), npk, hi2(acc[j][p])));
                        }
                    } else {
                        dn[u][j][p] = mul2(dv[p], wf[j][p]);
                        nxt = fma2(dv[p], xh[u][j][p], acc[j][p]);
                    }
                    a2 = fma2(dn[u][j][p], xh[u][j][p], a2);
                    // padded rows: keep the old sum, a select after the arithmetic
                    acc[j][p] = (!kMask || okr[u]) ? nxt : acc[j][p];
                }
            }
            s[u] = lo2(a2) + hi2(a2);
        }
        group_allreduce<W, T, U>(s, red, parity);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const f2 r2 = splat2(rs[u]), nm = splat2(-(s[u] * inv_n));
#pragma unroll
            for (int j = 0; j < KV; ++j) {
                f2 o[P];
#pragma unroll
                for (int p = 0; p < P; ++p) o[p] = mul2(r2, fma2(xh[u][j][p], nm, dn[u][j][p]));
                st_stream_if(alive && okr[u] && colok[j], dxb + u * grow + j * W * VEC, pack2<TX>(o));
            }
        }
    };

    Ring<2, kind_stages(S, kBwdRms)> rg;
    rg.src[0] = reinterpret_cast<const unsigned char*>(x);
    rg.src[1] = reinterpret_cast<const unsigned char*>(dy);
    rg.row_bytes = rb;
    rg.R = G * U;
    rg.M = M;
    rg.nblocks = nblocks;
    rg.slot = slot_bytes(S, kBwdRms);
    rg.fault = fault;
    const int64_t nfull = M / (G * U);  // blocks without padded rows
    const int64_t rstride = (int64_t)gridDim.x * (G * U);
    int64_t row0 = (int64_t)blockIdx.x * (G * U) + g;  // this thread's first row
    TX* dxb = dx + row0 * N + l * VEC;
    ring_loop(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        const unsigned char* xs = rg.tile(k, 0) + soff;
        const unsigned char* ds = rg.tile(k, 1) + soff;
        if (b < nfull)
            rows(xs, ds, dxb, row0, alive, std::false_type{});
        else
            rows(xs, ds, dxb, row0, alive, std::true_type{});
        row0 += rstride;
        dxb += rstride * N;
    });

    if (ws == nullptr) return;  // no weight gradient requested (uniform)
    float* wrow = ws + blockIdx.x * (int64_t)N;
    cta_store_columns_kv<W, KV, P, T>(acc, reinterpret_cast<float*>(dsm + 128), wrow, N);  // drained ring slots
}

// ------------------------------------------------------ general (any shape)
// The weight of column c as the expression variant uses it: w, or Gemma's
// 1 + w formed in float32.
__device__ __forceinline__ float rms_weight(const void* w, int pt, int c, int variant)
{
    const float v = ld_param(w, pt, c);
    return variant == 2 ? 1.f + v : v;
}

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
                    int pt, float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n,
                    int variant)
{
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kGenWarps;
    for (int64_t r = blockIdx.x * (int64_t)kGenWarps + (threadIdx.x >> 5); r < M; r += nw) {
        const TX* xr = x + r * N;
        const float rs = warp_row_rstd(xr, N, lane, eps, inv_n);
        for (int c = lane; c < N; c += 32) {
            const float xh = ld1(xr, c) * rs;
            st1(y, r * N + c, rms_weight(w, pt, c, variant) * (variant == 0 ? round_x<TX>(xh) : xh));
        }
        if (rstd && lane == 0) rstd[r] = rs;
    }
}

template <typename TX>
__global__ void __launch_bounds__(kGenThreads)
    rms_bwd_general(const TX* __restrict__ x, const TX* __restrict__ dy,
                    const void* __restrict__ w, int pt, const float* __restrict__ rstd,
                    TX* __restrict__ dx, float* __restrict__ ws, int64_t M, int N, float eps,
                    float inv_n, int variant)
{
    const int lane = threadIdx.x & 31;
    const int64_t wi = blockIdx.x * (int64_t)kGenWarps + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * kGenWarps;
    const bool cast_first = variant == 0;  // the Llama expression's rounding points
    const bool round_terms = cast_first && pt != kF32;
    float* wrow = ws ? ws + wi * (int64_t)N : nullptr;
    if (wrow)
        for (int c = lane; c < N; c += 32) wrow[c] = 0.f;
    for (int64_t r = wi; r < M; r += nw) {
        const TX* xr = x + r * N;
        const TX* dr = dy + r * N;
        const float rs = rstd ? rstd[r] : warp_row_rstd(xr, N, lane, eps, inv_n);
        float s[1] = {0.f};
        for (int c = lane; c < N; c += 32) {
            float dn = ld1(dr, c) * rms_weight(w, pt, c, variant);
            if (cast_first) dn = round_x<TX>(dn);
            s[0] = fmaf(dn, ld1(xr, c) * rs, s[0]);
        }
        butterfly<32, 1>(s);
        const float m = s[0] * inv_n;
        for (int c = lane; c < N; c += 32) {
            const float dv = ld1(dr, c);
            const float xh = ld1(xr, c) * rs;
            float dn = dv * rms_weight(w, pt, c, variant);
            if (cast_first) dn = round_x<TX>(dn);
            st1(dx, r * N + c, rs * (dn - xh * m));
            float term = dv * (cast_first ? round_x<TX>(xh) : xh);
            if (round_terms) term = round_x<TX>(term);
            if (wrow) wrow[c] += term;
        }
    }
}

// Launch schedule S of a fast kernel: the weight-first instance (kWF) for
// the weight-first and Gemma expressions with 16-bit activations; with
// float32 activations both expressions are the same float32 arithmetic.
#define GBN_RMS_LAUNCH(KERNEL, S, SMEM, ...)                                                       \
    do {                                                                                           \
        if constexpr (is16<TX>()) {                                                                \
            if (variant != 0) {                                                                    \
                ring_attributes<KERNEL<TX, S, true>>(SMEM);                                        \
                KERNEL<TX, S, true><<<L.grid, kSched[S].T, SMEM, L.stream>>>(__VA_ARGS__);         \
                break;                                                                             \
            }                                                                                      \
        }                                                                                          \
        ring_attributes<KERNEL<TX, S, false>>(SMEM);                                               \
        KERNEL<TX, S, false><<<L.grid, kSched[S].T, SMEM, L.stream>>>(__VA_ARGS__);                \
    } while (0)

template <typename TX>
cudaError_t fwd_dispatch(const Launch& L, int pt, const void* x, const void* w, void* y,
                         float* rstd, int64_t M, int N, float eps, int variant)
{
    const TX* xp = static_cast<const TX*>(x);
    TX* yp = static_cast<TX*>(y);
    const float inv_n = (float)(1.0 / (double)N);
    const int gemma = variant == 2;
    if (!L.fast) {
        rms_fwd_general<TX><<<L.grid, kGenThreads, 0, L.stream>>>(xp, yp, w, pt, rstd, M, N, eps,
                                                                  inv_n, variant);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE(S)                                                                                \
    case S: {                                                                                      \
        constexpr int smem = ring_smem_bytes(S, kFwdNorm, 1);                                      \
        GBN_RMS_LAUNCH(rms_fwd_fast, S, smem, xp, yp, w, pt, rstd, M, N, eps, inv_n, L.nblocks,    \
                       L.fault, gemma);                                                            \
        break;                                                                                     \
    }
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9) GBN_CASE(11)
        GBN_CASE(12)
#undef GBN_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename TX>
cudaError_t bwd_dispatch(const Launch& L, int pt, const void* x, const void* dy, const void* w,
                         const float* rstd, void* dx, float* ws, int64_t M, int N, float eps,
                         int variant)
{
    const TX* xp = static_cast<const TX*>(x);
    const TX* dyp = static_cast<const TX*>(dy);
    TX* dxp = static_cast<TX*>(dx);
    const float inv_n = (float)(1.0 / (double)N);
    const int gemma = variant == 2;
    if (!L.fast) {
        rms_bwd_general<TX><<<L.grid, kGenThreads, 0, L.stream>>>(xp, dyp, w, pt, rstd, dxp, ws,
                                                                  M, N, eps, inv_n, variant);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE(S)                                                                                \
    case S: {                                                                                      \
        constexpr int smem = ring_smem_bytes(S, kBwdRms, 2);                                       \
        GBN_RMS_LAUNCH(rms_bwd_fast, S, smem, xp, dyp, w, pt, rstd, dxp, ws, M, N, eps, inv_n,     \
                       L.nblocks, L.fault, gemma);                                                 \
        break;                                                                                     \
    }
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9) GBN_CASE(11)
        GBN_CASE(12)
#undef GBN_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}
#undef GBN_RMS_LAUNCH

}  // namespace

cudaError_t launch_rms_fwd(const Launch& L, int xt, int pt, const void* x, const void* w, void* y,
                           float* rstd, int64_t M, int N, float eps, int variant)
{
    if (xt == kF32) return fwd_dispatch<float>(L, pt, x, w, y, rstd, M, N, eps, variant);
    if (xt == kF16) return fwd_dispatch<__half>(L, pt, x, w, y, rstd, M, N, eps, variant);
    return fwd_dispatch<__nv_bfloat16>(L, pt, x, w, y, rstd, M, N, eps, variant);
}

cudaError_t launch_rms_bwd(const Launch& L, int xt, int pt, const void* x, const void* dy,
                           const void* w, const float* rstd, void* dx, float* ws, int64_t M,
                           int N, float eps, int variant)
{
    if (xt == kF32) return bwd_dispatch<float>(L, pt, x, dy, w, rstd, dx, ws, M, N, eps, variant);
    if (xt == kF16) return bwd_dispatch<__half>(L, pt, x, dy, w, rstd, dx, ws, M, N, eps, variant);
    return bwd_dispatch<__nv_bfloat16>(L, pt, x, dy, w, rstd, dx, ws, M, N, eps, variant);
}

}  // namespace gbn
