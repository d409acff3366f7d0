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
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace gbn {
namespace {

// The row mean s / N from the row sum by Markstein's correction step
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q = fl(s y) with
// y = fl(1/N), the residual r = s - q N in one fma, then fl(q + r y) in
// another.  Markstein's theorem: when y is 1/N rounded to nearest and q is
// within an ulp of s/N, r is exact and fl(q + r y) is s/N correctly rounded
// (barring underflow), where q alone may miss it by an ulp.  A constant row
// of value c has the exact sum s = N c; q is c or a neighbour of c, so
// r = N (c - q) is exact and q + r y = c + (c - q)(N y - 1), with
// |N y - 1| <= 2^-24, rounds to c: x - mean = 0 exactly and y = beta
// (rstd is 1/sqrt(eps) there, so any error in the mean would reach y
// magnified).
__device__ __forceinline__ float row_mean(float s, float n, float inv_n)
{
    const float mu = s * inv_n;
    return fmaf(fmaf(-mu, n, s), inv_n, mu);
}

// ------------------------------------------------------------ fast forward
// x streams through the ring; two row all-reduces (sum, then the centred sum
// of squares) per row.  Every thread runs every row (row reductions are
// collective); loads and stores are predicated, and only the ragged last
// block compares rows against M.
template <typename TX, int S, int kIn>
__global__ void __launch_bounds__(kSched[S].T, kind_minb(S, kFwdLN))
    ln_fwd_fast(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ gamma,
                const void* __restrict__ beta, int pt, float* __restrict__ mean,
                float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n,
                int64_t nblocks, unsigned* fault, RowMaps maps)
{
    grid_dependency_sync();
    constexpr int W = kSched[S].W, U = kind_U(S, kFwdLN), T = kSched[S].T, KV = kSched[S].KV;
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
    const float fN = (float)N;

    f2 gm[KV][P], bt[KV][P];
#pragma unroll
    for (int j = 0; j < KV; ++j) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int c = (l + j * W) * VEC + 2 * p;
            gm[j][p] = (colok[j] && gamma) ? ld_param2(gamma, pt, c) : splat2(1.f);
            bt[j][p] = (colok[j] && beta) ? ld_param2(beta, pt, c) : splat2(0.f);
        }
    }

    Ring<1, kind_stages(S, kFwdLN), kIn == kInRows> rg;
    rg.src[0] = reinterpret_cast<const unsigned char*>(x);
    if constexpr (kIn == kInRows) rg.map[0] = maps.m[0];
    rg.row_bytes = rb;
    rg.R = G * U;
    rg.M = M;
    rg.nblocks = nblocks;
    rg.slot = slot_bytes(S, kFwdLN);
    rg.fault = fault;
    // Row positions advance by a fixed stride from one of this CTA's blocks
    // to the next; blocks below nfull hold no padded rows.
    const int64_t nfull = M / (G * U);
    const int64_t rstride = (int64_t)gridDim.x * (G * U);
    int64_t row0 = (int64_t)blockIdx.x * (G * U) + g;  // this thread's first row
    TX* yb = y + row0 * N + l * VEC;
    const bool lead = l == 0 && in_group<W>();  // stores the row statistics
    // Full blocks of rows that fill every lane's vectors run without row,
    // column or fault predicates (a failed copy leaves stale bytes in the
    // slot, never an address outside it; the fault word reports it): up to
    // 1.5% faster (N = 128, 2048).
    const bool exact = !seg_groups(W) && N / VEC == W * KV;
    // rows wider than a warp: the row reduction's barrier releases the slot
    ring_loop<(W > 32)>(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        const unsigned char* xs = rg.tile(k, 0) + soff;
        const bool full = b < nfull;
        auto run = [&](auto clean_) {
            constexpr bool kClean = decltype(clean_)::value;
            bool okr[U];
            f2 xv[U][KV][P];
            float s[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                okr[u] = kClean || (alive && (full || row0 + u * G < M));
                s[u] = 0.f;
#pragma unroll
                for (int j = 0; j < KV; ++j) {
                    const bool ok = okr[u] && (kClean || colok[j]);
                    unpack2<TX>(lds128_if(ok, xs + u * srow + j * W * 16), xv[u][j]);
                    f2 a2 = xv[u][j][0];
#pragma unroll
                    for (int p = 1; p < P; ++p) a2 = add2(a2, xv[u][j][p]);
                    s[u] += lo2(a2) + hi2(a2);
                }
            }
            group_allreduce<W, T, U>(s, red, parity);
            float mu[U], q[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                mu[u] = row_mean(s[u], fN, inv_n);
                const f2 m2 = splat2(mu[u]);
                q[u] = 0.f;
#pragma unroll
                for (int j = 0; j < KV; ++j) {
                    f2 q2 = splat2(0.f);
#pragma unroll
                    for (int p = 0; p < P; ++p) {
                        xv[u][j][p] = sub2(xv[u][j][p], m2);  // x - mu, kept for the output
                        q2 = fma2(xv[u][j][p], xv[u][j][p], q2);
                    }
                    // vectors past the row's end add nothing
                    q[u] += (kClean || colok[j]) ? lo2(q2) + hi2(q2) : 0.f;
                }
            }
            group_allreduce<W, T, U>(q, red, parity);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float rs = rsqrtf(fmaf(q[u], inv_n, eps));
                const f2 r2 = splat2(rs);
                const int64_t orow = stat_row<kIn>(maps, row0 + u * G);
                TX* const yr = kIn == kInStorage ? y + orow * N + l * VEC : yb + u * grow;
#pragma unroll
                for (int j = 0; j < KV; ++j) {
                    f2 o[P];
#pragma unroll
                    for (int p = 0; p < P; ++p)
                        o[p] = fma2(mul2(xv[u][j][p], r2), gm[j][p], bt[j][p]);
                    st_stream_if(okr[u] && (kClean || colok[j]), yr + j * W * VEC, pack2<TX>(o));
                }
                if (mean) st_f32_if(lead && okr[u], mean + orow, mu[u]);
                if (rstd) st_f32_if(lead && okr[u], rstd + orow, rs);
            }
        };
        if (full && exact)
            run(std::true_type{});
        else
            run(std::false_type{});
        row0 += rstride;
        yb += rstride * N;
    });
}

// ----------------------------------------------------------- fast backward
// x and dy stream through the ring; the saved mean and rstd of the next row
// block are prefetched into registers while the current one is processed.
// Full row blocks run without masking; the ragged last block masks its
// padded rows by a select after the arithmetic.
template <typename TX, int S, int kIn>
__global__ void __launch_bounds__(kSched[S].T, kind_minb(S, kBwdLN))
    ln_bwd_fast(const TX* __restrict__ x, const TX* __restrict__ dy,
                const float* __restrict__ mean, const float* __restrict__ rstd,
                const void* __restrict__ gamma, int pt, TX* __restrict__ dx,
                float* __restrict__ ws, int64_t M, int N, float inv_n, int64_t nblocks,
                unsigned* fault, RowMaps maps)
{
    grid_dependency_sync();
    constexpr int W = kSched[S].W, U = kind_U(S, kBwdLN), T = kSched[S].T, KV = kSched[S].KV;
    constexpr int VEC = Vec<TX>::kN, P = Pairs<TX>::kP;
    constexpr int G = groups_per_cta(W, T);
    // xhat and g of every vector stay in registers across the row reduction;
    // with the column accumulators that caps the 16-bit kernel at 2 vectors
    // per thread (4 spill); float32 vectors hold half the elements, and 4 fit.
    // The lean form (16-bit rows of 1025-2048 vectors) holds only the column
    // accumulators: it reads the row from the ring slot again after the
    // reduction, and gamma from shared memory at each use.
    constexpr bool kLean = lean_bwd<TX>(S);
    static_assert(KV <= 2 || sizeof(TX) == 4 || kLean,
                  "the 16-bit LayerNorm backward takes at most 2 vectors per thread");
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ float red[GroupRed<W, T, 2 * U>::kFloats];
    int parity = 0;
    const int g = grp<W>(), l = lan<W>();
    // vector j of a row is vector l + j*W: in shared memory at +j*W*16 bytes
    bool colok[KV];
#pragma unroll
    for (int j = 0; j < KV; ++j) colok[j] = in_group<W>() && l + j * W < N / VEC;
    const int rb = N * (int)sizeof(TX);
    const int soff = g * rb + l * 16, srow = G * rb, grow = G * N;

    f2 gm[KV][P], acc_g[KV][P], acc_b[KV][P];
#pragma unroll
    for (int j = 0; j < KV; ++j) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
            if constexpr (!kLean)
                gm[j][p] = (colok[j] && gamma) ? ld_param2(gamma, pt, (l + j * W) * VEC + 2 * p)
                                               : splat2(1.f);
            acc_g[j][p] = acc_b[j][p] = splat2(0.f);
        }
    }
    // the lean form's gamma, as float32 past the ring
    const float* prm = reinterpret_cast<const float*>(dsm + bwd_ring_bytes<TX>(S, kBwdLN));
    if constexpr (kLean)
        if (gamma) stage_params<T>(const_cast<float*>(prm), gamma, pt, N);
    // gamma of pair p of vector j
    auto gam = [&](int j, int p) -> f2 {
        if constexpr (kLean)
            return (colok[j] && gamma) ? prm2(prm, (l + j * W) * VEC + 2 * p) : splat2(1.f);
        else
            return gm[j][p];
    };

    // saved statistics of this thread's rows, loaded one row block ahead of
    // use (*_n), or two (*_nn too) with one vector per thread: measured
    // faster for those rows, slower for the multi-vector ones
    constexpr bool kDeep = KV == 1;
    // and, where one CTA per SM (or two rows per block, or 160 rows of 8
    // bytes of statistics each) leaves too little work between the load and
    // its use to hide a DRAM miss, prefetched into L2 four blocks ahead: N =
    // 8192 0.866 -> 0.958 of measured copy, 2048 0.913 -> 0.925, 24 0.921 ->
    // 0.941; at N = 16, 128 and 4096 (two or more CTAs per SM hide it) the
    // prefetches cost 2-4%, and in the lean form (16-bit N = 16384) 0.50 ->
    // 0.36
    constexpr bool kPrefetch = kIn == kInContig && !kLean &&
                               (S == 14 || S == 17 || S == 19 || seg_groups(W));
    float mu_n[U], rs_n[U], mu_nn[U], rs_nn[U];
    auto load_stats = [&](int64_t row0, float (&mu_d)[U], float (&rs_d)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = row0 + u * G;
            const int64_t srow = row < M ? stat_row<kIn>(maps, row) : 0;
            mu_d[u] = row < M ? ld_stat<kIn>(mean, srow) : 0.f;
            rs_d[u] = row < M ? ld_stat<kIn>(rstd, srow) : 0.f;
        }
    };
    const int64_t bstride = (int64_t)gridDim.x * (G * U);
    load_stats((int64_t)blockIdx.x * (G * U) + g, mu_n, rs_n);
    if constexpr (kDeep) load_stats((int64_t)blockIdx.x * (G * U) + g + bstride, mu_nn, rs_nn);

    // Pass 1 (before the row reduction) also accumulates the parameter
    // gradients, which do not depend on it; pass 2 needs only xhat and g.
    auto rows = [&](const unsigned char* xs, const unsigned char* ds, TX* dxb, int64_t row0,
                    bool alive, auto masked, auto exact) {
        constexpr bool kMask = decltype(masked)::value;
        constexpr bool kExact = decltype(exact)::value;
        float rs[U], mu[U];
        f2 xh[U][KV][P], gg[U][KV][P];
        bool okr[U];
        float s[2 * U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            okr[u] = !kMask || row0 + u * G < M;
            rs[u] = rs_n[u];
            const f2 m2 = splat2(mu_n[u]), r2 = splat2(rs[u]);
            // (sum g, sum g*xhat); vectors past the row's end hold dy = 0
            f2 s1 = splat2(0.f), s2 = splat2(0.f);
#pragma unroll
            for (int j = 0; j < KV; ++j) {
                const bool ok = kExact ? okr[u] : alive && colok[j] && okr[u];
                f2 xv[P], dv[P];
                unpack2<TX>(lds128_if(ok, xs + u * srow + j * W * 16), xv);
                unpack2<TX>(lds128_if(ok, ds + u * srow + j * W * 16), dv);
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const f2 xhv = mul2(sub2(xv[p], m2), r2);
                    const f2 ggv = mul2(dv[p], gam(j, p));
                    s1 = add2(s1, ggv);
                    s2 = fma2(ggv, xhv, s2);
                    if constexpr (kMask) {
                        // padded rows: select after the arithmetic, never a 0/1 multiply
                        const f2 z = splat2(0.f);
                        acc_g[j][p] = add2(acc_g[j][p], sel2(okr[u], mul2(dv[p], xhv), z));
                        acc_b[j][p] = add2(acc_b[j][p], sel2(okr[u], dv[p], z));
                    } else {
                        acc_g[j][p] = fma2(dv[p], xhv, acc_g[j][p]);
                        acc_b[j][p] = add2(acc_b[j][p], dv[p]);
                    }
                    if constexpr (!kLean) {
                        xh[u][j][p] = xhv;
                        gg[u][j][p] = ggv;
                    }
                }
            }
            s[2 * u] = lo2(s1) + hi2(s1);
            s[2 * u + 1] = lo2(s2) + hi2(s2);
            mu[u] = mu_n[u];
        }
        if constexpr (kDeep) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                mu_n[u] = mu_nn[u];
                rs_n[u] = rs_nn[u];
            }
            load_stats(row0 + 2 * bstride, mu_nn, rs_nn);  // two blocks of this CTA ahead
        } else {
            load_stats(row0 + bstride, mu_n, rs_n);  // the next block of this CTA
        }
        if constexpr (kPrefetch) {
            prefetch_stats(mean, row0 - g + 4 * bstride, G * U, M);
            prefetch_stats(rstd, row0 - g + 4 * bstride, G * U, M);
        }
        group_allreduce<W, T, 2 * U>(s, red, parity);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const f2 ma = splat2(s[2 * u] * inv_n), nmb = splat2(-(s[2 * u + 1] * inv_n));
            const f2 r2 = splat2(rs[u]);
            TX* const dxr = out_at<kIn>(dxb, u * grow, dx, maps, row0 + u * G, N, l * VEC);
#pragma unroll
            for (int j = 0; j < KV; ++j) {
                const bool ok = kExact ? okr[u] : alive && colok[j] && okr[u];
                if constexpr (kLean) {  // the row again from the slot
                    const f2 m2 = splat2(mu[u]);
                    f2 xv[P], dv[P];
                    unpack2<TX>(lds128_if(ok, xs + u * srow + j * W * 16), xv);
                    unpack2<TX>(lds128_if(ok, ds + u * srow + j * W * 16), dv);
#pragma unroll
                    for (int p = 0; p < P; ++p) {
                        xh[u][j][p] = mul2(sub2(xv[p], m2), r2);
                        gg[u][j][p] = mul2(dv[p], gam(j, p));
                    }
                }
                // rstd * (g - mean(g) - xhat * mean(g xhat)); g - mean(g) first,
                // so a width-one row gives exactly zero
                f2 o[P];
#pragma unroll
                for (int p = 0; p < P; ++p)
                    o[p] = mul2(r2, fma2(xh[u][j][p], nmb, sub2(gg[u][j][p], ma)));
                st_stream_if(ok, dxr + j * W * VEC, pack2<TX>(o));
            }
        }
    };

    Ring<2, bwd_stages<TX>(S, kBwdLN), kIn == kInRows> rg;
    rg.src[0] = reinterpret_cast<const unsigned char*>(x);
    rg.src[1] = reinterpret_cast<const unsigned char*>(dy);
    if constexpr (kIn == kInRows) {
        rg.map[0] = maps.m[0];
        rg.map[1] = maps.m[1];
    }
    rg.row_bytes = rb;
    rg.R = G * U;
    rg.M = M;
    rg.nblocks = nblocks;
    rg.slot = slot_bytes(S, kBwdLN);
    rg.fault = fault;
    const int64_t nfull = M / (G * U);  // blocks without padded rows
    const int64_t rstride = (int64_t)gridDim.x * (G * U);
    int64_t row0 = (int64_t)blockIdx.x * (G * U) + g;  // this thread's first row
    TX* dxb = dx + row0 * N + l * VEC;
    // Rows that fill every lane's vectors (the row group's exact capacity)
    // run their full blocks without per-vector column predicates, and load
    // the slot without the fault predicate (a failed copy leaves stale bytes
    // in the slot, never an address outside it; the fault word reports it):
    // 0.5-1.2% faster at N = 256-8192.  The lean form keeps the predicates
    // (without them it spills more).
    const bool exact = !seg_groups(W) && N / VEC == W * KV;
    using ExactT = std::integral_constant<bool, !kLean>;
    // rows wider than a warp: the row reduction's barrier releases the slot,
    // unless the row is read again after it (the lean form)
    ring_loop<(W > 32) && !kLean>(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        const unsigned char* xs = rg.tile(k, 0) + soff;
        const unsigned char* ds = rg.tile(k, 1) + soff;
        if (b < nfull) {
            if (exact && !kLean)
                rows(xs, ds, dxb, row0, alive, std::false_type{}, ExactT{});
            else
                rows(xs, ds, dxb, row0, alive, std::false_type{}, std::false_type{});
        } else {
            rows(xs, ds, dxb, row0, alive, std::true_type{}, std::false_type{});
        }
        row0 += rstride;
        dxb += rstride * N;
    });

    if (ws == nullptr) return;  // no parameter gradient requested (uniform)
    float* wrow = ws + blockIdx.x * (2 * (int64_t)N);
    float* colbuf = reinterpret_cast<float*>(dsm + 128);  // drained ring slots, past the barriers
    cta_store_columns_kv<W, KV, P, T>(acc_g, colbuf, wrow, N);
    cta_store_columns_kv<W, KV, P, T>(acc_b, colbuf, wrow + N, N);
}

// ------------------------------------------------------ general (any shape)
// One warp per row, scalar loads, row re-read from cache per pass.
template <typename TX>
__global__ void __launch_bounds__(kGenThreads)
    ln_fwd_general(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ gamma,
                   const void* __restrict__ beta, int pt, float* __restrict__ mean,
                   float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n, RowMaps maps,
                   int scattered)
{
    grid_dependency_sync();
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kGenWarps;
    for (int64_t r = blockIdx.x * (int64_t)kGenWarps + (threadIdx.x >> 5); r < M; r += nw) {
        const TX* xr = in_row(x, maps, 0, scattered, r, N);
        float v[1] = {0.f};
        for (int c = lane; c < N; c += 32) v[0] += ld1c(xr, c);
        butterfly<32, 1>(v);
        const float mu = row_mean(v[0], (float)N, inv_n);
        float q[1] = {0.f};
        for (int c = lane; c < N; c += 32) {
            const float d = ld1c(xr, c) - mu;
            q[0] += d * d;
        }
        butterfly<32, 1>(q);
        const float rs = rsqrtf(fmaf(q[0], inv_n, eps));
        for (int c = lane; c < N; c += 32) {
            const float gm = gamma ? ld_param(gamma, pt, c) : 1.f;
            const float bt = beta ? ld_param(beta, pt, c) : 0.f;
            st1(y, r * N + c, fmaf((ld1c(xr, c) - mu) * rs, gm, bt));
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
                   float* __restrict__ ws, int64_t M, int N, float inv_n, RowMaps maps,
                   int scattered)
{
    grid_dependency_sync();
    __shared__ float accs[kGenWarps * kGenCols];
    const int lane = threadIdx.x & 31;
    const int64_t w = blockIdx.x * (int64_t)kGenWarps + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * kGenWarps;
    float* wrow = ws ? ws + w * (2 * (int64_t)N) : nullptr;
    // the warp's column sums: in shared memory when they fit, else in its
    // workspace row; lane c % 32 alone touches column c, rows in order
    const bool local = 2 * N <= kGenCols;
    float* arow = local ? accs + (threadIdx.x >> 5) * kGenCols : wrow;
    if (wrow)
        for (int c = lane; c < 2 * N; c += 32) arow[c] = 0.f;
    for (int64_t r = w; r < M; r += nw) {
        const TX* xr = in_row(x, maps, 0, scattered, r, N);
        const TX* dr = in_row(dy, maps, 1, scattered, r, N);
        const float mu = mean[r], rs = rstd[r];
        float s[2] = {0.f, 0.f};
        for (int c = lane; c < N; c += 32) {
            const float xh = (ld1c(xr, c) - mu) * rs;
            const float gg = __fmul_rn(ld1c(dr, c), gamma ? ld_param(gamma, pt, c) : 1.f);
            s[0] += gg;
            s[1] += gg * xh;
        }
        butterfly<32, 2>(s);
        const float ma = s[0] * inv_n, mb = s[1] * inv_n;
        for (int c = lane; c < N; c += 32) {
            const float xh = (ld1c(xr, c) - mu) * rs;
            const float dv = ld1c(dr, c);
            const float gg = __fmul_rn(dv, gamma ? ld_param(gamma, pt, c) : 1.f);
            st1(dx, r * N + c, rs * (gg - ma - xh * mb));
            if (wrow) {
                arow[c] += dv * xh;
                arow[N + c] += dv;
            }
        }
    }
    if (wrow && local)
        for (int c = lane; c < 2 * N; c += 32) wrow[c] = arow[c];
}

// ------------------------------------------------------ row-batched path
// Rows whose byte length is not a multiple of 16 (common.cuh, "row-batched"):
// blocks of R rows through the ring, one warp per row.  Units past the row's
// end read as zeros and are left out of every sum where a zero would count.
template <typename TX, int E, int KMAX>
__global__ void __launch_bounds__(kBatchThreads, batch_minb(false))
    ln_fwd_batch(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ gamma,
                 const void* __restrict__ beta, int pt, float* __restrict__ mean,
                 float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n,
                 int64_t nblocks, int R, unsigned* fault)
{
    grid_dependency_sync();
    using U = Unit<TX, E>;
    extern __shared__ __align__(128) unsigned char dsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nu = N / E;
    const int rb = N * (int)sizeof(TX);
    bool uok[KMAX];
    float gm[KMAX][E], bt[KMAX][E];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        uok[k] = lane + 32 * k < nu;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int c = (lane + 32 * k) * E + e;
            gm[k][e] = (uok[k] && gamma) ? ld_param(gamma, pt, c) : 1.f;
            bt[k][e] = (uok[k] && beta) ? ld_param(beta, pt, c) : 0.f;
        }
    }
    const float fN = (float)N;
    // elements from `tail` on were not bulk-copied (the last block's end)
    const int64_t tail = ((M * (int64_t)rb) & ~(int64_t)15) / (int64_t)sizeof(TX);
    Ring<1, batch_stages(1)> rg;
    rg.src[0] = reinterpret_cast<const unsigned char*>(x);
    rg.row_bytes = rb;
    rg.R = R;
    rg.M = M;
    rg.nblocks = nblocks;
    rg.slot = batch_slot(1);
    rg.fault = fault;
    constexpr int RB = batch_rb(KMAX, E);
    constexpr int UB = E * (int)sizeof(TX);  // bytes of a unit
    ring_loop(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        if (!alive) return;
        const uint32_t xs = smem_u32(rg.tile(k, 0)) + lane * UB;
        const int64_t r0 = b * R;
        const int rows = (int)(M - r0 < R ? M - r0 : R);
        // RB consecutive rows a warp at once.  A whole block (every row group
        // full, every unit in the slot) runs unmasked; otherwise rows past the
        // block read zeros and units past the copied bytes come from global
        // memory.
        auto pass = [&](auto masked) {
            constexpr bool kMask = decltype(masked)::value;
            for (int i0 = warp * RB; i0 < rows; i0 += kBatchWarps * RB) {
                float v[RB][KMAX][E], s[RB], q[RB];
#pragma unroll
                for (int rr = 0; rr < RB; ++rr) {
                    const int i = i0 + rr;
                    s[rr] = 0.f;
#pragma unroll
                    for (int kk = 0; kk < KMAX; ++kk) {
                        typename U::W w{};
                        if constexpr (kMask) {
                            const int64_t gi = (r0 + i) * N + (lane + 32 * kk) * E;
                            if (i < rows && uok[kk])
                                w = gi < tail ? U::lds(xs + i * rb + kk * 32 * UB) : U::ld(x + gi);
                        } else {
                            if (uok[kk]) w = U::lds(xs + i * rb + kk * 32 * UB);
                        }
                        U::unpack(w, v[rr][kk]);
#pragma unroll
                        for (int e = 0; e < E; ++e) s[rr] += v[rr][kk][e];
                    }
                }
                butterfly<32, RB>(s);
#pragma unroll
                for (int rr = 0; rr < RB; ++rr) {
                    s[rr] = row_mean(s[rr], fN, inv_n);  // the mean
                    q[rr] = 0.f;
#pragma unroll
                    for (int kk = 0; kk < KMAX; ++kk)
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            v[rr][kk][e] -= s[rr];
                            q[rr] = uok[kk] ? fmaf(v[rr][kk][e], v[rr][kk][e], q[rr]) : q[rr];
                        }
                }
                butterfly<32, RB>(q);
#pragma unroll
                for (int rr = 0; rr < RB; ++rr) {
                    const int i = i0 + rr;
                    if (kMask && i >= rows) break;  // the same for the whole warp
                    const int64_t r = r0 + i;
                    const float rs = rsqrtf(fmaf(q[rr], inv_n, eps));
                    TX* const yr = y + r * N + lane * E;
#pragma unroll
                    for (int kk = 0; kk < KMAX; ++kk) {
                        float o[E];
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            o[e] = fmaf(v[rr][kk][e] * rs, gm[kk][e], bt[kk][e]);
                        if (uok[kk]) U::st(yr + kk * 32 * E, U::pack(o));
                    }
                    if (lane == 0) {
                        if (mean) mean[r] = s[rr];
                        if (rstd) rstd[r] = rs;
                    }
                }
            }
        };
        // R is a multiple of 8 and RB divides 8: a full block has no partial row group
        if (rows == R && (r0 + R) * N <= tail)
            pass(std::false_type{});
        else
            pass(std::true_type{});
    });
}

template <typename TX, int E, int KMAX>
__global__ void __launch_bounds__(kBatchThreads, batch_minb(true))
    ln_bwd_batch(const TX* __restrict__ x, const TX* __restrict__ dy,
                 const float* __restrict__ mean, const float* __restrict__ rstd,
                 const void* __restrict__ gamma, int pt, TX* __restrict__ dx,
                 float* __restrict__ ws, int64_t M, int N, float inv_n, int64_t nblocks, int R,
                 unsigned* fault)
{
    grid_dependency_sync();
    using U = Unit<TX, E>;
    extern __shared__ __align__(128) unsigned char dsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nu = N / E;
    const int rb = N * (int)sizeof(TX);
    bool uok[KMAX];
    float gm[KMAX][E], acc_g[KMAX][E], acc_b[KMAX][E];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        uok[k] = lane + 32 * k < nu;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            gm[k][e] = (uok[k] && gamma) ? ld_param(gamma, pt, (lane + 32 * k) * E + e) : 1.f;
            acc_g[k][e] = acc_b[k][e] = 0.f;
        }
    }
    const int64_t tail = ((M * (int64_t)rb) & ~(int64_t)15) / (int64_t)sizeof(TX);
    Ring<2, batch_stages(2)> rg;
    rg.src[0] = reinterpret_cast<const unsigned char*>(x);
    rg.src[1] = reinterpret_cast<const unsigned char*>(dy);
    rg.row_bytes = rb;
    rg.R = R;
    rg.M = M;
    rg.nblocks = nblocks;
    rg.slot = batch_slot(2);
    rg.fault = fault;
    constexpr int RB = batch_rb(KMAX, E);
    constexpr int UB = E * (int)sizeof(TX);  // bytes of a unit
    ring_loop(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        if (!alive) return;
        const uint32_t xs = smem_u32(rg.tile(k, 0)) + lane * UB;
        const uint32_t ds = smem_u32(rg.tile(k, 1)) + lane * UB;
        const int64_t r0 = b * R;
        const int rows = (int)(M - r0 < R ? M - r0 : R);
        // RB consecutive rows a warp at once.  A whole block runs unmasked;
        // otherwise rows past the block read zeros (and then add exact zeros
        // to the column sums) and units past the copied bytes come from global
        // memory.
        auto pass = [&](auto masked) {
            constexpr bool kMask = decltype(masked)::value;
            for (int i0 = warp * RB; i0 < rows; i0 += kBatchWarps * RB) {
                float xh[RB][KMAX][E], g[RB][KMAX][E], s[2 * RB], rs[RB];
#pragma unroll
                for (int rr = 0; rr < RB; ++rr) {
                    const int i = i0 + rr;
                    const int64_t r = r0 + i;
                    const bool ok = !kMask || i < rows;
                    const float mu = ok ? __ldca(mean + r) : 0.f;
                    rs[rr] = ok ? __ldca(rstd + r) : 0.f;
                    s[2 * rr] = s[2 * rr + 1] = 0.f;
#pragma unroll
                    for (int kk = 0; kk < KMAX; ++kk) {
                        const uint32_t so = i * rb + kk * 32 * UB;
                        typename U::W wx{}, wd{};
                        if constexpr (kMask) {
                            const int64_t gi = r * N + (lane + 32 * kk) * E;
                            if (ok && uok[kk]) {
                                const bool sm = gi < tail;
                                wx = sm ? U::lds(xs + so) : U::ld(x + gi);
                                wd = sm ? U::lds(ds + so) : U::ld(dy + gi);
                            }
                        } else if (uok[kk]) {
                            wx = U::lds(xs + so);
                            wd = U::lds(ds + so);
                        }
                        float xv[E], dv[E];
                        U::unpack(wx, xv);
                        U::unpack(wd, dv);
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            xh[rr][kk][e] = (xv[e] - mu) * rs[rr];
                            g[rr][kk][e] = dv[e] * gm[kk][e];
                            s[2 * rr] += g[rr][kk][e];
                            s[2 * rr + 1] = fmaf(g[rr][kk][e], xh[rr][kk][e], s[2 * rr + 1]);
                            acc_g[kk][e] = fmaf(dv[e], xh[rr][kk][e], acc_g[kk][e]);
                            acc_b[kk][e] += dv[e];
                        }
                    }
                }
                butterfly<32, 2 * RB>(s);
#pragma unroll
                for (int rr = 0; rr < RB; ++rr) {
                    const int i = i0 + rr;
                    if (kMask && i >= rows) break;  // the same for the whole warp
                    const float ma = s[2 * rr] * inv_n, mb = s[2 * rr + 1] * inv_n;
                    TX* const dxr = dx + (r0 + i) * N + lane * E;
#pragma unroll
                    for (int kk = 0; kk < KMAX; ++kk) {
                        float o[E];
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            o[e] = rs[rr] * fmaf(-xh[rr][kk][e], mb, g[rr][kk][e] - ma);
                        if (uok[kk]) U::st(dxr + kk * 32 * E, U::pack(o));
                    }
                }
            }
        };
        // R is a multiple of 8 and RB divides 8: a full block has no partial row group
        if (rows == R && (r0 + R) * N <= tail)
            pass(std::false_type{});
        else
            pass(std::true_type{});
    });
    if (ws == nullptr) return;  // no parameter gradient requested (uniform)
    // the warps' column sums, added in warp order into the CTA's partial row
    // (the drained ring slots hold them: 8 x 2N floats, at most 32 KB)
    float* cols = reinterpret_cast<float*>(dsm + 128);
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int c = (lane + 32 * k) * E + e;
            if (uok[k]) {
                cols[warp * 2 * N + c] = acc_g[k][e];
                cols[warp * 2 * N + N + c] = acc_b[k][e];
            }
        }
    __syncthreads();
    float* wrow = ws + blockIdx.x * (2 * (int64_t)N);
    for (int c = threadIdx.x; c < 2 * N; c += kBatchThreads) {
        float t = cols[c];
#pragma unroll
        for (int w = 1; w < kBatchWarps; ++w) t += cols[w * 2 * N + c];
        wrow[c] = t;
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
    if (L.batch) {
        constexpr int smem = batch_smem(1);
        if (!with_batch(L.E, L.KMAX, [&](auto e_, auto k_) {
                constexpr int E_ = decltype(e_)::value, K_ = decltype(k_)::value;
                ring_attributes<ln_fwd_batch<TX, E_, K_>>(smem);
                launch_pdl(ln_fwd_batch<TX, E_, K_>, L.grid, kBatchThreads, smem, L.stream, xp, yp,
                           gamma, beta, pt, mean, rstd, M, N, eps, inv_n, L.nblocks, L.R, L.fault);
            }))
            return cudaErrorInvalidValue;
        return cudaGetLastError();
    }
    if (!L.fast) {
        launch_pdl(ln_fwd_general<TX>, L.grid, kGenThreads, 0, L.stream,
            xp, yp, gamma, beta, pt, mean, rstd, M, N, eps, inv_n, L.maps, L.scattered);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE(S)                                                                                \
    case S: {                                                                                      \
        constexpr int smem = ring_smem_bytes(S, kFwdLN, 1);                                        \
        with_mode(L.in_mode, [&](auto m_) {                                                        \
            constexpr int kIn_ = decltype(m_)::value;                                              \
            ring_attributes<ln_fwd_fast<TX, S, kIn_>>(smem);                                       \
            launch_pdl(ln_fwd_fast<TX, S, kIn_>, L.grid, kSched[S].T, smem, L.stream,              \
                xp, yp, gamma, beta, pt, mean, rstd, M, N, eps, inv_n, L.nblocks, L.fault,         \
                L.maps);                                                                           \
        });                                                                                        \
        break;                                                                                     \
    }
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9)
        GBN_CASE(13) GBN_CASE(16) GBN_CASE(17) GBN_CASE(18) GBN_CASE(20) GBN_CASE(21)
        GBN_CASE(22)
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
    if (L.batch) {
        constexpr int smem = batch_smem(2);
        if (!with_batch(L.E, L.KMAX, [&](auto e_, auto k_) {
                constexpr int E_ = decltype(e_)::value, K_ = decltype(k_)::value;
                ring_attributes<ln_bwd_batch<TX, E_, K_>>(smem);
                launch_pdl(ln_bwd_batch<TX, E_, K_>, L.grid, kBatchThreads, smem, L.stream, xp,
                           dyp, mean, rstd, gamma, pt, dxp, ws, M, N, inv_n, L.nblocks, L.R,
                           L.fault);
            }))
            return cudaErrorInvalidValue;
        return cudaGetLastError();
    }
    if (!L.fast) {
        launch_pdl(ln_bwd_general<TX>, L.grid, kGenThreads, 0, L.stream,
            xp, dyp, mean, rstd, gamma, pt, dxp, ws, M, N, inv_n, L.maps, L.scattered);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE_BODY(S)                                                                           \
    {                                                                                              \
        constexpr int smem = bwd_smem_bytes<TX>(S, kBwdLN);                                        \
        with_mode(L.in_mode, [&](auto m_) {                                                        \
            constexpr int kIn_ = decltype(m_)::value;                                              \
            ring_attributes<ln_bwd_fast<TX, S, kIn_>>(smem);                                       \
            launch_pdl(ln_bwd_fast<TX, S, kIn_>, L.grid, kSched[S].T, smem, L.stream,              \
                xp, dyp, mean, rstd, gamma, pt, dxp, ws, M, N, inv_n, L.nblocks, L.fault, L.maps); \
        });                                                                                        \
    }
#define GBN_CASE(S)                                                                                \
    case S:                                                                                        \
        GBN_CASE_BODY(S)                                                                           \
        break;
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9)
        GBN_CASE(12) GBN_CASE(14) GBN_CASE(15) GBN_CASE(17) GBN_CASE(19) GBN_CASE(23)
#undef GBN_CASE
#undef GBN_CASE_BODY
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
    if (xt == kF16) return fwd_dispatch<__half>(L, pt, x, gamma, beta, y, mean, rstd, M, N, eps);
    return fwd_dispatch<__nv_bfloat16>(L, pt, x, gamma, beta, y, mean, rstd, M, N, eps);
}

cudaError_t launch_ln_bwd(const Launch& L, int xt, int pt, const void* x, const void* dy,
                          const float* mean, const float* rstd, const void* gamma, void* dx,
                          float* ws, int64_t M, int N)
{
    if (xt == kF32) return bwd_dispatch<float>(L, pt, x, dy, mean, rstd, gamma, dx, ws, M, N);
    if (xt == kF16) return bwd_dispatch<__half>(L, pt, x, dy, mean, rstd, gamma, dx, ws, M, N);
    return bwd_dispatch<__nv_bfloat16>(L, pt, x, dy, mean, rstd, gamma, dx, ws, M, N);
}

}  // namespace gbn
