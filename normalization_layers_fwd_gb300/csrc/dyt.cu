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
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace gbn {
namespace {

// The flush-to-zero form: e = 2^v only reaches the subnormal range for
// |z| > 43.6, where tanh rounds to +-1 either way and sech^2 (below 2^-124)
// becomes 0, and the ex2 then needs no subnormal handling around it, which
// the DyT kernels, bound by instruction issue, cannot afford.
__device__ __forceinline__ float ex2_approx(float v)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float rcp_approx(float v)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// tanh and sech^2 in float32, from two identities:
//  * with e = exp(-2|z|) = 2^(-2 |z| log2(e)) (hardware ex2):
//      tanh|z| = (1 - e) / (1 + e),  sech^2 z = 4e / (1 + e)^2;
//    sech^2 keeps full relative accuracy for every z this way (no
//    1 - tanh^2 cancellation), so it needs no second branch;
//  * |z| < 1/8: 1 - e cancels, so tanh takes the Maclaurin series
//    z - z^3/3 + 2z^5/15 - 17z^7/315 (the next term is below 2e-10 relative).
// z = +-inf gives tanh = +-1 and sech^2 = 0; NaN propagates.  For |z| > 43.6
// sech^2 is 0 (flushed), against a true value below 2^-124.
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
    t = a < kSmall ? tanh_series(z) : copysignf((1.0f - e) * q, z);
    s = (4.0f * e) * (q * q);
}

// The same two identities on a pair of lanes: the exponential and the
// reciprocal are per lane (MUFU), everything else runs as .f32x2.
__device__ __forceinline__ f2 tanh_series2(f2 z)
{
    const f2 z2 = mul2(z, z);
    f2 p = fma2(z2, splat2(kT7), splat2(kT5));
    p = fma2(z2, p, splat2(kT3));
    p = fma2(z2, p, splat2(1.0f));
    return mul2(z, p);
}

__device__ __forceinline__ f2 pick_tanh2(f2 z, f2 ts, f2 tb)
{
    const float z0 = lo2(z), z1 = hi2(z);
    return mk2(fabsf(z0) < kSmall ? lo2(ts) : copysignf(lo2(tb), z0),
               fabsf(z1) < kSmall ? hi2(ts) : copysignf(hi2(tb), z1));
}

__device__ __forceinline__ f2 dyt_tanh2(f2 z)
{
    const f2 e = mk2(ex2_approx(fabsf(lo2(z)) * kM2Log2e), ex2_approx(fabsf(hi2(z)) * kM2Log2e));
    const f2 d = add2(e, splat2(1.0f));
    const f2 q = mk2(rcp_approx(lo2(d)), rcp_approx(hi2(d)));
    const f2 tb = mul2(sub2(splat2(1.0f), e), q);
    return pick_tanh2(z, tanh_series2(z), tb);
}

__device__ __forceinline__ void dyt_tanh_sech2_2(f2 z, f2& t, f2& s)
{
    const f2 e = mk2(ex2_approx(fabsf(lo2(z)) * kM2Log2e), ex2_approx(fabsf(hi2(z)) * kM2Log2e));
    const f2 d = add2(e, splat2(1.0f));
    const f2 q = mk2(rcp_approx(lo2(d)), rcp_approx(hi2(d)));
    t = pick_tanh2(z, tanh_series2(z), mul2(sub2(splat2(1.0f), e), q));
    s = mul2(mul2(e, splat2(4.0f)), mul2(q, q));
}

// ------------------------------------------------------------ fast forward
// Addressing: a thread's vector of row u of a block sits at soff + u*srow in
// the ring slot and at row0*N + l*VEC + u*grow in HBM (row0 = the block's
// first row + g); only the ragged last block compares rows against M.
template <typename TX, int S, int kIn>
__global__ void __launch_bounds__(kSched[S].T, kind_minb(S, kFwdDyT))
    dyt_fwd_fast(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ alpha,
                 const void* __restrict__ gamma, const void* __restrict__ beta, int pt,
                 int64_t M, int N, int64_t nblocks, unsigned* fault, RowMaps maps)
{
    grid_dependency_sync();
    constexpr int W = kSched[S].W, U = kind_U(S, kFwdDyT), T = kSched[S].T, KV = kSched[S].KV;
    constexpr int VEC = Vec<TX>::kN, P = Pairs<TX>::kP;
    constexpr int G = groups_per_cta(W, T);
    extern __shared__ __align__(128) unsigned char dsm[];
    const int g = grp<W>(), l = lan<W>();
    // vector j of a row is vector l + j*W: in shared memory at +j*W*16 bytes
    bool colok[KV];
#pragma unroll
    for (int j = 0; j < KV; ++j) colok[j] = in_group<W>() && l + j * W < N / VEC;
    const int rb = N * (int)sizeof(TX);
    const int soff = g * rb + l * 16, srow = G * rb, grow = G * N;

    const f2 a2 = splat2(ld_param(alpha, pt, 0));
    f2 gm[KV][P], bt[KV][P];
#pragma unroll
    for (int j = 0; j < KV; ++j) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int c = (l + j * W) * VEC + 2 * p;
            gm[j][p] = colok[j] ? ld_param2(gamma, pt, c) : splat2(0.f);
            bt[j][p] = colok[j] ? ld_param2(beta, pt, c) : splat2(0.f);
        }
    }

    Ring<1, kind_stages(S, kFwdDyT), kIn == kInRows> rg;
    rg.src[0] = reinterpret_cast<const unsigned char*>(x);
    if constexpr (kIn == kInRows) rg.map[0] = maps.m[0];
    rg.row_bytes = rb;
    rg.R = G * U;
    rg.M = M;
    rg.nblocks = nblocks;
    rg.slot = slot_bytes(S, kFwdDyT);
    rg.fault = fault;
    const int64_t nfull = M / (G * U);  // blocks without padded rows
    const int64_t rstride = (int64_t)gridDim.x * (G * U);
    int64_t row0 = (int64_t)blockIdx.x * (G * U) + g;  // this thread's first row
    TX* yb = y + row0 * N + l * VEC;
    // Full blocks of rows that fill every lane's vectors run without row,
    // column or fault predicates (a failed copy leaves stale bytes in the
    // slot, never an address outside it; the fault word reports it): N =
    // 4096 0.917 -> 0.931, 8192 0.888 -> 0.909 of measured copy.
    const bool exact = !seg_groups(W) && N / VEC == W * KV;
    ring_loop(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        const unsigned char* xs = rg.tile(k, 0) + soff;
        const bool full = b < nfull;
        auto run = [&](auto clean_) {
            constexpr bool kClean = decltype(clean_)::value;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool okr = kClean || (alive && (full || row0 + u * G < M));
                TX* const yr = out_at<kIn>(yb, u * grow, y, maps, row0 + u * G, N, l * VEC);
#pragma unroll
                for (int j = 0; j < KV; ++j) {
                    const bool ok = kClean || (okr && colok[j]);
                    f2 v[P];
                    unpack2<TX>(lds128_if(ok, xs + u * srow + j * W * 16), v);
#pragma unroll
                    for (int p = 0; p < P; ++p)
                        v[p] = fma2(gm[j][p], dyt_tanh2(mul2(a2, v[p])), bt[j][p]);
                    st_stream_if(ok, yr + j * W * VEC, pack2<TX>(v));
                }
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
// x and dy stream through the ring.  Full row blocks run without masking;
// only the ragged last block masks its padded rows, by a select after the
// arithmetic (its slots past the last row hold stale data).
template <typename TX, int S, int kIn>
__global__ void __launch_bounds__(kSched[S].T, kind_minb(S, kBwdDyT))
    dyt_bwd_fast(const TX* __restrict__ x, const TX* __restrict__ dy, TX* __restrict__ dx,
                 const void* __restrict__ alpha, const void* __restrict__ gamma, int pt,
                 float* __restrict__ ws, int64_t M, int N, int64_t nblocks, unsigned* fault,
                 RowMaps maps)
{
    grid_dependency_sync();
    constexpr int W = kSched[S].W, U = kind_U(S, kBwdDyT), T = kSched[S].T, KV = kSched[S].KV;
    constexpr int VEC = Vec<TX>::kN, P = Pairs<TX>::kP;
    constexpr int G = groups_per_cta(W, T);
    // The lean form (16-bit rows of 1025-2048 vectors) reads gamma from shared
    // memory at each use and sums gamma * dy * x * sech^2 per thread instead
    // of per column, so that only two column accumulators stay in registers.
    constexpr bool kLean = lean_bwd<TX>(S);
    // At 2 vectors a thread (16-bit) the same per-thread sum of
    // gamma * dy * x * sech^2, with gamma in registers: 16 fewer registers
    // than a per-column accumulator (DyT backward N = 4096 0.871 -> 0.885 of
    // measured copy; float32 rows measured slower with it).
    constexpr bool kDaT = kLean || (KV == 2 && sizeof(TX) == 2);
    static_assert(KV <= 2 || sizeof(TX) == 4 || kLean,
                  "the 16-bit DyT backward takes at most 2 vectors per thread");
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ float red[T / 32];
    const int g = grp<W>(), l = lan<W>();
    // vector j of a row is vector l + j*W: in shared memory at +j*W*16 bytes
    bool colok[KV];
#pragma unroll
    for (int j = 0; j < KV; ++j) colok[j] = in_group<W>() && l + j * W < N / VEC;
    const int rb = N * (int)sizeof(TX);
    const int soff = g * rb + l * 16, srow = G * rb, grow = G * N;

    const f2 a2 = splat2(ld_param(alpha, pt, 0));
    f2 gm[KV][P];
    // gamma*alpha: precomputed with one vector per thread; with two it is
    // recomputed at each use (the same product, so the same bits), which
    // keeps the kernel within 128 registers
    f2 ga[KV == 1 ? P : 1];
    // Per-column accumulators: sum dy*t, sum dy, sum dy*x*sech^2 (gamma is
    // applied to the last one once, at the end).
    f2 acc_g[KV][P], acc_b[KV][P], acc_a[KV][P];
    f2 da2 = splat2(0.f);  // the lean form's sum of gamma * dy * x * sech^2
    // the lean form's gamma, as float32 past the ring
    const float* prm = reinterpret_cast<const float*>(dsm + bwd_ring_bytes<TX>(S, kBwdDyT));
    if constexpr (kLean) stage_params<T>(const_cast<float*>(prm), gamma, pt, N);
    auto gm_at = [&](int j, int p) -> f2 {
        const int c = (l + j * W) * VEC + 2 * p;
        if constexpr (kLean)
            return colok[j] ? prm2(prm, c) : splat2(0.f);
        else
            return colok[j] ? ld_param2(gamma, pt, c) : splat2(0.f);
    };
#pragma unroll
    for (int j = 0; j < KV; ++j) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
            if constexpr (!kLean) gm[j][p] = gm_at(j, p);
            if constexpr (KV == 1) ga[p] = mul2(gm[0][p], a2);
            acc_g[j][p] = acc_b[j][p] = splat2(0.f);
            if constexpr (!kDaT) acc_a[j][p] = splat2(0.f);
        }
    }

    auto rows = [&](const unsigned char* xs, const unsigned char* ds, TX* dxb, int64_t row0,
                    bool alive, auto masked, auto exact_) {
        constexpr bool kExact = decltype(exact_)::value;  // every lane's vectors in the row
        constexpr bool kMask = decltype(masked)::value;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool okr = !kMask || row0 + u * G < M;
            TX* const dxr = out_at<kIn>(dxb, u * grow, dx, maps, row0 + u * G, N, l * VEC);
#pragma unroll
            for (int j = 0; j < KV; ++j) {
                const bool ok = kExact ? okr : alive && colok[j] && okr;
                f2 xv[P], dv[P], o[P];
                unpack2<TX>(lds128_if(ok, xs + u * srow + j * W * 16), xv);
                unpack2<TX>(lds128_if(ok, ds + u * srow + j * W * 16), dv);
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    f2 t, s;
                    dyt_tanh_sech2_2(mul2(a2, xv[p]), t, s);
                    const f2 dsd = mul2(dv[p], s);
                    if constexpr (kDaT) {
                        f2 gmv;
                        if constexpr (kLean)
                            gmv = gm_at(j, p);
                        else
                            gmv = gm[j][p];
                        o[p] = mul2(dsd, mul2(gmv, a2));
                        // lanes past the row's end and padded rows add nothing
                        // (their x may be anything)
                        da2 = sel2(ok, fma2(gmv, mul2(dsd, xv[p]), da2), da2);
                        if constexpr (kMask) {
                            const f2 z = splat2(0.f);
                            acc_g[j][p] = add2(acc_g[j][p], sel2(okr, mul2(dv[p], t), z));
                            acc_b[j][p] = add2(acc_b[j][p], sel2(okr, dv[p], z));
                        } else {
                            acc_g[j][p] = fma2(dv[p], t, acc_g[j][p]);
                            acc_b[j][p] = add2(acc_b[j][p], dv[p]);
                        }
                        continue;
                    }
                    if constexpr (KV == 1)
                        o[p] = mul2(dsd, ga[p]);
                    else
                        o[p] = mul2(dsd, mul2(gm[j][p], a2));
                    if constexpr (kMask) {
                        // padded rows: select after the arithmetic, never a 0/1 multiply
                        const f2 z = splat2(0.f);
                        acc_g[j][p] = add2(acc_g[j][p], sel2(okr, mul2(dv[p], t), z));
                        acc_b[j][p] = add2(acc_b[j][p], sel2(okr, dv[p], z));
                        acc_a[j][p] = add2(acc_a[j][p], sel2(okr, mul2(dsd, xv[p]), z));
                    } else {
                        acc_g[j][p] = fma2(dv[p], t, acc_g[j][p]);
                        acc_b[j][p] = add2(acc_b[j][p], dv[p]);
                        acc_a[j][p] = fma2(dsd, xv[p], acc_a[j][p]);
                    }
                }
                st_stream_if(ok, dxr + j * W * VEC, pack2<TX>(o));
            }
        }
    };

    Ring<2, bwd_stages<TX>(S, kBwdDyT), kIn == kInRows> rg;
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
    rg.slot = slot_bytes(S, kBwdDyT);
    rg.fault = fault;
    const int64_t nfull = M / (G * U);  // blocks without padded rows
    const int64_t rstride = (int64_t)gridDim.x * (G * U);
    int64_t row0 = (int64_t)blockIdx.x * (G * U) + g;  // this thread's first row
    TX* dxb = dx + row0 * N + l * VEC;
    // Rows that fill every lane's vectors run their full blocks without
    // per-vector column predicates and load the slot without the fault
    // predicate (a failed copy leaves stale bytes in the slot, never an
    // address outside it; the fault word reports it).  Measured at several
    // vectors a thread or 1024 threads: N = 4096 0.885 -> 0.916, 8192 0.927
    // -> 0.935 of measured copy; at one vector in 256 threads 1% slower, so
    // those keep the predicates, and so does the lean form.
    constexpr bool kUseExact = !kLean && (KV > 1 || T > 256);
    using ExactT = std::integral_constant<bool, kUseExact>;
    const bool exact = kUseExact && !seg_groups(W) && N / VEC == W * KV;
    ring_loop(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        const unsigned char* xs = rg.tile(k, 0) + soff;
        const unsigned char* ds = rg.tile(k, 1) + soff;
        if (b < nfull)
            if (exact)
                rows(xs, ds, dxb, row0, alive, std::false_type{}, ExactT{});
            else
                rows(xs, ds, dxb, row0, alive, std::false_type{}, std::false_type{});
        else
            rows(xs, ds, dxb, row0, alive, std::true_type{}, std::false_type{});
        row0 += rstride;
        dxb += rstride * N;
    });

    if (ws == nullptr) return;  // no parameter gradient requested (uniform)
    const int64_t L = 2 * (int64_t)N + 1;
    float* wrow = ws + blockIdx.x * L;
    float* colbuf = reinterpret_cast<float*>(dsm + 128);  // drained ring slots, past the barriers
    cta_store_columns_kv<W, KV, P, T>(acc_g, colbuf, wrow, N);
    cta_store_columns_kv<W, KV, P, T>(acc_b, colbuf, wrow + N, N);
    // lanes past the row's end hold garbage (tanh(alpha*0) for alpha = inf);
    // they are never stored above and are excluded here
    float da = 0.f;
    if constexpr (kDaT) {
        da = lo2(da2) + hi2(da2);
    } else {
#pragma unroll
        for (int j = 0; j < KV; ++j) {
            if (colok[j]) {
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const f2 q = mul2(gm[j][p], acc_a[j][p]);
                    da += lo2(q) + hi2(q);
                }
            }
        }
    }
    const float tot = cta_sum<T>(da, red);
    if (threadIdx.x == 0) wrow[2 * N] = tot;
}

// ------------------------------------------------------ general (any shape)
template <typename TX>
__global__ void __launch_bounds__(kGenThreads)
    dyt_fwd_general(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ alpha,
                    const void* __restrict__ gamma, const void* __restrict__ beta, int pt,
                    int64_t M, int N, RowMaps maps, int scattered)
{
    grid_dependency_sync();
    const float a = ld_param(alpha, pt, 0);
    const int64_t E = M * (int64_t)N;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < E;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % N);
        const float xv = scattered ? ld1(in_row(x, maps, 0, 1, i / N, N), c) : ld1(x, i);
        st1(y, i, fmaf(ld_param(gamma, pt, c), dyt_tanh(a * xv), ld_param(beta, pt, c)));
    }
}

// One warp per row; warp w owns workspace row w and accumulates into it
// (read-modify-write by the lane that owns each column, rows in order).
template <typename TX>
__global__ void __launch_bounds__(kGenThreads)
    dyt_bwd_general(const TX* __restrict__ x, const TX* __restrict__ dy, TX* __restrict__ dx,
                    const void* __restrict__ alpha, const void* __restrict__ gamma, int pt,
                    float* __restrict__ ws, int64_t M, int N, RowMaps maps, int scattered)
{
    grid_dependency_sync();
    __shared__ float accs[kGenWarps * kGenCols];
    const int lane = threadIdx.x & 31;
    const int64_t w = blockIdx.x * (int64_t)kGenWarps + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * kGenWarps;
    const int64_t L = 2 * (int64_t)N + 1;
    float* wrow = ws ? ws + w * L : nullptr;
    // the warp's column sums: in shared memory when they fit, else in its
    // workspace row; lane c % 32 alone touches column c, rows in order
    const bool local = 2 * N <= kGenCols;
    float* arow = local ? accs + (threadIdx.x >> 5) * kGenCols : wrow;
    if (wrow)
        for (int c = lane; c < 2 * N; c += 32) arow[c] = 0.f;
    const float a = ld_param(alpha, pt, 0);
    float da = 0.f;
    for (int64_t r = w; r < M; r += nw) {
        const TX* xr = in_row(x, maps, 0, scattered, r, N);
        const TX* dr = in_row(dy, maps, 1, scattered, r, N);
        for (int c = lane; c < N; c += 32) {
            const int64_t i = r * N + c;
            const float xv = ld1(xr, c), dv = ld1(dr, c), gmv = ld_param(gamma, pt, c);
            float t, s;
            dyt_tanh_sech2(a * xv, t, s);
            const float ds = dv * s;
            st1(dx, i, ds * (gmv * a));
            if (wrow) {
                arow[c] += dv * t;
                arow[N + c] += dv;
            }
            da = fmaf(gmv, ds * xv, da);
        }
    }
    if (wrow && local)
        for (int c = lane; c < 2 * N; c += 32) wrow[c] = arow[c];
    float v[1] = {da};
    butterfly<32, 1>(v);
    if (wrow && lane == 0) wrow[2 * N] = v[0];
}

// ------------------------------------------------------ row-batched path
// Rows whose byte length is not a multiple of 16 (common.cuh, "row-batched"):
// blocks of R rows through the ring, one warp per row, lane l taking units
// l, l + 32, ... of it.
template <typename TX, int E, int KMAX>
__global__ void __launch_bounds__(kBatchThreads, batch_minb(false))
    dyt_fwd_batch(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ alpha,
                  const void* __restrict__ gamma, const void* __restrict__ beta, int pt,
                  int64_t M, int N, int64_t nblocks, int R, unsigned* fault)
{
    grid_dependency_sync();
    using U = Unit<TX, E>;
    extern __shared__ __align__(128) unsigned char dsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nu = N / E;
    const int rb = N * (int)sizeof(TX);
    const float a = ld_param(alpha, pt, 0);
    bool uok[KMAX];
    float gm[KMAX][E], bt[KMAX][E];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        uok[k] = lane + 32 * k < nu;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int c = (lane + 32 * k) * E + e;
            gm[k][e] = uok[k] ? ld_param(gamma, pt, c) : 0.f;
            bt[k][e] = uok[k] ? ld_param(beta, pt, c) : 0.f;
        }
    }
    const int64_t tail = ((M * (int64_t)rb) & ~(int64_t)15) / (int64_t)sizeof(TX);
    Ring<1, batch_stages(1)> rg;
    rg.src[0] = reinterpret_cast<const unsigned char*>(x);
    rg.row_bytes = rb;
    rg.R = R;
    rg.M = M;
    rg.nblocks = nblocks;
    rg.slot = batch_slot(1);
    rg.fault = fault;
    constexpr int UB = E * (int)sizeof(TX);  // bytes of a unit
    ring_loop(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        if (!alive) return;
        const uint32_t xs = smem_u32(rg.tile(k, 0)) + lane * UB;
        const int64_t r0 = b * R;
        const int rows = (int)(M - r0 < R ? M - r0 : R);
        // one row a warp at a time (no row reduction to share), its units all
        // loaded before any is used.  A block whose units are all in the slot
        // runs unmasked; the last one takes units past the copied bytes from
        // global memory.
        auto pass = [&](auto masked) {
            constexpr bool kMask = decltype(masked)::value;
            for (int i = warp; i < rows; i += kBatchWarps) {
                const int64_t gr = (r0 + i) * N + lane * E;
                typename U::W w[KMAX];
#pragma unroll
                for (int kk = 0; kk < KMAX; ++kk) {
                    w[kk] = typename U::W{};
                    if constexpr (kMask) {
                        const int64_t gi = gr + kk * 32 * E;
                        if (uok[kk])
                            w[kk] = gi < tail ? U::lds(xs + i * rb + kk * 32 * UB) : U::ld(x + gi);
                    } else {
                        if (uok[kk]) w[kk] = U::lds(xs + i * rb + kk * 32 * UB);
                    }
                }
#pragma unroll
                for (int kk = 0; kk < KMAX; ++kk) {
                    float v[E];
                    U::unpack(w[kk], v);
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        v[e] = fmaf(gm[kk][e], dyt_tanh(a * v[e]), bt[kk][e]);
                    if (uok[kk]) U::st(y + gr + kk * 32 * E, U::pack(v));
                }
            }
        };
        if ((r0 + rows) * N <= tail)
            pass(std::false_type{});
        else
            pass(std::true_type{});
    });
}

template <typename TX, int E, int KMAX>
__global__ void __launch_bounds__(kBatchThreads, batch_minb(true))
    dyt_bwd_batch(const TX* __restrict__ x, const TX* __restrict__ dy, TX* __restrict__ dx,
                  const void* __restrict__ alpha, const void* __restrict__ gamma, int pt,
                  float* __restrict__ ws, int64_t M, int N, int64_t nblocks, int R,
                  unsigned* fault)
{
    grid_dependency_sync();
    using U = Unit<TX, E>;
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ float red[kBatchWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nu = N / E;
    const int rb = N * (int)sizeof(TX);
    const float a = ld_param(alpha, pt, 0);
    bool uok[KMAX];
    float gm[KMAX][E], acc_g[KMAX][E], acc_b[KMAX][E];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        uok[k] = lane + 32 * k < nu;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            gm[k][e] = uok[k] ? ld_param(gamma, pt, (lane + 32 * k) * E + e) : 0.f;
            acc_g[k][e] = acc_b[k][e] = 0.f;
        }
    }
    float da = 0.f;
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
    constexpr int UB = E * (int)sizeof(TX);  // bytes of a unit
    ring_loop(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        if (!alive) return;
        const uint32_t xs = smem_u32(rg.tile(k, 0)) + lane * UB;
        const uint32_t ds = smem_u32(rg.tile(k, 1)) + lane * UB;
        const int64_t r0 = b * R;
        const int rows = (int)(M - r0 < R ? M - r0 : R);
        // one row a warp at a time (no row reduction to share), its units all
        // loaded before any is used.  A block whose units are all in the slot
        // runs unmasked; the last one takes units past the copied bytes from
        // global memory.
        auto pass = [&](auto masked) {
            constexpr bool kMask = decltype(masked)::value;
            for (int i = warp; i < rows; i += kBatchWarps) {
                const int64_t gr = (r0 + i) * N + lane * E;
                typename U::W wx[KMAX], wd[KMAX];
#pragma unroll
                for (int kk = 0; kk < KMAX; ++kk) {
                    wx[kk] = wd[kk] = typename U::W{};
                    const int so = i * rb + kk * 32 * UB;
                    if constexpr (kMask) {
                        const int64_t gi = gr + kk * 32 * E;
                        if (uok[kk]) {
                            const bool sm = gi < tail;
                            wx[kk] = sm ? U::lds(xs + so) : U::ld(x + gi);
                            wd[kk] = sm ? U::lds(ds + so) : U::ld(dy + gi);
                        }
                    } else if (uok[kk]) {
                        wx[kk] = U::lds(xs + so);
                        wd[kk] = U::lds(ds + so);
                    }
                }
#pragma unroll
                for (int kk = 0; kk < KMAX; ++kk) {
                    if (!uok[kk]) continue;
                    float xv[E], dv[E], o[E];
                    U::unpack(wx[kk], xv);
                    U::unpack(wd[kk], dv);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        float t, sc;
                        dyt_tanh_sech2(a * xv[e], t, sc);
                        const float dsd = dv[e] * sc;
                        o[e] = dsd * (gm[kk][e] * a);
                        acc_g[kk][e] = fmaf(dv[e], t, acc_g[kk][e]);
                        acc_b[kk][e] += dv[e];
                        da = fmaf(gm[kk][e], dsd * xv[e], da);
                    }
                    U::st(dx + gr + kk * 32 * E, U::pack(o));
                }
            }
        };
        if ((r0 + rows) * N <= tail)
            pass(std::false_type{});
        else
            pass(std::true_type{});
    });
    if (ws == nullptr) return;  // no parameter gradient requested (uniform)
    const int64_t L = 2 * (int64_t)N + 1;
    float* cols = reinterpret_cast<float*>(dsm + 128);  // drained ring slots: 8 x 2N floats
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
    float v[1] = {da};
    butterfly<32, 1>(v);
    if (lane == 0) red[warp] = v[0];
    __syncthreads();
    float* wrow = ws + blockIdx.x * L;
    for (int c = threadIdx.x; c < 2 * N; c += kBatchThreads) {
        float t = cols[c];
#pragma unroll
        for (int w = 1; w < kBatchWarps; ++w) t += cols[w * 2 * N + c];
        wrow[c] = t;
    }
    if (threadIdx.x == 0) {
        float t = red[0];
#pragma unroll
        for (int w = 1; w < kBatchWarps; ++w) t += red[w];
        wrow[2 * N] = t;
    }
}

template <typename TX>
cudaError_t fwd_dispatch(const Launch& L, int pt, const void* x, const void* alpha,
                         const void* gamma, const void* beta, void* y, int64_t M, int N)
{
    const TX* xp = static_cast<const TX*>(x);
    TX* yp = static_cast<TX*>(y);
    if (L.batch) {
        constexpr int smem = batch_smem(1);
        if (!with_batch(L.E, L.KMAX, [&](auto e_, auto k_) {
                constexpr int E_ = decltype(e_)::value, K_ = decltype(k_)::value;
                ring_attributes<dyt_fwd_batch<TX, E_, K_>>(smem);
                launch_pdl(dyt_fwd_batch<TX, E_, K_>, L.grid, kBatchThreads, smem, L.stream, xp,
                           yp, alpha, gamma, beta, pt, M, N, L.nblocks, L.R, L.fault);
            }))
            return cudaErrorInvalidValue;
        return cudaGetLastError();
    }
    if (!L.fast) {
        launch_pdl(dyt_fwd_general<TX>, L.grid, kGenThreads, 0, L.stream, xp, yp, alpha, gamma,
                   beta, pt, M, N, L.maps, L.scattered);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE(S)                                                                                \
    case S: {                                                                                      \
        constexpr int smem = ring_smem_bytes(S, kFwdDyT, 1);                                       \
        with_mode(L.in_mode, [&](auto m_) {                                                        \
            constexpr int kIn_ = decltype(m_)::value;                                              \
            ring_attributes<dyt_fwd_fast<TX, S, kIn_>>(smem);                                      \
            launch_pdl(dyt_fwd_fast<TX, S, kIn_>, L.grid, kSched[S].T, smem, L.stream,             \
                xp, yp, alpha, gamma, beta, pt, M, N, L.nblocks, L.fault, L.maps);                 \
        });                                                                                        \
        break;                                                                                     \
    }
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9)
        GBN_CASE(12) GBN_CASE(13) GBN_CASE(17)
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
    if (L.batch) {
        constexpr int smem = batch_smem(2);
        if (!with_batch(L.E, L.KMAX, [&](auto e_, auto k_) {
                constexpr int E_ = decltype(e_)::value, K_ = decltype(k_)::value;
                ring_attributes<dyt_bwd_batch<TX, E_, K_>>(smem);
                launch_pdl(dyt_bwd_batch<TX, E_, K_>, L.grid, kBatchThreads, smem, L.stream, xp,
                           dyp, dxp, alpha, gamma, pt, ws, M, N, L.nblocks, L.R, L.fault);
            }))
            return cudaErrorInvalidValue;
        return cudaGetLastError();
    }
    if (!L.fast) {
        launch_pdl(dyt_bwd_general<TX>, L.grid, kGenThreads, 0, L.stream, xp, dyp, dxp, alpha,
                   gamma, pt, ws, M, N, L.maps, L.scattered);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE_BODY(S)                                                                           \
    {                                                                                              \
        constexpr int smem = bwd_smem_bytes<TX>(S, kBwdDyT);                                       \
        with_mode(L.in_mode, [&](auto m_) {                                                        \
            constexpr int kIn_ = decltype(m_)::value;                                              \
            ring_attributes<dyt_bwd_fast<TX, S, kIn_>>(smem);                                      \
            launch_pdl(dyt_bwd_fast<TX, S, kIn_>, L.grid, kSched[S].T, smem, L.stream,             \
                xp, dyp, dxp, alpha, gamma, pt, ws, M, N, L.nblocks, L.fault, L.maps);             \
        });                                                                                        \
    }
#define GBN_CASE(S)                                                                                \
    case S:                                                                                        \
        GBN_CASE_BODY(S)                                                                           \
        break;
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9) GBN_CASE(11)
        GBN_CASE(12)
        GBN_CASE(17)
#undef GBN_CASE
#undef GBN_CASE_BODY
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dyt_fwd(const Launch& L, int xt, int pt, const void* x, const void* alpha,
                           const void* gamma, const void* beta, void* y, int64_t M, int N)
{
    if (xt == kF32) return fwd_dispatch<float>(L, pt, x, alpha, gamma, beta, y, M, N);
    if (xt == kF16) return fwd_dispatch<__half>(L, pt, x, alpha, gamma, beta, y, M, N);
    return fwd_dispatch<__nv_bfloat16>(L, pt, x, alpha, gamma, beta, y, M, N);
}

cudaError_t launch_dyt_bwd(const Launch& L, int xt, int pt, const void* x, const void* dy,
                           const void* alpha, const void* gamma, void* dx, float* ws, int64_t M,
                           int N)
{
    if (xt == kF32) return bwd_dispatch<float>(L, pt, x, dy, alpha, gamma, dx, ws, M, N);
    if (xt == kF16) return bwd_dispatch<__half>(L, pt, x, dy, alpha, gamma, dx, ws, M, N);
    return bwd_dispatch<__nv_bfloat16>(L, pt, x, dy, alpha, gamma, dx, ws, M, N);
}

}  // namespace gbn
