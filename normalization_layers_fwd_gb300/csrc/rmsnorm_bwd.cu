// rmsnorm_bwd.cu -- RMSNorm backward: the fast (bulk-copy ring) and general
// kernels, their dispatch and launch_rms_bwd.  The rounding points and the
// expression variants are described in rmsnorm.cuh.
#include "rmsnorm.cuh"

namespace gbn {
namespace {

// ----------------------------------------------------------- fast backward
// x and dy stream through the ring; a given rstd of the next row block is
// prefetched into registers, otherwise r is recomputed with the forward's
// code.  Full row blocks run without masking; the ragged last block masks its
// padded rows by a select after the arithmetic.
template <typename TX, int S, bool kWF, int kIn>
__global__ void __launch_bounds__(kSched[S].T, kind_minb(S, kBwdRms))
    rms_bwd_fast(const TX* __restrict__ x, const TX* __restrict__ dy, const void* __restrict__ w,
                 int pt, const float* __restrict__ rstd, TX* __restrict__ dx,
                 float* __restrict__ ws, int64_t M, int N, float eps, float inv_n,
                 int64_t nblocks, unsigned* fault, int gemma, RowMaps maps)
{
    grid_dependency_sync();
    constexpr int W = kSched[S].W, U = kind_U(S, kBwdRms), T = kSched[S].T, KV = kSched[S].KV;
    constexpr int VEC = Vec<TX>::kN, P = Pairs<TX>::kP;
    constexpr int G = groups_per_cta(W, T);
    // The lean form (16-bit rows of 1025-2048 vectors) holds only the weight
    // gradient accumulators: it reads the row from the ring slot again after
    // the row reduction, and the weight from shared memory at each use.
    constexpr bool kLean = lean_bwd<TX>(S);
    static_assert(KV <= 2 || sizeof(TX) == 4 || kLean,
                  "the 16-bit RMSNorm backward takes at most 2 vectors per thread");
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
    // the weight of pair p of vector j, as float32 (1 + w for Gemma) and as a
    // packed 16-bit pair (used when w16)
    // the lean form's weight, as float32 past the ring (a 16-bit weight
    // converts back to its own bits exactly)
    const float* prm = reinterpret_cast<const float*>(dsm + bwd_ring_bytes<TX>(S, kBwdRms));
    if constexpr (kLean) stage_params<T>(const_cast<float*>(prm), w, pt, N);
    auto wf_at = [&](int j, int p) -> f2 {
        const int c = (l + j * W) * VEC + 2 * p;
        const f2 v = !colok[j] ? splat2(0.f) : kLean ? prm2(prm, c) : ld_param2(w, pt, c);
        return gemma ? add2(splat2(1.f), v) : v;  // 1 + w in float32
    };
    auto wpk_at = [&](int j, int p) -> uint32_t {
        const int c = (l + j * W) * VEC + 2 * p;
        if (!(w16 && colok[j])) return 0u;
        if constexpr (kLean)
            return P16<TX>::from_f2(prm2(prm, c));
        else
            return static_cast<const uint32_t*>(w)[c / 2];
    };
#pragma unroll
    for (int j = 0; j < KV; ++j) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
            if constexpr (!kLean) {
                wf[j][p] = wf_at(j, p);
                wpk[j][p] = wpk_at(j, p);
            }
            acc[j][p] = splat2(0.f);
        }
    }
    auto wfv = [&](int j, int p) -> f2 {
        if constexpr (kLean)
            return wf_at(j, p);
        else
            return wf[j][p];
    };
    auto wpkv = [&](int j, int p) -> uint32_t {
        if constexpr (kLean)
            return wpk_at(j, p);
        else
            return wpk[j][p];
    };
    // dn = dy w (rounded as the expression says) of one pair, and the weight
    // gradient accumulator with this row's term dy n added (n = xhat rounded)
    auto pair_terms = [&](int j, int p, uint32_t dyw, f2 dv, f2 xh, f2 a, f2& dn) -> f2 {
        if constexpr (is16<TX>() && !kWF) {
            const uint32_t npk = P16<TX>::from_f2(xh);  // n = round_x(xhat)
            if (w16) {
                dn = P16<TX>::to_f2(P16<TX>::mul(dyw, wpkv(j, p)));
                return add2(a, P16<TX>::to_f2(P16<TX>::mul(dyw, npk)));
            }
            // float32 weight: dy*n unrounded, exact product of two 16-bit values
            dn = round2<TX>(mul2(dv, wfv(j, p)));
            return mk2(P16<TX>::fma_lo(dyw, npk, lo2(a)), P16<TX>::fma_hi(dyw, npk, hi2(a)));
        } else {
            dn = mul2(dv, wfv(j, p));
            return fma2(dv, xh, a);
        }
    };
    // the given rstd of this thread's rows, loaded one row block ahead of use
    // (rs_n), or two (rs_nn too) with several vectors per thread: measured
    // faster for those wide rows, slower for the narrow ones
    constexpr bool kDeep = KV > 1;
    // and, for the segmented rows of 3 vectors, prefetched into L2 four
    // blocks ahead: N = 24 0.902 -> 0.931 of measured copy (elsewhere the
    // prefetches cost 1-10%)
    constexpr bool kPrefetch = kIn == kInContig && seg_groups(W);
    float rs_n[U], rs_nn[U];
    auto load_rstd = [&](int64_t row0, float (&dst)[U]) {
        if (rstd) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t row = row0 + u * G;
                dst[u] = row < M ? ld_stat<kIn>(rstd, stat_row<kIn>(maps, row)) : 0.f;
            }
        }
    };
    const int64_t bstride = (int64_t)gridDim.x * (G * U);
    load_rstd((int64_t)blockIdx.x * (G * U) + g, rs_n);
    if constexpr (kDeep) load_rstd((int64_t)blockIdx.x * (G * U) + g + bstride, rs_nn);

    // Pass 1 (after r is known) computes dn and xhat, the reduction term and
    // the weight-gradient term (independent of the row reduction); pass 2
    // keeps only xhat and dn.
    auto rows = [&](const unsigned char* xs, const unsigned char* ds, TX* dxb, int64_t row0,
                    bool alive_, auto masked, auto exact_) {
        constexpr bool kMask = decltype(masked)::value;
        // every lane's vectors in the row: no column or fault predicates
        // (the fault word still reports a failed copy)
        constexpr bool kExact = decltype(exact_)::value;
        const bool alive = kExact || alive_;
        bool col[KV];
#pragma unroll
        for (int j = 0; j < KV; ++j) col[j] = kExact || colok[j];
        float rs[U];
        bool okr[U];
        f2 xh[U][KV][P], dn[U][KV][P];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            okr[u] = !kMask || row0 + u * G < M;
#pragma unroll
            for (int j = 0; j < KV; ++j)  // x, scaled by r below
                unpack2<TX>(lds128_if(alive && okr[u] && col[j], xs + u * srow + j * W * 16),
                        xh[u][j]);
            rs[u] = rs_n[u];
            if constexpr (kDeep) rs_n[u] = rs_nn[u];
        }
        if constexpr (kDeep)
            load_rstd(row0 + 2 * bstride, rs_nn);
        else
            load_rstd(row0 + bstride, rs_n);
        if constexpr (kPrefetch)
            if (rstd) prefetch_stats(rstd, row0 - g + 4 * bstride, G * U, M);
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
                const uint4 dr = lds128_if(alive && okr[u] && col[j], ds + u * srow + j * W * 16);
                f2 dv[P];
                unpack2<TX>(dr, dv);
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    xh[u][j][p] = mul2(xh[u][j][p], r2);
                    // the accumulator with this row's dw term added
                    const f2 nxt = pair_terms(j, p, word(dr, p), dv[p], xh[u][j][p], acc[j][p],
                                              dn[u][j][p]);
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
            TX* const dxr = out_at<kIn>(dxb, u * grow, dx, maps, row0 + u * G, N, l * VEC);
#pragma unroll
            for (int j = 0; j < KV; ++j) {
                f2 o[P];
#pragma unroll
                for (int p = 0; p < P; ++p) o[p] = mul2(r2, fma2(xh[u][j][p], nm, dn[u][j][p]));
                st_stream_if(alive && okr[u] && col[j], dxr + j * W * VEC, pack2<TX>(o));
            }
        }
    };

    // The lean form of `rows`: x for the recomputed r, then x and dy for the
    // reduction and the weight gradient, then x and dy again for dx.
    auto rows_lean = [&](const unsigned char* xs, const unsigned char* ds, TX* dxb, int64_t row0,
                         bool alive, auto masked) {
        constexpr bool kMask = decltype(masked)::value;
        float rs[U], s[U];
        bool okr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            okr[u] = !kMask || row0 + u * G < M;
            rs[u] = rs_n[u];
            if constexpr (kDeep) rs_n[u] = rs_nn[u];
        }
        if constexpr (kDeep)
            load_rstd(row0 + 2 * bstride, rs_nn);
        else
            load_rstd(row0 + bstride, rs_n);
        if (!rstd) {  // uniform branch: recompute r exactly as the forward does
#pragma unroll
            for (int u = 0; u < U; ++u) {
                rs[u] = 0.f;
#pragma unroll
                for (int j = 0; j < KV; ++j) {
                    f2 xv[P];
                    unpack2<TX>(lds128_if(alive && okr[u] && colok[j], xs + u * srow + j * W * 16),
                                xv);
                    rs[u] += vec_sumsq2<P>(xv);
                }
            }
            group_allreduce<W, T, U>(rs, red, parity);
#pragma unroll
            for (int u = 0; u < U; ++u) rs[u] = rsqrtf(fmaf(rs[u], inv_n, eps));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const f2 r2 = splat2(rs[u]);
            f2 a2 = splat2(0.f);
#pragma unroll
            for (int j = 0; j < KV; ++j) {
                const bool ok = alive && okr[u] && colok[j];
                const uint4 dr = lds128_if(ok, ds + u * srow + j * W * 16);
                f2 xv[P], dv[P];
                unpack2<TX>(lds128_if(ok, xs + u * srow + j * W * 16), xv);
                unpack2<TX>(dr, dv);
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const f2 xh = mul2(xv[p], r2);
                    f2 dn;
                    const f2 nxt = pair_terms(j, p, word(dr, p), dv[p], xh, acc[j][p], dn);
                    a2 = fma2(dn, xh, a2);
                    acc[j][p] = (!kMask || okr[u]) ? nxt : acc[j][p];
                }
            }
            s[u] = lo2(a2) + hi2(a2);
        }
        group_allreduce<W, T, U>(s, red, parity);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const f2 r2 = splat2(rs[u]), nm = splat2(-(s[u] * inv_n));
            TX* const dxr = out_at<kIn>(dxb, u * grow, dx, maps, row0 + u * G, N, l * VEC);
#pragma unroll
            for (int j = 0; j < KV; ++j) {
                const bool ok = alive && okr[u] && colok[j];
                const uint4 dr = lds128_if(ok, ds + u * srow + j * W * 16);
                f2 xv[P], dv[P], o[P];
                unpack2<TX>(lds128_if(ok, xs + u * srow + j * W * 16), xv);
                unpack2<TX>(dr, dv);
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const f2 xh = mul2(xv[p], r2);
                    f2 dn;
                    pair_terms(j, p, word(dr, p), dv[p], xh, splat2(0.f), dn);
                    o[p] = mul2(r2, fma2(xh, nm, dn));
                }
                st_stream_if(ok, dxr + j * W * VEC, pack2<TX>(o));
            }
        }
    };

    Ring<2, bwd_stages<TX>(S, kBwdRms), kIn == kInRows> rg;
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
    rg.slot = slot_bytes(S, kBwdRms);
    rg.fault = fault;
    const int64_t nfull = M / (G * U);  // blocks without padded rows
    const int64_t rstride = (int64_t)gridDim.x * (G * U);
    int64_t row0 = (int64_t)blockIdx.x * (G * U) + g;  // this thread's first row
    TX* dxb = dx + row0 * N + l * VEC;
    // rows wider than a warp: the row reduction's barrier releases the slot;
    // except at 1024 threads (one CTA per SM), where the ring's own barrier
    // measured 7% faster
    // Rows that fill every lane's vectors run their full blocks without
    // per-vector column predicates and load the slot without the fault
    // predicate (a failed copy leaves stale bytes in the slot, never an
    // address outside it; the fault word reports it): up to 0.8% faster.
    const bool exact = !seg_groups(W) && N / VEC == W * KV;
    ring_loop<(W > 32 && T < 1024 && !kLean)>(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        const unsigned char* xs = rg.tile(k, 0) + soff;
        const unsigned char* ds = rg.tile(k, 1) + soff;
        if constexpr (kLean) {
            if (b < nfull)
                rows_lean(xs, ds, dxb, row0, alive, std::false_type{});
            else
                rows_lean(xs, ds, dxb, row0, alive, std::true_type{});
        } else {
            if (b < nfull) {
                if (exact)
                    rows(xs, ds, dxb, row0, alive, std::false_type{}, std::true_type{});
                else
                    rows(xs, ds, dxb, row0, alive, std::false_type{}, std::false_type{});
            } else {
                rows(xs, ds, dxb, row0, alive, std::true_type{}, std::false_type{});
            }
        }
        row0 += rstride;
        dxb += rstride * N;
    });

    if (ws == nullptr) return;  // no weight gradient requested (uniform)
    float* wrow = ws + blockIdx.x * (int64_t)N;
    // the column buffer: drained ring slots, past the barriers
    cta_store_columns_kv<W, KV, P, T>(acc, reinterpret_cast<float*>(dsm + 128), wrow, N);
}

template <typename TX>
__global__ void __launch_bounds__(kGenThreads)
    rms_bwd_general(const TX* __restrict__ x, const TX* __restrict__ dy,
                    const void* __restrict__ w, int pt, const float* __restrict__ rstd,
                    TX* __restrict__ dx, float* __restrict__ ws, int64_t M, int N, float eps,
                    float inv_n, int variant, RowMaps maps, int scattered)
{
    grid_dependency_sync();
    __shared__ float accs[kGenWarps * kGenCols];
    const int lane = threadIdx.x & 31;
    const int64_t wi = blockIdx.x * (int64_t)kGenWarps + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * kGenWarps;
    const bool cast_first = variant == 0;  // the Llama expression's rounding points
    const bool round_terms = cast_first && pt != kF32;
    float* wrow = ws ? ws + wi * (int64_t)N : nullptr;
    // the warp's column sums: in shared memory when they fit, else in its
    // workspace row; lane c % 32 alone touches column c, rows in order
    const bool local = N <= kGenCols;
    float* arow = local ? accs + (threadIdx.x >> 5) * kGenCols : wrow;
    if (wrow)
        for (int c = lane; c < N; c += 32) arow[c] = 0.f;
    for (int64_t r = wi; r < M; r += nw) {
        const TX* xr = in_row(x, maps, 0, scattered, r, N);
        const TX* dr = in_row(dy, maps, 1, scattered, r, N);
        const float rs = rstd ? rstd[r] : warp_row_rstd(xr, N, lane, eps, inv_n);
        float s[1] = {0.f};
        for (int c = lane; c < N; c += 32) {
            float dn = ld1c(dr, c) * rms_weight(w, pt, c, variant);
            if (cast_first) dn = round_x<TX>(dn);
            s[0] = fmaf(dn, ld1c(xr, c) * rs, s[0]);
        }
        butterfly<32, 1>(s);
        const float m = s[0] * inv_n;
        for (int c = lane; c < N; c += 32) {
            const float dv = ld1c(dr, c);
            const float xh = ld1c(xr, c) * rs;
            float dn = dv * rms_weight(w, pt, c, variant);
            if (cast_first) dn = round_x<TX>(dn);
            st1(dx, r * N + c, rs * (dn - xh * m));
            float term = dv * (cast_first ? round_x<TX>(xh) : xh);
            if (round_terms) term = round_x<TX>(term);
            if (wrow) arow[c] += term;
        }
    }
    if (wrow && local)
        for (int c = lane; c < N; c += 32) wrow[c] = arow[c];
}

// ------------------------------------------------------ row-batched path
// Rows whose byte length is not a multiple of 16 (common.cuh, "row-batched"):
// blocks of R rows through the ring, one warp per row; a recomputed r uses
// the forward's batch_row_rstd.  The rounding points are the general path's.
template <typename TX, int E, int KMAX>
__global__ void __launch_bounds__(kBatchThreads, batch_minb(true))
    rms_bwd_batch(const TX* __restrict__ x, const TX* __restrict__ dy, const void* __restrict__ w,
                  int pt, const float* __restrict__ rstd, TX* __restrict__ dx,
                  float* __restrict__ ws, int64_t M, int N, float eps, float inv_n, int variant,
                  int64_t nblocks, int R, unsigned* fault)
{
    grid_dependency_sync();
    using U = Unit<TX, E>;
    extern __shared__ __align__(128) unsigned char dsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nu = N / E;
    const int rb = N * (int)sizeof(TX);
    const bool cast_first = variant == 0;  // the Llama expression's rounding points
    const bool round_terms = cast_first && pt != kF32;
    bool uok[KMAX];
    float wv[KMAX][E], acc[KMAX][E];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        uok[k] = lane + 32 * k < nu;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            wv[k][e] = uok[k] ? rms_weight(w, pt, (lane + 32 * k) * E + e, variant) : 0.f;
            acc[k][e] = 0.f;
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
                float xv[RB][KMAX][E], dv[RB][KMAX][E], rs[RB], s[RB];
#pragma unroll
                for (int rr = 0; rr < RB; ++rr) {
                    const int i = i0 + rr;
                    const int64_t r = r0 + i;
                    const bool ok = !kMask || i < rows;
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
                        U::unpack(wx, xv[rr][kk]);
                        U::unpack(wd, dv[rr][kk]);
                    }
                    rs[rr] = rstd ? (ok ? __ldca(rstd + r) : 0.f) : batch_sumsq<KMAX, E>(xv[rr]);
                }
                if (!rstd) batch_rstd<RB>(rs, eps, inv_n);  // uniform branch
#pragma unroll
                for (int rr = 0; rr < RB; ++rr) {
                    s[rr] = 0.f;
#pragma unroll
                    for (int kk = 0; kk < KMAX; ++kk)
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            float dn = dv[rr][kk][e] * wv[kk][e];
                            if (cast_first) dn = round_x<TX>(dn);
                            s[rr] = fmaf(dn, xv[rr][kk][e] * rs[rr], s[rr]);
                        }
                }
                butterfly<32, RB>(s);
#pragma unroll
                for (int rr = 0; rr < RB; ++rr) {
                    const int i = i0 + rr;
                    const bool ok = !kMask || i < rows;
                    const float m = s[rr] * inv_n;
                    TX* const dxr = dx + (r0 + i) * N + lane * E;
#pragma unroll
                    for (int kk = 0; kk < KMAX; ++kk) {
                        float o[E];
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            const float xh = xv[rr][kk][e] * rs[rr];
                            float dn = dv[rr][kk][e] * wv[kk][e];
                            if (cast_first) dn = round_x<TX>(dn);
                            o[e] = rs[rr] * (dn - xh * m);
                            float term = dv[rr][kk][e] * (cast_first ? round_x<TX>(xh) : xh);
                            if (round_terms) term = round_x<TX>(term);
                            acc[kk][e] += term;
                        }
                        if (ok && uok[kk]) U::st(dxr + kk * 32 * E, U::pack(o));
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
    if (ws == nullptr) return;  // no weight gradient requested (uniform)
    float* cols = reinterpret_cast<float*>(dsm + 128);  // drained ring slots: 8 x N floats
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e)
            if (uok[k]) cols[warp * N + (lane + 32 * k) * E + e] = acc[k][e];
    __syncthreads();
    float* wrow = ws + blockIdx.x * (int64_t)N;
    for (int c = threadIdx.x; c < N; c += kBatchThreads) {
        float t = cols[c];
#pragma unroll
        for (int q = 1; q < kBatchWarps; ++q) t += cols[q * N + c];
        wrow[c] = t;
    }
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
    if (L.batch) {
        constexpr int smem = batch_smem(2);
        if (!with_batch(L.E, L.KMAX, [&](auto e_, auto k_) {
                constexpr int E_ = decltype(e_)::value, K_ = decltype(k_)::value;
                ring_attributes<rms_bwd_batch<TX, E_, K_>>(smem);
                launch_pdl(rms_bwd_batch<TX, E_, K_>, L.grid, kBatchThreads, smem, L.stream, xp,
                           dyp, w, pt, rstd, dxp, ws, M, N, eps, inv_n, variant, L.nblocks, L.R,
                           L.fault);
            }))
            return cudaErrorInvalidValue;
        return cudaGetLastError();
    }
    if (!L.fast) {
        launch_pdl(rms_bwd_general<TX>, L.grid, kGenThreads, 0, L.stream,
            xp, dyp, w, pt, rstd, dxp, ws, M, N, eps, inv_n, variant, L.maps, L.scattered);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE_BODY(S)                                                                           \
    {                                                                                              \
        constexpr int smem = bwd_smem_bytes<TX>(S, kBwdRms);                                       \
        GBN_RMS_LAUNCH(rms_bwd_fast, S, smem, xp, dyp, w, pt, rstd, dxp, ws, M, N, eps, inv_n,     \
                       L.nblocks, L.fault, gemma);                                                 \
    }
#define GBN_CASE(S)                                                                                \
    case S:                                                                                        \
        GBN_CASE_BODY(S)                                                                           \
        break;
        GBN_CASE(0) GBN_CASE(1) GBN_CASE(2) GBN_CASE(3) GBN_CASE(4) GBN_CASE(5)
        GBN_CASE(6) GBN_CASE(7) GBN_CASE(8) GBN_CASE(9) GBN_CASE(11)
        GBN_CASE(12) GBN_CASE(14) GBN_CASE(15) GBN_CASE(19) GBN_CASE(23)
        GBN_CASE(17)
#undef GBN_CASE
#undef GBN_CASE_BODY
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}
#undef GBN_RMS_LAUNCH

}  // namespace

cudaError_t launch_rms_bwd(const Launch& L, int xt, int pt, const void* x, const void* dy,
                           const void* w, const float* rstd, void* dx, float* ws, int64_t M,
                           int N, float eps, int variant)
{
    if (xt == kF32) return bwd_dispatch<float>(L, pt, x, dy, w, rstd, dx, ws, M, N, eps, variant);
    if (xt == kF16) return bwd_dispatch<__half>(L, pt, x, dy, w, rstd, dx, ws, M, N, eps, variant);
    return bwd_dispatch<__nv_bfloat16>(L, pt, x, dy, w, rstd, dx, ws, M, N, eps, variant);
}

}  // namespace gbn
