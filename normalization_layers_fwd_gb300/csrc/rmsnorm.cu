// rmsnorm.cu -- RMSNorm forward: the fast (bulk-copy ring) and general
// kernels, their dispatch and launch_rms_fwd.  The rounding points and the
// expression variants are described in rmsnorm.cuh.
#include "rmsnorm.cuh"

namespace gbn {
namespace {

// ------------------------------------------------------------ fast forward
template <typename TX, int S, bool kWF, int kIn>
__global__ void __launch_bounds__(kSched[S].T, kind_minb(S, kFwdNorm))
    rms_fwd_fast(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ w,
                 int pt, float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n,
                 int64_t nblocks, unsigned* fault, int gemma, RowMaps maps)
{
    grid_dependency_sync();
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

    Ring<1, kind_stages(S, kFwdNorm), kIn == kInRows> rg;
    rg.src[0] = reinterpret_cast<const unsigned char*>(x);
    if constexpr (kIn == kInRows) rg.map[0] = maps.m[0];
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
    // rows wider than a warp: the row reduction's barrier releases the slot
    ring_loop<(W > 32)>(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
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
            const int64_t orow = stat_row<kIn>(maps, row0 + u * G);
            TX* const yr = kIn == kInStorage ? y + orow * N + l * VEC : yb + u * grow;
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
                st_stream_if(okr[u] && colok[j], yr + j * W * VEC, out);
            }
            if (rstd) st_f32_if(lead && okr[u], rstd + orow, rs);
        }
        row0 += rstride;
        yb += rstride * N;
    });
}

template <typename TX>
__global__ void __launch_bounds__(kGenThreads)
    rms_fwd_general(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ w,
                    int pt, float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n,
                    int variant, RowMaps maps, int scattered)
{
    grid_dependency_sync();
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kGenWarps;
    for (int64_t r = blockIdx.x * (int64_t)kGenWarps + (threadIdx.x >> 5); r < M; r += nw) {
        const TX* xr = in_row(x, maps, 0, scattered, r, N);
        const float rs = warp_row_rstd(xr, N, lane, eps, inv_n);
        for (int c = lane; c < N; c += 32) {
            const float xh = ld1c(xr, c) * rs;
            const float n = variant == 0 ? round_x<TX>(xh) : xh;
            st1(y, r * N + c, rms_weight(w, pt, c, variant) * n);
        }
        if (rstd && lane == 0) rstd[r] = rs;
    }
}

// ------------------------------------------------------ row-batched path
// Rows whose byte length is not a multiple of 16 (common.cuh, "row-batched"):
// blocks of R rows through the ring, one warp per row.
template <typename TX, int E, int KMAX>
__global__ void __launch_bounds__(kBatchThreads, batch_minb(false))
    rms_fwd_batch(const TX* __restrict__ x, TX* __restrict__ y, const void* __restrict__ w,
                  int pt, float* __restrict__ rstd, int64_t M, int N, float eps, float inv_n,
                  int variant, int64_t nblocks, int R, unsigned* fault)
{
    grid_dependency_sync();
    using U = Unit<TX, E>;
    extern __shared__ __align__(128) unsigned char dsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nu = N / E;
    const int rb = N * (int)sizeof(TX);
    bool uok[KMAX];
    float wv[KMAX][E];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        uok[k] = lane + 32 * k < nu;
#pragma unroll
        for (int e = 0; e < E; ++e)
            wv[k][e] = uok[k] ? rms_weight(w, pt, (lane + 32 * k) * E + e, variant) : 0.f;
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
    constexpr int RB = batch_rb(KMAX, E);
    constexpr int UB = E * (int)sizeof(TX);  // bytes of a unit
    ring_loop(rg, dsm, [&](int64_t b, int64_t k, bool alive) {
        if (!alive) return;
        const uint32_t xs = smem_u32(rg.tile(k, 0)) + lane * UB;
        const int64_t r0 = b * R;
        const int rows = (int)(M - r0 < R ? M - r0 : R);
        // RB consecutive rows a warp at once.  A whole block runs unmasked;
        // otherwise rows past the block read zeros and units past the copied
        // bytes come from global memory.
        auto pass = [&](auto masked) {
            constexpr bool kMask = decltype(masked)::value;
            for (int i0 = warp * RB; i0 < rows; i0 += kBatchWarps * RB) {
                float v[RB][KMAX][E], rs[RB];
#pragma unroll
                for (int rr = 0; rr < RB; ++rr) {
                    const int i = i0 + rr;
#pragma unroll
                    for (int kk = 0; kk < KMAX; ++kk) {
                        typename U::W wd{};
                        if constexpr (kMask) {
                            const int64_t gi = (r0 + i) * N + (lane + 32 * kk) * E;
                            if (i < rows && uok[kk])
                                wd = gi < tail ? U::lds(xs + i * rb + kk * 32 * UB) : U::ld(x + gi);
                        } else {
                            if (uok[kk]) wd = U::lds(xs + i * rb + kk * 32 * UB);
                        }
                        U::unpack(wd, v[rr][kk]);
                    }
                    rs[rr] = batch_sumsq<KMAX, E>(v[rr]);
                }
                batch_rstd<RB>(rs, eps, inv_n);
#pragma unroll
                for (int rr = 0; rr < RB; ++rr) {
                    const int i = i0 + rr;
                    if (kMask && i >= rows) break;  // the same for the whole warp
                    const int64_t r = r0 + i;
                    TX* const yr = y + r * N + lane * E;
#pragma unroll
                    for (int kk = 0; kk < KMAX; ++kk) {
                        float o[E];
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            const float xh = v[rr][kk][e] * rs[rr];
                            o[e] = wv[kk][e] * (variant == 0 ? round_x<TX>(xh) : xh);
                        }
                        if (uok[kk]) U::st(yr + kk * 32 * E, U::pack(o));
                    }
                    if (rstd && lane == 0) rstd[r] = rs[rr];
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

template <typename TX>
cudaError_t fwd_dispatch(const Launch& L, int pt, const void* x, const void* w, void* y,
                         float* rstd, int64_t M, int N, float eps, int variant)
{
    const TX* xp = static_cast<const TX*>(x);
    TX* yp = static_cast<TX*>(y);
    const float inv_n = (float)(1.0 / (double)N);
    const int gemma = variant == 2;
    if (L.batch) {
        constexpr int smem = batch_smem(1);
        if (!with_batch(L.E, L.KMAX, [&](auto e_, auto k_) {
                constexpr int E_ = decltype(e_)::value, K_ = decltype(k_)::value;
                ring_attributes<rms_fwd_batch<TX, E_, K_>>(smem);
                launch_pdl(rms_fwd_batch<TX, E_, K_>, L.grid, kBatchThreads, smem, L.stream, xp,
                           yp, w, pt, rstd, M, N, eps, inv_n, variant, L.nblocks, L.R, L.fault);
            }))
            return cudaErrorInvalidValue;
        return cudaGetLastError();
    }
    if (!L.fast) {
        launch_pdl(rms_fwd_general<TX>, L.grid, kGenThreads, 0, L.stream,
            xp, yp, w, pt, rstd, M, N, eps, inv_n, variant, L.maps, L.scattered);
        return cudaGetLastError();
    }
    switch (L.sid) {
#define GBN_CASE_BODY(S)                                                                           \
    {                                                                                              \
        constexpr int smem = ring_smem_bytes(S, kFwdNorm, 1);                                      \
        GBN_RMS_LAUNCH(rms_fwd_fast, S, smem, xp, yp, w, pt, rstd, M, N, eps, inv_n, L.nblocks,    \
                       L.fault, gemma);                                                            \
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

cudaError_t launch_rms_fwd(const Launch& L, int xt, int pt, const void* x, const void* w, void* y,
                           float* rstd, int64_t M, int N, float eps, int variant)
{
    if (xt == kF32) return fwd_dispatch<float>(L, pt, x, w, y, rstd, M, N, eps, variant);
    if (xt == kF16) return fwd_dispatch<__half>(L, pt, x, w, y, rstd, M, N, eps, variant);
    return fwd_dispatch<__nv_bfloat16>(L, pt, x, w, y, rstd, M, N, eps, variant);
}

}  // namespace gbn
