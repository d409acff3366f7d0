// rmsnorm.cuh -- shared parts of the RMSNorm forward (rmsnorm.cu) and
// backward (rmsnorm_bwd.cu): row helpers and the launch macros.
//
// The Llama expression (variant 0):
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
// The weight-first expressions (variant 1, and Gemma's 1 + w as variant 2)
// round only their outputs: the fast kernels' kWF instances use the float32
// formulas for every activation dtype.
#pragma once

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
        const float f = ld1c(xr, c);
        v[0] = fmaf(f, f, v[0]);
    }
    butterfly<32, 1>(v);
    return rsqrtf(fmaf(v[0], inv_n, eps));
}

// The row-batched kernels' r of a row: this lane's sum of squares of its
// units in unit order (units past the row's end are zeros), then the warp
// butterfly (one butterfly for several rows adds each value in the same
// order), then rsqrt.  The forward and the backward's recomputation share
// these, so both give the same bits.
template <int KMAX, int E>
__device__ __forceinline__ float batch_sumsq(const float (&v)[KMAX][E])
{
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) s = fmaf(v[k][e], v[k][e], s);
    return s;
}
template <int RB>
__device__ __forceinline__ void batch_rstd(float (&s)[RB], float eps, float inv_n)
{
    butterfly<32, RB>(s);
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) s[rr] = rsqrtf(fmaf(s[rr], inv_n, eps));
}

// Launch schedule S of a fast kernel: the weight-first instance (kWF) for
// the weight-first and Gemma expressions with 16-bit activations (with
// float32 activations both expressions are the same float32 arithmetic),
// and the scattered-row instance (kRows) for inputs that follow row maps.
#define GBN_RMS_LAUNCH(KERNEL, S, SMEM, ...)                                                       \
    with_mode(L.in_mode, [&](auto m_) {                                                            \
        constexpr int kIn_ = decltype(m_)::value;                                                  \
        if constexpr (is16<TX>()) {                                                                \
            if (variant != 0) {                                                                    \
                ring_attributes<KERNEL<TX, S, true, kIn_>>(SMEM);                                  \
                launch_pdl(KERNEL<TX, S, true, kIn_>, L.grid, kSched[S].T, SMEM, L.stream,         \
                           __VA_ARGS__, L.maps);                                                   \
                return;                                                                            \
            }                                                                                      \
        }                                                                                          \
        ring_attributes<KERNEL<TX, S, false, kIn_>>(SMEM);                                         \
        launch_pdl(KERNEL<TX, S, false, kIn_>, L.grid, kSched[S].T, SMEM, L.stream, __VA_ARGS__,   \
                   L.maps);                                                                        \
    })

}  // namespace
}  // namespace gbn
