// common.cuh -- device helpers shared by the DyT, LayerNorm and RMSNorm kernels.
//
// Data movement: every hot kernel streams 16-byte vectors (8 bf16 or 4 f32)
// with evict-first cache hints (each activation byte is touched once), keeps
// a row (or a few rows) in registers, and reduces within a "row group" of W
// threads: warp shuffles when W <= 32, shuffles plus one shared-memory step
// when a row spans several warps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gbn {

enum DType : int { kF32 = 0, kBF16 = 1 };

// ------------------------------------------------------------------ schedule
// One row group = W threads, each holding KV 16-byte vectors of a row
// (capacity W*KV*VEC columns).  A CTA of T threads holds G = T/W groups; each
// group handles UF (forward kernels that read one tensor) or UB (kernels
// that read two tensors, and LayerNorm's two-reduction forward) rows per
// iteration, so a CTA iteration covers G*U rows ("a row block").  MINB CTAs
// per SM stay resident; the register budget follows from it through
// __launch_bounds__.  The per-row summation order depends only on (W, KV),
// never on U, so a forward and a backward with different U reduce a row
// identically.
struct SchedEntry {
    int max_nvec, W, KV, UF, UB, T, MINB;
};

constexpr int kNumSched = 11;
constexpr SchedEntry kSched[kNumSched] = {
    {1, 1, 1, 4, 2, 256, 3},     {2, 2, 1, 4, 2, 256, 3},     {4, 4, 1, 4, 2, 256, 3},
    {8, 8, 1, 4, 2, 256, 3},     {16, 16, 1, 4, 2, 256, 3},   {32, 32, 1, 4, 2, 256, 3},
    {64, 32, 2, 2, 2, 256, 2},   {128, 64, 2, 2, 2, 256, 2},  {256, 128, 2, 2, 2, 256, 2},
    {512, 256, 2, 2, 2, 256, 2}, {1024, 512, 2, 1, 1, 512, 1},
};
constexpr int kMaxFastVec = 1024;

// Threads per CTA and warps per CTA of the general (any width, any
// alignment) kernels, which give every warp one row at a time.
constexpr int kGenThreads = 256;
constexpr int kGenWarps = kGenThreads / 32;

// ------------------------------------------------------------- vector types
template <typename TX> struct Vec;
template <> struct Vec<float> { static constexpr int kN = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int kN = 8; };

__device__ __forceinline__ uint4 ld_stream(const void* p)
{
    return __ldcs(static_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_stream(void* p, const uint4& v)
{
    __stcs(static_cast<uint4*>(p), v);
}

__device__ __forceinline__ void unpack(const uint4& u, float (&f)[4])
{
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
}

// bfloat16 is the upper half of a float32; element 2k sits in the low half
// of 32-bit word k.
__device__ __forceinline__ void unpack(const uint4& u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[2 * k] = __uint_as_float(w[k] << 16);
        f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 pack(const float (&f)[4])
{
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    uint32_t r;
    memcpy(&r, &h, sizeof r);
    return r;
}

__device__ __forceinline__ uint4 pack(const float (&f)[8])
{
    return make_uint4(pack2_bf16(f[0], f[1]), pack2_bf16(f[2], f[3]), pack2_bf16(f[4], f[5]),
                      pack2_bf16(f[6], f[7]));
}

// Scalar access (general path).
__device__ __forceinline__ float ld1(const float* p, int64_t i) { return __ldcs(p + i); }
__device__ __forceinline__ float ld1(const __nv_bfloat16* p, int64_t i)
{
    return __bfloat162float(__ldcs(p + i));
}
__device__ __forceinline__ void st1(float* p, int64_t i, float v) { __stcs(p + i, v); }
__device__ __forceinline__ void st1(__nv_bfloat16* p, int64_t i, float v)
{
    __stcs(p + i, __float2bfloat16_rn(v));
}

// Round a float32 value to the activation dtype's precision (identity for f32).
template <typename TX> __device__ __forceinline__ float round_x(float v);
template <> __device__ __forceinline__ float round_x<float>(float v) { return v; }
template <> __device__ __forceinline__ float round_x<__nv_bfloat16>(float v)
{
    return __bfloat162float(__float2bfloat16_rn(v));
}

// Parameters (gamma, beta, alpha, weight) are f32 or bf16 per a runtime code.
__device__ __forceinline__ float ld_param(const void* p, int pt, int64_t j)
{
    if (pt == kF32) return static_cast<const float*>(p)[j];
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[j]);
}

__device__ __forceinline__ void st_param(void* p, int pt, int64_t j, float v)
{
    if (pt == kF32)
        static_cast<float*>(p)[j] = v;
    else
        static_cast<__nv_bfloat16*>(p)[j] = __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------- reductions
// Sum across the 32 lanes of a warp by an xor butterfly.  Every lane ends
// with the same bits: at each step a lane adds the same two partial sums as
// its partner, and float addition is commutative.
template <int WIDTH, int NV>
__device__ __forceinline__ void butterfly(float (&v)[NV])
{
#pragma unroll
    for (int off = WIDTH / 2; off >= 1; off >>= 1) {
#pragma unroll
        for (int k = 0; k < NV; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], off);
    }
}

// Shared memory a group all-reduce of NV values needs (floats), for a CTA
// of T threads in groups of W.
template <int W, int T, int NV>
struct GroupRed {
    static constexpr int kWarps = W / 32;
    static constexpr int kG = T / W;
    static constexpr int kFloats = (W > 32) ? 2 * kG * kWarps * NV : 1;
};

// All-reduce NV values over the W threads of a row group.  W <= 32: the
// group is an aligned slice of a warp and the butterfly stays inside it.
// W > 32: butterfly per warp, then every thread sums the warps' results in
// warp order from a double-buffered shared slot (one __syncthreads per call;
// every thread of the CTA must make the same sequence of calls).
template <int W, int T, int NV>
__device__ __forceinline__ void group_allreduce(float (&v)[NV], float* red, int& parity)
{
    if constexpr (W <= 32) {
        butterfly<W, NV>(v);
    } else {
        constexpr int kWarps = W / 32;
        constexpr int kG = T / W;
        butterfly<32, NV>(v);
        const int lane = threadIdx.x & 31;
        const int g = threadIdx.x / W;
        const int wig = (threadIdx.x % W) >> 5;
        float* slot = red + (parity * kG + g) * kWarps * NV;
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < NV; ++k) slot[wig * NV + k] = v[k];
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            float s = slot[k];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) s += slot[w * NV + k];
            v[k] = s;
        }
        parity ^= 1;
    }
}

// Sum one float per thread over the whole CTA in a fixed order (butterfly
// per warp, then warps in index order).  Result valid in thread 0.
template <int T>
__device__ __forceinline__ float cta_sum(float v, float* red /* >= T/32 floats */)
{
    float a[1] = {v};
    butterfly<32, 1>(a);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a[0];
    __syncthreads();
    float s = 0.f;
    if (threadIdx.x == 0) {
        s = red[0];
#pragma unroll
        for (int w = 1; w < T / 32; ++w) s += red[w];
    }
    __syncthreads();
    return s;
}

// Write the CTA's per-column partial sums of one quantity to its workspace
// row.  acc holds, for this thread, columns (kv*W + l)*VEC + e.  With more
// than one group per CTA the groups' values are summed in group order
// through shared memory (buf: G*W*KV*VEC floats); one group writes directly.
template <int W, int KV, int VEC, int T>
__device__ __forceinline__ void cta_store_columns(const float (&acc)[KV][VEC], float* buf,
                                                  float* __restrict__ out_row, int N)
{
    constexpr int kG = T / W;
    constexpr int kCap = W * KV * VEC;
    const int g = threadIdx.x / W;
    const int l = threadIdx.x % W;
    if constexpr (kG == 1) {
#pragma unroll
        for (int kv = 0; kv < KV; ++kv)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int c = (kv * W + l) * VEC + e;
                if (c < N) out_row[c] = acc[kv][e];
            }
    } else {
#pragma unroll
        for (int kv = 0; kv < KV; ++kv)
#pragma unroll
            for (int e = 0; e < VEC; ++e) buf[g * kCap + (kv * W + l) * VEC + e] = acc[kv][e];
        __syncthreads();
        for (int c = threadIdx.x; c < kCap && c < N; c += T) {
            float s = buf[c];
#pragma unroll 4
            for (int gg = 1; gg < kG; ++gg) s += buf[gg * kCap + c];
            out_row[c] = s;
        }
        __syncthreads();
    }
}

}  // namespace gbn
