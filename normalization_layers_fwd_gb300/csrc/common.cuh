// common.cuh -- device helpers shared by the DyT, LayerNorm and RMSNorm kernels.
//
// Data movement: every hot kernel streams 16-byte vectors (8 bf16 or f16, or 4 f32)
// with evict-first cache hints (each activation byte is touched once), keeps
// a row (or a few rows) in registers, and reduces within a "row group" of W
// threads: warp shuffles when W <= 32, shuffles plus one shared-memory step
// when a row spans several warps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>
#include <utility>

#include "ctx_cache.h"
#include "internal.h"

namespace gbn {

enum DType : int { kF32 = 0, kBF16 = 1, kF16 = 2 };

// ------------------------------------------------------------------ schedule
// One row group = W threads, each holding KV 16-byte vectors of a row
// (capacity W*KV*VEC columns).  A CTA of T threads holds G = T/W groups; each
// group handles UF (forward kernels, which read one tensor) or UB (backward
// kernels, which read two) rows per iteration, so a CTA iteration covers
// G*U rows ("a row block").  MINB CTAs
// per SM stay resident; the register budget follows from it through
// __launch_bounds__.  The per-row summation order depends only on (W, KV),
// never on U, so a forward and a backward with different U reduce a row
// identically.
struct SchedEntry {
    int max_nvec, W, T, KV;
};

// Schedules 0-11: one 16-byte vector per thread per row: a row of nvec
// vectors takes W = next_pow2(nvec) threads, so register pressure stays flat
// from N = 8 to N = 8192 bf16.  A CTA has T = max(256, W) threads.
// Rows of exactly 3 vectors (bf16 N = 24, the tall-narrow LayerNorm of the
// torch-xpu-ops page) take segmented groups of W = 3 lanes, 10 per warp,
// instead of 4-lane groups with a lane idle.
// Schedules 12-14: wide rows (257-1024 vectors) held by 256 or 512 threads
// with KV = 2 or 4 vectors each (vector l + j*W for j < KV), one row per
// CTA.  Against schedules 10-11 they divide the per-row reduction and
// barrier cost by KV; at 256 threads two independent CTAs share an SM.
// Schedule 17: rows of 1025-2048 vectors (bf16 N <= 16384, f32 N <= 8192)
// held by 512 threads with KV = 4 vectors each, one row per CTA, one CTA
// per SM.  The backwards keep the row's xhat (and g, dn) in registers as
// well as their column accumulators, which fits the 128-register budget
// only with float32 activations (half the elements per vector); the
// planner gives it to the 16-bit backwards never, and to the 16-bit RMSNorm
// forward never either (its backward must reduce a row in its order).
// Schedules 15-16: rows of 33-64 and 65-128 vectors held by one warp with
// KV = 2 or 4 vectors per lane, 8 rows per pass: the row reductions stay
// inside the warp (shuffles, no barrier), where one vector per lane would
// spread a row over 2-4 warps and a __syncthreads per reduction.  They pay
// where a kernel reduces more than once per row (the LayerNorm backward
// takes 15, the LayerNorm forward 16).
// Schedules 18-23 complete two families for the LayerNorm kernels, which
// reduce twice per row: 4 vectors per lane for the forward (W = capacity / 4:
// 22, 20, 16, 18, 21, 13 for rows of up to 32 ... 1024 vectors) and 2 for
// the backward (W = capacity / 2: 15, 23, 19, 12, 14), so each row's
// reductions span a quarter or half as many lanes and warps as one vector
// per lane would.  Measured on GB300 (fraction of measured copy, bf16,
// against the one-vector schedule or schedule 12): forward N = 256 0.947 ->
// 0.974, 512 0.850 -> 0.970, 2048 0.860 -> 0.932, 4096 0.904 -> 0.937,
// float32 N = 2048 0.908 -> 1.002; backward N = 1024 0.893 -> 0.913, 2048
// 0.879 -> 0.906.
// Which kernel takes which is decided per kernel by the planner (api.cu),
// within each kernel's register budget.
constexpr int kNumSched = 24;
constexpr int kNumSched1 = 12;  // the one-vector schedules
constexpr SchedEntry kSched[kNumSched] = {
    {1, 1, 256, 1},     {2, 2, 256, 1},     {3, 3, 256, 1},     {4, 4, 256, 1},
    {8, 8, 256, 1},     {16, 16, 256, 1},   {32, 32, 256, 1},   {64, 64, 256, 1},
    {128, 128, 256, 1}, {256, 256, 256, 1}, {512, 512, 512, 1}, {1024, 1024, 1024, 1},
    {512, 256, 256, 2}, {1024, 256, 256, 4}, {1024, 512, 512, 2},
    {64, 32, 256, 2},   {128, 32, 256, 4},  {2048, 512, 512, 4},
    {256, 64, 256, 4},  {256, 128, 256, 2}, {64, 16, 256, 4},   {512, 128, 256, 4},
    {32, 8, 256, 4},    {128, 64, 256, 2},
};

// Row groups of a power-of-two width tile the CTA; a width that is not a
// power of two packs floor(32/W) groups per warp and leaves the rest of the
// warp's lanes idle.
constexpr bool seg_groups(int W) { return (W & (W - 1)) != 0; }
constexpr int groups_per_cta(int W, int T) { return seg_groups(W) ? (T / 32) * (32 / W) : T / W; }

template <int W>
__device__ __forceinline__ int grp()
{
    if constexpr (seg_groups(W))
        return (threadIdx.x >> 5) * (32 / W) + (threadIdx.x & 31) / W;
    else
        return threadIdx.x / W;
}
template <int W>
__device__ __forceinline__ int lan()
{
    if constexpr (seg_groups(W))
        return (threadIdx.x & 31) % W;
    else
        return threadIdx.x % W;
}
// false for the idle lanes of a segmented warp
template <int W>
__device__ __forceinline__ bool in_group()
{
    if constexpr (seg_groups(W))
        return (threadIdx.x & 31) < (32 / W) * W;
    else
        return true;
}

// Launch traits per kernel kind: U rows per thread per row block, CTAs per
// SM (registers through __launch_bounds__, shared memory through the ring),
// and ring depth.  Row blocks of T/W * U rows are 8-32 KB per staged tensor.
// DyT's kernels have no row reduction and the most arithmetic per byte, so
// they take the largest blocks; the backward kernels stage two tensors and
// keep more per-row state, so they run 2 CTAs per SM.  At the widest rows
// (512 threads at 2 CTAs per SM, 64 registers) the backwards keep one row
// per thread: two spill.
// kFwdNorm is the RMSNorm forward; the LayerNorm forward (kFwdLN) shares its
// traits except at 2 vectors per thread, where it runs 3 CTAs per SM.
enum KernelKind : int {
    kFwdDyT = 0, kFwdNorm = 1, kFwdLN = 2, kBwdLN = 3, kBwdDyT = 4, kBwdRms = 5
};

constexpr bool is_bwd(int kind) { return kind >= kBwdLN; }

constexpr int kind_U1(int S, int kind)
{
    return kind == kBwdDyT ? (kSched[S].T == 512 ? 1 : 2)
           : is_bwd(kind)  ? (kSched[S].T == 256 ? 2 : 1)
           : kind == kFwdDyT && kSched[S].T == 256 ? 4
                                                   : 2;
}
// Several vectors per thread take proportionally fewer rows.
constexpr int kind_U(int S, int kind)
{
    return kind_U1(S, kind) / kSched[S].KV > 1 ? kind_U1(S, kind) / kSched[S].KV : 1;
}
// RMSNorm's backward keeps the least per-row state (84 registers), so it
// fits 3 CTAs per SM and more bytes in flight.  DyT's backward at 512
// threads needs about 80 registers (three column accumulators besides the
// row), so it runs one CTA per SM rather than spill at two.
constexpr int kind_minb(int S, int kind)
{
    return kSched[S].KV > 1 ? (kSched[S].T == 512 ? 1 : kind == kFwdLN && kSched[S].KV == 2 ? 3 : 2)
           : kSched[S].T == 1024 ? 1
           : kSched[S].T == 512 ? (kind == kBwdDyT ? 1 : 2)
           : kind == kBwdRms    ? 3
           : is_bwd(kind)       ? 2
           : kind == kFwdDyT    ? 3
                                : 4;
}
// The lean backward form: 16-bit rows of 1025-2048 vectors (schedule 17, 4
// vectors a thread), whose row and parameters do not fit the registers next
// to the column accumulators.  Those kernels keep only the accumulators in
// registers, read the row from the ring slot again after the row reduction,
// and read the parameters from L1 at each use.
template <typename TX>
constexpr bool lean_bwd(int S)
{
    return sizeof(TX) == 2 && S == 17;
}

// Ring depth.  Every SM keeps (CTAs x stages) row blocks of loads in
// flight.  The one-vector forward kernels at 256 threads (4 or 3 CTAs per
// SM) stream best with 2 stages: at 4 the whole GPU holds about 20 MB of
// outstanding bulk copies and the forward sweep loses 5-15%.  The wide-row
// RMSNorm forward wants 4; at 256 threads, the LayerNorm forward at 4
// vectors per thread and the DyT forward at 2 or 4 want 2 (DyT N = 4096
// 0.909 -> 0.920 of measured copy).  The backward kernels,
// which spend longer per block, want 3 (RMSNorm) or 4; the RMSNorm backward
// at 512 threads (one CTA per SM) 4 (N = 8192: 0.91 -> 0.95 of measured
// copy, where 4 stages cost the 256-thread schedules 1-4%).  Backward slots
// of 4 vectors per thread (32 KB per tensor) take 3.
constexpr int kind_stages(int S, int kind)
{
    return !is_bwd(kind) ? (kSched[S].KV == 1 ? (kSched[S].T == 256 ? 2 : 4)
                            : kSched[S].T == 256 && (kind == kFwdDyT ||
                                                      (kind == kFwdLN && kSched[S].KV == 4))
                                ? 2
                                : 4)
           : kSched[S].KV == 4                      ? 3
           : kind == kBwdRms                        ? (kSched[S].T == 512 ? 4 : 3)
           : kind == kBwdDyT && kSched[S].T == 1024 ? 3
                                                    : 4;
}

// Bytes of one ring slot for one staged tensor, and of the whole dynamic
// shared memory a kernel with NT staged tensors needs (barriers first).
constexpr int slot_bytes(int S, int kind)
{
    return groups_per_cta(kSched[S].W, kSched[S].T) * kSched[S].W * kSched[S].KV *
           kind_U(S, kind) * 16;
}
constexpr int ring_smem_bytes(int S, int kind, int NT)
{
    return 128 + kind_stages(S, kind) * NT * slot_bytes(S, kind);
}

// A backward kernel's ring depth and dynamic shared memory.  The lean form
// runs a 2-stage ring and keeps the row's parameters, as float32, in shared
// memory past the ring (kLeanParams floats, loaded once per CTA): read from
// L1 at each use they cost a scattered load per element pair.
constexpr int kLeanParams = 2048 * 8;  // the widest lean row, 2048 16-bit vectors
template <typename TX>
constexpr int bwd_stages(int S, int kind)
{
    return lean_bwd<TX>(S) ? 2 : kind_stages(S, kind);
}
template <typename TX>
constexpr int bwd_ring_bytes(int S, int kind)
{
    return 128 + bwd_stages<TX>(S, kind) * 2 * slot_bytes(S, kind);
}
template <typename TX>
constexpr int bwd_smem_bytes(int S, int kind)
{
    return bwd_ring_bytes<TX>(S, kind) + (lean_bwd<TX>(S) ? kLeanParams * 4 : 0);
}

// Threads per CTA and warps per CTA of the general (any width, any
// alignment) kernels, which give every warp one row at a time.
constexpr int kGenThreads = 256;
constexpr int kGenWarps = kGenThreads / 32;
// Columns of parameter-gradient partials a general backward warp accumulates
// in shared memory (8 warps x 1536 floats = 48 KB per CTA); wider partial
// rows accumulate in the warp's workspace row in global memory.
constexpr int kGenCols = 1536;

// --------------------------------------------------- row-batched (any width)
// Contiguous rows whose byte length is not a multiple of 16 cannot take the
// 16-byte vectors of the schedules above.  The row-batched kernels still
// stream them through the bulk-copy ring: a block of R rows, R a multiple of
// 8, spans R * row_bytes bytes, a multiple of 16 for every element size, so
// with a 16-byte aligned base every full block starts and ends on a 16-byte
// boundary and moves as one bulk copy (the last block's final bytes below a
// 16-byte multiple come from global memory).  In shared memory a warp takes
// one row at a time and lane l reads units l, l + 32, ... of it: a unit is an
// element pair when rows hold whole pairs, else one element.  Row
// reductions are warp butterflies; a backward's column sums stay in
// registers and are combined across the CTA's warps in warp order at the
// end.  Widths up to batch_max_units(E) * 32 units, and rows of at most
// batch_slot / 8 bytes.
constexpr int kBatchThreads = 256;
constexpr int kBatchWarps = kBatchThreads / 32;
// KMAX, the units a lane holds per row: up to 4, so rows up to 256 elements
// in pairs and 128 single elements.  8 units a lane are left out: ptxas 13.0
// crashes on the LayerNorm kernels' 8-pair instance, and a build whose
// 8-element LayerNorm instances ran unchecked faulted once on GB300 (the
// same sequence with every access bounds-checked ran clean).
constexpr int batch_max_units(int) { return 4; }
// Rows a warp takes at once (their reductions share one butterfly, so the
// shuffle chains of RB rows overlap), by the values a lane holds per row
// (KMAX * E): 4 rows up to 2 values, 2 up to 6, 1 at 8 (more spill in the
// backwards).  A ring block holds a multiple of 8 * RB rows where the slot
// allows.
constexpr int batch_rb(int KMAX, int E) { return KMAX * E <= 2 ? 4 : KMAX * E <= 6 ? 2 : 1; }
static_assert(8 % batch_rb(1, 1) == 0 && 8 % batch_rb(3, 2) == 0 && 8 % batch_rb(4, 2) == 0,
              "a block of R rows, R a multiple of 8, holds whole groups of RB rows");
// Bytes per staged tensor per ring slot and ring depth, by the tensors a
// kernel stages (NT: 1 for a forward, 2 for a backward): 24 KB x 2 and
// 16 KB x 2, so that a block holds several row groups per warp (a 260-byte
// row fills 80 or 48 rows of them, where 8 KB held 16: one row group per
// warp between ring barriers).  Measured against 8 KB x 4 (fraction of
// measured copy, bf16 N = 130, forward / backward): DyT 0.54 / 0.49 ->
// 0.63 / 0.53, LayerNorm 0.48 / 0.55 -> 0.63 / 0.66, RMSNorm 0.61 / 0.47 ->
// 0.84 / 0.55; 16 KB and 12 KB slots 3 deep came in between.
constexpr int batch_slot(int NT) { return NT == 1 ? 24576 : 16384; }
constexpr int batch_stages(int) { return 2; }
// CTAs per SM: 4 for a forward (one staged tensor), 3 for a backward.
constexpr int batch_minb(bool bwd) { return bwd ? 3 : 4; }
constexpr int batch_smem(int NT) { return 128 + batch_stages(NT) * NT * batch_slot(NT); }

// One unit of E consecutive elements (E = 2: a pair, E = 1: one element),
// moved as one word: loaded through L1 (ld.global.ca, coherent with the
// previous kernel's writes once griddepcontrol.wait has returned) or from
// the ring slot by shared-memory address (lds), and stored with the
// streaming hint.
template <typename TX, int E> struct Unit;
template <> struct Unit<float, 1> {
    using W = float;
    static __device__ __forceinline__ W ld(const float* p) { return __ldca(p); }
    static __device__ __forceinline__ W lds(uint32_t a)
    {
        float v;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
        return v;
    }
    static __device__ __forceinline__ void st(float* p, W w) { __stcs(p, w); }
    static __device__ __forceinline__ void unpack(W w, float (&v)[1]) { v[0] = w; }
    static __device__ __forceinline__ W pack(const float (&v)[1]) { return v[0]; }
};
template <> struct Unit<float, 2> {
    using W = float2;
    static __device__ __forceinline__ W ld(const float* p)
    {
        return __ldca(reinterpret_cast<const float2*>(p));
    }
    static __device__ __forceinline__ W lds(uint32_t a)
    {
        float2 v;
        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
        return v;
    }
    static __device__ __forceinline__ void st(float* p, W w)
    {
        __stcs(reinterpret_cast<float2*>(p), w);
    }
    static __device__ __forceinline__ void unpack(W w, float (&v)[2])
    {
        v[0] = w.x;
        v[1] = w.y;
    }
    static __device__ __forceinline__ W pack(const float (&v)[2])
    {
        return make_float2(v[0], v[1]);
    }
};
template <typename TX> struct Unit16 {
    static __device__ __forceinline__ float to_f(unsigned short h)
    {
        if constexpr (std::is_same<TX, __half>::value)
            return __half2float(__ushort_as_half(h));
        else
            return __uint_as_float((unsigned)h << 16);
    }
    static __device__ __forceinline__ unsigned short from_f(float v)
    {
        if constexpr (std::is_same<TX, __half>::value)
            return __half_as_ushort(__float2half_rn(v));
        else
            return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
};
template <typename TX> struct Unit16x1 {
    using W = unsigned short;
    static __device__ __forceinline__ W ld(const TX* p)
    {
        return __ldca(reinterpret_cast<const unsigned short*>(p));
    }
    static __device__ __forceinline__ W lds(uint32_t a)
    {
        unsigned short v;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
        return v;
    }
    static __device__ __forceinline__ void st(TX* p, W w)
    {
        __stcs(reinterpret_cast<unsigned short*>(p), w);
    }
    static __device__ __forceinline__ void unpack(W w, float (&v)[1])
    {
        v[0] = Unit16<TX>::to_f(w);
    }
    static __device__ __forceinline__ W pack(const float (&v)[1])
    {
        return Unit16<TX>::from_f(v[0]);
    }
};
template <typename TX> struct Unit16x2 {
    using W = unsigned int;
    static __device__ __forceinline__ W ld(const TX* p)
    {
        return __ldca(reinterpret_cast<const unsigned int*>(p));
    }
    static __device__ __forceinline__ W lds(uint32_t a)
    {
        unsigned v;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
        return v;
    }
    static __device__ __forceinline__ void st(TX* p, W w)
    {
        __stcs(reinterpret_cast<unsigned int*>(p), w);
    }
    static __device__ __forceinline__ void unpack(W w, float (&v)[2])
    {
        v[0] = Unit16<TX>::to_f((unsigned short)(w & 0xffffu));
        v[1] = Unit16<TX>::to_f((unsigned short)(w >> 16));
    }
    static __device__ __forceinline__ W pack(const float (&v)[2])
    {
        // one two-lane conversion, round to nearest even (element 0 low)
        if constexpr (std::is_same<TX, __half>::value) {
            const __half2 h = __floats2half2_rn(v[0], v[1]);
            return *reinterpret_cast<const unsigned*>(&h);
        } else {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[0], v[1]);
            return *reinterpret_cast<const unsigned*>(&h);
        }
    }
};
template <> struct Unit<__nv_bfloat16, 1> : Unit16x1<__nv_bfloat16> {};
template <> struct Unit<__nv_bfloat16, 2> : Unit16x2<__nv_bfloat16> {};
template <> struct Unit<__half, 1> : Unit16x1<__half> {};
template <> struct Unit<__half, 2> : Unit16x2<__half> {};

// Call f(std::integral_constant<int, E>, std::integral_constant<int, KMAX>)
// for a row-batched launch (host side).
template <class F>
inline bool with_batch(int E, int KMAX, F&& f)
{
    using std::integral_constant;
    auto k = [&](auto e) {
        switch (KMAX) {
            case 1: f(e, integral_constant<int, 1>{}); return true;
            case 2: f(e, integral_constant<int, 2>{}); return true;
            case 3: f(e, integral_constant<int, 3>{}); return true;
            case 4: f(e, integral_constant<int, 4>{}); return true;
            default: return false;
        }
    };
    return E == 2 ? k(integral_constant<int, 2>{}) : k(integral_constant<int, 1>{});
}

// ------------------------------------------------------------- vector types
template <typename TX> struct Vec;
template <> struct Vec<float> { static constexpr int kN = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int kN = 8; };
template <> struct Vec<__half> { static constexpr int kN = 8; };

// The dtype code of an activation type, and whether it is a 16-bit type.
template <typename TX>
constexpr int dtype_code()
{
    return std::is_same<TX, float>::value ? kF32 : std::is_same<TX, __half>::value ? kF16 : kBF16;
}
template <typename TX>
constexpr bool is16()
{
    return !std::is_same<TX, float>::value;
}

__device__ __forceinline__ uint4 ld_stream(const void* p)
{
    return __ldcs(static_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_stream(void* p, const uint4& v)
{
    __stcs(static_cast<uint4*>(p), v);
}

// Predicated stores: every lane issues one instruction and the predicate
// decides, so a per-lane condition costs no divergent branch.
__device__ __forceinline__ void st_stream_if(bool p, void* addr, const uint4& v)
{
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t"
        "@q st.global.cs.v4.b32 [%1], {%2, %3, %4, %5};\n\t}" ::"r"((int)p),
        "l"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}
__device__ __forceinline__ void st_f32_if(bool p, float* addr, float v)
{
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t@q st.global.f32 [%1], %2;\n\t}" ::"r"(
            (int)p),
        "l"(addr), "f"(v));
}

// Scalar access (general path).
__device__ __forceinline__ float ld1(const float* p, int64_t i) { return __ldcs(p + i); }
__device__ __forceinline__ float ld1(const __nv_bfloat16* p, int64_t i)
{
    return __bfloat162float(__ldcs(p + i));
}
__device__ __forceinline__ float ld1(const __half* p, int64_t i)
{
    return __half2float(__ldcs(p + i));
}
// Cached element loads for the general kernels, whose passes re-read a row
// (the first pass brings it into L1, the others hit there).
__device__ __forceinline__ float ld1c(const float* p, int64_t i) { return __ldg(p + i); }
__device__ __forceinline__ float ld1c(const __nv_bfloat16* p, int64_t i)
{
    return __bfloat162float(__ldg(p + i));
}
__device__ __forceinline__ float ld1c(const __half* p, int64_t i)
{
    return __half2float(__ldg(p + i));
}
__device__ __forceinline__ void st1(float* p, int64_t i, float v) { __stcs(p + i, v); }
__device__ __forceinline__ void st1(__nv_bfloat16* p, int64_t i, float v)
{
    __stcs(p + i, __float2bfloat16_rn(v));
}
__device__ __forceinline__ void st1(__half* p, int64_t i, float v)
{
    __stcs(p + i, __float2half_rn(v));
}

// Round a float32 value to the activation dtype's precision (identity for f32).
template <typename TX> __device__ __forceinline__ float round_x(float v);
template <> __device__ __forceinline__ float round_x<float>(float v) { return v; }
template <> __device__ __forceinline__ float round_x<__nv_bfloat16>(float v)
{
    return __bfloat162float(__float2bfloat16_rn(v));
}
template <> __device__ __forceinline__ float round_x<__half>(float v)
{
    return __half2float(__float2half_rn(v));
}

// Parameters (gamma, beta, alpha, weight) are f32, bf16 or f16 per a
// runtime code.
__device__ __forceinline__ float ld_param(const void* p, int pt, int64_t j)
{
    if (pt == kF32) return static_cast<const float*>(p)[j];
    if (pt == kBF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[j]);
    return __half2float(static_cast<const __half*>(p)[j]);
}

// Parameter vector p (N columns of dtype pt) into prm as float32, by all T
// threads of the CTA; the caller's next __syncthreads publishes it.
template <int T>
__device__ __forceinline__ void stage_params(float* prm, const void* p, int pt, int N)
{
    for (int c = threadIdx.x; c < N; c += T) prm[c] = ld_param(p, pt, c);
}

__device__ __forceinline__ void st_param(void* p, int pt, int64_t j, float v)
{
    if (pt == kF32)
        static_cast<float*>(p)[j] = v;
    else if (pt == kBF16)
        static_cast<__nv_bfloat16*>(p)[j] = __float2bfloat16_rn(v);
    else
        static_cast<__half*>(p)[j] = __float2half_rn(v);
}

// ---------------------------------------------------- bulk-copy ring (TMA)
// A CTA streams its row blocks through a ring of kStages shared-memory
// slots.  Thread 0 issues one 1D bulk copy (cp.async.bulk, the Tensor
// Memory Accelerator's untiled form) per staged tensor per block, with the
// slot's mbarrier expecting the bytes; every thread waits on the barrier's
// phase, reads its vectors from shared memory, and after a __syncthreads
// thread 0 refills the slot kStages blocks ahead.  Every wait is bounded:
// after kWaitCycles it records kFaultWaitTimeout in the library's fault
// word and the CTA finishes its remaining iterations without waiting,
// loading or storing, then waits (bounded again) for its copies in flight.

constexpr long long kWaitCycles = 1LL << 31;  // ~1 s at 2 GHz
constexpr unsigned kFaultWaitTimeout = 1u;

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for a barrier phase; false (and a fault bit) on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* fault,
                                          long long limit = kWaitCycles)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) {
            if (fault) atomicOr(fault, kFaultWaitTimeout);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// One 16-byte vector from shared memory, re-read at every use: each pass
// over a row reads the ring slot again rather than keeping the row in
// registers across the row reductions (volatile, so it is not merged).
__device__ __forceinline__ uint4 lds128(const void* p)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ uint4 lds128_if(bool ok, const unsigned char* p)
{
    return ok ? lds128(p) : make_uint4(0, 0, 0, 0);
}

// Where each row of a non-contiguous input starts: row r begins at byte
//   (r % n1) * s1 + ((r / n1) % n2) * s2 + (r / (n1 * n2)) * s3
// from the tensor's base (the row itself is contiguous).  A row stride is
// (n1 = M, s1 = stride); a head-major [B, S, H, D] view of [B, H, S, D]
// storage, rows ordered (b, s, h), is (H, S*D*e, S, D*e, H*S*D*e), e the
// element size.
__device__ __forceinline__ int64_t row_byte_offset(const RowMap& m, int64_t r)
{
    const int64_t q = r / m.n1;
    return (r - q * m.n1) * m.s1 + (q % m.n2) * m.s2 + (q / m.n2) * m.s3;
}

// The output row of storage row q (kInStorage), in 32-bit arithmetic:
// q < 2^31 and every output row (padded rows' included) below 2^32.
__device__ __forceinline__ int64_t out_row(const OutMap& o, int64_t q)
{
    const uint32_t uq = (uint32_t)q;
    const uint32_t q1 = (uint32_t)(((uint64_t)uq * o.ma) >> o.sa);
    const uint32_t q2 = (uint32_t)(((uint64_t)q1 * o.mb) >> o.sb);
    return (int64_t)((uq - q1 * o.a) * o.wa + (q1 - q2 * o.b) * o.wb + q2 * o.wc);
}

// A saved per-row statistic of row r, loaded through L1 with the normal L2
// policy (ld.global.ca).  Every warp of a row group reads the same value,
// and L1 serves all but the first; in storage order a 32-byte sector's
// eight values serve rows a level stride apart, far apart in time, and L2
// keeps the sector for them.  The streaming (evict-first) hint measured
// 1-4% slower in the backwards that read statistics (RMSNorm N = 2048
// 0.927 -> 0.959 of measured copy without it, LayerNorm N = 24 0.913 ->
// 0.927), and on head-major storage order 8-9%.  The load is coherent with
// the forward that wrote the statistics once griddepcontrol.wait returns.
template <int kIn>
__device__ __forceinline__ float ld_stat(const float* p, int64_t r)
{
    return __ldca(p + r);
}

// Bring the saved statistics of R rows from row r0 on into L2, one 128-byte
// line per lane of the CTA's last warp (not the ring issuer's warp, whose
// delays hold up the bulk copies); no register holds them.
__device__ __forceinline__ void prefetch_stats(const float* p, int64_t r0, int R, int64_t M)
{
    const int t = (int)threadIdx.x - (int)(blockDim.x - 32);  // the last warp's lanes
    const int64_t r = r0 + (int64_t)t * 32;
    if (t >= 0 && t * 32 < R && r < M)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p + r));
}

// The row whose outputs (and saved statistics) belong to this thread's row q.
template <int kIn>
__device__ __forceinline__ int64_t stat_row(const RowMaps& maps, int64_t q)
{
    if constexpr (kIn == kInStorage)
        return out_row(maps.o, q);
    else
        return q;
}

// Where this thread's vectors of row q go: at yb + off while rows are in
// order, else at the storage-order map's row (lvec: the thread's column).
template <int kIn, typename TX>
__device__ __forceinline__ TX* out_at(TX* yb, int64_t off, TX* y, const RowMaps& maps, int64_t q,
                                      int N, int lvec)
{
    if constexpr (kIn == kInStorage)
        return y + out_row(maps.o, q) * N + lvec;
    else
        return yb + off;
}

// Row r of input t (0: x, 1: dy) for the general kernels: r * N elements
// in, or where the row map puts it.
template <typename TX>
__device__ __forceinline__ const TX* in_row(const TX* base, const RowMaps& maps, int t,
                                            int scattered, int64_t r, int N)
{
    if (!scattered) return base + r * N;
    return reinterpret_cast<const TX*>(reinterpret_cast<const unsigned char*>(base) +
                                       row_byte_offset(maps.m[t], r));
}

// The ring of one CTA.  NT staged tensors, each row `row_bytes` long; row
// block b covers rows [b*R, min(b*R + R, M)).  Blocks b = blockIdx.x +
// k*gridDim.x, k = 0..K-1, belong to this CTA.  With kRows the tensors'
// rows are scattered (map[t]): warp 0 issues one bulk copy per row, and the
// slot still holds the block's rows back to back.  Contiguous blocks are
// copied whole; a bulk copy moves a multiple of 16 bytes, so when the last
// block's byte count is not one, its final (count mod 16) bytes are not
// copied (tail_bytes below) and the row-batched kernels, the only ones whose
// rows are not 16-byte multiples, read them from global memory.
template <int NT, int kStages, bool kRows = false>
struct Ring {
    uint64_t* bar;             // [kStages]
    unsigned char* buf;        // [kStages][NT][slot]
    uint32_t slot;             // bytes per tensor per slot
    const unsigned char* src[NT];
    RowMap map[kRows ? NT : 1];
    int64_t row_bytes, R, M, nblocks;
    unsigned* fault;

    __device__ int64_t count() const
    {
        return nblocks > (int64_t)blockIdx.x ? (nblocks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    }
    __device__ int64_t block(int64_t k) const { return blockIdx.x + k * (int64_t)gridDim.x; }
    __device__ const unsigned char* tile(int64_t k, int t) const
    {
        return buf + ((k % kStages) * NT + t) * (size_t)slot;
    }
    // contiguous rows: thread 0 only; kRows: every lane of warp 0
    __device__ void issue(int64_t k)
    {
        const int s = (int)(k % kStages);
        const int64_t r0 = block(k) * R;
        const int64_t rows = (M - r0) < R ? (M - r0) : R;
        const uint32_t bytes = (uint32_t)(rows * row_bytes) & ~15u;
        if constexpr (!kRows) {
            mbar_expect_tx(&bar[s], NT * bytes);
            if (bytes != 0) {  // a last block narrower than 16 bytes copies nothing
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    bulk_g2s(buf + (s * NT + t) * (size_t)slot, src[t] + r0 * row_bytes, bytes,
                             &bar[s]);
            }
        } else {
            const int lane = threadIdx.x & 31;
            if (lane == 0) mbar_expect_tx(&bar[s], NT * bytes);
            __syncwarp();  // the expected byte count is set before any copy lands
#pragma unroll
            for (int t = 0; t < NT; ++t)
                for (int64_t i = lane; i < rows; i += 32)
                    bulk_g2s(buf + (s * NT + t) * (size_t)slot + i * row_bytes,
                             src[t] + row_byte_offset(map[t], r0 + i), (uint32_t)row_bytes,
                             &bar[s]);
        }
    }
    __device__ bool issuer() const { return kRows ? threadIdx.x < 32 : threadIdx.x == 0; }
};

// Run `body(b, k, alive)` over this CTA's row blocks with the ring full
// kStages deep.  `dsm` is the kernel's dynamic shared memory (128-byte
// aligned).  Every thread makes the same calls (body may __syncthreads).
// kBodySyncs: every call of body passes a __syncthreads after its last read
// of the slot (a row reduction across warps, with the row kept in registers
// past it), so the slot can be refilled as soon as body returns, without a
// barrier of its own.
template <bool kBodySyncs = false, int NT, int kStages, bool kRows, class Body>
__device__ __forceinline__ void ring_loop(Ring<NT, kStages, kRows>& rg, unsigned char* dsm,
                                          Body&& body)
{
    rg.bar = reinterpret_cast<uint64_t*>(dsm);
    rg.buf = dsm + 128;
    const int64_t K = rg.count();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&rg.bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (rg.issuer())
        for (int64_t k = 0; k < K && k < kStages; ++k) rg.issue(k);
    bool alive = true;
    int64_t failed_at = K;
    for (int64_t k = 0; k < K; ++k) {
        if (alive) {
            alive = mbar_wait(&rg.bar[k % kStages], (uint32_t)((k / kStages) & 1), rg.fault);
            if (!alive) failed_at = k;
        }
        body(rg.block(k), k, alive);
        if constexpr (!kBodySyncs) __syncthreads();  // every thread is done with slot k % kStages
        if (rg.issuer() && alive && k + kStages < K) {
            fence_proxy_async();
            rg.issue(k + kStages);
        }
    }
    if (!alive) {  // wait, bounded, for copies this thread may have in flight
        for (int64_t k = failed_at; k < K && k < failed_at + kStages; ++k)
            mbar_wait(&rg.bar[k % kStages], (uint32_t)((k / kStages) & 1), nullptr, kWaitCycles);
    }
    __syncthreads();
}

// ------------------------------------------------------------ paired fp32
// Two float32 lanes in one 64-bit register pair.  sm_100 and later run add,
// sub, mul and fma on both lanes in one instruction (the .f32x2 forms), which
// halves the instruction count of the elementwise arithmetic; these kernels
// are issue-bound once their loads are staged through shared memory.
struct f2 {
    uint64_t v;
};

__device__ __forceinline__ f2 mk2(float lo, float hi)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ f2 splat2(float a) { return mk2(a, a); }
__device__ __forceinline__ float lo2(f2 a)
{
    float l, h;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(l), "=f"(h) : "l"(a.v));
    return l;
}
__device__ __forceinline__ float hi2(f2 a)
{
    float l, h;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(l), "=f"(h) : "l"(a.v));
    return h;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b)
{
    f2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b)
{
    f2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b)
{
    f2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c)
{
    f2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return r;
}
// lane-wise select: c ? a : b
__device__ __forceinline__ f2 sel2(bool c, f2 a, f2 b)
{
    f2 r;
    r.v = c ? a.v : b.v;
    return r;
}

// A bf16 pair (one 32-bit word, element 2k in the low half) as two floats.
__device__ __forceinline__ f2 bf2_to_f2(uint32_t w)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "r"(w << 16), "r"(w & 0xffff0000u));
    return r;
}
// Two floats to a bf16 pair, each rounded to nearest even.
__device__ __forceinline__ uint32_t f2_to_bf2(f2 a)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi2(a)), "f"(lo2(a)));
    return r;
}

// One 16-byte vector as pairs: 4 pairs of bf16 or f16, or 2 pairs of f32.
template <typename TX> struct Pairs;
template <> struct Pairs<__nv_bfloat16> { static constexpr int kP = 4; };
template <> struct Pairs<__half> { static constexpr int kP = 4; };
template <> struct Pairs<float> { static constexpr int kP = 2; };

// acc + a*b for bf16 a, b (the low or high halves of packed pairs): one
// instruction, the exact product added with one rounding to float32.
__device__ __forceinline__ float fma_bf16_lo(uint32_t a, uint32_t b, float acc)
{
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}
__device__ __forceinline__ float fma_bf16_hi(uint32_t a, uint32_t b, float acc)
{
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}

// Two bf16 products of bf16 pairs, each rounded once to bf16 (the exact
// product of two bf16 values fits in float32, so this equals rounding the
// float32 product).
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// The same operations for IEEE binary16 pairs: f16 -> f32 is exact, f32 ->
// f16 rounds to nearest even, and an f16 x f16 product (at most 22
// significant bits) is exact in float32 before its one rounding.
__device__ __forceinline__ f2 h2_to_f2(uint32_t w)
{
    float lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
    return mk2(lo, hi);
}
__device__ __forceinline__ uint32_t f2_to_h2(f2 a)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi2(a)), "f"(lo2(a)));
    return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ float fma_f16_lo(uint32_t a, uint32_t b, float acc)
{
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}
__device__ __forceinline__ float fma_f16_hi(uint32_t a, uint32_t b, float acc)
{
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}

// Packed-pair operations of a 16-bit activation type.
template <typename TX> struct P16;
template <> struct P16<__nv_bfloat16> {
    static __device__ __forceinline__ f2 to_f2(uint32_t w) { return bf2_to_f2(w); }
    static __device__ __forceinline__ uint32_t from_f2(f2 a) { return f2_to_bf2(a); }
    static __device__ __forceinline__ uint32_t mul(uint32_t a, uint32_t b) { return bmul2(a, b); }
    static __device__ __forceinline__ float fma_lo(uint32_t a, uint32_t b, float c)
    {
        return fma_bf16_lo(a, b, c);
    }
    static __device__ __forceinline__ float fma_hi(uint32_t a, uint32_t b, float c)
    {
        return fma_bf16_hi(a, b, c);
    }
};
template <> struct P16<__half> {
    static __device__ __forceinline__ f2 to_f2(uint32_t w) { return h2_to_f2(w); }
    static __device__ __forceinline__ uint32_t from_f2(f2 a) { return f2_to_h2(a); }
    static __device__ __forceinline__ uint32_t mul(uint32_t a, uint32_t b) { return hmul2(a, b); }
    static __device__ __forceinline__ float fma_lo(uint32_t a, uint32_t b, float c)
    {
        return fma_f16_lo(a, b, c);
    }
    static __device__ __forceinline__ float fma_hi(uint32_t a, uint32_t b, float c)
    {
        return fma_f16_hi(a, b, c);
    }
};

// One 16-byte vector of activations <-> its float32 pairs.
template <typename TX>
__device__ __forceinline__ void unpack2(const uint4& u, f2 (&p)[Pairs<TX>::kP])
{
    if constexpr (is16<TX>()) {
        p[0] = P16<TX>::to_f2(u.x);
        p[1] = P16<TX>::to_f2(u.y);
        p[2] = P16<TX>::to_f2(u.z);
        p[3] = P16<TX>::to_f2(u.w);
    } else {
        asm("mov.b64 %0, {%1, %2};" : "=l"(p[0].v) : "r"(u.x), "r"(u.y));
        asm("mov.b64 %0, {%1, %2};" : "=l"(p[1].v) : "r"(u.z), "r"(u.w));
    }
}
template <typename TX>
__device__ __forceinline__ uint4 pack2(const f2 (&p)[Pairs<TX>::kP])
{
    if constexpr (is16<TX>()) {
        return make_uint4(P16<TX>::from_f2(p[0]), P16<TX>::from_f2(p[1]), P16<TX>::from_f2(p[2]),
                          P16<TX>::from_f2(p[3]));
    } else {
        uint4 u;
        asm("mov.b64 {%0, %1}, %2;" : "=r"(u.x), "=r"(u.y) : "l"(p[0].v));
        asm("mov.b64 {%0, %1}, %2;" : "=r"(u.z), "=r"(u.w) : "l"(p[1].v));
        return u;
    }
}

// Round both lanes to the activation dtype's precision (identity for f32).
template <typename TX>
__device__ __forceinline__ f2 round2(f2 a)
{
    if constexpr (is16<TX>())
        return P16<TX>::to_f2(P16<TX>::from_f2(a));
    else
        return a;
}

// Parameters of columns c, c+1 as a pair.
__device__ __forceinline__ f2 ld_param2(const void* p, int pt, int64_t c)
{
    return mk2(ld_param(p, pt, c), ld_param(p, pt, c + 1));
}
// The staged parameters of columns c, c + 1 (a plain load, which the
// compiler schedules with the arithmetic: measured 2x faster in the lean DyT
// backward than a volatile one issued in program order)
__device__ __forceinline__ f2 prm2(const float* prm, int c)
{
    const float2 v = *reinterpret_cast<const float2*>(prm + c);
    return mk2(v.x, v.y);
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
    static constexpr int kFloats = (W > 32) ? 2 * kG * NV * 32 : 1;
};

// All-reduce NV values over the W threads of a row group.  W <= 32: the
// group is an aligned slice of a warp and the butterfly stays inside it.
// W > 32: butterfly per warp; lane 0 of each warp stores its partial into a
// double-buffered shared slot (one __syncthreads per call); then lane l of
// every warp loads partial (l mod kWarps) and each aligned run of kWarps
// lanes runs the same butterfly over the same values in the same positions,
// so every thread ends with identical bits.  Every thread of the CTA must
// make the same sequence of calls.
template <int W, int T, int NV>
__device__ __forceinline__ void group_allreduce(float (&v)[NV], float* red, int& parity)
{
    if constexpr (seg_groups(W)) {
        // gather the group's W values in lane order: the same sum on every lane
        const int base = ((threadIdx.x & 31) / W) * W;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            float sum = __shfl_sync(0xffffffffu, v[k], base);
#pragma unroll
            for (int j = 1; j < W; ++j) sum += __shfl_sync(0xffffffffu, v[k], base + j);
            v[k] = sum;
        }
    } else if constexpr (W <= 32) {
        butterfly<W, NV>(v);
    } else {
        constexpr int kWarps = W / 32;
        constexpr int kG = T / W;
        static_assert(kWarps <= 32, "a row group spans at most 32 warps");
        butterfly<32, NV>(v);
        const int lane = threadIdx.x & 31;
        const int g = threadIdx.x / W;
        const int wig = (threadIdx.x % W) >> 5;
        float* slot = red + (parity * kG + g) * NV * 32;  // [NV][32]
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < NV; ++k) slot[k * 32 + wig] = v[k];
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < NV; ++k) v[k] = slot[k * 32 + (lane & (kWarps - 1))];
        butterfly<kWarps, NV>(v);
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
// row.  acc holds, for this thread, columns l*VEC + e (l = lane in its row
// group).  With more than one group per CTA the groups' values are summed in
// group order through shared memory (buf: T*VEC floats); a single group
// writes directly.
template <int W, int VEC, int T>
__device__ __forceinline__ void cta_store_columns(const float (&acc)[VEC], float* buf,
                                                  float* __restrict__ out_row, int N)
{
    constexpr int kG = groups_per_cta(W, T);
    constexpr int kCap = W * VEC;
    const int g = grp<W>();
    const int l = lan<W>();
    if constexpr (kG == 1) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int c = l * VEC + e;
            if (c < N) out_row[c] = acc[e];
        }
    } else {
        if (in_group<W>()) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) buf[g * kCap + l * VEC + e] = acc[e];
        }
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

// Pair form: acc[p] holds columns l*2P + 2p and l*2P + 2p + 1.
template <int W, int P, int T>
__device__ __forceinline__ void cta_store_columns2(const f2 (&acc)[P], float* buf,
                                                   float* __restrict__ out_row, int N)
{
    float a[2 * P];
#pragma unroll
    for (int p = 0; p < P; ++p) {
        a[2 * p] = lo2(acc[p]);
        a[2 * p + 1] = hi2(acc[p]);
    }
    cta_store_columns<W, 2 * P, T>(a, buf, out_row, N);
}

// KV vectors per thread (vector l + j*W holds columns (l + j*W)*VEC ...).
// With several row groups per CTA, vector j's columns go through
// cta_store_columns2 at column offset j*W*VEC; with one group per CTA each
// thread writes its own columns.
template <int W, int KV, int P, int T>
__device__ __forceinline__ void cta_store_columns_kv(const f2 (&acc)[KV][P], float* buf,
                                                     float* __restrict__ out_row, int N)
{
    if constexpr (KV == 1) {
        cta_store_columns2<W, P, T>(acc[0], buf, out_row, N);
    } else if constexpr (groups_per_cta(W, T) > 1) {
#pragma unroll
        for (int j = 0; j < KV; ++j)
            cta_store_columns2<W, P, T>(acc[j], buf, out_row + j * W * 2 * P, N - j * W * 2 * P);
    } else {
        const int l = lan<W>();
#pragma unroll
        for (int j = 0; j < KV; ++j) {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const int c = (l + j * W) * 2 * P + 2 * p;
                if (c < N) out_row[c] = lo2(acc[j][p]);
                if (c + 1 < N) out_row[c + 1] = hi2(acc[j][p]);
            }
        }
    }
}

// ------------------------------------------- programmatic dependent launch
// Every kernel here is launched with programmatic stream serialization
// (launch_pdl below): the GPU may schedule it while the kernel before it on
// the stream is still running, once every CTA of that kernel has executed
// griddepcontrol.launch_dependents (or exited).  Each kernel executes
// launch_dependents first, so its successor is scheduled as soon as all of
// its own CTAs are running, and then griddepcontrol.wait, which returns
// once every prerequisite grid has completed and its memory is visible,
// before its first global-memory access.  The data dependences are those of
// plain stream order (nothing is read or written before the wait, and a
// predecessor that never signals releases its successor when it exits);
// what overlaps is the successor's launch and CTA scheduling with the
// predecessor's tail.  A successor is only launched once all of its
// predecessor's CTAs have started, so waiting CTAs never keep a
// predecessor's CTAs off the SMs.
__device__ __forceinline__ void grid_dependency_sync()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch `kernel` on `stream` with programmatic stream serialization.  A
// failed launch is left in the runtime's last error, which the callers read
// with cudaGetLastError.
template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t stream, Args&&... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Call f(std::integral_constant<int, m>) for the launch's input mode m.
template <class F>
inline void with_mode(int in_mode, F&& f)
{
    if (in_mode == kInRows)
        f(std::integral_constant<int, kInRows>{});
    else if (in_mode == kInStorage)
        f(std::integral_constant<int, kInStorage>{});
    else
        f(std::integral_constant<int, kInContig>{});
}

// Raise a kernel's dynamic shared-memory limit and prefer the maximum
// shared-memory carve-out, once per kernel per context (host side: function
// attributes belong to the context that loaded the module).  The template
// parameter is the kernel itself, so every kernel has its own cache.  A
// failed attempt is not cached (the launch then fails and reports it).
template <auto Kernel>
inline void ring_attributes(int smem)
{
    static CtxCache<char> done;
    char ok = 0;
    done.get(current_ctx_id, [smem](char& v) {
        if (cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess ||
            cudaFuncSetAttribute(Kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        v = 1;
        return true;
    }, ok);
}

}  // namespace gbn
