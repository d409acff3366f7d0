// colsum.cu -- second stage of the parameter-gradient column reduction.
//
// The backward kernels leave P fp32 partial rows (one per CTA, or one per
// warp on the general path).  This kernel sums each column over the P rows
// in a fixed order and writes the result in the parameter dtype; the
// torch-xpu-ops page "Layernorm bwd OPT #1880" runs the same second stage as
// its "two sum" launches after GammaBetaReduceFunctor.  There are no float
// atomics anywhere, so the result is bit-identical from run to run.
//
// Block = 32 columns x kSlices slices: slice s sums rows s, s+kSlices, ...
// in increasing order, then slice 0 adds the kSlices slice sums in order.
// The partial rows were just written and sit in L2, so the kernel is bound
// by load latency, not bandwidth: 32 slices with up to 16 loads in flight
// per thread cover the usual P (a few hundred rows) in one round trip.
#include "common.cuh"
#include "internal.h"

namespace gbn {
namespace {

constexpr int kCols = 32;
constexpr int kSlices = 32;
constexpr int kBatch = 16;  // independent loads in flight per thread

__global__ void __launch_bounds__(kCols * kSlices)
    colsum_kernel(const float* __restrict__ ws, int64_t P, int64_t rowlen, int64_t N, int pt,
                  void* __restrict__ out0, void* __restrict__ out1, void* __restrict__ out2)
{
    grid_dependency_sync();
    __shared__ float part[kSlices][kCols + 1];
    const int tx = threadIdx.x % kCols, ty = threadIdx.x / kCols;
    const int64_t c = blockIdx.x * (int64_t)kCols + tx;
    float s = 0.f;
    if (c < rowlen) {
        // batches of kBatch independent loads (all in flight, the rows past P
        // masked), added in row order
        for (int64_t p0 = ty; p0 < P; p0 += kBatch * kSlices) {
            float v[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int64_t p = p0 + i * kSlices;
                v[i] = p < P ? __ldcg(ws + p * rowlen + c) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                if (p0 + i * kSlices < P) s += v[i];
        }
    }
    part[ty][tx] = s;
    __syncthreads();
    if (ty == 0 && c < rowlen) {
        float t = part[0][tx];
#pragma unroll
        for (int k = 1; k < kSlices; ++k) t += part[k][tx];
        if (c < N) {
            if (out0) st_param(out0, pt, c, t);
        } else if (c < 2 * N) {
            if (out1) st_param(out1, pt, c - N, t);
        } else {
            if (out2) st_param(out2, pt, c - 2 * N, t);
        }
    }
}

}  // namespace

cudaError_t launch_colsum(cudaStream_t s, const float* ws, int64_t P, int64_t rowlen, int64_t N,
                          int pt, void* out0, void* out1, void* out2)
{
    const int64_t blocks = (rowlen + kCols - 1) / kCols;
    launch_pdl(colsum_kernel, (unsigned)blocks, kCols * kSlices, 0, s, ws, P, rowlen, N, pt, out0,
               out1, out2);
    return cudaGetLastError();
}

}  // namespace gbn
