// internal.h -- launch descriptors shared by the host dispatch (api.cu) and
// the per-layer kernel files.  Not part of the public C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gbn {

// Where each row of a non-contiguous input starts: row r begins at byte
//   (r % n1) * s1 + ((r / n1) % n2) * s2 + (r / (n1 * n2)) * s3
// from the tensor's base (the row itself is contiguous).
struct RowMap {
    int64_t n1, s1, n2, s2, s3;
};
// Storage-order reads.  When x (and dy, with the same map) place their M
// rows on the M contiguous rows of their storage in some order, the fast
// kernels stream storage row q and write its outputs at row
//   out_row(q) = (q % a) * wa + ((q / a) % b) * wb + (q / (a * b)) * wc.
// q / a is (q * ma) >> sa and (q / a) / b is ((q / a) * mb) >> sb: division
// by an invariant integer as a multiplication by its rounded-up reciprocal
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994), exact for dividends and divisors below 2^31.
struct OutMap {
    uint32_t ma, mb;
    int sa, sb;
    uint32_t a, b, wa, wb, wc;  // out_row stays below 2^32 for every q < M + 2^20
};
struct RowMaps {
    RowMap m[2];  // x, then dy
    OutMap o;     // storage order (in_mode 2)
};

// Input modes of the fast kernels.
enum InMode {
    kInContig = 0,   // rows at r * N
    kInRows = 1,     // rows where maps.m put them: one bulk copy per row
    kInStorage = 2,  // storage rows in order, outputs through maps.o
};

// How one call is laid out on the GPU.  Decided on the host from (M, N,
// dtypes, pointer alignment, SM count) by a fixed table, never by runtime
// tuning, so the same inputs always give the same summation order.
struct Launch {
    int fast;           // 1: 16-byte vector path (schedule `sid`); 0: general path
    int sid;            // index into kSched (fast path only)
    int batch;          // 1: row-batched path (when not fast): `E`-element units, at
    int E, KMAX, R;     //    most KMAX units a lane per row, R rows a ring block
    int grid;           // CTAs launched (persistent: each loops over row blocks)
    int64_t nblocks;    // row blocks of the fast and row-batched paths
    int64_t P;          // partial rows the backward writes into the workspace
    cudaStream_t stream;
    unsigned* fault;    // the device's fault word (bounded waits that ran out)
    int scattered;      // 1: x (and dy) rows follow maps rather than r * N
    int in_mode;        // InMode of the fast path
    RowMaps maps;
};

// The unique id of the calling thread's current CUDA context, plus one; 0
// when no context is current or the driver cannot be reached (api.cu).
// Host-side caches of device addresses and function attributes key on it.
uint64_t current_ctx_id();

// Workspace row length (floats) per layer: the per-column partial sums of
// every parameter gradient, plus one scalar for DyT's alpha.
inline int64_t ws_row_floats(int op, int64_t N)
{
    return op == 0 ? 2 * N + 1 : (op == 1 ? 2 * N : N);
}

cudaError_t launch_dyt_fwd(const Launch& L, int xt, int pt, const void* x, const void* alpha,
                           const void* gamma, const void* beta, void* y, int64_t M, int N);
cudaError_t launch_dyt_bwd(const Launch& L, int xt, int pt, const void* x, const void* dy,
                           const void* alpha, const void* gamma, void* dx, float* ws,
                           int64_t M, int N);

cudaError_t launch_ln_fwd(const Launch& L, int xt, int pt, const void* x, const void* gamma,
                          const void* beta, void* y, float* mean, float* rstd, int64_t M, int N,
                          float eps);
cudaError_t launch_ln_bwd(const Launch& L, int xt, int pt, const void* x, const void* dy,
                          const float* mean, const float* rstd, const void* gamma, void* dx,
                          float* ws, int64_t M, int N);

// variant: the RMSNorm expression (0 cast then weight, 1 weight then cast,
// 2 Gemma's (1 + weight) then cast), as gbn_rms_variant in gbnorm.h.
cudaError_t launch_rms_fwd(const Launch& L, int xt, int pt, const void* x, const void* w,
                           void* y, float* rstd, int64_t M, int N, float eps, int variant);
cudaError_t launch_rms_bwd(const Launch& L, int xt, int pt, const void* x, const void* dy,
                           const void* w, const float* rstd, void* dx, float* ws, int64_t M,
                           int N, float eps, int variant);

// Second stage of the parameter-gradient reduction: out[c] = sum over the P
// workspace rows of column c, in a fixed order, written in the parameter
// dtype.  Columns [0,N) go to out0, [N,2N) to out1, [2N] to out2 (each
// nullable: skipped).
cudaError_t launch_colsum(cudaStream_t s, const float* ws, int64_t P, int64_t rowlen, int64_t N,
                          int pt, void* out0, void* out1, void* out2);

}  // namespace gbn
