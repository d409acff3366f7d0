/*
 * gbnorm.h -- C ABI of the GB300 row-normalization library (libgbnorm.so).
 *
 * Forward and backward of three row-wise normalization layers over a
 * row-major activation x of shape [M, N] (M rows, normalized over N):
 *
 *   DyT        y = gamma_j * tanh(alpha * x_ij) + beta_j, scalar alpha
 *              (the fused DyT kernels of Liger-Kernel PR 1617, "fix(dyt):
 *              use a 1D grid and tile small-width rows", Summary)
 *   LayerNorm  y = (x - mean) * rstd * gamma_j + beta_j, biased variance,
 *              rstd = 1/sqrt(var + eps) (the backward's saved-statistics
 *              interface follows torch-xpu-ops "Layernorm bwd OPT #1880")
 *   RMSNorm    y = weight * (x.float() * rsqrt(mean(x.float()^2) + eps))
 *              .to(x.dtype), with the rounding points of DeepSpeed PR 8645
 *              (quoted in PR 8664), section "Semantics"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every tensor argument is a DEVICE pointer on the current CUDA
 *   device (cudaGetDevice()).  Activations (x, dy, y, dx) are contiguous
 *   row-major [M, N] in the activation dtype `xt`; parameters (alpha [1],
 *   gamma/beta/weight [N]) and parameter gradients are in the parameter
 *   dtype `pt`/`wt`; saved statistics (mean, rstd) are float32 [M].
 *   Every pointer must be aligned to its element size (else GBN_EINVAL).
 *   Beyond that any alignment is accepted: 16-byte aligned activations with
 *   N*sizeof a multiple of 16 take the vector path, up to N = 16384 (16-bit
 *   activations) or 8192 (float32);
 *   other contiguous rows up to N = 256 (even N) or 128 (odd N) whose inputs
 *   start on a 16-byte boundary take the row-batched path; the rest the
 *   general path.
 * Ownership.  The caller owns all memory.  The library never allocates,
 *   never frees, never synchronizes and launches only on `stream` (which may
 *   be 0, the legacy default stream).  Calls are asynchronous: a GBN_OK
 *   return means the work was enqueued.
 * Outputs.  y and dx take x's dtype; parameter gradients take the
 *   parameters' dtype (Liger-Kernel PR 1617, Summary).  Parameter-gradient
 *   outputs are nullable: a null pointer skips that output.
 * Workspace.  A backward call needs `gbn_bwd_workspace_bytes(...)` bytes of
 *   4-byte aligned device scratch for its per-CTA partial column sums.  It
 *   needs no initialization: every launch writes every partial row it later
 *   reads.  One workspace must not serve two calls that may overlap on the
 *   GPU.  With every parameter-gradient output null, ws may be null.
 * Determinism.  The launch layout is a fixed function of (M, N, dtypes,
 *   alignment, row layout, SM count) and no float atomics are used:
 *   identical inputs give bit-identical outputs on the same device.
 * Empty input.  M == 0 is a successful call that writes zero parameter
 *   gradients (it still needs `stream` to be valid).
 * Errors.  Invalid arguments return an error status BEFORE anything is
 *   launched; a failed launch returns GBN_ELAUNCH.  No error is fatal and
 *   no kernel traps.
 */
#ifndef GBNORM_H
#define GBNORM_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types: float32, bfloat16, IEEE binary16. */
typedef enum { GBN_F32 = 0, GBN_BF16 = 1, GBN_F16 = 2 } gbn_dtype;

/* Return codes. */
typedef enum {
    GBN_OK = 0,
    GBN_EINVAL = 1,     /* null required pointer, M < 0, N < 1, N > INT32_MAX, bad eps, a pointer
                           not aligned to its element size, misaligned ws */
    GBN_EDTYPE = 2,     /* dtype code not in gbn_dtype, or an RMSNorm dtype pair without
                           defined rounding (see rmsnorm_fwd) */
    GBN_EWORKSPACE = 3, /* ws_bytes smaller than the call needs */
    GBN_ELAUNCH = 4,    /* a kernel launch failed (cudaGetLastError after the launch) */
    GBN_EDEVICE = 5,    /* the current device could not be queried */
    GBN_ESCRATCH = 6    /* rmsnorm_bwd_static_ws: the call needs more scratch than
                           GBN_STATIC_WS_BYTES */
} gbn_status;

/* Layer selector of gbn_bwd_workspace_bytes. */
typedef enum { GBN_OP_DYT = 0, GBN_OP_LAYERNORM = 1, GBN_OP_RMSNORM = 2 } gbn_op;

/* Human-readable name of a gbn_status value (static storage). */
const char* gbn_status_string(int status);

/* Workspace bytes a backward call of layer `op` on [M, N] activations of
 * dtype xt with parameters of dtype pt needs on `device` (an upper bound
 * over both pointer-alignment paths).  Returns 0 for M == 0 and (size_t)-1
 * on invalid arguments or when the device cannot be queried. */
size_t gbn_bwd_workspace_bytes(int op, int64_t M, int64_t N, int xt, int pt, int device);

/* Fault word of the current device: bit 0 (GBN_FAULT_WAIT_TIMEOUT) is set
 * when a kernel's bounded shared-memory barrier wait ran out (about one
 * second); that kernel then finished without further waits (writing, on some
 * paths, values computed from stale shared memory into its own outputs, never
 * outside them) and its outputs are not valid.  Copies the word to host memory *out (this call
 * synchronizes with the device) and zeroes it when `clear` is nonzero.  No
 * counterpart on the pages: it reports the safety bound of the bulk-copy
 * pipeline. */
#define GBN_FAULT_WAIT_TIMEOUT 1u
int gbn_read_faults(unsigned* out, int clear);

/* Self-test of the bounded wait: launches one CTA on `stream` whose barrier
 * never completes, with a wait limit of `limit_cycles` SM clock cycles
 * (1..2^32).  The kernel must give up, set GBN_FAULT_WAIT_TIMEOUT and write 0
 * to *result_device (an int in device memory; 1 would mean the wait
 * completed).  No counterpart on the pages. */
int gbn_selftest_wait_timeout(long long limit_cycles, int* result_device, cudaStream_t stream);

/* ---------------------------------------------------------------- DyT
 * dyt_fwd: y[i,j] = gamma[j] * tanh(alpha[0] * x[i,j]) + beta[j].
 *   x, y [M,N] xt; alpha [1], gamma [N], beta [N] pt (all required).
 * dyt_bwd: dx = dy * gamma * alpha * sech^2(alpha x);
 *   dgamma[j] = sum_i dy tanh(alpha x), dbeta[j] = sum_i dy,
 *   dalpha[0] = sum_ij dy gamma_j x sech^2(alpha x).
 *   Padded rows of a tile are masked after the arithmetic, so alpha = +inf
 *   gives finite dgamma, dbeta, dalpha (Liger-Kernel PR 1617, Summary);
 *   dx itself is NaN there (dy * gamma * inf * 0 under IEEE rules).
 *   x, dy, dx [M,N] xt (required); dalpha [1], dgamma/dbeta [N] pt (nullable). */
int dyt_fwd(const void* x, const void* alpha, const void* gamma, const void* beta, void* y,
            int64_t M, int64_t N, int xt, int pt, cudaStream_t stream);
int dyt_bwd(const void* x, const void* dy, const void* alpha, const void* gamma, void* dx,
            void* dalpha, void* dgamma, void* dbeta, int64_t M, int64_t N, int xt, int pt,
            void* ws, size_t ws_bytes, cudaStream_t stream);

/* ----------------------------------------------------------- LayerNorm
 * layernorm_fwd: mean_i, rstd_i = 1/sqrt(var_i + eps) (biased variance);
 *   y = (x - mean) * rstd * gamma + beta.  gamma, beta nullable (1 and 0);
 *   mean, rstd [M] f32 nullable (written when given).  eps >= 0, finite.
 * layernorm_bwd: with xhat = (x - mean) rstd and g = dy * gamma,
 *   dx = rstd * (g - mean_j g - xhat * mean_j(g xhat)),
 *   dgamma[j] = sum_i dy xhat, dbeta[j] = sum_i dy.
 *   mean, rstd (required) are the forward's saved statistics; gamma
 *   nullable (1); dgamma, dbeta nullable.  The column sums run as per-CTA
 *   partials plus a second pass (torch-xpu-ops "Layernorm bwd OPT #1880"). */
int layernorm_fwd(const void* x, const void* gamma, const void* beta, void* y, float* mean,
                  float* rstd, int64_t M, int64_t N, float eps, int xt, int pt,
                  cudaStream_t stream);
int layernorm_bwd(const void* x, const void* dy, const float* mean, const float* rstd,
                  const void* gamma, void* dx, void* dgamma, void* dbeta, int64_t M, int64_t N,
                  int xt, int pt, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------- RMSNorm
 * rmsnorm_fwd: r_i = rsqrt(mean_j x^2 + eps) in f32, n = round_x(x r),
 *   y = round_x(w * n).  w [N] wt (required); rstd [M] f32 nullable.
 * rmsnorm_bwd: xhat = x r, dn = round_x(dy w),
 *   dx = round_x(r (dn - xhat mean_j(dn xhat))),
 *   dw[j] = sum_i round_x(dy n) when wt == xt, sum_i dy n when wt is f32
 *   (DeepSpeed PR 8645 quoted in PR 8664, "Semantics").  With 16-bit
 *   activations (bf16 or f16) the weight is f32 or of the activation dtype;
 *   any other pair returns GBN_EDTYPE.  rstd nullable:
 *   when null r is recomputed with the forward's exact arithmetic, so the
 *   result is bit-identical either way.  dw nullable.  eps >= 0, finite. */
int rmsnorm_fwd(const void* x, const void* w, void* y, float* rstd, int64_t M, int64_t N,
                float eps, int xt, int wt, cudaStream_t stream);
int rmsnorm_bwd(const void* x, const void* dy, const void* w, const float* rstd, void* dx,
                void* dw, int64_t M, int64_t N, float eps, int xt, int wt, void* ws,
                size_t ws_bytes, cudaStream_t stream);

/* RMSNorm expression variants (the fused-RMSNorm page, DeepSpeed PR 8645
 * quoted in PR 8664, "Which modules are replaced" and "Not covered"):
 *   GBN_RMS_CAST_FIRST   y = w * (x r).to(x.dtype): the Llama expression of
 *                        rmsnorm_fwd / rmsnorm_bwd above;
 *   GBN_RMS_WEIGHT_FIRST y = (w * (x r)).to(x.dtype): the weight multiplies
 *                        the float32 normalized value (GptOss, OLMo 2/3
 *                        style);
 *   GBN_RMS_GEMMA        y = ((x r) * (1 + w)).to(x.dtype), 1 + w in float32.
 * The weight-first forms round only their outputs; their backward is
 *   dn = dy w' (float32, w' = w or 1 + w), dx = round_x(r (dn - xhat
 *   mean_j(dn xhat))), dw[j] = sum_i dy xhat (float32, one final rounding).
 * They accept any weight dtype. */
typedef enum {
    GBN_RMS_CAST_FIRST = 0,
    GBN_RMS_WEIGHT_FIRST = 1,
    GBN_RMS_GEMMA = 2
} gbn_rms_variant;

/* rmsnorm_fwd / rmsnorm_bwd with an expression variant (gbn_rms_variant;
 * anything else returns GBN_EINVAL).  Arguments otherwise as above; the
 * backward's rstd recomputation (rstd null) is the same in every variant. */
int rmsnorm_fwd_ex(const void* x, const void* w, void* y, float* rstd, int64_t M, int64_t N,
                   float eps, int xt, int wt, int variant, cudaStream_t stream);
int rmsnorm_bwd_ex(const void* x, const void* dy, const void* w, const float* rstd, void* dx,
                   void* dw, int64_t M, int64_t N, float eps, int xt, int wt, int variant,
                   void* ws, size_t ws_bytes, cudaStream_t stream);

/* Row layouts of the inputs.
 *   DeepSpeed PR 8645 ("fused RMSNorm", section "Where the kernels run",
 *   row "Layout") takes any leading shape and copies a non-contiguous input
 *   before its kernels run; its tests (section "Correctness evidence", 1)
 *   feed a head-major input and the head-major upstream gradient that
 *   attention produces.  The *_rows entry points below read such inputs in
 *   place instead of copying them.
 * gbn_rows describes where the M rows of an input lie, in ELEMENTS of the
 *   activation dtype from the input's pointer: row r starts at
 *     (r % n1) * s1 + ((r / n1) % n2) * s2 + (r / (n1 * n2)) * s3
 *   and its N elements are contiguous.  That covers every tensor of up to
 *   four dimensions whose last stride is 1 ([B, S, H, D] viewed as M = B*S*H
 *   rows of D with n1 = H, n2 = S: s1, s2, s3 its H, S and B strides; the
 *   head-major [B, H, S, D] transposed to [B, S, H, D] is one such tensor).
 *   n1, n2 >= 1, s1, s2, s3 >= 0 and every row start below 2^62 bytes,
 *   else GBN_EINVAL.  Rows may overlap (broadcast strides of 0 are allowed);
 *   the outputs (y, dx, the statistics) stay contiguous [M, N] and must not
 *   overlap any input.
 * A null layout means contiguous rows (row r at r * N), so the *_rows entry
 *   points with null layouts are the plain entry points.  A layout that
 *   happens to describe contiguous rows is treated as null.  Otherwise the
 *   vector path needs the input pointer and s1, s2, s3 times the element size
 *   to be multiples of 16 bytes (besides the contiguous conditions above);
 *   other layouts take the general path.
 * Results.  y, dx and the saved statistics are the bits that a contiguous
 *   copy of the same rows gives.  So are the parameter gradients, except
 *   when x's layout (and dy's, the same layout) puts the M rows on the M
 *   contiguous rows of the storage in another order, as a head-major tensor
 *   does, and M < 2^31 - 2^20: the vector path then reads the storage in
 *   order and writes each row's outputs to its own row, and the parameter
 *   gradients are the bits of the call on the storage itself read as
 *   contiguous rows (the same sums, added in another order). */
typedef struct {
    int64_t n1, s1, n2, s2, s3;
} gbn_rows;

int dyt_fwd_rows(const void* x, const gbn_rows* xl, const void* alpha, const void* gamma,
                 const void* beta, void* y, int64_t M, int64_t N, int xt, int pt,
                 cudaStream_t stream);
int dyt_bwd_rows(const void* x, const gbn_rows* xl, const void* dy, const gbn_rows* dyl,
                 const void* alpha, const void* gamma, void* dx, void* dalpha, void* dgamma,
                 void* dbeta, int64_t M, int64_t N, int xt, int pt, void* ws, size_t ws_bytes,
                 cudaStream_t stream);
int layernorm_fwd_rows(const void* x, const gbn_rows* xl, const void* gamma, const void* beta,
                       void* y, float* mean, float* rstd, int64_t M, int64_t N, float eps, int xt,
                       int pt, cudaStream_t stream);
int layernorm_bwd_rows(const void* x, const gbn_rows* xl, const void* dy, const gbn_rows* dyl,
                       const float* mean, const float* rstd, const void* gamma, void* dx,
                       void* dgamma, void* dbeta, int64_t M, int64_t N, int xt, int pt, void* ws,
                       size_t ws_bytes, cudaStream_t stream);
int rmsnorm_fwd_rows(const void* x, const gbn_rows* xl, const void* w, void* y, float* rstd,
                     int64_t M, int64_t N, float eps, int xt, int wt, int variant,
                     cudaStream_t stream);
int rmsnorm_bwd_rows(const void* x, const gbn_rows* xl, const void* dy, const gbn_rows* dyl,
                     const void* w, const float* rstd, void* dx, void* dw, int64_t M, int64_t N,
                     float eps, int xt, int wt, int variant, void* ws, size_t ws_bytes,
                     cudaStream_t stream);

/* rmsnorm_bwd_static_ws: rmsnorm_bwd without a caller workspace.  The pages
 *   have no counterpart; it exists for callers that cannot allocate device
 *   memory (a host program with no device allocator of its own, code under a
 *   pool that already holds the device's memory, a loop that must not call
 *   cudaMalloc/cudaFree because they can synchronize the device).  Arguments,
 *   kernels, launch layout and results are those of rmsnorm_bwd; the partial
 *   column sums of dw go to a static device array of GBN_STATIC_WS_BYTES
 *   (8 MiB) inside the library, held by every device (every context) that
 *   loads the library until the process exits.  The call allocates nothing.
 *   Limit: a call with dw non-null and M > 0 whose partial sums need more than
 *   GBN_STATIC_WS_BYTES returns GBN_ESCRATCH before launching anything.  The
 *   need is (rows of partials) x N x 4 bytes, which grows with the device's
 *   SM count S: on the vector path (16-byte aligned activations, N a multiple
 *   of 8 for 16-bit or 4 for f32 activations) at most 32 KiB x S for
 *   N <= 8192, within the array for S <= 256, and 4 x N x S bytes for 16-bit
 *   N up to 16384 (one partial row per SM), within the array while
 *   N x S <= 2^21; on the general path, with
 *   S' = S rounded up to an even number, at most 8 MiB while N <= 2^19 / S'
 *   (the number of warps adapts) and 16 x S' x N bytes beyond (for M of at
 *   least 4 S' rows).  gbn_bwd_workspace_bytes(GBN_OP_RMSNORM, ...), an upper
 *   bound over both paths, <= GBN_STATIC_WS_BYTES is a sufficient check
 *   ahead of a call.  With dw null the array is not used.
 *   Set-up: the array's device address belongs to the CUDA context that
 *   loaded the library's module, so it is looked up with
 *   cudaGetSymbolAddress on the first call in each context (made current)
 *   and cached under that context's id; a new context (after
 *   cudaDeviceReset, or a second context on the device) looks it up again.
 *   Make the first call in a context before any stream capture.  Returns
 *   GBN_EDEVICE when the lookup fails.
 *   Sharing: every call in a context uses the same array, which keeps the
 *   last call's contents (nothing in it needs to start at zero: each call
 *   writes every partial row before reading it).  Calls that may overlap on
 *   the GPU (different streams, or host threads without ordering) race on the
 *   array and give wrong dw. */
#define GBN_STATIC_WS_BYTES (8u << 20)
int rmsnorm_bwd_static_ws(const void* x, const void* dy, const void* w, const float* rstd,
                          void* dx, void* dw, int64_t M, int64_t N, float eps, int xt, int wt,
                          cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GBNORM_H */
