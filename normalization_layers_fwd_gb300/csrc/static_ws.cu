// static_ws.cu -- RMSNorm backward whose scratch is a library-owned static
// device array, for callers that cannot allocate device memory.
//
// The backward entry points take their partial-column-sum scratch from the
// caller.  Some callers have no way to hand one over:
//   * a plain C, C++ or Fortran host program that links this library but has
//     no device allocator of its own to pair allocations with frees;
//   * code running under a memory pool that has already reserved the
//     device's memory, where a private cudaMalloc fails or fragments the pool;
//   * a latency-bound loop that must not call cudaMalloc or cudaFree, since
//     both can synchronize the whole device.
// rmsnorm_bwd_static_ws serves them.  It runs the same kernels, with the same
// launch layout and the same results, as rmsnorm_bwd, but puts the per-CTA
// partial column sums of dw into g_static_ws below.  It allocates nothing and
// calls no allocating routine.
#include "ctx_cache.h"
#include "gbnorm.h"
#include "internal.h"

// The scratch.  Every device (every context) that loads this library holds
// these GBN_STATIC_WS_BYTES bytes until the process exits.  In host code the
// name g_static_ws only stands for the device variable; its device address
// comes from cudaGetSymbolAddress (static_ws_ptr below).
static __device__ __align__(256) unsigned char g_static_ws[GBN_STATIC_WS_BYTES];

namespace {

gbn::CtxCache<void*> g_static_ws_ptr;

// Device address of g_static_ws in the current context.  Looked up with
// cudaGetSymbolAddress on the first call in each context and cached under
// the context's id: the address belongs to the context that loaded the
// module, so a new context (after cudaDeviceReset, or a second context on
// the device) looks it up again.  Returns null when the lookup fails.
void* static_ws_ptr()
{
    void* p = nullptr;
    const bool ok = g_static_ws_ptr.get(gbn::current_ctx_id, [](void*& v) {
        if (cudaGetSymbolAddress(&v, g_static_ws) != cudaSuccess || !v) {
            cudaGetLastError();  // leave no sticky error behind
            return false;
        }
        return true;
    }, p);
    return ok ? p : nullptr;
}

}  // namespace

extern "C" int rmsnorm_bwd_static_ws(const void* x, const void* dy, const void* w,
                                     const float* rstd, void* dx, void* dw, int64_t M, int64_t N,
                                     float eps, int xt, int wt, cudaStream_t stream)
{
    void* ws = static_ws_ptr();
    if (!ws) return GBN_EDEVICE;
    // Nothing in the array has to start at zero: the first kernel writes
    // every partial row that the column-sum kernel then reads, so what an
    // earlier call left there is never read.  rmsnorm_bwd checks the size
    // before launching anything; a call that needs more than the array holds
    // is reported as GBN_ESCRATCH.
    const int rc = rmsnorm_bwd(x, dy, w, rstd, dx, dw, M, N, eps, xt, wt, ws,
                               (size_t)GBN_STATIC_WS_BYTES, stream);
    return rc == GBN_EWORKSPACE ? GBN_ESCRATCH : rc;
}
