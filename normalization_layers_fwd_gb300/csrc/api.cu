// api.cu -- the extern "C" entry points of libgbnorm.so: argument checks,
// the fixed launch-layout table, and the launches (kernel files hold the
// kernels).  Nothing here allocates memory or synchronizes.
#include <cuda.h>  // CUcontext and CUresult only: the driver is reached through entry points

#include <atomic>
#include <climits>
#include <cmath>
#include <initializer_list>

#include "common.cuh"
#include "ctx_cache.h"
#include "gbnorm.h"
#include "internal.h"

using gbn::Launch;

namespace gbn {

// The unique id of the calling thread's current context, plus one (0 means
// no context is current, or the driver cannot be reached).  cuCtxGetCurrent
// and cuCtxGetId come from the runtime's driver entry-point table, so the
// library needs no link-time dependency on the driver library and loads on
// a host without one.
uint64_t current_ctx_id()
{
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static std::atomic<void*> s_cur{nullptr}, s_id{nullptr};
    void* cur = s_cur.load(std::memory_order_acquire);
    void* gid = s_id.load(std::memory_order_acquire);
    if (!cur || !gid) {
        cudaDriverEntryPointQueryResult qa{}, qb{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &cur, 12000, cudaEnableDefault,
                                             &qa) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &gid, 12000, cudaEnableDefault, &qb) !=
                cudaSuccess ||
            qa != cudaDriverEntryPointSuccess || qb != cudaDriverEntryPointSuccess || !cur ||
            !gid) {
            cudaGetLastError();
            return 0;
        }
        s_cur.store(cur, std::memory_order_release);
        s_id.store(gid, std::memory_order_release);
    }
    CUcontext c = nullptr;
    if (reinterpret_cast<GetCurrent>(cur)(&c) != CUDA_SUCCESS || !c) return 0;
    unsigned long long id = 0;
    if (reinterpret_cast<GetId>(gid)(c, &id) != CUDA_SUCCESS) return 0;
    return (uint64_t)id + 1;
}

}  // namespace gbn

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];  // 0 = not yet queried

// Fault word: bit 0 = a kernel's bounded barrier wait ran out (the kernel then
// finished without loading or storing; its outputs are not valid).  One per
// device and context (a __device__ variable), read and cleared by
// gbn_read_faults().  Its address is cached per context.
__device__ unsigned int g_fault_word;
gbn::CtxCache<unsigned*> g_fault_ptr;

int sm_count(int device)
{
    if (device < 0 || device >= kMaxDevices) return -1;
    int v = g_sms[device].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        v <= 0) {
        cudaGetLastError();  // do not leave a sticky error for the caller
        return -1;
    }
    g_sms[device].store(v, std::memory_order_relaxed);
    return v;
}

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return dev;
}

int current_sms() { return sm_count(current_device()); }

// Device address of the fault word in the current context (cached per
// context: the address belongs to the context that loaded the module).
unsigned* fault_ptr()
{
    unsigned* p = nullptr;
    const bool ok = g_fault_ptr.get(gbn::current_ctx_id, [](unsigned*& v) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_fault_word) != cudaSuccess || !a) {
            cudaGetLastError();
            return false;
        }
        v = static_cast<unsigned*>(a);
        return true;
    }, p);
    return ok ? p : nullptr;
}

bool dtype_ok(int t) { return t == gbn::kF32 || t == gbn::kBF16 || t == gbn::kF16; }
int elem_bytes(int t) { return t == gbn::kF32 ? 4 : 2; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Every pointer must at least be aligned to its element size (null passes):
// even the general path's scalar loads need that.
bool elem_aligned(const void* p, int t)
{
    return (reinterpret_cast<uintptr_t>(p) & (uintptr_t)(elem_bytes(t) - 1)) == 0;
}
bool all_aligned(int t, std::initializer_list<const void*> ps)
{
    for (const void* p : ps)
        if (!elem_aligned(p, t)) return false;
    return true;
}

// Warps of the general path: up to 32 per SM.  In a backward each warp owns
// one workspace row of L floats, so there the count also stays where the
// workspace is at most 8 MB (GBN_STATIC_WS_BYTES), but not below 4 per SM.
int64_t general_warps(int64_t M, int sms, int64_t L)
{
    int64_t w = 32LL * sms;
    if (L > 0) {
        // whole CTAs of kGenWarps: the workspace holds a row per launched warp
        const int64_t fit = (int64_t(8) << 20) / (4 * L) / gbn::kGenWarps * gbn::kGenWarps;
        const int64_t floor4 = 4LL * sms;
        w = fit < w ? (fit > floor4 ? fit : floor4) : w;
    }
    return M < w ? M : w;
}

// Workspace row length (floats) of a backward kernel kind; 0 for a forward.
int64_t general_ws_floats(int kind, int64_t N)
{
    return kind == gbn::kBwdDyT ? gbn::ws_row_floats(0, N)
           : kind == gbn::kBwdLN ? gbn::ws_row_floats(1, N)
           : kind == gbn::kBwdRms ? gbn::ws_row_floats(2, N)
                                  : 0;
}

// Whether [M, N] of dtype xt can take the 16-byte vector path (alignment
// aside), and its schedule index.
// Multi-vector schedules a kernel may take, as a set (bit s - kNumSched1 for
// schedule s), chosen per kernel within its register budget and by
// measurement.  Schedule s serves rows of more than half its capacity and at
// most its capacity (max_nvec / 2 < nvec <= max_nvec), the first in table
// order that the set holds; other rows take the one-vector schedules.
constexpr unsigned kWide12 = 1u, kWide13 = 2u, kWide14 = 4u, kWide15 = 8u, kWide16 = 16u,
                   kWide17 = 32u, kWide18 = 64u, kWide19 = 128u, kWide20 = 256u,
                   kWide21 = 512u, kWide22 = 1024u, kWide23 = 2048u;

// Each kernel's set: the DyT forward 12-13 and backward 12; the LayerNorm
// forward 4 vectors per lane at every capacity from 32 vectors (22, 20, 16,
// 18, 21, 13) and the backward 2 (15, 23, 19, 12, 14); the RMSNorm forward
// and backward 2 as well (one set, so the backward's recomputed rstd
// reduces a row in the forward's order).  The 16-bit backwards hold at most
// 2 vectors per thread.
// Rows of 1025-2048 vectors take schedule 17 in every kernel; the 16-bit
// backwards in their lean form (common.cuh, lean_bwd).
unsigned wide_set(int kind, int)
{
    const unsigned w17 = kWide17;
    switch (kind) {
        case gbn::kFwdDyT: return kWide12 | kWide13 | w17;
        case gbn::kBwdDyT: return kWide12 | w17;
        case gbn::kFwdLN:
            return kWide22 | kWide20 | kWide16 | kWide18 | kWide21 | kWide13 | w17;
        case gbn::kBwdLN: return kWide15 | kWide23 | kWide19 | kWide12 | kWide14 | w17;
        default:  // RMSNorm forward and backward
            return kWide15 | kWide23 | kWide19 | kWide12 | kWide14 | w17;
    }
}

int fast_sid(int64_t N, int xt, unsigned wide)
{
    const int vec = 16 / elem_bytes(xt);
    if (N % vec != 0) return -1;
    const int64_t nvec = N / vec;
    for (int s = gbn::kNumSched1; s < gbn::kNumSched; ++s) {
        const int cap = gbn::kSched[s].max_nvec;
        if (((wide >> (s - gbn::kNumSched1)) & 1u) && cap / 2 < nvec && nvec <= cap) return s;
    }
    for (int s = 0; s < gbn::kNumSched1; ++s)
        if (nvec <= gbn::kSched[s].max_nvec) return s;
    return -1;
}

// The launch layout of one row-wise kernel of the given kind (gbn::KernelKind).
Launch plan(int64_t M, int64_t N, int xt, bool aligned, int sms, cudaStream_t stream, int kind,
            unsigned wide = 0)
{
    Launch L{};
    L.stream = stream;
    const int sid = aligned ? fast_sid(N, xt, wide) : -1;
    if (sid >= 0) {
        const gbn::SchedEntry& e = gbn::kSched[sid];
        const int64_t rows_per_block =
            (int64_t)gbn::groups_per_cta(e.W, e.T) * gbn::kind_U(sid, kind);
        L.fast = 1;
        L.sid = sid;
        L.nblocks = (M + rows_per_block - 1) / rows_per_block;
        const int64_t cap = (int64_t)sms * gbn::kind_minb(sid, kind);
        L.grid = (int)(L.nblocks < cap ? L.nblocks : cap);
        L.P = L.grid;
    } else {
        const int64_t warps = general_warps(M, sms, general_ws_floats(kind, N));
        L.fast = 0;
        L.grid = (int)((warps + gbn::kGenWarps - 1) / gbn::kGenWarps);
        L.P = (int64_t)L.grid * gbn::kGenWarps;
    }
    return L;
}

// The row-batched layout (common.cuh): contiguous rows whose staged inputs
// start on 16-byte boundaries, units of an element pair when N is even and
// every pointer holds whole pairs (pair_ok), else of one element, at most
// batch_max_units(E) units a lane, and ring blocks of at least 8 rows.  Returns
// a Launch with batch == 0 when the path does not apply.
Launch plan_batch(int64_t M, int64_t N, int xt, bool base16, bool pair_ok, int sms,
                  cudaStream_t stream, int kind)
{
    Launch L{};
    L.stream = stream;
    if (!base16 || M <= 0) return L;
    const int E = (N % 2 == 0 && pair_ok) ? 2 : 1;
    const int64_t nu = N / E;
    const int64_t kmax = (nu + 31) / 32;  // units a lane
    if (kmax > gbn::batch_max_units(E)) return L;
    // rows a block: a multiple of 8 * RB (every warp busy) where the slot
    // holds that many, else of 8
    const int64_t fit = gbn::batch_slot(gbn::is_bwd(kind) ? 2 : 1) / (N * elem_bytes(xt));
    const int64_t step =
        8 * (kind == gbn::kFwdDyT || kind == gbn::kBwdDyT ? 1 : gbn::batch_rb((int)kmax, E));
    const int64_t R = fit >= step ? fit / step * step : fit / 8 * 8;
    if (R < 8) return L;
    L.batch = 1;
    L.E = E;
    L.KMAX = (int)kmax;
    L.R = (int)R;
    L.nblocks = (M + R - 1) / R;
    const int64_t cap = (int64_t)sms * gbn::batch_minb(gbn::is_bwd(kind));
    L.grid = (int)(L.nblocks < cap ? L.nblocks : cap);
    L.P = L.grid;
    return L;
}

bool shape_ok(int64_t M, int64_t N)
{
    if (M < 0 || N < 1 || N > INT_MAX) return false;
    // keep M*N*8 (the widest byte offset computed anywhere) inside int64
    return M <= (INT64_MAX / 8) / N;
}

bool eps_ok(float eps) { return std::isfinite(eps) && eps >= 0.f; }

int launch_status(cudaError_t e)
{
    if (e == cudaSuccess) return GBN_OK;
    return GBN_ELAUNCH;
}

size_t ws_needed(int op, const Launch& L, int64_t N)
{
    return (size_t)L.P * (size_t)gbn::ws_row_floats(op, N) * sizeof(float);
}

// Common tail of every backward: the second reduction stage (also for M ==
// 0, where it writes zeros).
int finish_bwd(cudaStream_t s, const float* ws, int64_t P, int op, int64_t N, int pt, void* o0,
               void* o1, void* o2)
{
    if (!o0 && !o1 && !o2) return GBN_OK;
    const int64_t rowlen = gbn::ws_row_floats(op, N);
    return launch_status(gbn::launch_colsum(s, ws, P, rowlen, N, pt, o0, o1, o2));
}

// A one-CTA kernel whose barrier never completes: it expects bytes that no
// copy delivers, so its bounded wait must run out, record the timeout in the
// fault word and return.  It exercises the same wait as the ring kernels.
__global__ void selftest_wait_kernel(unsigned* fault, long long limit, int* result)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        gbn::mbar_init(&bar, 1);
        gbn::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) gbn::mbar_expect_tx(&bar, 16);  // 16 bytes that never arrive
    const bool ok = gbn::mbar_wait(&bar, 0, fault, limit);
    if (threadIdx.x == 0) *result = ok ? 1 : 0;
}

// Row layouts of the inputs (x, dy), null for contiguous rows.
struct Inputs {
    bool ok;         // every layout given is valid
    bool vec_ok;     // every row start is 16-byte aligned (vector path possible)
    int scattered;   // some input's rows are not at r * N
    int mode;        // gbn::InMode of the fast path
    gbn::RowMaps maps;
};

// x / d as (q * m) >> s for every x < 2^31, for a divisor 1 <= d < 2^31:
// with l = ceil(log2 d), m = ceil(2^(31+l) / d) < 2^32 and s = 31 + l
// (the rounded-up reciprocal of Granlund and Montgomery, 1994: the
// multiplier's excess over 2^(31+l)/d is below 1, so for x < 2^31 the error
// of x*m / 2^(31+l) against x/d is below 2^-l <= 1/d).
void invariant_divisor(int64_t d, uint32_t& m, int& s)
{
    int l = 0;
    while ((int64_t(1) << l) < d) ++l;
    const uint64_t p = uint64_t(1) << (31 + l);
    m = (uint32_t)((p + (uint64_t)d - 1) / (uint64_t)d);
    s = 31 + l;
}

// Whether a row map (in bytes, rows of rb bytes) puts the M rows on the M
// contiguous rows of the storage in some order; if so, the map from storage
// row to output row.
bool storage_order(const gbn::RowMap& m, int64_t M, int64_t rb, gbn::OutMap& o)
{
    if (M < 2 || M > (int64_t(1) << 31) - (int64_t(1) << 20)) return false;
    if (M % (m.n1 * m.n2) != 0) return false;
    struct Level { int64_t n, s, w; };
    Level lv[3] = {{m.n1, m.s1, 1}, {m.n2, m.s2, m.n1}, {M / (m.n1 * m.n2), m.s3, m.n1 * m.n2}};
    Level use[3];
    int k = 0;
    for (const Level& v : lv)
        if (v.n > 1) use[k++] = v;
    for (int i = 1; i < k; ++i)  // by storage stride
        for (int j = i; j > 0 && use[j].s < use[j - 1].s; --j) {
            const Level t = use[j];
            use[j] = use[j - 1];
            use[j - 1] = t;
        }
    int64_t expect = rb;
    for (int i = 0; i < k; ++i) {
        if (use[i].s != expect) return false;
        expect *= use[i].n;
    }
    for (int i = k; i < 3; ++i) use[i] = Level{1, 0, 0};
    o.a = (uint32_t)use[0].n;
    o.b = (uint32_t)use[1].n;
    o.wa = (uint32_t)use[0].w;
    o.wb = (uint32_t)use[1].w;
    o.wc = (uint32_t)use[2].w;
    invariant_divisor(o.a, o.ma, o.sa);
    invariant_divisor(o.b, o.mb, o.sb);
    return true;
}

// Whether layout l places row r at r * N for every r < M (levels that no
// row reaches are ignored; products are checked, so huge sizes of unused
// levels cannot overflow).
bool contiguous_rows(const gbn_rows& l, int64_t M, int64_t N)
{
    if (M <= 1) return true;
    if (l.s1 != N) return false;
    if (M <= l.n1) return true;
    int64_t n12;
    if (l.s2 != l.n1 * N) return false;  // n1 < M here, so n1 * N <= M * N fits
    if (__builtin_mul_overflow(l.n1, l.n2, &n12) || M <= n12) return true;
    return l.s3 == n12 * N;  // n12 < M here
}

// Whether every row start of layout l over M rows, in bytes (e per element),
// stays below 2^62: the kernels compute row offsets in int64.
bool layout_extent_ok(const gbn_rows& l, int64_t M, int64_t e)
{
    if (M <= 0) return true;
    const int64_t last = M - 1;
    const int64_t i1 = last < l.n1 - 1 ? last : l.n1 - 1;
    const int64_t q = last / l.n1;
    const int64_t i2 = q < l.n2 - 1 ? q : l.n2 - 1;
    const int64_t i3 = q / l.n2;
    int64_t a, b, c, t;
    if (__builtin_mul_overflow(i1, l.s1, &a) || __builtin_mul_overflow(i2, l.s2, &b) ||
        __builtin_mul_overflow(i3, l.s3, &c) || __builtin_add_overflow(a, b, &t) ||
        __builtin_add_overflow(t, c, &t) || __builtin_mul_overflow(t, e, &t))
        return false;
    return t < (int64_t(1) << 62);
}

Inputs input_layouts(const gbn_rows* xl, const gbn_rows* dyl, const void* x, const void* dy,
                     int64_t M, int64_t N, int xt)
{
    Inputs in{};
    in.ok = true;
    in.vec_ok = true;
    const int64_t e = elem_bytes(xt);
    const gbn_rows* ls[2] = {xl, dyl};
    const void* base[2] = {x, dy};
    for (int t = 0; t < 2; ++t) {
        gbn::RowMap& m = in.maps.m[t];
        m = gbn::RowMap{M > 0 ? M : 1, N * e, 1, 0, 0};
        const gbn_rows* l = ls[t];
        if (!l) continue;
        if (l->n1 < 1 || l->n2 < 1 || l->s1 < 0 || l->s2 < 0 || l->s3 < 0 ||
            !layout_extent_ok(*l, M, e)) {
            in.ok = false;
            continue;
        }
        if (contiguous_rows(*l, M, N)) continue;
        // Levels beyond the M rows change no row offset; capping them keeps
        // n1 * n2 <= 2 M in the kernels' index arithmetic.
        const int64_t n1 = l->n1 < M ? l->n1 : M;
        const int64_t q = (M + n1 - 1) / n1;
        const int64_t n2 = l->n2 < q ? l->n2 : q;
        // The stride of a level that no row reaches multiplies only zero
        // (n1 == 1: every r % n1 is 0; n2 == 1: every (r / n1) % n2 is 0;
        // n1 * n2 >= M: every r / (n1 n2) is 0), so it is dropped before it
        // is scaled to bytes: a huge unused stride must not overflow.  The
        // strides that are reached were bounded by layout_extent_ok.
        int64_t b1 = 0, b2 = 0, b3 = 0;
        if ((n1 > 1 && __builtin_mul_overflow(l->s1, e, &b1)) ||
            (n2 > 1 && __builtin_mul_overflow(l->s2, e, &b2)) ||
            (n1 * n2 < M && __builtin_mul_overflow(l->s3, e, &b3))) {
            in.ok = false;
            continue;
        }
        m = gbn::RowMap{n1, b1, n2, b2, b3};
        in.scattered |= 1 << t;
        if (!aligned16(base[t]) || (m.s1 | m.s2 | m.s3) % 16 != 0) in.vec_ok = false;
    }
    // Storage order when every input follows one map that permutes whole
    // storage rows (x alone in a forward; x and dy alike in a backward).
    const gbn::RowMap& a = in.maps.m[0];
    const gbn::RowMap& b = in.maps.m[1];
    const bool both = dy != nullptr;
    const bool same = !both || (in.scattered == 3 && a.n1 == b.n1 && a.s1 == b.s1 &&
                                a.n2 == b.n2 && a.s2 == b.s2 && a.s3 == b.s3);
    if (in.scattered)
        in.mode = (in.scattered & 1) && same && storage_order(a, M, N * e, in.maps.o)
                      ? gbn::kInStorage
                      : gbn::kInRows;
    in.scattered = in.scattered ? 1 : 0;
    return in;
}

// Every pointer aligned to an element pair (null passes).
bool pair_aligned(int t, std::initializer_list<const void*> ps)
{
    for (const void* p : ps)
        if ((reinterpret_cast<uintptr_t>(p) & (uintptr_t)(2 * elem_bytes(t) - 1)) != 0)
            return false;
    return true;
}

// The row-batched layout in place of the general one where it applies.
void prefer_batch(Launch& L, const Inputs& in, int64_t M, int64_t N, int xt, bool base16,
                  bool pair_ok, int sms, cudaStream_t stream, int kind)
{
    if (L.fast || in.scattered) return;
    const Launch B = plan_batch(M, N, xt, base16, pair_ok, sms, stream, kind);
    if (B.batch) L = B;
}

}  // namespace

extern "C" {

int gbn_read_faults(unsigned* out, int clear)
{
    if (!out) return GBN_EINVAL;
    if (current_device() < 0) return GBN_EDEVICE;
    if (cudaMemcpyFromSymbol(out, g_fault_word, sizeof(unsigned)) != cudaSuccess) {
        cudaGetLastError();
        return GBN_ELAUNCH;
    }
    if (clear) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(unsigned)) != cudaSuccess) {
            cudaGetLastError();
            return GBN_ELAUNCH;
        }
    }
    return GBN_OK;
}

int gbn_selftest_wait_timeout(long long limit_cycles, int* result_device, cudaStream_t stream)
{
    if (!result_device || limit_cycles <= 0 || limit_cycles > (1LL << 32)) return GBN_EINVAL;
    unsigned* f = fault_ptr();
    if (!f) return GBN_EDEVICE;
    selftest_wait_kernel<<<1, 32, 0, stream>>>(f, limit_cycles, result_device);
    return launch_status(cudaGetLastError());
}

const char* gbn_status_string(int status)
{
    switch (status) {
        case GBN_OK: return "GBN_OK";
        case GBN_EINVAL: return "GBN_EINVAL: invalid argument";
        case GBN_EDTYPE: return "GBN_EDTYPE: unsupported dtype";
        case GBN_EWORKSPACE: return "GBN_EWORKSPACE: workspace too small";
        case GBN_ELAUNCH: return "GBN_ELAUNCH: kernel launch failed";
        case GBN_EDEVICE: return "GBN_EDEVICE: cannot query the CUDA device";
        case GBN_ESCRATCH:
            return "GBN_ESCRATCH: the call needs more scratch than the static array "
                   "(GBN_STATIC_WS_BYTES) holds";
        default: return "GBN_UNKNOWN";
    }
}

size_t gbn_bwd_workspace_bytes(int op, int64_t M, int64_t N, int xt, int pt, int device)
{
    if (op < GBN_OP_DYT || op > GBN_OP_RMSNORM || !shape_ok(M, N) || !dtype_ok(xt) ||
        !dtype_ok(pt))
        return (size_t)-1;
    if (M == 0) return 0;
    const int sms = sm_count(device);
    if (sms <= 0) return (size_t)-1;
    const int kind =
        op == GBN_OP_DYT ? gbn::kBwdDyT : op == GBN_OP_LAYERNORM ? gbn::kBwdLN : gbn::kBwdRms;
    // the vector path with the kernel's wide set, or the general path
    const Launch a = plan(M, N, xt, true, sms, nullptr, kind, wide_set(kind, xt));
    const Launch b = plan(M, N, xt, false, sms, nullptr, kind);
    const Launch c = plan_batch(M, N, xt, true, true, sms, nullptr, kind);
    const Launch& ab = a.P > b.P ? a : b;
    const size_t need = ws_needed(op, c.batch && c.P > ab.P ? c : ab, N);
    return (need + 255) & ~(size_t)255;
}

// ---------------------------------------------------------------------- DyT
int dyt_fwd_rows(const void* x, const gbn_rows* xl, const void* alpha, const void* gamma,
                 const void* beta, void* y, int64_t M, int64_t N, int xt, int pt,
                 cudaStream_t stream)
{
    if (!dtype_ok(xt) || !dtype_ok(pt)) return GBN_EDTYPE;
    if (!shape_ok(M, N) || !alpha || !gamma || !beta) return GBN_EINVAL;
    if (M > 0 && (!x || !y)) return GBN_EINVAL;
    if (!all_aligned(xt, {x, y}) || !all_aligned(pt, {alpha, gamma, beta})) return GBN_EINVAL;
    const Inputs in = input_layouts(xl, nullptr, x, nullptr, M, N, xt);
    if (!in.ok) return GBN_EINVAL;
    if (M == 0) return GBN_OK;
    const int sms = current_sms();
    if (sms <= 0) return GBN_EDEVICE;
    Launch L = plan(M, N, xt, aligned16(x) && aligned16(y) && in.vec_ok, sms, stream,
                    gbn::kFwdDyT, wide_set(gbn::kFwdDyT, xt));
    prefer_batch(L, in, M, N, xt, aligned16(x), pair_aligned(xt, {y}), sms, stream, gbn::kFwdDyT);
    if (!(L.fault = fault_ptr())) return GBN_EDEVICE;
    L.scattered = in.scattered;
    L.in_mode = in.mode;
    L.maps = in.maps;
    if (!L.fast && !L.batch) {  // elementwise general path: one thread per element
        const int64_t E = M * N;
        const int64_t blocks = (E + gbn::kGenThreads - 1) / gbn::kGenThreads;
        const int64_t cap = 8LL * sms;
        L.grid = (int)(blocks < cap ? blocks : cap);
    }
    return launch_status(gbn::launch_dyt_fwd(L, xt, pt, x, alpha, gamma, beta, y, M, (int)N));
}

int dyt_fwd(const void* x, const void* alpha, const void* gamma, const void* beta, void* y,
            int64_t M, int64_t N, int xt, int pt, cudaStream_t stream)
{
    return dyt_fwd_rows(x, nullptr, alpha, gamma, beta, y, M, N, xt, pt, stream);
}

int dyt_bwd_rows(const void* x, const gbn_rows* xl, const void* dy, const gbn_rows* dyl,
                 const void* alpha, const void* gamma, void* dx, void* dalpha, void* dgamma,
                 void* dbeta, int64_t M, int64_t N, int xt, int pt, void* ws, size_t ws_bytes,
                 cudaStream_t stream)
{
    if (!dtype_ok(xt) || !dtype_ok(pt)) return GBN_EDTYPE;
    if (!shape_ok(M, N) || !alpha || !gamma) return GBN_EINVAL;
    if (M > 0 && (!x || !dy || !dx)) return GBN_EINVAL;
    if (!all_aligned(xt, {x, dy, dx}) || !all_aligned(pt, {alpha, gamma, dalpha, dgamma, dbeta}))
        return GBN_EINVAL;
    const bool grads = dalpha || dgamma || dbeta;
    if (grads && ws && !aligned4(ws)) return GBN_EINVAL;
    const Inputs in = input_layouts(xl, dyl, x, dy, M, N, xt);
    if (!in.ok) return GBN_EINVAL;
    const int sms = current_sms();
    if (sms <= 0) return GBN_EDEVICE;
    Launch L = plan(M, N, xt, aligned16(x) && aligned16(dy) && aligned16(dx) && in.vec_ok, sms,
                    stream, gbn::kBwdDyT, wide_set(gbn::kBwdDyT, xt));
    prefer_batch(L, in, M, N, xt, aligned16(x) && aligned16(dy), pair_aligned(xt, {dx}), sms,
                 stream, gbn::kBwdDyT);
    if (!(L.fault = fault_ptr())) return GBN_EDEVICE;
    L.scattered = in.scattered;
    L.in_mode = in.mode;
    L.maps = in.maps;
    if (grads && M > 0 && (!ws || ws_bytes < ws_needed(GBN_OP_DYT, L, N))) return GBN_EWORKSPACE;
    float* wsf = grads ? static_cast<float*>(ws) : nullptr;
    if (M > 0) {
        const int rc = launch_status(
            gbn::launch_dyt_bwd(L, xt, pt, x, dy, alpha, gamma, dx, wsf, M, (int)N));
        if (rc != GBN_OK) return rc;
    }
    return finish_bwd(stream, wsf, M > 0 ? L.P : 0, GBN_OP_DYT, N, pt, dgamma, dbeta, dalpha);
}

int dyt_bwd(const void* x, const void* dy, const void* alpha, const void* gamma, void* dx,
            void* dalpha, void* dgamma, void* dbeta, int64_t M, int64_t N, int xt, int pt,
            void* ws, size_t ws_bytes, cudaStream_t stream)
{
    return dyt_bwd_rows(x, nullptr, dy, nullptr, alpha, gamma, dx, dalpha, dgamma, dbeta, M, N,
                        xt, pt, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- LayerNorm
int layernorm_fwd_rows(const void* x, const gbn_rows* xl, const void* gamma, const void* beta,
                       void* y, float* mean, float* rstd, int64_t M, int64_t N, float eps, int xt,
                       int pt, cudaStream_t stream)
{
    if (!dtype_ok(xt) || !dtype_ok(pt)) return GBN_EDTYPE;
    if (!shape_ok(M, N) || !eps_ok(eps)) return GBN_EINVAL;
    if (M > 0 && (!x || !y)) return GBN_EINVAL;
    if (!all_aligned(xt, {x, y}) || !all_aligned(pt, {gamma, beta}) ||
        !all_aligned(GBN_F32, {mean, rstd}))
        return GBN_EINVAL;
    const Inputs in = input_layouts(xl, nullptr, x, nullptr, M, N, xt);
    if (!in.ok) return GBN_EINVAL;
    if (M == 0) return GBN_OK;
    const int sms = current_sms();
    if (sms <= 0) return GBN_EDEVICE;
    Launch L = plan(M, N, xt, aligned16(x) && aligned16(y) && in.vec_ok, sms, stream,
                    gbn::kFwdLN, wide_set(gbn::kFwdLN, xt));
    prefer_batch(L, in, M, N, xt, aligned16(x), pair_aligned(xt, {y}), sms, stream, gbn::kFwdLN);
    if (!(L.fault = fault_ptr())) return GBN_EDEVICE;
    L.scattered = in.scattered;
    L.in_mode = in.mode;
    L.maps = in.maps;
    return launch_status(
        gbn::launch_ln_fwd(L, xt, pt, x, gamma, beta, y, mean, rstd, M, (int)N, eps));
}

int layernorm_fwd(const void* x, const void* gamma, const void* beta, void* y, float* mean,
                  float* rstd, int64_t M, int64_t N, float eps, int xt, int pt,
                  cudaStream_t stream)
{
    return layernorm_fwd_rows(x, nullptr, gamma, beta, y, mean, rstd, M, N, eps, xt, pt, stream);
}

int layernorm_bwd_rows(const void* x, const gbn_rows* xl, const void* dy, const gbn_rows* dyl,
                       const float* mean, const float* rstd, const void* gamma, void* dx,
                       void* dgamma, void* dbeta, int64_t M, int64_t N, int xt, int pt, void* ws,
                       size_t ws_bytes, cudaStream_t stream)
{
    if (!dtype_ok(xt) || !dtype_ok(pt)) return GBN_EDTYPE;
    if (!shape_ok(M, N)) return GBN_EINVAL;
    if (M > 0 && (!x || !dy || !dx || !mean || !rstd)) return GBN_EINVAL;
    if (!all_aligned(xt, {x, dy, dx}) || !all_aligned(pt, {gamma, dgamma, dbeta}) ||
        !all_aligned(GBN_F32, {mean, rstd}))
        return GBN_EINVAL;
    const bool grads = dgamma || dbeta;
    if (grads && ws && !aligned4(ws)) return GBN_EINVAL;
    const Inputs in = input_layouts(xl, dyl, x, dy, M, N, xt);
    if (!in.ok) return GBN_EINVAL;
    const int sms = current_sms();
    if (sms <= 0) return GBN_EDEVICE;
    Launch L = plan(M, N, xt, aligned16(x) && aligned16(dy) && aligned16(dx) && in.vec_ok, sms,
                    stream, gbn::kBwdLN, wide_set(gbn::kBwdLN, xt));
    prefer_batch(L, in, M, N, xt, aligned16(x) && aligned16(dy), pair_aligned(xt, {dx}), sms,
                 stream, gbn::kBwdLN);
    if (!(L.fault = fault_ptr())) return GBN_EDEVICE;
    L.scattered = in.scattered;
    L.in_mode = in.mode;
    L.maps = in.maps;
    if (grads && M > 0 && (!ws || ws_bytes < ws_needed(GBN_OP_LAYERNORM, L, N)))
        return GBN_EWORKSPACE;
    float* wsf = grads ? static_cast<float*>(ws) : nullptr;
    if (M > 0) {
        const int rc = launch_status(
            gbn::launch_ln_bwd(L, xt, pt, x, dy, mean, rstd, gamma, dx, wsf, M, (int)N));
        if (rc != GBN_OK) return rc;
    }
    return finish_bwd(stream, wsf, M > 0 ? L.P : 0, GBN_OP_LAYERNORM, N, pt, dgamma, dbeta,
                      nullptr);
}

int layernorm_bwd(const void* x, const void* dy, const float* mean, const float* rstd,
                  const void* gamma, void* dx, void* dgamma, void* dbeta, int64_t M, int64_t N,
                  int xt, int pt, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    return layernorm_bwd_rows(x, nullptr, dy, nullptr, mean, rstd, gamma, dx, dgamma, dbeta, M, N,
                              xt, pt, ws, ws_bytes, stream);
}

// ------------------------------------------------------------------ RMSNorm
// The Llama expression (variant 0) rounds w*n, dy*w and dy*n to the
// activation dtype; with 16-bit activations its weight is float32 or of the
// activation dtype (a bf16 x with an f16 weight, or the reverse, has no
// defined rounding point).  The weight-first variants round only their
// outputs and take any weight dtype.
bool rms_dtypes_ok(int xt, int wt, int variant)
{
    if (!dtype_ok(xt) || !dtype_ok(wt)) return false;
    return variant != GBN_RMS_CAST_FIRST || xt == GBN_F32 || wt == GBN_F32 || wt == xt;
}

bool rms_variant_ok(int v) { return v >= GBN_RMS_CAST_FIRST && v <= GBN_RMS_GEMMA; }

int rmsnorm_fwd_rows(const void* x, const gbn_rows* xl, const void* w, void* y, float* rstd,
                     int64_t M, int64_t N, float eps, int xt, int wt, int variant,
                     cudaStream_t stream)
{
    if (!rms_variant_ok(variant)) return GBN_EINVAL;
    if (!rms_dtypes_ok(xt, wt, variant)) return GBN_EDTYPE;
    if (!shape_ok(M, N) || !eps_ok(eps) || !w) return GBN_EINVAL;
    if (M > 0 && (!x || !y)) return GBN_EINVAL;
    if (!all_aligned(xt, {x, y}) || !all_aligned(wt, {w}) || !all_aligned(GBN_F32, {rstd}))
        return GBN_EINVAL;
    const Inputs in = input_layouts(xl, nullptr, x, nullptr, M, N, xt);
    if (!in.ok) return GBN_EINVAL;
    if (M == 0) return GBN_OK;
    const int sms = current_sms();
    if (sms <= 0) return GBN_EDEVICE;
    Launch L = plan(M, N, xt, aligned16(x) && aligned16(y) && in.vec_ok, sms, stream,
                    gbn::kFwdNorm, wide_set(gbn::kFwdNorm, xt));
    prefer_batch(L, in, M, N, xt, aligned16(x), pair_aligned(xt, {y}), sms, stream,
                 gbn::kFwdNorm);
    if (!(L.fault = fault_ptr())) return GBN_EDEVICE;
    L.scattered = in.scattered;
    L.in_mode = in.mode;
    L.maps = in.maps;
    return launch_status(gbn::launch_rms_fwd(L, xt, wt, x, w, y, rstd, M, (int)N, eps, variant));
}

int rmsnorm_fwd_ex(const void* x, const void* w, void* y, float* rstd, int64_t M, int64_t N,
                   float eps, int xt, int wt, int variant, cudaStream_t stream)
{
    return rmsnorm_fwd_rows(x, nullptr, w, y, rstd, M, N, eps, xt, wt, variant, stream);
}

int rmsnorm_bwd_rows(const void* x, const gbn_rows* xl, const void* dy, const gbn_rows* dyl,
                     const void* w, const float* rstd, void* dx, void* dw, int64_t M, int64_t N,
                     float eps, int xt, int wt, int variant, void* ws, size_t ws_bytes,
                     cudaStream_t stream)
{
    if (!rms_variant_ok(variant)) return GBN_EINVAL;
    if (!rms_dtypes_ok(xt, wt, variant)) return GBN_EDTYPE;
    if (!shape_ok(M, N) || !eps_ok(eps) || !w) return GBN_EINVAL;
    if (M > 0 && (!x || !dy || !dx)) return GBN_EINVAL;
    if (!all_aligned(xt, {x, dy, dx}) || !all_aligned(wt, {w, dw}) || !all_aligned(GBN_F32, {rstd}))
        return GBN_EINVAL;
    if (dw && ws && !aligned4(ws)) return GBN_EINVAL;
    const Inputs in = input_layouts(xl, dyl, x, dy, M, N, xt);
    if (!in.ok) return GBN_EINVAL;
    const int sms = current_sms();
    if (sms <= 0) return GBN_EDEVICE;
    // the forward's set: a recomputed rstd reduces each row in its order
    Launch L = plan(M, N, xt, aligned16(x) && aligned16(dy) && aligned16(dx) && in.vec_ok, sms,
                    stream, gbn::kBwdRms, wide_set(gbn::kBwdRms, xt));
    prefer_batch(L, in, M, N, xt, aligned16(x) && aligned16(dy), pair_aligned(xt, {dx}), sms,
                 stream, gbn::kBwdRms);
    if (!(L.fault = fault_ptr())) return GBN_EDEVICE;
    L.scattered = in.scattered;
    L.in_mode = in.mode;
    L.maps = in.maps;
    if (dw && M > 0 && (!ws || ws_bytes < ws_needed(GBN_OP_RMSNORM, L, N))) return GBN_EWORKSPACE;
    float* wsf = dw ? static_cast<float*>(ws) : nullptr;
    if (M > 0) {
        const int rc = launch_status(
            gbn::launch_rms_bwd(L, xt, wt, x, dy, w, rstd, dx, wsf, M, (int)N, eps, variant));
        if (rc != GBN_OK) return rc;
    }
    return finish_bwd(stream, wsf, M > 0 ? L.P : 0, GBN_OP_RMSNORM, N, wt, dw, nullptr, nullptr);
}

int rmsnorm_bwd_ex(const void* x, const void* dy, const void* w, const float* rstd, void* dx,
                   void* dw, int64_t M, int64_t N, float eps, int xt, int wt, int variant,
                   void* ws, size_t ws_bytes, cudaStream_t stream)
{
    return rmsnorm_bwd_rows(x, nullptr, dy, nullptr, w, rstd, dx, dw, M, N, eps, xt, wt, variant,
                            ws, ws_bytes, stream);
}

int rmsnorm_fwd(const void* x, const void* w, void* y, float* rstd, int64_t M, int64_t N,
                float eps, int xt, int wt, cudaStream_t stream)
{
    return rmsnorm_fwd_ex(x, w, y, rstd, M, N, eps, xt, wt, GBN_RMS_CAST_FIRST, stream);
}

int rmsnorm_bwd(const void* x, const void* dy, const void* w, const float* rstd, void* dx,
                void* dw, int64_t M, int64_t N, float eps, int xt, int wt, void* ws,
                size_t ws_bytes, cudaStream_t stream)
{
    return rmsnorm_bwd_ex(x, dy, w, rstd, dx, dw, M, N, eps, xt, wt, GBN_RMS_CAST_FIRST, ws,
                          ws_bytes, stream);
}

}  // extern "C"
