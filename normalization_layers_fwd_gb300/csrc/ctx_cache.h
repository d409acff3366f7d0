// ctx_cache.h -- host-side values cached per CUDA context.
//
// The device address of a __device__ variable, and a kernel's function
// attributes, belong to one CUDA context: every context loads the module
// again, with the variable at its own address.  A value cached per device
// number alone goes stale when the context changes under it (after
// cudaDeviceReset, or in a second context on the same device created with
// the driver API, a green context included) and would hand the new
// context's kernels an address that is not theirs.  CtxCache keys each
// value on the context's unique id (the driver's cuCtxGetId, never reused
// within a process), holding the values of up to kSlots contexts.
//
// This header is plain C++ (no CUDA types) so that its logic can be
// compiled and tested on a host without a GPU.
#pragma once

#include <stdint.h>

#include <mutex>

namespace gbn {

template <class T, int kSlots = 8>
class CtxCache {
public:
    // The value for the calling thread's current context.  `ctx_id()`
    // returns that context's id, or 0 when no context is current or the id
    // cannot be read; `fetch(T&)` computes the value in the current context
    // and returns false on failure (then nothing is cached and get returns
    // false).  The id is read again after a fetch, because the fetch may be
    // the runtime call that makes the device's primary context current; a
    // value fetched while no id can be read is returned but not cached.
    template <class CtxId, class Fetch>
    bool get(CtxId&& ctx_id, Fetch&& fetch, T& out)
    {
        uint64_t id = ctx_id();
        if (id != 0 && find(id, out)) return true;
        T v{};
        if (!fetch(v)) return false;
        id = ctx_id();
        if (id != 0) insert(id, v);
        out = v;
        return true;
    }

private:
    std::mutex mu_;
    uint64_t ids_[kSlots] = {};
    T vals_[kSlots] = {};
    int next_ = 0;  // the slot the next new context takes (round robin)

    bool find(uint64_t id, T& out)
    {
        std::lock_guard<std::mutex> g(mu_);
        for (int i = 0; i < kSlots; ++i)
            if (ids_[i] == id) {
                out = vals_[i];
                return true;
            }
        return false;
    }
    void insert(uint64_t id, const T& v)
    {
        std::lock_guard<std::mutex> g(mu_);
        for (int i = 0; i < kSlots; ++i)
            if (ids_[i] == id) {
                vals_[i] = v;
                return;
            }
        ids_[next_] = id;
        vals_[next_] = v;
        next_ = (next_ + 1) % kSlots;
    }
};

}  // namespace gbn
