// scratch_cache.h -- the per-context cache of the no-allocation entry point's
// scratch address (host code only, no CUDA types, so host tests can drive it
// with a fake context query and lookup).
//
// A __device__ array has one address per CUDA context that loaded the
// library's device code.  The entry point looks that address up once per
// context and reuses it.  Entries are keyed by the driver's context ID, which
// the driver never reuses within a process, so a device reset (after which
// the device code is loaded afresh, perhaps at another address) is a new key
// and gets a new lookup instead of a stale address.
#pragma once

#include <mutex>

namespace basp {

template <int kSlots>
class ScratchAddressCache {
  public:
    // `ctx_id()` returns the current context's ID, or 0 if there is none (or
    // it cannot be read); `lookup(&addr)` returns true and the address in the
    // current context, making a context current if none was.  Returns false
    // if the lookup fails; nothing is cached then.
    template <class CtxId, class Lookup>
    bool get(CtxId ctx_id, Lookup lookup, void **out) {
        std::lock_guard<std::mutex> lock(mu_);
        unsigned long long id = ctx_id();
        if (id != 0) {
            for (const Entry &e : entries_)
                if (e.ctx_id == id) {
                    *out = e.addr;
                    return true;
                }
        }
        void *p = nullptr;
        if (!lookup(&p) || p == nullptr) return false;
        if (id == 0) id = ctx_id();       // the lookup made a context current
        if (id != 0) {
            entries_[next_] = Entry{id, p};
            next_ = (next_ + 1) % kSlots;
        }
        *out = p;
        return true;
    }

  private:
    struct Entry {
        unsigned long long ctx_id;
        void *addr;
    };
    std::mutex mu_;
    Entry entries_[kSlots] = {};
    int next_ = 0;
};

}  // namespace basp
