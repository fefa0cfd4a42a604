// vc_ctx_cache.h -- per-CUDA-context records of one-time settings.
//
// Some settings the library makes act on the CUDA context that is current on
// the calling host thread (cudaFuncSetAttribute, for instance).  They must be
// made once in every context that launches the kernel, and again after a device
// reset (the new context has a new handle).  Pure C++ without CUDA headers, so
// that a host-only test can exercise it.
#pragma once
#include <mutex>
#include <vector>

namespace vc {

// The CUDA context current on a host thread and its device: the key of every
// per-context record (a context destroyed by a device reset and recreated gets
// a new handle, so nothing recorded for the old one is reused).
struct CtxKey {
    int device = -1;
    const void* ctx = nullptr;
    bool operator==(const CtxKey& o) const { return device == o.device && ctx == o.ctx; }
};

// For each (context, kernel), the largest size a setting has been made with.
// ensure() runs `apply` only when no record covers the request and records the
// request only when `apply` returns 0 (success); `apply` may complete the key
// (a context that its own call created).  Thread safe: one lock around the
// lookup, the setting and the record, so concurrent callers apply a setting once.
class CtxAttrCache {
public:
    template <class Apply>
    auto ensure(CtxKey key, const void* kern, int bytes, Apply apply) -> decltype(apply(&key)) {
        using Status = decltype(apply(&key));
        std::lock_guard<std::mutex> lock(mu_);
        for (const Entry& e : done_)
            if (e.kern == kern && e.key == key && e.bytes >= bytes) return static_cast<Status>(0);
        const Status status = apply(&key);
        if (status == static_cast<Status>(0)) done_.push_back(Entry{key, kern, bytes});
        return status;
    }

private:
    struct Entry {
        CtxKey key;
        const void* kern;
        int bytes;
    };
    std::mutex mu_;
    std::vector<Entry> done_;
};

}  // namespace vc
