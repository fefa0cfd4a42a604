// Host-only checks of the per-context setting cache (vc_ctx_cache.h), built
// and run by test_ctx_cache_host.py.  Prints OK, or the failed check and exits 1.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <thread>
#include <vector>

#include "vc_ctx_cache.h"

#define CHECK(c)                                                      \
    do {                                                              \
        if (!(c)) {                                                   \
            std::printf("FAILED line %d: %s\n", __LINE__, #c);        \
            std::exit(1);                                             \
        }                                                             \
    } while (0)

static const void* ctx_handle(uintptr_t v) { return reinterpret_cast<const void*>(v); }

int main() {
    using vc::CtxKey;
    int kern1 = 0, kern2 = 0;  // stand-ins for two kernels' addresses
    int calls = 0;
    auto ok = [&](CtxKey*) { ++calls; return 0; };

    vc::CtxAttrCache c;
    const CtxKey dev0{0, ctx_handle(0x10)}, dev1{1, ctx_handle(0x20)}, dev0_reset{0, ctx_handle(0x30)};
    CHECK(c.ensure(dev0, &kern1, 1000, ok) == 0 && calls == 1);        // first use: applied
    CHECK(c.ensure(dev0, &kern1, 1000, ok) == 0 && calls == 1);        // same context: recorded
    CHECK(c.ensure(dev0, &kern1, 500, ok) == 0 && calls == 1);         // a smaller size is covered
    CHECK(c.ensure(dev0, &kern1, 2000, ok) == 0 && calls == 2);        // a larger one applies again
    CHECK(c.ensure(dev0, &kern1, 2000, ok) == 0 && calls == 2);
    CHECK(c.ensure(dev1, &kern1, 1000, ok) == 0 && calls == 3);        // another device
    CHECK(c.ensure(dev0_reset, &kern1, 1000, ok) == 0 && calls == 4);  // a new context after a reset
    CHECK(c.ensure(dev0, &kern2, 1000, ok) == 0 && calls == 5);        // another kernel

    // a failed setting is not recorded: the next call tries again
    auto fail = [&](CtxKey*) { ++calls; return 4; };
    CHECK(c.ensure(dev1, &kern2, 1000, fail) == 4 && calls == 6);
    CHECK(c.ensure(dev1, &kern2, 1000, ok) == 0 && calls == 7);
    CHECK(c.ensure(dev1, &kern2, 1000, ok) == 0 && calls == 7);

    // a key the setting completes (a context its own call created) is recorded complete
    auto create = [&](CtxKey* k) { ++calls; k->ctx = ctx_handle(0x40); return 0; };
    CHECK(c.ensure(CtxKey{2, nullptr}, &kern1, 100, create) == 0 && calls == 8);
    CHECK(c.ensure(CtxKey{2, ctx_handle(0x40)}, &kern1, 100, ok) == 0 && calls == 8);

    // host threads racing on four contexts apply the setting once per context
    vc::CtxAttrCache shared;
    std::atomic<int> applied{0};
    std::vector<std::thread> threads;
    for (int t = 0; t < 8; ++t)
        threads.emplace_back([&] {
            for (int i = 0; i < 2000; ++i)
                shared.ensure(CtxKey{i % 4, ctx_handle(0x100 + i % 4)}, &kern1, 4096, [&](CtxKey*) {
                    applied.fetch_add(1);
                    return 0;
                });
        });
    for (std::thread& th : threads) th.join();
    CHECK(applied.load() == 4);
    std::printf("OK\n");
    return 0;
}
