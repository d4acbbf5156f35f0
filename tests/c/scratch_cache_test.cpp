// scratch_cache_test.cpp -- host test of the no-allocation entry point's
// per-context scratch address cache (sequence_re_layout_gb300/csrc/
// scratch_cache.h), driven by a fake context query and a fake symbol lookup.
// Test program: exit status 0 and "scratch_cache ok" on success.
#include <cstdio>
#include <cstdlib>

#include "scratch_cache.h"

#define CHECK(cond, msg)                                                  \
    do {                                                                  \
        if (!(cond)) {                                                    \
            std::fprintf(stderr, "scratch_cache: %s\n", msg);             \
            std::exit(1);                                                 \
        }                                                                 \
    } while (0)

namespace {
unsigned long long g_ctx = 0;        // the "current context" (0: none)
unsigned long long g_bound = 7;      // context a lookup makes current if none is
int g_lookups = 0;
bool g_fail = false;

unsigned long long ctx_id() { return g_ctx; }

// The device array's address depends on the context it was loaded into.
bool lookup(void **p) {
    ++g_lookups;
    if (g_fail) return false;
    if (g_ctx == 0) g_ctx = g_bound;
    *p = reinterpret_cast<void *>(0x10000ull * g_ctx);
    return true;
}
}  // namespace

int main() {
    basp::ScratchAddressCache<4> cache;
    void *a = nullptr;

    // no context current yet: the lookup binds one, and its address is cached
    CHECK(cache.get(ctx_id, lookup, &a) && a == reinterpret_cast<void *>(0x70000ull),
          "first call");
    CHECK(g_lookups == 1, "first call looks the address up");
    CHECK(cache.get(ctx_id, lookup, &a) && g_lookups == 1, "second call reuses it");

    // a device reset: a new context with a new ID, the device code loaded
    // afresh at another address -- the cache must not return the old one
    g_ctx = 8;
    CHECK(cache.get(ctx_id, lookup, &a) && a == reinterpret_cast<void *>(0x80000ull),
          "new context gets its own address");
    CHECK(g_lookups == 2, "new context looks the address up");
    CHECK(cache.get(ctx_id, lookup, &a) && g_lookups == 2, "and reuses it after");

    // back on the first context (another device, say): still cached
    g_ctx = 7;
    CHECK(cache.get(ctx_id, lookup, &a) && a == reinterpret_cast<void *>(0x70000ull) &&
              g_lookups == 2, "first context still cached");

    // a failed lookup caches nothing and reports failure
    g_ctx = 9;
    g_fail = true;
    CHECK(!cache.get(ctx_id, lookup, &a), "failed lookup is reported");
    g_fail = false;
    CHECK(cache.get(ctx_id, lookup, &a) && a == reinterpret_cast<void *>(0x90000ull) &&
              g_lookups == 4, "a later lookup in that context succeeds");

    // more contexts than slots: the oldest entries are replaced, never mixed up
    for (unsigned long long c = 10; c < 20; ++c) {
        g_ctx = c;
        CHECK(cache.get(ctx_id, lookup, &a) && a == reinterpret_cast<void *>(0x10000ull * c),
              "address follows its context");
    }
    std::printf("scratch_cache ok\n");
    return 0;
}
