"""The per-context cache of device addresses and kernel attributes
(csrc/ctx_cache.h), compiled with the host C++ compiler and driven with fake
context ids: no GPU.  A __device__ variable lives at a new address in every
CUDA context, so a cached address must be looked up again when the current
context's id changes (after cudaDeviceReset, or in a second context on the
same device), and reused while it stays the same."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "normalization_layers_fwd_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <thread>
#include <vector>
#include "ctx_cache.h"

static uint64_t g_ctx = 0;   // the fake current context id (0: none)
static int g_fetches = 0;    // lookups made
static uint64_t fake_id() { return g_ctx; }

#define CHECK(c)                                                      \
    do {                                                              \
        if (!(c)) {                                                   \
            std::printf("FAIL line %d: %s\n", __LINE__, #c);          \
            return 1;                                                 \
        }                                                             \
    } while (0)

int main()
{
    gbn::CtxCache<long, 4> c;
    long v = 0;
    // a fetch records which context it ran in; context c's value is 1000 c
    auto fetch = [](long& out) { ++g_fetches; out = 1000 * (long)g_ctx; return true; };
    g_ctx = 1;
    CHECK(c.get(fake_id, fetch, v) && v == 1000 && g_fetches == 1);
    CHECK(c.get(fake_id, fetch, v) && v == 1000 && g_fetches == 1);   // cached
    g_ctx = 2;                                                         // a new context
    CHECK(c.get(fake_id, fetch, v) && v == 2000 && g_fetches == 2);   // looked up again
    g_ctx = 1;
    CHECK(c.get(fake_id, fetch, v) && v == 1000 && g_fetches == 2);   // both kept
    // no context current before the fetch: the fetch makes one current, and
    // the value is cached under the id read after it
    g_ctx = 0;
    auto fetch_makes_ctx = [](long& out) { ++g_fetches; g_ctx = 7; out = 7000; return true; };
    CHECK(c.get(fake_id, fetch_makes_ctx, v) && v == 7000 && g_fetches == 3);
    CHECK(c.get(fake_id, fetch, v) && v == 7000 && g_fetches == 3);
    // no id readable at all: the value is returned, never cached
    g_ctx = 0;
    CHECK(c.get(fake_id, fetch, v) && v == 0 && g_fetches == 4);
    CHECK(c.get(fake_id, fetch, v) && g_fetches == 5);
    // a failed fetch caches nothing and reports failure
    g_ctx = 9;
    auto fail = [](long&) { ++g_fetches; return false; };
    CHECK(!c.get(fake_id, fail, v) && g_fetches == 6);
    CHECK(c.get(fake_id, fetch, v) && v == 9000 && g_fetches == 7);
    // more contexts than slots: evicted ones are looked up again, correctly
    for (uint64_t k = 10; k < 20; ++k) {
        g_ctx = k;
        CHECK(c.get(fake_id, fetch, v) && v == 1000 * (long)k);
    }
    const int before = g_fetches;
    g_ctx = 10;  // evicted long ago
    CHECK(c.get(fake_id, fetch, v) && v == 10000 && g_fetches == before + 1);
    g_ctx = 19;  // still held
    CHECK(c.get(fake_id, fetch, v) && v == 19000 && g_fetches == before + 1);
    // concurrent readers of one context see its value
    gbn::CtxCache<long, 4> shared;
    g_ctx = 3;
    std::vector<std::thread> ts;
    std::vector<long> got(8, -1);
    for (int t = 0; t < 8; ++t)
        ts.emplace_back([&, t] {
            long r = -1;
            for (int i = 0; i < 1000; ++i)
                if (!shared.get(fake_id, [](long& o) { o = 3000; return true; }, r) || r != 3000)
                    return;
            got[t] = r;
        });
    for (auto& t : ts) t.join();
    for (long r : got) CHECK(r == 3000);
    std::printf("OK\n");
    return 0;
}
"""


def test_ctx_cache_refetches_when_the_context_changes(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "t.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "t"
    subprocess.run([cxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC, str(src), "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr
