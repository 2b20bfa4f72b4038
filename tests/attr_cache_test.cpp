// Host test of the per-device kernel-attribute cache (attr_cache.h): the
// setter runs once per (kernel, device) and again only for a larger size,
// failures are not recorded, and concurrent callers set each pair once.
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "attr_cache.h"

static int failures = 0;
#define EXPECT(c)                                              \
  do {                                                         \
    if (!(c)) {                                                \
      std::printf("FAILED line %d: %s\n", __LINE__, #c);      \
      ++failures;                                              \
    }                                                          \
  } while (0)

int main() {
  static int k1, k2;  // two distinct "kernels"
  {
    mla::AttrCache c;
    int calls = 0;
    auto set = [&](const void*, int) { ++calls; return 0; };
    EXPECT(c.ensure(&k1, 0, 1000, set) == 0 && calls == 1);
    EXPECT(c.ensure(&k1, 0, 1000, set) == 0 && calls == 1);   // same device: cached
    EXPECT(c.ensure(&k1, 0, 500, set) == 0 && calls == 1);    // smaller: still covered
    EXPECT(c.ensure(&k1, 1, 1000, set) == 0 && calls == 2);   // another device: set there too
    EXPECT(c.ensure(&k2, 0, 1000, set) == 0 && calls == 3);   // another kernel
    EXPECT(c.ensure(&k1, 0, 2000, set) == 0 && calls == 4);   // larger: set again
    EXPECT(c.ensure(&k1, 0, 2000, set) == 0 && calls == 4);
  }
  {
    mla::AttrCache c;
    int calls = 0;
    auto bad = [&](const void*, int) { ++calls; return 98; };
    auto good = [&](const void*, int) { ++calls; return 0; };
    EXPECT(c.ensure(&k1, 3, 1000, bad) == 98 && calls == 1);  // the error is returned ...
    EXPECT(c.ensure(&k1, 3, 1000, good) == 0 && calls == 2);  // ... and not remembered
    EXPECT(c.ensure(&k1, 3, 1000, good) == 0 && calls == 2);
  }
  {
    mla::AttrCache c;
    std::atomic<int> calls{0};
    std::vector<std::thread> ts;
    for (int t = 0; t < 16; ++t)
      ts.emplace_back([&, t] {
        for (int i = 0; i < 2000; ++i)
          c.ensure((i & 1) ? (const void*)&k1 : (const void*)&k2, (t + i) % 4, 4096,
                   [&](const void*, int) { calls.fetch_add(1); return 0; });
      });
    for (auto& t : ts) t.join();
    EXPECT(calls.load() == 8);                                 // 2 kernels x 4 devices
  }
  if (failures == 0) std::printf("ok\n");
  return failures == 0 ? 0 : 1;
}
