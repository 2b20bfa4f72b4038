// Per-device record of the dynamic shared-memory limit each kernel has been
// given.  cudaFuncSetAttribute(MaxDynamicSharedMemorySize) acts on the current
// device only, so a process that launches a kernel on several GPUs must set it
// once per (kernel, device).  Plain C++ (no CUDA types): the setter is passed
// in, so host tests can drive the cache with a fake.
#pragma once

#include <mutex>
#include <vector>

namespace mla {

class AttrCache {
 public:
  // Ensures `set(func, bytes)` has succeeded on `device` for at least `bytes`.
  // The setter runs under the cache's lock, at most once per (func, device,
  // larger size); its return value (0 = success) is returned and a failure is
  // not recorded, so the next call tries again.
  template <class SetFn>
  int ensure(const void* func, int device, int bytes, SetFn&& set) {
    std::lock_guard<std::mutex> lock(mu_);
    for (Entry& e : entries_)
      if (e.func == func && e.device == device) {
        if (e.bytes >= bytes) return 0;
        const int r = set(func, bytes);
        if (r == 0) e.bytes = bytes;
        return r;
      }
    const int r = set(func, bytes);
    if (r == 0) entries_.push_back(Entry{func, device, bytes});
    return r;
  }

 private:
  struct Entry {
    const void* func;
    int device;
    int bytes;
  };
  std::mutex mu_;
  std::vector<Entry> entries_;
};

}  // namespace mla
