// A small map from CUDA context ID to a device address, for the scratch array
// of kla_forward_chunked_noalloc (kla_noalloc.cu). Host code only, no CUDA
// calls: kla_noalloc.cu supplies the key (the driver's unique ID of the
// current context) and the lookup that fills a miss.
//
// Keyed on the context rather than the device number: a __device__ array has
// one address per context that loads the module, so after cudaDeviceReset
// (a new primary context) or under a context the caller created and made
// current, the address cached for the device number would belong to a
// context that no longer exists or to another one. Context IDs are never
// reused within a process, so a new context always misses and is looked up.
#pragma once

#include <cstddef>
#include <cstdint>

namespace kla {

template <int N>
class ContextAddressCache {
 public:
  // The address cached for context `id`, or nullptr.
  void* find(unsigned long long id) const {
    for (int s = 0; s < N; ++s)
      if (used_[s] && ids_[s] == id) return ptrs_[s];
    return nullptr;
  }
  // Remember `ptr` for context `id` (replacing an entry for the same id; when
  // full, the oldest entry makes room: a context whose entry was dropped is
  // looked up again on its next call).
  void insert(unsigned long long id, void* ptr) {
    for (int s = 0; s < N; ++s)
      if (used_[s] && ids_[s] == id) {
        ptrs_[s] = ptr;
        return;
      }
    const int s = next_;
    next_ = (next_ + 1) % N;
    used_[s] = true;
    ids_[s] = id;
    ptrs_[s] = ptr;
  }
  int size() const {
    int n = 0;
    for (int s = 0; s < N; ++s) n += used_[s] ? 1 : 0;
    return n;
  }

 private:
  unsigned long long ids_[N] = {};
  void* ptrs_[N] = {};
  bool used_[N] = {};
  int next_ = 0;
};

}  // namespace kla
