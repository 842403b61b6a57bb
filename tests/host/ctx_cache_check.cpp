// Host-only check of kla::ContextAddressCache (the per-context address cache
// of the allocation-free forward). Prints one line per check; exit 0 if all hold.
#include <cstdio>

#include "kla_ctx_cache.h"

int main() {
  int fails = 0;
  auto check = [&](bool ok, const char* what) {
    std::printf("%s %s\n", ok ? "ok" : "FAIL", what);
    fails += ok ? 0 : 1;
  };
  kla::ContextAddressCache<4> c;
  int a, b, d, e, f;
  check(c.find(1) == nullptr, "empty cache misses");
  c.insert(1, &a);
  check(c.find(1) == &a, "hit after insert");
  check(c.find(2) == nullptr, "another context misses (a reset gives a new context ID)");
  c.insert(2, &b);
  check(c.find(1) == &a && c.find(2) == &b, "two contexts on one device keep their own addresses");
  c.insert(1, &d);
  check(c.find(1) == &d && c.size() == 2, "re-insert replaces, no duplicate entry");
  c.insert(3, &e);
  c.insert(4, &f);
  check(c.size() == 4, "fills to capacity");
  c.insert(5, &a);  // evicts the oldest slot (context 1)
  check(c.find(1) == nullptr && c.find(5) == &a && c.find(2) == &b, "full cache drops the oldest entry");
  return fails == 0 ? 0 : 1;
}
