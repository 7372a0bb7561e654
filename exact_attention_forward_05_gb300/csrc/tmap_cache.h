// tmap_cache.h -- a small least-recently-used cache of encoded TMA tensor
// maps, so that repeated launches on the same buffers skip the host-side
// encoding.  The key is every argument the 4-D tiled encoding takes, so a hit
// returns exactly the descriptor a fresh encoding would produce (the encoding
// is a pure function of its arguments and does not depend on the device).
// Internal: not part of the C ABI.  Header-only and free of CUDA types so that
// its logic can be compiled and tested on a machine without a GPU.
#pragma once

#include <cstdint>
#include <cstring>
#include <mutex>

namespace attn_internal {

struct TmapKey {
  uint64_t base;        // global address of element (0, 0, 0, 0)
  uint64_t dims[4];     // extents, innermost first
  uint64_t strides[3];  // byte strides of dims[1..3]
  uint32_t box[4];      // box extents, innermost first
  uint32_t dtype;       // CUtensorMapDataType
  uint32_t swizzle;     // CUtensorMapSwizzle
};
static_assert(sizeof(TmapKey) == 88, "TmapKey has no padding, so memcmp compares every field");

inline bool same_key(const TmapKey& a, const TmapKey& b) { return std::memcmp(&a, &b, sizeof(TmapKey)) == 0; }

// SLOTS entries of (key, value); a lookup that hits refreshes the entry, an
// insertion replaces an empty slot or else the least recently used one.
// Thread-safe (one mutex).
template <typename V, int SLOTS>
class TmapCache {
 public:
  bool find(const TmapKey& key, V* out) {
    std::lock_guard<std::mutex> lock(mu_);
    for (int i = 0; i < SLOTS; ++i)
      if (used_[i] && same_key(keys_[i], key)) {
        *out = vals_[i];
        stamp_[i] = ++clock_;
        ++hits_;
        return true;
      }
    ++misses_;
    return false;
  }

  void insert(const TmapKey& key, const V& value) {
    std::lock_guard<std::mutex> lock(mu_);
    int slot = -1;
    for (int i = 0; i < SLOTS && slot < 0; ++i)
      if (used_[i] && same_key(keys_[i], key)) slot = i;  // another thread encoded it first
    for (int i = 0; i < SLOTS && slot < 0; ++i)
      if (!used_[i]) slot = i;
    if (slot < 0) {
      slot = 0;
      for (int i = 1; i < SLOTS; ++i)
        if (stamp_[i] < stamp_[slot]) slot = i;
    }
    keys_[slot] = key;
    vals_[slot] = value;
    used_[slot] = true;
    stamp_[slot] = ++clock_;
  }

  void clear() {
    std::lock_guard<std::mutex> lock(mu_);
    for (int i = 0; i < SLOTS; ++i) used_[i] = false;
  }

  uint64_t hits() {
    std::lock_guard<std::mutex> lock(mu_);
    return hits_;
  }
  uint64_t misses() {
    std::lock_guard<std::mutex> lock(mu_);
    return misses_;
  }

 private:
  std::mutex mu_;
  TmapKey keys_[SLOTS] = {};
  V vals_[SLOTS] = {};
  bool used_[SLOTS] = {};
  uint64_t stamp_[SLOTS] = {};
  uint64_t clock_ = 0, hits_ = 0, misses_ = 0;
};

}  // namespace attn_internal
