// tmap.h — host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled,
// reached through the runtime's driver entry point so the library needs no
// link-time libcuda), with a small cache so that a pass with unchanged
// pointers pays no encoding cost.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <map>
#include <mutex>
#include <tuple>

namespace moe {

struct TmapKey {
  uint64_t ptr;
  int dtype, rank, swizzle;
  uint64_t dims[5];
  uint64_t strides[4];
  uint32_t box[5];
  bool operator<(const TmapKey& o) const { return memcmp(this, &o, sizeof *this) < 0; }
};

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// Encodes (or fetches from the cache) a tiled tensor map over a row-major
// tensor (no swizzle unless asked). dims/box are innermost-first; strides (bytes) are those of
// dims[1..rank-1]; rank ≤ 5. Out-of-bounds elements of a box read as zero.
inline bool make_tmap(CUtensorMap* out, const void* ptr, CUtensorMapDataType dtype, int rank,
                      const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                      CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  if (rank < 1 || rank > 5) return false;
  static std::mutex mu;
  static std::map<TmapKey, CUtensorMap> cache;
  TmapKey key;
  memset(&key, 0, sizeof key);
  key.ptr = reinterpret_cast<uint64_t>(ptr);
  key.dtype = (int)dtype;
  key.rank = rank;
  key.swizzle = (int)swizzle;
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) key.strides[i] = strides[i];
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return true;
  }
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], es[5] = {1, 1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) s[i] = strides[i];
  CUresult r = fn(out, dtype, (cuuint32_t)rank, const_cast<void*>(ptr), d, s, b, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (cache.size() > 4096) cache.clear();
  cache[key] = *out;
  return true;
}

// Values computed for recent keys, compared bytewise (Key must be a POD:
// zero it before filling it, so padding compares equal). A launcher keeps its
// whole set of tensor maps here, so that a call with the same pointers and
// sizes as an earlier one reuses them with one lookup. Bounded: cleared when
// it passes 1024 entries.
template <class Key, class Val>
class RecentCache {
 public:
  bool get(const Key& k, Val* v) {
    std::lock_guard<std::mutex> lock(mu_);
    auto it = map_.find(Bytes(k));
    if (it == map_.end()) return false;
    *v = it->second;
    return true;
  }
  void put(const Key& k, const Val& v) {
    std::lock_guard<std::mutex> lock(mu_);
    if (map_.size() >= 1024) map_.clear();
    map_[Bytes(k)] = v;
  }

 private:
  struct Bytes {
    Key k;
    explicit Bytes(const Key& key) : k(key) {}
    bool operator<(const Bytes& o) const { return memcmp(&k, &o.k, sizeof(Key)) < 0; }
  };
  std::mutex mu_;
  std::map<Bytes, Val> map_;
};

}  // namespace moe
