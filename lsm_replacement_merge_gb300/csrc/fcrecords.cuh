// fcrecords.cuh -- one thread's run of merged records, loaded for the flat
// front-compression length passes (bit profile in fc.cu, byte profile in
// bytefc.cu).
//
// "Everett: GPU construction experiment" (exact lengths) and "Everett:
// byte-profile GPU merge" ("Pipeline"): a record's length needs its key's
// extent, its LCP with the preceding record's key, its value's extent and
// its tombstone bit. A thread takes I consecutive output records and the
// record before them and issues every load of them before using any: the
// refs, then the key extents and each key's first 16 bytes (from the key
// prefix table of the record's source), the value extents and the tombstone
// words. The passes wait on these loads, so one round of independent loads
// per dependency level is what sets their time.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace lsm {

// Src: a source of records with members key, val (lsm_bytes), tomb (bitmap
// or null) and prefix (the key prefix table, 2 words per key; required for
// every source a loaded record comes from).
template <class Src>
__device__ __forceinline__ const Src &source_of(const Src &a, const Src &b, uint32_t ref) {
  return (ref & LSM_REF_FROM_B) ? b : a;
}

template <class Src, int I>
struct FlatRecords {
  static constexpr int Q = I + 1;  // slot 0: the record before the first
  uint32_t rr[Q];
  uint64_t kb[Q], ke[Q], p0[Q], p1[Q];
  uint64_t vb[I], ve[I];
  uint32_t tw[I];

  __device__ __forceinline__ void load(const Src &sa, const Src &sb,
                                       const uint32_t *__restrict__ refs, int64_t N,
                                       int64_t first) {
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const int64_t i = first - 1 + q;
      rr[q] = (i >= 0 && i < N) ? __ldg(refs + i) : 0u;
    }
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const int64_t i = first - 1 + q;
      const bool live = i >= 0 && i < N;
      const uint32_t idx = rr[q] & ~LSM_REF_FROM_B;
      const Src &src = source_of(sa, sb, rr[q]);
      kb[q] = live ? __ldg(src.key.off + idx) : 0;
      ke[q] = live ? __ldg(src.key.off + idx + 1) : 0;
      ulonglong2 v = make_ulonglong2(0, 0);
      if (live) v = __ldg(reinterpret_cast<const ulonglong2 *>(src.prefix) + idx);
      p0[q] = v.x;
      p1[q] = v.y;
    }
#pragma unroll
    for (int q = 0; q < I; ++q) {
      const int64_t i = first + q;
      const bool live = i < N;
      const uint32_t idx = rr[q + 1] & ~LSM_REF_FROM_B;
      const Src &src = source_of(sa, sb, rr[q + 1]);
      vb[q] = live ? __ldg(src.val.off + idx) : 0;
      ve[q] = live ? __ldg(src.val.off + idx + 1) : 0;
      tw[q] = (live && src.tomb) ? __ldg(src.tomb + (idx >> 5)) : 0u;
    }
  }

  // Record first + q is a tombstone.
  __device__ __forceinline__ bool tomb(int q) const {
    return (tw[q] >> ((rr[q + 1] & ~LSM_REF_FROM_B) & 31)) & 1u;
  }

  // Leading bits (of 128) on which the first 16 bytes of record first + q
  // and its predecessor agree (128 when they all do; bytes past a key's end
  // read as zero).
  __device__ __forceinline__ uint32_t prefix_agree_bits(int q) const {
    const uint64_t d0 = p0[q] ^ p0[q + 1], d1 = p1[q] ^ p1[q + 1];
    return d0 ? static_cast<uint32_t>(__clzll(static_cast<long long>(d0)))
              : (d1 ? 64u + static_cast<uint32_t>(__clzll(static_cast<long long>(d1))) : 128u);
  }
};

}  // namespace lsm
