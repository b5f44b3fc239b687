// lookback.cuh -- decoupled lookback over per-CTA aggregates (device side).
//
// CTA t publishes its aggregate in state[t], then walks back over its
// predecessors' states, 32 at a time (one per lane of warp 0), summing
// aggregates until it meets an inclusive prefix; it then publishes its own
// inclusive prefix. A state word is kPublished | inclusive << 31 | value
// (31-bit values); the caller zeroes the states before every launch (a zero
// word reads as "not yet published"), inside a kernel that runs earlier on
// the same stream or with a memset node, so that a launch never depends on
// what an earlier call, or an earlier replay of a captured graph, left in
// them. Every CTA a wait depends on must be resident (callers launch only as
// many CTAs as fit at once); each wait is bounded in time, after which the
// missing aggregate counts as zero and LSM_ERR_TIMEOUT is recorded.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace lsm {

// The high half of every published state word.
constexpr uint64_t kPublished = 1ull << 32;

// Called by the 32 lanes of warp 0 of CTA t; returns the sum of the
// aggregates of CTAs 0 .. t-1 (in every lane).
__device__ __forceinline__ uint32_t lookback_exclusive(uint64_t *state, uint32_t t, uint32_t agg,
                                                       int32_t *status) {
  const int lane = threadIdx.x & 31;
  constexpr uint64_t tag = kPublished;
  if (t == 0) {
    if (lane == 0) st_relaxed_u64(state, tag | (1ull << 31) | agg);
    return 0;
  }
  if (lane == 0) st_relaxed_u64(state + t, tag | agg);
  uint32_t prefix = 0;
  int64_t base = static_cast<int64_t>(t) - 1;
  const uint64_t t0 = globaltimer_ns();
  bool late = false;
  for (;;) {
    const int64_t idx = base - lane;
    uint64_t v = idx >= 0 ? ld_relaxed_u64(state + idx) : (tag | (1ull << 31));
    uint32_t polls = 0;
    while (!__all_sync(0xffffffffu, (v >> 32) == 1u)) {
      if ((v >> 32) != 1u) v = ld_relaxed_u64(state + idx);
      if ((++polls & 31) == 0 &&
          __any_sync(0xffffffffu, globaltimer_ns() - t0 > static_cast<uint64_t>(kWaitLimitNs))) {
        late = true;
        if ((v >> 32) != 1u) v = tag | (1ull << 31);  // give up: count it as zero
      }
    }
    const uint32_t inc = __ballot_sync(0xffffffffu, (v >> 31) & 1u);
    uint32_t c = static_cast<uint32_t>(v & 0x7FFFFFFFu);
    if (inc) {
      const int first = __ffs(inc) - 1;
      c = lane <= first ? c : 0u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    prefix += c;
    if (inc) break;
    base -= 32;
  }
  if (lane == 0) {
    if (late) report(status, LSM_ERR_TIMEOUT);
    st_relaxed_u64(state + t, tag | (1ull << 31) | ((prefix + agg) & 0x7FFFFFFFu));
  }
  return prefix;
}

// The sum of the aggregates in state[lo, hi), called by a whole warp: 32 K
// states per round of loads (K per lane, issued together), each polled
// until its word is published (bounded: past the limit a
// missing one counts as zero and LSM_ERR_TIMEOUT is recorded). For callers
// that know the prefix at an earlier tile and need only the aggregates
// since, so that no tile waits for another tile's prefix.
template <int K>
__device__ __forceinline__ uint32_t window_sum(const uint64_t *state, int64_t lo, int64_t hi,
                                               int32_t *status) {
  const int lane = threadIdx.x & 31;
  constexpr uint64_t tag = kPublished;
  const uint64_t t0 = globaltimer_ns();
  bool late = false;
  uint32_t sum = 0;
  for (int64_t b = lo; b < hi; b += 32 * K) {
    uint64_t v[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int64_t idx = b + 32 * k + lane;
      v[k] = idx < hi ? ld_relaxed_u64(state + idx) : tag;
    }
    uint32_t polls = 0;
    for (;;) {
      bool pub = true;
#pragma unroll
      for (int k = 0; k < K; ++k) pub = pub && (v[k] >> 32) == 1u;
      if (__all_sync(0xffffffffu, pub)) break;
#pragma unroll
      for (int k = 0; k < K; ++k)
        if ((v[k] >> 32) != 1u) v[k] = ld_relaxed_u64(state + b + 32 * k + lane);
      if ((++polls & 31) == 0 &&
          __any_sync(0xffffffffu, globaltimer_ns() - t0 > static_cast<uint64_t>(kWaitLimitNs))) {
        late = true;
#pragma unroll
        for (int k = 0; k < K; ++k)
          if ((v[k] >> 32) != 1u) v[k] = tag;  // give up: counts as zero
      }
    }
#pragma unroll
    for (int k = 0; k < K; ++k) sum += static_cast<uint32_t>(v[k] & 0x7FFFFFFFu);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (late && lane == 0) report(status, LSM_ERR_TIMEOUT);
  return sum;
}

}  // namespace lsm
