// rank512.cuh -- the 512-bit rank directory's query (device side).
//
// "Everett: collision bitmap and rank experiment", "Temporary rank layouts":
// each 512-bit block has a 32-bit absolute prefix and seven packed 9-bit
// prefixes for its 64-bit pairs; an exclusive rank query uses the
// directory, at most one preceding 32-bit word and a masked current word:
// at most two popcounts. Layout: dir[3b] = R(512 b); dir[3b+1] | dir[3b+2]
// << 32 holds the popcount of the block's first s 64-bit words at bits
// [9(s-1), 9s) for s = 1..7.
#pragma once

#include <cstdint>

namespace lsm {

// R(p) for p in [0, m]: directory entry, packed sub-prefix, at most one
// preceding 32-bit word and the masked current word.
__device__ __forceinline__ uint32_t rank512_at(const uint32_t *__restrict__ C,
                                               const uint32_t *__restrict__ dir, int64_t p) {
  const int64_t b = p >> 9;
  uint32_t r = dir[3 * b];
  const int s = static_cast<int>((p >> 6) & 7);
  if (s) {
    const uint64_t packed = static_cast<uint64_t>(dir[3 * b + 1]) |
                            (static_cast<uint64_t>(dir[3 * b + 2]) << 32);
    r += static_cast<uint32_t>((packed >> (9 * (s - 1))) & 0x1FFu);
  }
  const int64_t w = p >> 5;
  if (p & 32) r += __popc(C[w - 1]);
  if (p & 31) r += __popc(C[w] & ((1u << (p & 31)) - 1u));
  return r;
}

}  // namespace lsm
