// rank2048.cuh -- the 2048-bit rank directory's query (device side).
//
// "Everett: collision bitmap and rank experiment", "Temporary rank layouts":
// one 8-byte entry per 2048 bits with three packed populations of its
// 512-bit runs, and absolute counts at epochs of 2^32 bits. Entry b:
//   bits  0..31  R(2048 b) minus the count at the start of its epoch
//   bits 32..61  populations of the block's first three 512-bit runs,
//                ten bits each (run r at bit 32 + 10 r)
// epochs[e] = R(2^32 e). A query adds the epoch, the entry's count, the
// earlier runs' populations, the whole words of the current run before p
// (up to fifteen: more bitmap loads than the 512-bit layout's one) and the
// masked word holding p.
#pragma once

#include <cstdint>

namespace lsm {

constexpr int kRank2048Threads = 256;  // 2048-bit blocks per CTA of the build

__device__ __forceinline__ uint64_t rank2048_at(const uint32_t *__restrict__ C,
                                                const uint64_t *__restrict__ dir,
                                                const uint64_t *__restrict__ epochs, int64_t p) {
  const uint64_t e = dir[p >> 11];
  uint64_t r = epochs[p >> 32] + (e & 0xFFFFFFFFu);
  const int runs = static_cast<int>((p >> 9) & 3);
#pragma unroll
  for (int q = 0; q < 3; ++q)
    if (q < runs) r += (e >> (32 + 10 * q)) & 0x3FFu;
  // whole words of the current 512-bit run before p, four at a time when aligned
  const int64_t w0 = (p >> 9) * 16, w1 = p >> 5;
  int64_t w = w0;
  for (; w + 4 <= w1; w += 4) {
    const uint4 v = *reinterpret_cast<const uint4 *>(C + w);
    r += __popc(v.x) + __popc(v.y) + __popc(v.z) + __popc(v.w);
  }
  for (; w < w1; ++w) r += __popc(C[w]);
  if (p & 31) r += __popc(C[w1] & ((1u << (p & 31)) - 1u));
  return r;
}

}  // namespace lsm
