// strings.cuh -- byte-string keys on the device.
//
// Keys live in CSR arenas (bytes + uint64 offsets). They are read as
// big-endian 8-byte windows built from aligned 8-byte loads, so that one
// comparison step covers eight bytes; bytes past a key's end are masked to
// zero. Order is unsigned lexicographic with a proper prefix first
// ("Everett: GPU construction experiment", prefix-cache paragraph: zero
// padding plus the original length keeps proper-prefix order exact; the
// LCP clamps to the shorter key).
//
// Readability contract (checked on the host): each arena starts on an
// 8-byte boundary and stays readable up to the next multiple of 8 bytes
// past its last byte. A window load touches the aligned word holding `pos`
// and, only when the key continues past it, the next aligned word.
#pragma once

#include <cstdint>

#include "lsmmerge.h"

namespace lsm {

__device__ __forceinline__ uint64_t bswap64(uint64_t x) {
  const uint32_t lo = static_cast<uint32_t>(x), hi = static_cast<uint32_t>(x >> 32);
  return (static_cast<uint64_t>(__byte_perm(lo, 0, 0x0123)) << 32) | __byte_perm(hi, 0, 0x0123);
}

// Bytes [pos, min(pos + 8, end)) of `arena` as a big-endian word: byte pos
// in bits 63..56. Requires pos < end.
__device__ __forceinline__ uint64_t load_be64(const uint8_t *__restrict__ arena, uint64_t pos,
                                              uint64_t end) {
  const uint64_t *w = reinterpret_cast<const uint64_t *>(arena);
  const uint64_t q = pos >> 3;
  const unsigned r = static_cast<unsigned>(pos & 7);
  uint64_t x = __ldg(w + q) >> (8 * r);
  if (r && 8 * q + 8 < end) x |= __ldg(w + q + 1) << (64 - 8 * r);
  uint64_t be = bswap64(x);
  const uint64_t avail = end - pos;
  if (avail < 8) be &= ~uint64_t(0) << (8 * (8 - avail));
  return be;
}

// Bytes [kb, min(kb + 16, ke)) as two big-endian words (bytes kb..kb+7 in
// w0, kb+8..kb+15 in w1, zero past ke). Only the aligned 8-byte words that
// hold key bytes are loaded (at most three); each output 32-bit word is one
// byte permute of two consecutive 32-bit source words, which does the
// byte shift and the byte swap at once.
__device__ __forceinline__ void load_prefix16(const uint8_t *__restrict__ arena, uint64_t kb,
                                              uint64_t ke, uint64_t &w0, uint64_t &w1) {
  if (ke <= kb) {
    w0 = w1 = 0;
    return;
  }
  const uint64_t *w = reinterpret_cast<const uint64_t *>(arena);
  const uint64_t q = kb >> 3;
  const uint64_t lastb = kb + 15 < ke - 1 ? kb + 15 : ke - 1;  // last byte needed
  const uint64_t lim = lastb >> 3;
  const uint64_t a = __ldg(w + q);
  const uint64_t b = q + 1 <= lim ? __ldg(w + q + 1) : 0;
  const uint64_t c = q + 2 <= lim ? __ldg(w + q + 2) : 0;
  const uint32_t t[6] = {static_cast<uint32_t>(a), static_cast<uint32_t>(a >> 32),
                         static_cast<uint32_t>(b), static_cast<uint32_t>(b >> 32),
                         static_cast<uint32_t>(c), static_cast<uint32_t>(c >> 32)};
  const unsigned r = static_cast<unsigned>(kb & 7);
  const unsigned s = r & 3;
  const unsigned sel = (s << 12) | ((s + 1) << 8) | ((s + 2) << 4) | (s + 3);
  const bool hi4 = r >= 4;  // the window starts in the second 32-bit word
  const uint32_t u0 = hi4 ? t[1] : t[0], u1 = hi4 ? t[2] : t[1], u2 = hi4 ? t[3] : t[2];
  const uint32_t u3 = hi4 ? t[4] : t[3], u4 = hi4 ? t[5] : t[4];
  uint32_t o0 = __byte_perm(u0, u1, sel), o1 = __byte_perm(u1, u2, sel);
  uint32_t o2 = __byte_perm(u2, u3, sel), o3 = __byte_perm(u3, u4, sel);
  const uint64_t len = ke - kb;
  if (len < 16) {  // zero the bytes past the key's end
    const int n = static_cast<int>(len);
    auto keep = [n](int k) -> uint32_t {  // bytes 4k..4k+3 of the window
      const int have = n - 4 * k;
      return have >= 4 ? ~0u : (have <= 0 ? 0u : ~0u << (8 * (4 - have)));
    };
    o0 &= keep(0);
    o1 &= keep(1);
    o2 &= keep(2);
    o3 &= keep(3);
  }
  w0 = (static_cast<uint64_t>(o0) << 32) | o1;
  w1 = (static_cast<uint64_t>(o2) << 32) | o3;
}

struct KeyRef {
  const uint8_t *arena;
  uint64_t begin, end;
};

__device__ __forceinline__ KeyRef key_at(const lsm_bytes &col, int64_t idx) {
  return KeyRef{col.arena, __ldg(col.off + idx), __ldg(col.off + idx + 1)};
}

// Three-way comparison of two keys whose first `from` bytes are known to be
// equal (from a multiple of 8, at most the shorter length): negative, zero
// or positive.
__device__ __forceinline__ int key_cmp_from(const KeyRef &a, const KeyRef &b, uint64_t from) {
  const uint64_t la = a.end - a.begin, lb = b.end - b.begin;
  const uint64_t l = la < lb ? la : lb;
  for (uint64_t t = from; t < l; t += 8) {
    const uint64_t x = load_be64(a.arena, a.begin + t, a.begin + l);
    const uint64_t y = load_be64(b.arena, b.begin + t, b.begin + l);
    if (x != y) return x < y ? -1 : 1;
  }
  return la == lb ? 0 : (la < lb ? -1 : 1);
}

// Three-way comparison: negative, zero or positive.
__device__ __forceinline__ int key_cmp(const KeyRef &a, const KeyRef &b) {
  return key_cmp_from(a, b, 0);
}

// The same comparison with both keys' first 16 bytes loaded in one round
// (zero-padded prefix words: equal words with one key at most 16 bytes long
// make the shorter key a proper prefix of the other, or the keys equal);
// bytes past 16 only when both keys are longer and their first 16 agree.
// Keys that share their first 8 bytes then cost one dependent load round
// instead of two.
__device__ __forceinline__ int key_cmp_prefix16(const KeyRef &a, const KeyRef &b) {
  uint64_t a0, a1, b0, b1;
  load_prefix16(a.arena, a.begin, a.end, a0, a1);
  load_prefix16(b.arena, b.begin, b.end, b0, b1);
  if (a0 != b0) return a0 < b0 ? -1 : 1;
  if (a1 != b1) return a1 < b1 ? -1 : 1;
  const uint64_t la = a.end - a.begin, lb = b.end - b.begin;
  if (la <= 16 || lb <= 16) return la == lb ? 0 : (la < lb ? -1 : 1);
  return key_cmp_from(a, b, 16);
}

}  // namespace lsm
