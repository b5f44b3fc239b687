// bytefc.cu -- byte-profile front compression of the merged string records.
//
// "Everett: byte-profile GPU merge", "Pipeline": the byte profile's records
// carry byte LEB128 counts, FC literals and optional-value tags, with
// 15-record blocks; a common encoded value width drops the value length
// ("width seventeen means a one-byte presence tag and sixteen payload
// bytes"); records are sized, scanned and emitted in order. Record i (the
// bit profile's grammar of "Everett: GPU construction experiment" with
// bytes for bits and LEB128 for Exp-Golomb):
//   p_i = byte LCP with record i-1's key (p_0 = 0), K_i = key bytes,
//   b_i = 1 + p_i when i mod 15 = 0, else K_{i-1} - p_i;
//   LEB128(b_i) LEB128(K_i - p_i) key bytes [p_i, K_i) then tag 0 for a
//   tombstone, else tag 1, LEB128(value length) (left out under a common
//   width W) and the value bytes.
//
//   bytefc_lengths_kernel  one tile of 1024 records per CTA, four records
//                          per thread: key extents, byte LCP with the
//                          predecessor from aligned 8-byte loads, control,
//                          record length; the tile's total for the scan
//                          (bytefc_lengths_flat_kernel when the inputs
//                          carry key prefix tables: 512 threads of two
//                          records, every load issued before any is used)
//   (scan)                 the FC pipeline's one-CTA tile scan and offsets
//                          pass turn the lengths into byte offsets
//   bytefc_emit_kernel     one CTA per 256 consecutive records: each thread
//                          writes its record into a shared copy of their
//                          contiguous byte span (records never share a
//                          byte), one bulk store moves the aligned interior
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "fcrecords.cuh"
#include "internal.h"

namespace lsm {

namespace {

constexpr int kBfThreads = 256;
constexpr int kBfItems = 4;
constexpr int kBfTile = kBfThreads * kBfItems;

struct BSource {
  lsm_bytes key, val;
  const uint32_t *tomb;
  const uint64_t *prefix;  // the key prefix table (bytes 0..15 big-endian), or NULL
};

__device__ __forceinline__ const BSource &bpick(const BSource &a, const BSource &b, uint32_t ref) {
  return (ref & LSM_REF_FROM_B) ? b : a;
}

// `need` (1..8) bytes of an 8-byte aligned arena from byte offset o, byte t
// of the window in bits [8t, 8t+8) of the result (little-endian words); the
// second aligned word is read only when the window reaches into it.
__device__ __forceinline__ uint64_t bytes8_at(const uint8_t *arena, uint64_t o, int need) {
  const uint64_t *w = reinterpret_cast<const uint64_t *>(arena);
  const uint64_t t = o >> 3;
  const int sh = static_cast<int>(o & 7);
  uint64_t v = __ldg(w + t) >> (8 * sh);
  if (sh + need > 8) v |= __ldg(w + t + 1) << (64 - 8 * sh);
  return v;
}

// Byte LCP of two byte strings, clamped to the shorter one.
__device__ __forceinline__ uint64_t byte_lcp(const uint8_t *aa, uint64_t ao, uint64_t alen,
                                             const uint8_t *ba, uint64_t bo, uint64_t blen) {
  const uint64_t L = alen < blen ? alen : blen;
  for (uint64_t t = 0; t < L; t += 8) {
    const int need = L - t < 8 ? static_cast<int>(L - t) : 8;
    uint64_t x = bytes8_at(aa, ao + t, need) ^ bytes8_at(ba, bo + t, need);
    if (need < 8) x &= (1ull << (8 * need)) - 1;
    if (x) return t + (__ffsll(static_cast<long long>(x)) - 1) / 8;
  }
  return L;
}

__device__ __forceinline__ uint32_t leb_len(uint64_t x) {
  uint32_t n = 1;
  while (x >= 128) {
    x >>= 7;
    ++n;
  }
  return n;
}

__device__ __forceinline__ bool is_tomb(const BSource &src, uint32_t idx) {
  return src.tomb && ((__ldg(src.tomb + (idx >> 5)) >> (idx & 31)) & 1u);
}

__global__ void __launch_bounds__(kBfThreads) bytefc_lengths_kernel(
    BSource sa, BSource sb, const uint32_t *__restrict__ refs, int64_t N, uint64_t W,
    uint32_t *__restrict__ lcp, uint32_t *__restrict__ ctrl, uint32_t *__restrict__ rec,
    uint64_t *__restrict__ tile_sum, int32_t *status) {
  pdl_begin();
  __shared__ uint64_t scratch[kBfThreads / 32 + 1];
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kBfTile + int64_t(threadIdx.x) * kBfItems;
  uint64_t local = 0;
#pragma unroll
  for (int q = 0; q < kBfItems; ++q) {
    const int64_t i = first + q;
    if (i >= N) break;
    const uint32_t r = __ldg(refs + i), idx = r & 0x7FFFFFFFu;
    const BSource &src = bpick(sa, sb, r);
    const uint64_t ks = __ldg(src.key.off + idx), K = __ldg(src.key.off + idx + 1) - ks;
    uint64_t p = 0, Kp = 0;
    if (i > 0) {
      const uint32_t pr = __ldg(refs + i - 1), pidx = pr & 0x7FFFFFFFu;
      const BSource &ps = bpick(sa, sb, pr);
      const uint64_t pks = __ldg(ps.key.off + pidx);
      Kp = __ldg(ps.key.off + pidx + 1) - pks;
      if (src.prefix && ps.prefix) {
        // the first 16 bytes from the prefix tables: the first differing
        // byte of the big-endian words, clamped to the shorter key; bytes
        // past 16 only when both keys are longer and the 16 agree
        const ulonglong2 u = __ldg(reinterpret_cast<const ulonglong2 *>(ps.prefix) + pidx);
        const ulonglong2 v = __ldg(reinterpret_cast<const ulonglong2 *>(src.prefix) + idx);
        const uint64_t L = Kp < K ? Kp : K;
        const uint64_t d0 = u.x ^ v.x, d1 = u.y ^ v.y;
        if (d0) p = static_cast<uint64_t>(__clzll(static_cast<long long>(d0))) / 8;
        else if (d1) p = 8 + static_cast<uint64_t>(__clzll(static_cast<long long>(d1))) / 8;
        else p = L > 16 ? 16 + byte_lcp(ps.key.arena, pks + 16, Kp - 16, src.key.arena, ks + 16,
                                        K - 16)
                        : 16;
        p = p < L ? p : L;
      } else {
        p = byte_lcp(ps.key.arena, pks, Kp, src.key.arena, ks, K);
      }
    }
    const uint64_t b = (i % 15 == 0) ? 1 + p : Kp - p;
    uint64_t v;
    if (is_tomb(src, idx)) {
      v = 1;
      if (W) report(status, LSM_ERR_ARG);  // a tombstone breaks the common width
    } else {
      const uint64_t vb = __ldg(src.val.off + idx + 1) - __ldg(src.val.off + idx);
      if (W && vb + 1 != W) report(status, LSM_ERR_ARG);
      v = W ? W : 1 + leb_len(vb) + vb;
    }
    const uint64_t L = leb_len(b) + leb_len(K - p) + (K - p) + v;
    if (L > 0xFFFFFFFFull || b > 0xFFFFFFFFull) report(status, LSM_ERR_OVERFLOW);
    lcp[i] = static_cast<uint32_t>(p);
    ctrl[i] = static_cast<uint32_t>(b);
    rec[i] = static_cast<uint32_t>(L);
    local += static_cast<uint32_t>(L);
  }
  const uint64_t total = block_sum<kBfThreads, uint64_t>(local, scratch);
  if (threadIdx.x == 0) tile_sum[blockIdx.x] = total;
}

// The same lengths when both sources carry key prefix tables: each of 512
// threads takes two consecutive records and the record before them
// (FlatRecords: every load issued before any is used), two CTAs per SM.
// The byte LCP is the first byte at which the 16-byte prefixes differ,
// clamped to the shorter key; bytes past 16 come from the arenas only when
// both keys are longer and all 16 agree. Measured on the 4M + 4M strings
// (lengths + scan + offsets, L2 flushed): 115 us against 141 us for
// bytefc_lengths_kernel on the same tables (four records per thread, each
// record's loads after the previous record's).
constexpr int kBfFlatThreads = 512;
constexpr int kBfFlatItems = kBfTile / kBfFlatThreads;
static_assert(kBfFlatItems * kBfFlatThreads == kBfTile, "a flat tile is one scan tile");

__global__ void __launch_bounds__(kBfFlatThreads, 2) bytefc_lengths_flat_kernel(
    BSource sa, BSource sb, const uint32_t *__restrict__ refs, int64_t N, uint64_t W,
    uint32_t *__restrict__ lcp, uint32_t *__restrict__ ctrl, uint32_t *__restrict__ rec,
    uint64_t *__restrict__ tile_sum, int32_t *status) {
  pdl_begin();
  __shared__ uint64_t scratch[kBfFlatThreads / 32 + 1];
  const int64_t first =
      static_cast<int64_t>(blockIdx.x) * kBfTile + int64_t(threadIdx.x) * kBfFlatItems;
  FlatRecords<BSource, kBfFlatItems> R;
  R.load(sa, sb, refs, N, first);
  uint64_t local = 0;
  bool bad_width = false, overflow = false;
#pragma unroll
  for (int q = 0; q < kBfFlatItems; ++q) {
    const int64_t i = first + q;
    if (i >= N) break;
    const uint64_t K = R.ke[q + 1] - R.kb[q + 1];
    uint64_t p = 0, Kp = 0;
    if (i > 0) {
      Kp = R.ke[q] - R.kb[q];
      const uint64_t L = Kp < K ? Kp : K;
      p = R.prefix_agree_bits(q) / 8;
      if (p == 16 && L > 16)
        p = 16 + byte_lcp(bpick(sa, sb, R.rr[q]).key.arena, R.kb[q] + 16, Kp - 16,
                          bpick(sa, sb, R.rr[q + 1]).key.arena, R.kb[q + 1] + 16, K - 16);
      p = p < L ? p : L;
    }
    const uint64_t b = (i % 15 == 0) ? 1 + p : Kp - p;
    uint64_t v;
    if (R.tomb(q)) {
      v = 1;
      bad_width |= W != 0;  // a tombstone breaks the common width
    } else {
      const uint64_t vb = R.ve[q] - R.vb[q];
      bad_width |= W && vb + 1 != W;
      v = W ? W : 1 + leb_len(vb) + vb;
    }
    const uint64_t L = leb_len(b) + leb_len(K - p) + (K - p) + v;
    overflow |= L > 0xFFFFFFFFull || b > 0xFFFFFFFFull;
    lcp[i] = static_cast<uint32_t>(p);
    ctrl[i] = static_cast<uint32_t>(b);
    rec[i] = static_cast<uint32_t>(L);
    local += static_cast<uint32_t>(L);
  }
  if (bad_width) report(status, LSM_ERR_ARG);
  if (overflow) report(status, LSM_ERR_OVERFLOW);
  const uint64_t total = block_sum<kBfFlatThreads, uint64_t>(local, scratch);
  if (threadIdx.x == 0) tile_sum[blockIdx.x] = total;
}

// Common encoded value width ("Pipeline": detected before the records are
// sized). acc[1] = the smallest value length, acc[2] = the largest, acc[3]
// = 1 when a record is a tombstone; the finish step writes acc[0] = 1 +
// the length when every record is present with one length, else 0.
__global__ void __launch_bounds__(256) bytefc_width_reduce_kernel(
    BSource sa, BSource sb, const uint32_t *__restrict__ refs, int64_t N,
    unsigned long long *acc) {
  pdl_begin();
  __shared__ unsigned long long s_min[8], s_max[8];
  __shared__ int s_tomb[8];
  unsigned long long mn = ~0ull, mx = 0;
  int tomb = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < N; i += stride) {
    const uint32_t r = __ldg(refs + i), idx = r & 0x7FFFFFFFu;
    const BSource &src = bpick(sa, sb, r);
    if (is_tomb(src, idx)) {
      tomb = 1;
    } else {
      const unsigned long long vb = __ldg(src.val.off + idx + 1) - __ldg(src.val.off + idx);
      mn = vb < mn ? vb : mn;
      mx = vb > mx ? vb : mx;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long a = __shfl_xor_sync(0xffffffffu, mn, o);
    const unsigned long long b = __shfl_xor_sync(0xffffffffu, mx, o);
    mn = a < mn ? a : mn;
    mx = b > mx ? b : mx;
  }
  tomb = __any_sync(0xffffffffu, tomb);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    s_min[w] = mn;
    s_max[w] = mx;
    s_tomb[w] = tomb;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int t = 1; t < static_cast<int>(blockDim.x >> 5); ++t) {
      mn = s_min[t] < mn ? s_min[t] : mn;
      mx = s_max[t] > mx ? s_max[t] : mx;
      tomb |= s_tomb[t];
    }
    if (mn != ~0ull) atomicMin(acc + 1, mn);
    if (mx) atomicMax(acc + 2, mx);
    if (tomb) atomicOr(acc + 3, 1ull);
  }
}

__global__ void bytefc_width_finish_kernel(int64_t N, unsigned long long *acc) {
  pdl_begin();
  acc[0] = (N > 0 && !acc[3] && acc[1] == acc[2]) ? 1 + acc[1] : 0;
}

// Record i's checked extent: its bytes [pos, end) when the offsets, lcp and
// control give exactly its own length (the lengths pass's output for these
// inputs and W); otherwise false (the record is reported and not written).
struct RecordPlan {
  uint64_t ks, K, p, b, vs, vlen, pos, end;
  bool tomb;
};

__device__ __forceinline__ bool plan_record(const BSource &sa, const BSource &sb,
                                            const uint32_t *__restrict__ refs,
                                            const uint32_t *__restrict__ lcp,
                                            const uint32_t *__restrict__ ctrl,
                                            const uint64_t *__restrict__ off, int64_t i,
                                            uint64_t W, RecordPlan &r, const BSource *&srcp) {
  const uint32_t ref = __ldg(refs + i), idx = ref & 0x7FFFFFFFu;
  const BSource &src = bpick(sa, sb, ref);
  srcp = &src;
  r.ks = __ldg(src.key.off + idx);
  r.K = __ldg(src.key.off + idx + 1) - r.ks;
  r.p = __ldg(lcp + i);
  r.b = __ldg(ctrl + i);
  r.pos = __ldg(off + i);
  r.end = __ldg(off + i + 1);
  r.tomb = is_tomb(src, idx);
  r.vs = r.tomb ? 0 : __ldg(src.val.off + idx);
  r.vlen = r.tomb ? 0 : __ldg(src.val.off + idx + 1) - r.vs;
  const uint64_t v = r.tomb ? 1 : (W ? W : 1 + leb_len(r.vlen) + r.vlen);
  return r.p <= r.K && r.end >= r.pos &&
         leb_len(r.b) + leb_len(r.K - r.p) + (r.K - r.p) + v == r.end - r.pos &&
         !(W && (r.tomb || r.vlen + 1 != W));
}

// Writes a planned record through `put(position, byte)`: LEB128(b),
// LEB128(K - p), the key bytes [p, K) (read as aligned 8-byte words), the tag
// byte, LEB128(value length) unless a common width W is given, the value
// bytes.
template <class Put>
__device__ __forceinline__ void write_record(const BSource &src, const RecordPlan &r, uint64_t W,
                                             const Put &put) {
  uint64_t pos = r.pos;
  auto leb = [&](uint64_t x) {
    do {
      uint8_t byte = static_cast<uint8_t>(x & 0x7F);
      x >>= 7;
      if (x) byte |= 0x80;
      put(pos++, byte);
    } while (x);
  };
  auto copy = [&](const uint8_t *arena, uint64_t from, uint64_t len) {
    for (uint64_t t = 0; t < len; t += 8) {
      const int need = len - t < 8 ? static_cast<int>(len - t) : 8;
      const uint64_t w = bytes8_at(arena, from + t, need);
      for (int q = 0; q < need; ++q) put(pos++, static_cast<uint8_t>(w >> (8 * q)));
    }
  };
  leb(r.b);
  leb(r.K - r.p);
  copy(src.key.arena, r.ks + r.p, r.K - r.p);
  put(pos++, r.tomb ? 0 : 1);
  if (!r.tomb) {
    if (!W) leb(r.vlen);
    copy(src.val.arena, r.vs, r.vlen);
  }
}

// write_record into a shared copy of the span (dst = the copy at the
// record's first byte): the counts and the tag as single bytes; the key and
// value bytes by 4-byte stores once the destination is 4-byte aligned (each
// 8-byte read of the arena gives two), single bytes at either end.
__device__ __forceinline__ void write_record_smem(const BSource &src, const RecordPlan &r,
                                                  uint64_t W, uint8_t *dst) {
  uint32_t at = 0;
  auto leb = [&](uint64_t x) {
    do {
      uint8_t byte = static_cast<uint8_t>(x & 0x7F);
      x >>= 7;
      if (x) byte |= 0x80;
      dst[at++] = byte;
    } while (x);
  };
  auto copy = [&](const uint8_t *arena, uint64_t from, uint64_t len) {
    uint64_t t = 0;
    // bytes until the destination is 4-byte aligned
    const uint32_t lead = static_cast<uint32_t>((4 - (smem_u32(dst + at) & 3)) & 3);
    const uint64_t h = lead < len ? lead : len;
    if (h) {
      const uint64_t w = bytes8_at(arena, from, static_cast<int>(h));
      for (uint64_t q = 0; q < h; ++q) dst[at++] = static_cast<uint8_t>(w >> (8 * q));
      t = h;
    }
    for (; t + 8 <= len; t += 8) {
      const uint64_t w = bytes8_at(arena, from + t, 8);
      *reinterpret_cast<uint32_t *>(dst + at) = static_cast<uint32_t>(w);
      *reinterpret_cast<uint32_t *>(dst + at + 4) = static_cast<uint32_t>(w >> 32);
      at += 8;
    }
    if (t < len) {
      const int need = static_cast<int>(len - t);
      const uint64_t w = bytes8_at(arena, from + t, need);
      for (int q = 0; q < need; ++q) dst[at++] = static_cast<uint8_t>(w >> (8 * q));
    }
  };
  leb(r.b);
  leb(r.K - r.p);
  copy(src.key.arena, r.ks + r.p, r.K - r.p);
  dst[at++] = r.tomb ? 0 : 1;
  if (!r.tomb) {
    if (!W) leb(r.vlen);
    copy(src.val.arena, r.vs, r.vlen);
  }
}

// One CTA per kBeRecords consecutive records: their bytes are one
// contiguous span [s0, s1) of the payload. Each thread writes its record into
// a shared copy of the span (records never share a byte), then the
// 16-byte-aligned interior leaves with one bulk store and the at most 15
// bytes at either end with plain stores. A span larger than the shared
// buffer (very long keys or values) is written record by record straight to
// global memory instead. A record whose extent does not match its fields is
// reported (LSM_ERR_ARG) and its bytes in the span are zero.
constexpr int kBeRecords = 256;
constexpr int kBeBuf = 24 * 1024;

__global__ void __launch_bounds__(kBeRecords) bytefc_emit_kernel(
    BSource sa, BSource sb, const uint32_t *__restrict__ refs, int64_t N, uint64_t W,
    const uint32_t *__restrict__ lcp, const uint32_t *__restrict__ ctrl,
    const uint64_t *__restrict__ off, uint8_t *__restrict__ payload, int64_t nbytes,
    int32_t *status) {
  pdl_begin();
  __shared__ __align__(16) uint8_t buf[kBeBuf];
  const int64_t R0 = static_cast<int64_t>(blockIdx.x) * kBeRecords;
  const int64_t R1 = R0 + kBeRecords < N ? R0 + kBeRecords : N;
  const int64_t i = R0 + threadIdx.x;
  const uint64_t s0 = __ldg(off + R0), s1 = __ldg(off + R1);
  // buf[0] mirrors the 16-byte boundary of the payload at or below s0, so
  // that shared and global addresses agree modulo 16
  const uint64_t pa = reinterpret_cast<uintptr_t>(payload);
  const uint64_t base = s0 - ((pa + s0) & 15);
  const bool staged = s1 >= s0 && s1 <= static_cast<uint64_t>(nbytes) &&
                      s1 - base + 16 <= static_cast<uint64_t>(kBeBuf);
  if (!staged) {
    // record by record, straight to global memory
    if (i < R1) {
      RecordPlan r;
      const BSource *src;
      if (!plan_record(sa, sb, refs, lcp, ctrl, off, i, W, r, src) ||
          r.end > static_cast<uint64_t>(nbytes)) {
        report(status, LSM_ERR_ARG);
      } else {
        write_record(*src, r, W, [&](uint64_t q, uint8_t v) { payload[q] = v; });
      }
    }
    return;
  }
  if (i < R1) {
    RecordPlan r;
    const BSource *src;
    const bool ok = plan_record(sa, sb, refs, lcp, ctrl, off, i, W, r, src) && r.pos >= s0 &&
                    r.end <= s1;
    if (ok) {
      write_record_smem(*src, r, W, buf + (r.pos - base));
    } else {
      report(status, LSM_ERR_ARG);
      // the record's bytes inside the span read as zero
      const uint64_t a = r.pos < s0 ? s0 : (r.pos > s1 ? s1 : r.pos);
      const uint64_t e = r.end > s1 ? s1 : (r.end < a ? a : r.end);
      for (uint64_t q = a; q < e; ++q) buf[q - base] = 0;
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  const uint64_t a0 = s0 + ((16 - ((pa + s0) & 15)) & 15), a1 = s1 - ((pa + s1) & 15);
  if (a1 > a0) {
    if (threadIdx.x == 0) {
      bulk_s2g(payload + a0, buf + (a0 - base), static_cast<uint32_t>(a1 - a0));
      bulk_commit();
    }
    // the bytes before a0 and from a1 on
    const int head = static_cast<int>(a0 - s0), tail = static_cast<int>(s1 - a1);
    const int t = threadIdx.x - 1;
    if (t >= 0 && t < head) payload[s0 + t] = buf[s0 + t - base];
    if (t >= 16 && t < 16 + tail) payload[a1 + (t - 16)] = buf[a1 + (t - 16) - base];
  } else {
    const int t = threadIdx.x;
    for (uint64_t q = s0 + t; q < s1; q += blockDim.x) payload[q] = buf[q - base];
  }
  if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

BSource bsource(const lsm_bytes &key, const lsm_bytes &val, const uint32_t *tomb,
                const uint64_t *prefix = nullptr) {
  return BSource{key, val, tomb, prefix};
}

}  // namespace

cudaError_t launch_bytefc_lengths_scan(const lsm_fc_input &in, const uint32_t *refs, int64_t N,
                                       uint64_t W, uint32_t *lcp, uint32_t *ctrl,
                                       uint32_t *rec_bytes, uint64_t *byte_off, void *ws,
                                       int32_t *status, cudaStream_t s) {
  static_assert(kBfTile == 1024, "the offsets pass scans tiles of 1024 records");
  if (fc_tile_records() != kBfTile) return cudaErrorInvalidValue;
  uint64_t *tile_sum = static_cast<uint64_t *>(ws);
  const int64_t tiles = (N + kBfTile - 1) / kBfTile;
  // prefix tables on both sources (an empty one needs none): the flat form
  const bool flat = (in.prefixA || in.m == 0) && (in.prefixB || in.n == 0) &&
                    (in.prefixA || in.prefixB);
  profile_before(s);
  cudaError_t err =
      flat ? launch_kernel(false, bytefc_lengths_flat_kernel,
                           static_cast<unsigned>(tiles > 0 ? tiles : 1), kBfFlatThreads, 0, s,
                           bsource(in.keyA, in.valA, in.tombA, in.prefixA),
                           bsource(in.keyB, in.valB, in.tombB, in.prefixB), refs, N, W, lcp, ctrl,
                           rec_bytes, tile_sum, status)
           : launch_kernel(false, bytefc_lengths_kernel,
                           static_cast<unsigned>(tiles > 0 ? tiles : 1), kBfThreads, 0, s,
                           bsource(in.keyA, in.valA, in.tombA, in.prefixA),
                           bsource(in.keyB, in.valB, in.tombB, in.prefixB), refs, N, W, lcp, ctrl,
                           rec_bytes, tile_sum, status);
  if (err == cudaSuccess) err = launch_fc_offsets(rec_bytes, N, tile_sum, byte_off, s);
  profile_after(s);
  return err;
}

cudaError_t launch_bytefc_value_width(const lsm_fc_input &in, const uint32_t *refs, int64_t N,
                                      uint64_t *d_width, cudaStream_t s) {
  auto *acc = reinterpret_cast<unsigned long long *>(d_width);
  cudaError_t err = cudaMemsetAsync(acc + 1, 0xFF, sizeof(uint64_t), s);
  if (err == cudaSuccess) err = cudaMemsetAsync(acc + 2, 0, 2 * sizeof(uint64_t), s);
  if (err != cudaSuccess) return err;
  if (N > 0) {
    int64_t blocks = (N + 255) / 256;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    if (blocks > cap && cap > 0) blocks = cap;
    err = launch_kernel(false, bytefc_width_reduce_kernel, static_cast<unsigned>(blocks), 256, 0,
                        s, bsource(in.keyA, in.valA, in.tombA), bsource(in.keyB, in.valB, in.tombB),
                        refs, N, acc);
    if (err != cudaSuccess) return err;
  }
  return launch_kernel(false, bytefc_width_finish_kernel, 1, 1, 0, s, N, acc);
}

cudaError_t launch_bytefc_emit(const lsm_fc_input &in, const uint32_t *refs, int64_t N, uint64_t W,
                               const uint32_t *lcp, const uint32_t *ctrl, const uint64_t *byte_off,
                               uint8_t *payload, int64_t nbytes, int32_t *status, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  const int64_t blocks = (N + kBeRecords - 1) / kBeRecords;
  profile_before(s);
  const cudaError_t err = launch_kernel(false, bytefc_emit_kernel, static_cast<unsigned>(blocks),
                                        kBeRecords, 0, s, bsource(in.keyA, in.valA, in.tombA),
                                        bsource(in.keyB, in.valB, in.tombB), refs, N, W, lcp, ctrl,
                                        byte_off, payload, nbytes, status);
  profile_after(s);
  return err;
}

}  // namespace lsm
