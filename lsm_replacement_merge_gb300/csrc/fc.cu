// fc.cu -- exact front-compression lengths, their bit-offset scan, and the
// word-owned payload emit.
//
// "Everett: GPU construction experiment":
//   - the control argument: c_i = 1 + l_i when i mod 15 = 0, else
//     k_{i-1} - l_i, with l_i the exact bit LCP with the preceding surviving
//     key (l_0 = 0) and k_i the key length in bits;
//   - the record: EG0(c_i) EG0(k_i - l_i) key bits [l_i, k_i) value, value =
//     0 for a tombstone, else 1 EG0(byte length) bytes; E(x) = 2 floor(log2
//     (x+1)) + 1, so the record length is E(c_i) + E(k_i - l_i) + (k_i - l_i)
//     + v_i; bits MSB first, no padding between records;
//   - exact length scans into bit offsets (no independently encoded chunks,
//     no FC reset at a cut), and a word-owned emit that writes every final
//     32-bit word once; unused final bits are zero. Here the owner of a word
//     is the CTA that owns its run (below), not one thread per word: the
//     thread-per-word gather measured 1130 us on the 4M + 4M strings, the
//     run composition 335 us.
// EG0(x) is the order-0 Exp-Golomb code word: floor(log2(x+1)) zero bits,
// then x+1 in binary; as a number of E(x) bits it is simply x + 1.
//
// fc_lengths_kernel: one CTA per tile of 1024 records; four consecutive
// records per thread: LCP, control, record length; the tile's total goes to
// the workspace. The LCP comes from each key's first 16 bytes, cached once
// per tile (from the key prefix tables when the input carries them, else
// from the arenas); only keys agreeing on all 128 bits read further. fc_tile_scan_kernel (one CTA) turns the tile totals into
// exclusive prefixes, and fc_offsets_kernel adds each tile's prefix to a
// block scan of its record lengths to write the 64-bit bit offsets. (A
// single pass with a decoupled lookback was measured slower: tiles finish
// out of order and a finished tile waits for its predecessors' totals.)
//
// fc_emit_kernel: persistent; each CTA writes a contiguous range of runs of
// 8192 payload words (the word-owned emit at CTA granularity: every global
// word is written once, by the CTA that owns it). The CTA's first run finds
// its first record by 32-way probes over bit_off; in every run one thread
// per record loads that record's metadata and writes its fields into the
// run's word buffer in shared memory (words shared by two fields or records
// are ORed, words inside a key or value field are stored whole), and the run
// leaves with one bulk store.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "fcrecords.cuh"
#include "internal.h"
#include "strings.cuh"

namespace lsm {

namespace {

constexpr int kFcThreads = 256;
constexpr int kFcItems = 4;
constexpr int kFcTile = kFcThreads * kFcItems;
constexpr int kEmitThreads = 256;
constexpr int kEmitWords = 32;  // words per thread
constexpr int kEmitRun = kEmitThreads * kEmitWords;
constexpr int kEmitMaxRec = 1024;  // records one chunk of a run loads at a time

__device__ __forceinline__ uint64_t eg0_len(uint64_t x) {
  return 2 * static_cast<uint64_t>(63 - __clzll(static_cast<long long>(x + 1))) + 1;
}

struct Source {
  lsm_bytes key, val;
  const uint32_t *tomb;
  const uint64_t *prefix;  // the key prefix table (2 words per key), or NULL
};

__device__ __forceinline__ const Source &pick(const Source &a, const Source &b, uint32_t ref) {
  return (ref & LSM_REF_FROM_B) ? b : a;
}



struct FcLayout {
  static constexpr int64_t kRefs = 0;                                   // u32[tile + 1]
  static constexpr int64_t kKb = align_up((kFcTile + 1) * 4, 16);       // u64[tile + 1]
  static constexpr int64_t kKl = kKb + (kFcTile + 1) * 8;               // u32[tile + 1]
  static constexpr int64_t kV = align_up(kKl + (kFcTile + 1) * 4, 16);  // u32[tile] value bits
  static constexpr int64_t kSrc = kV + kFcTile * 4;                     // u8[tile + 1] from B
  static constexpr int64_t kLcp = align_up(kSrc + kFcTile + 1, 16);     // u32[tile]
  static constexpr int64_t kCtrl = kLcp + kFcTile * 4;
  static constexpr int64_t kRec = kCtrl + kFcTile * 4;
  static constexpr int64_t kP0 = align_up(kRec + kFcTile * 4, 16);    // u64[tile + 1] bytes 0..7
  static constexpr int64_t kP1 = kP0 + (kFcTile + 1) * 8;               // u64[tile + 1] bytes 8..15
  static constexpr int64_t kScan = align_up(kP1 + (kFcTile + 1) * 8, 16);  // u64[T/32 + 1]
  static constexpr int64_t kBytes = kScan + (kFcThreads / 32 + 2) * 8 + 16;
};

// 64 bits of an arena's bit stream (MSB first within bytes) starting at bit
// sb, of which the first `need` (1..64) are used: aligned 8-byte loads,
// byte-swapped; the second word is loaded only when the window crosses into
// it, so nothing past the last needed byte's 8-byte word is read.
__device__ __forceinline__ uint64_t bits64_at(const uint8_t *arena, uint64_t sb, int need) {
  const uint64_t *w = reinterpret_cast<const uint64_t *>(arena);
  const uint64_t t = sb >> 6;
  const int sh = static_cast<int>(sb & 63);
  uint64_t v = bswap64(__ldg(w + t)) << sh;
  if (sh + need > 64) v |= bswap64(__ldg(w + t + 1)) >> (64 - sh);
  return v;
}

// Exact bit LCP of two byte strings, clamped to the shorter one.
__device__ __forceinline__ uint64_t bit_lcp(const uint8_t *aa, uint64_t ab, uint64_t alen,
                                            const uint8_t *ba, uint64_t bb, uint64_t blen) {
  const uint64_t L = 8 * (alen < blen ? alen : blen);
  for (uint64_t t = 0; t < L; t += 64) {
    const int need = L - t < 64 ? static_cast<int>(L - t) : 64;
    uint64_t x = bits64_at(aa, 8 * ab + t, need);
    uint64_t y = bits64_at(ba, 8 * bb + t, need);
    if (need < 64) {
      const uint64_t mask = ~uint64_t(0) << (64 - need);
      x &= mask;
      y &= mask;
    }
    if (x != y) return t + static_cast<uint64_t>(__clzll(static_cast<long long>(x ^ y)));
  }
  return L;
}

// One tile of 1024 records per CTA, in phases whose loads are independent
// across records: (1) the refs, (2) every record's key offsets, value bits
// and source, (3) each thread's four consecutive records: bit LCP with the
// predecessor, control, record length; the tile's total is written for the
// offset scan.
__global__ void __launch_bounds__(kFcThreads) fc_lengths_kernel(
    Source sa, Source sb, const uint32_t *__restrict__ refs, int64_t N, uint32_t *__restrict__ lcp,
    uint32_t *__restrict__ ctrl, uint32_t *__restrict__ rec_bits, uint64_t *__restrict__ bit_off,
    uint64_t *tile_sum, int32_t *status) {
  pdl_begin();
  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t *sRefs = reinterpret_cast<uint32_t *>(smem + FcLayout::kRefs);
  uint64_t *sKb = reinterpret_cast<uint64_t *>(smem + FcLayout::kKb);
  uint32_t *sKl = reinterpret_cast<uint32_t *>(smem + FcLayout::kKl);
  uint32_t *sV = reinterpret_cast<uint32_t *>(smem + FcLayout::kV);
  uint8_t *sSrc = smem + FcLayout::kSrc;
  uint32_t *sLcp = reinterpret_cast<uint32_t *>(smem + FcLayout::kLcp);
  uint32_t *sCtrl = reinterpret_cast<uint32_t *>(smem + FcLayout::kCtrl);
  uint32_t *sRec = reinterpret_cast<uint32_t *>(smem + FcLayout::kRec);
  uint64_t *sP0 = reinterpret_cast<uint64_t *>(smem + FcLayout::kP0);
  uint64_t *sP1 = reinterpret_cast<uint64_t *>(smem + FcLayout::kP1);
  uint64_t *sScan = reinterpret_cast<uint64_t *>(smem + FcLayout::kScan);
  const int tid = threadIdx.x;
  if (N == 0) {
    if (tid == 0) bit_off[0] = 0;
    return;
  }
  const uint32_t t = blockIdx.x;
  const int64_t start = static_cast<int64_t>(t) * kFcTile;
  const int cnt = static_cast<int>(N - start < kFcTile ? N - start : kFcTile);
  // slot x holds record start - 1 + x (slot 0: the predecessor, if any)
  const int first = start > 0 ? 0 : 1;
  for (int x = first + tid; x <= cnt; x += kFcThreads) sRefs[x] = refs[start - 1 + x];
  __syncthreads();
  // with prefix tables (the call checks that every non-empty source has
  // one; records name non-empty sources only) the keys' first 16 bytes come
  // with the offsets; otherwise from the arenas, in phase (3)
  const bool tables = sa.prefix != nullptr || sb.prefix != nullptr;
  // (2) four records per thread per round: every load is issued before any
  // result is stored
  for (int x0 = first + tid; x0 <= cnt; x0 += 4 * kFcThreads) {
    uint64_t kb[4], ke[4], vb[4], ve[4], p0[4], p1[4];
    uint32_t tw[4], rr[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int x = x0 + u * kFcThreads;
      const uint32_t r = sRefs[x <= cnt ? x : first];
      rr[u] = r;
      const uint32_t idx = r & ~LSM_REF_FROM_B;
      const Source &src = pick(sa, sb, r);
      kb[u] = __ldg(src.key.off + idx);
      ke[u] = __ldg(src.key.off + idx + 1);
      vb[u] = __ldg(src.val.off + idx);
      ve[u] = __ldg(src.val.off + idx + 1);
      tw[u] = src.tomb ? __ldg(src.tomb + (idx >> 5)) : 0u;
      p0[u] = p1[u] = 0;
      if (tables) {
        const ulonglong2 v = __ldg(reinterpret_cast<const ulonglong2 *>(src.prefix) + idx);
        p0[u] = v.x;
        p1[u] = v.y;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int x = x0 + u * kFcThreads;
      if (x > cnt) continue;
      const uint32_t idx = rr[u] & ~LSM_REF_FROM_B;
      sKb[x] = kb[u];
      sKl[x] = static_cast<uint32_t>(ke[u] - kb[u]);
      sSrc[x] = (rr[u] & LSM_REF_FROM_B) ? 1 : 0;
      sP0[x] = p0[u];
      sP1[x] = p1[u];
      if (x > 0) {
        uint64_t v = 1;  // a tombstone is one bit
        if (!((tw[u] >> (idx & 31)) & 1u)) {
          const uint64_t vbytes = ve[u] - vb[u];
          v = 1 + eg0_len(vbytes) + 8 * vbytes;
        }
        sV[x - 1] = v > 0xFFFFFFFFull ? 0xFFFFFFFFu : static_cast<uint32_t>(v);
      }
    }
  }
  __syncthreads();

  // (3) without prefix tables, every slot's key: its first 16 bytes as two
  // big-endian words (zero past the key's end), each key loaded once
  // although two records compare it; every load is issued before any
  // result is stored
  if (!tables) {
    constexpr int kSlotsPerThread = (kFcTile + 1 + kFcThreads - 1) / kFcThreads;
    uint64_t w0[kSlotsPerThread], w1[kSlotsPerThread];
#pragma unroll
    for (int q = 0; q < kSlotsPerThread; ++q) {
      const int x = first + tid + q * kFcThreads;
      w0[q] = w1[q] = 0;
      if (x <= cnt) {
        const uint8_t *ar = sSrc[x] ? sb.key.arena : sa.key.arena;
        const uint64_t kb = sKb[x], ke = kb + sKl[x];
        load_prefix16(ar, kb, ke, w0[q], w1[q]);
      }
    }
#pragma unroll
    for (int q = 0; q < kSlotsPerThread; ++q) {
      const int x = first + tid + q * kFcThreads;
      if (x <= cnt) {
        sP0[x] = w0[q];
        sP1[x] = w1[q];
      }
    }
  }
  __syncthreads();

  // (4) this thread's four consecutive records: the bit LCP with the
  // predecessor from the cached words (the first differing bit, clamped to
  // the shorter key; past 128 equal bits the keys' further bytes decide),
  // control and record length
  const int b0 = tid * kFcItems;
  uint64_t sum = 0;
  bool overflow = false;
#pragma unroll
  for (int q = 0; q < kFcItems; ++q) {
    if (b0 + q >= cnt) break;
    const int x = b0 + q + 1;  // this record's slot; x - 1 is its predecessor
    const int64_t i = start + b0 + q;
    const uint64_t k = 8 * static_cast<uint64_t>(sKl[x]);
    uint64_t l = 0, k_prev = 0;
    if (i > 0) {
      k_prev = 8 * static_cast<uint64_t>(sKl[x - 1]);
      const uint64_t L = k_prev < k ? k_prev : k;
      const uint64_t d0 = sP0[x - 1] ^ sP0[x], d1 = sP1[x - 1] ^ sP1[x];
      l = d0 ? static_cast<uint64_t>(__clzll(static_cast<long long>(d0)))
             : (d1 ? 64 + static_cast<uint64_t>(__clzll(static_cast<long long>(d1))) : 128);
      if (l > L) l = L;
      if (l == 128 && L > 128) {
        const uint8_t *pa = sSrc[x - 1] ? sb.key.arena : sa.key.arena;
        const uint8_t *ca = sSrc[x] ? sb.key.arena : sa.key.arena;
        l = 128 + bit_lcp(pa, sKb[x - 1] + 16, sKl[x - 1] - 16, ca, sKb[x] + 16, sKl[x] - 16);
      }
    }
    const uint64_t c = (i % 15 == 0) ? 1 + l : k_prev - l;
    const uint64_t Lrec = eg0_len(c) + eg0_len(k - l) + (k - l) + sV[x - 1];
    overflow |= (Lrec > 0xFFFFFFFFull) || (c > 0xFFFFFFFFull) || sV[x - 1] == 0xFFFFFFFFu;
    sLcp[b0 + q] = static_cast<uint32_t>(l);
    sCtrl[b0 + q] = static_cast<uint32_t>(c);
    sRec[b0 + q] = static_cast<uint32_t>(Lrec);
    sum += Lrec;
  }
  if (overflow) report(status, LSM_ERR_OVERFLOW);
  const uint64_t agg = block_sum<kFcThreads, uint64_t>(sum, sScan);
  if (tid == 0) tile_sum[t] = agg;
  for (int x = tid; x < cnt; x += kFcThreads) {
    lcp[start + x] = sLcp[x];
    ctrl[start + x] = sCtrl[x];
    rec_bits[start + x] = sRec[x];
  }
}

// The same lengths when both sources carry key prefix tables, without the
// shared-memory phases: each thread takes kFlatItems consecutive records and
// the record before them (FlatRecords: every load issued before any is
// used) and computes the bit LCP, control and length of each;
// the tile's total goes to tile_sum as above. A record's predecessor is
// loaded again by the thread before it (measured faster than staging the
// tile). The pass waits on those loads, so warps per SM decide its time:
// measured on the 4M + 4M strings (lengths + scan + offsets, L2 flushed),
// 512 threads of two records at two CTAs per SM (64 registers, 32 warps)
// 116-119 us, against 137-144 us for 256 threads of four (107 registers,
// 16 warps), 131-137 us for those at three CTAs per SM (80 registers, with
// spills), 179-182 us for 512 threads at one CTA per SM (72 registers) and
// 175-178 us for 1024 threads of one record (48 registers, one CTA).
#ifndef FC_FLAT_MIN_BLOCKS
#define FC_FLAT_MIN_BLOCKS 2
#endif
#ifndef FC_FLAT_THREADS
#define FC_FLAT_THREADS 512
#endif
constexpr int kFlatThreads = FC_FLAT_THREADS;  // threads of one tile of kFcTile records
constexpr int kFlatItems = kFcTile / kFlatThreads;
static_assert(kFlatItems * kFlatThreads == kFcTile, "a flat tile is one scan tile");
__global__ void __launch_bounds__(kFlatThreads, FC_FLAT_MIN_BLOCKS) fc_lengths_flat_kernel(
    Source sa, Source sb, const uint32_t *__restrict__ refs, int64_t N, uint32_t *__restrict__ lcp,
    uint32_t *__restrict__ ctrl, uint32_t *__restrict__ rec_bits, uint64_t *__restrict__ bit_off,
    uint64_t *tile_sum, int32_t *status) {
  pdl_begin();
  __shared__ uint64_t scratch[kFlatThreads / 32 + 1];
  const int tid = threadIdx.x;
  if (N == 0) {
    if (tid == 0 && blockIdx.x == 0) bit_off[0] = 0;
    return;
  }
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kFcTile + int64_t(tid) * kFlatItems;
  FlatRecords<Source, kFlatItems> R;
  R.load(sa, sb, refs, N, first);
  uint64_t sum = 0;
  bool overflow = false;
#pragma unroll
  for (int q = 0; q < kFlatItems; ++q) {
    const int64_t i = first + q;
    if (i >= N) break;
    const uint64_t k = 8 * (R.ke[q + 1] - R.kb[q + 1]);
    uint64_t l = 0, k_prev = 0;
    if (i > 0) {
      k_prev = 8 * (R.ke[q] - R.kb[q]);
      const uint64_t L = k_prev < k ? k_prev : k;
      l = R.prefix_agree_bits(q);
      if (l > L) l = L;
      if (l == 128 && L > 128) {
        const uint8_t *pa = pick(sa, sb, R.rr[q]).key.arena;
        const uint8_t *ca = pick(sa, sb, R.rr[q + 1]).key.arena;
        l = 128 + bit_lcp(pa, R.kb[q] + 16, R.ke[q] - R.kb[q] - 16, ca, R.kb[q + 1] + 16,
                          R.ke[q + 1] - R.kb[q + 1] - 16);
      }
    }
    uint64_t v = 1;  // a tombstone is one bit
    if (!R.tomb(q)) {
      const uint64_t vbytes = R.ve[q] - R.vb[q];
      v = 1 + eg0_len(vbytes) + 8 * vbytes;
    }
    const uint64_t c = (i % 15 == 0) ? 1 + l : k_prev - l;
    const uint64_t Lrec = eg0_len(c) + eg0_len(k - l) + (k - l) + v;
    overflow |= (Lrec > 0xFFFFFFFFull) || (c > 0xFFFFFFFFull) || (v > 0xFFFFFFFFull);
    lcp[i] = static_cast<uint32_t>(l);
    ctrl[i] = static_cast<uint32_t>(c);
    rec_bits[i] = static_cast<uint32_t>(Lrec);
    sum += Lrec;
  }
  if (overflow) report(status, LSM_ERR_OVERFLOW);
  const uint64_t agg = block_sum<kFlatThreads, uint64_t>(sum, scratch);
  if (tid == 0) tile_sum[blockIdx.x] = agg;
}

// The exclusive prefix sums of the tile totals, in place, by one CTA in
// chunks of kScanThreads * 8; tile_sum[tiles] receives the grand total.
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads) fc_tile_scan_kernel(uint64_t *tile_sum,
                                                                    int64_t tiles) {
  pdl_begin();
  __shared__ uint64_t scratch[kScanThreads / 32 + 1];
  const int tid = threadIdx.x;
  uint64_t carry = 0;
  for (int64_t base = 0; base < tiles; base += kScanThreads * 8) {
    uint64_t v[8];
    uint64_t local = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t idx = base + int64_t(tid) * 8 + u;
      v[u] = idx < tiles ? tile_sum[idx] : 0;
      local += v[u];
    }
    uint64_t total;
    uint64_t run = carry + block_exclusive_sum<kScanThreads, uint64_t>(local, scratch, &total);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t idx = base + int64_t(tid) * 8 + u;
      if (idx < tiles) tile_sum[idx] = run;
      run += v[u];
    }
    carry += total;
  }
  if (tid == 0) tile_sum[tiles] = carry;
}

// bit_off for tile t: its exclusive tile prefix plus a block scan of its
// records' lengths; the last tile also writes bit_off[N], the total.
__global__ void __launch_bounds__(kFcThreads) fc_offsets_kernel(
    const uint32_t *__restrict__ rec_bits, int64_t N, const uint64_t *tile_sum, int64_t tiles,
    uint64_t *__restrict__ bit_off) {
  pdl_begin();
  __shared__ uint64_t scratch[kFcThreads / 32 + 1];
  const int tid = threadIdx.x;
  const int64_t t = blockIdx.x;
  const int64_t start = t * kFcTile;
  const int64_t b0 = start + int64_t(tid) * kFcItems;
  static_assert(kFcItems == 4, "one 16-byte load of lengths per thread");
  // 16-byte accesses when both arrays allow them (a full group of four)
  const uintptr_t addr_bits =
      reinterpret_cast<uintptr_t>(rec_bits) | reinterpret_cast<uintptr_t>(bit_off);
  const bool vec = b0 + 4 <= N && (addr_bits & 15) == 0;
  uint32_t r[4];
  if (vec) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(rec_bits + b0));
    r[0] = v.x;
    r[1] = v.y;
    r[2] = v.z;
    r[3] = v.w;
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) r[q] = b0 + q < N ? __ldg(rec_bits + b0 + q) : 0u;
  }
  const uint64_t local = uint64_t(r[0]) + r[1] + r[2] + r[3];
  uint64_t total;
  uint64_t run = tile_sum[t] + block_exclusive_sum<kFcThreads, uint64_t>(local, scratch, &total);
  uint64_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    o[q] = run;
    run += r[q];
  }
  if (vec) {
    ulonglong2 *dst = reinterpret_cast<ulonglong2 *>(bit_off + b0);
    dst[0] = make_ulonglong2(o[0], o[1]);
    dst[1] = make_ulonglong2(o[2], o[3]);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (b0 + q < N) bit_off[b0 + q] = o[q];
  }
  if (t == tiles - 1 && tid == 0) bit_off[N] = tile_sum[tiles];
}

// ---- emit ------------------------------------------------------------------------
struct RecordMeta {
  int64_t s, e;        // stream bits [s, e)
  uint64_t c, l, k;    // control, LCP bits, key bits
  KeyRef key;
  bool tomb;
  KeyRef val;
};

// Last index r in [lo, hi] with bit_off[r] <= bit (bit_off[lo] <= bit).
__device__ __forceinline__ int64_t warp_record_at(const uint64_t *bit_off, int64_t lo, int64_t hi,
                                                  uint64_t bit) {
  const int lane = threadIdx.x & 31;
  // invariant: bit_off[lo] <= bit; answer in [lo, hi]
  while (hi > lo) {
    const int64_t span = hi - lo;
    const bool last = span <= 32;
    const int64_t p = last ? lo + 1 + lane : lo + 1 + ((int64_t)lane * span) / 32;
    const bool le = (p <= hi) && (__ldg(bit_off + p) <= bit);
    const int cntle = __popc(__ballot_sync(0xffffffffu, le));
    if (last) {
      lo += cntle;
      break;
    }
    // probes are increasing; the cntle first ones satisfy bit_off[p] <= bit
    const int64_t p_le = cntle > 0 ? lo + 1 + ((int64_t)(cntle - 1) * span) / 32 : lo;
    const int64_t p_gt = cntle < 32 ? lo + 1 + ((int64_t)cntle * span) / 32 - 1 : hi;
    lo = p_le;
    hi = p_gt;
  }
  return lo;
}

// Shared-memory layout of one emit run: its output words.
struct EmitLayout {
  static constexpr int64_t kOut = 0;                           // u32[run]
  static constexpr int64_t kBytes = kOut + int64_t(kEmitRun) * 4 + 64;
};

// ---- record-centric composition into a run's word buffer ------------------------
// buf holds the run's words [w0, w0 + wn); only bits in the window [lo, hi)
// are written. Numeric fields (W <= 64 bits, MSB first) OR their chunks in;
// fields copied from an arena store whole words plainly (no other field or
// record shares such a word) and OR the partial ones at their two ends.
__device__ __forceinline__ void put_num_smem(uint32_t *buf, int64_t w0, int64_t lo, int64_t hi,
                                             int64_t p, int W, uint64_t V) {
  int64_t a = p > lo ? p : lo;
  const int64_t e = p + W < hi ? p + W : hi;
  while (a < e) {
    const int64_t wb = a & ~int64_t(31);
    const int64_t ce = e < wb + 32 ? e : wb + 32;
    const int len = static_cast<int>(ce - a);
    const int q0 = static_cast<int>(a - p);
    const uint64_t chunk = (V >> (W - q0 - len)) & ((uint64_t(1) << len) - 1);
    atomicOr(&buf[(wb >> 5) - w0], static_cast<uint32_t>(chunk << (32 - (a - wb) - len)));
    a = ce;
  }
}

// The arena's bit stream (MSB first within each byte) is the concatenation of
// its aligned 32-bit words read big-endian, so the 32 source bits starting
// at any bit are a funnel shift of two such words. A word past the field's
// last byte is never loaded.
__device__ __forceinline__ uint32_t be32_at(const uint8_t *arena, uint64_t t) {
  return __byte_perm(__ldg(reinterpret_cast<const uint32_t *>(arena) + t), 0, 0x0123);
}

// `len` (1..32) bits of the arena's stream starting at bit sb, right-aligned.
__device__ __forceinline__ uint32_t arena_bits(const uint8_t *arena, uint64_t sb, int len) {
  const uint64_t t = sb >> 5;
  const int sh = static_cast<int>(sb & 31);
  uint32_t v = be32_at(arena, t) << sh;
  if (sh + len > 32) v |= be32_at(arena, t + 1) >> (32 - sh);
  return v >> (32 - len);
}

// Copies the bits [p, p + W) of a field read from `arena` at src_bit into the
// run's words, only where they fall in [lo, hi): a partial first word and a
// partial last word are ORed (other fields share them); the full words in
// between, which no other field touches, are stored. Source and destination
// advance together, so every full word is one funnel shift of two
// consecutive source words at a fixed offset.
__device__ __forceinline__ void put_arena_smem(uint32_t *buf, int64_t w0, int64_t lo, int64_t hi,
                                               int64_t p, int64_t W, const uint8_t *arena,
                                               uint64_t src_bit, uint64_t /*src_end*/) {
  int64_t x = p > lo ? p : lo;
  const int64_t e = p + W < hi ? p + W : hi;
  if (x >= e) return;
  uint64_t sb = src_bit + static_cast<uint64_t>(x - p);
  if (x & 31) {  // partial first word
    const int64_t wb = x & ~int64_t(31);
    const int64_t ce = e < wb + 32 ? e : wb + 32;
    const int len = static_cast<int>(ce - x);
    atomicOr(&buf[(wb >> 5) - w0], arena_bits(arena, sb, len) << (wb + 32 - ce));
    sb += static_cast<uint64_t>(len);
    x = ce;
  }
  const int nfull = static_cast<int>((e - x) >> 5);
  if (nfull > 0) {
    // batches of up to 8 words: all source loads of a batch are issued
    // before any is used, so a field costs one load latency per batch
    uint32_t *dst = &buf[(x >> 5) - w0];
    const uint32_t *src = reinterpret_cast<const uint32_t *>(arena) + (sb >> 5);
    const int sh = static_cast<int>(sb & 31);
    const int extra = sh ? 1 : 0;  // a shifted word also takes bits of the next
    if (nfull <= 4) {  // short fields (most values): one batch of at most five loads
      uint32_t w[5];
#pragma unroll
      for (int u = 0; u < 5; ++u)
        w[u] = u < nfull + extra ? __byte_perm(__ldg(src + u), 0, 0x0123) : 0u;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (u < nfull) dst[u] = sh ? __funnelshift_l(w[u + 1], w[u], sh) : w[u];
    } else
    for (int q0 = 0; q0 < nfull; q0 += 8) {
      const int cnt = nfull - q0 < 8 ? nfull - q0 : 8;
      uint32_t w[9];
#pragma unroll
      for (int u = 0; u < 9; ++u)
        w[u] = u < cnt + extra ? __byte_perm(__ldg(src + q0 + u), 0, 0x0123) : 0u;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (u < cnt) dst[q0 + u] = sh ? __funnelshift_l(w[u + 1], w[u], sh) : w[u];
    }
    x += int64_t(32) * nfull;
    sb += uint64_t(32) * nfull;
  }
  if (x < e) {  // partial last word
    const int len = static_cast<int>(e - x);
    atomicOr(&buf[(x >> 5) - w0], arena_bits(arena, sb, len) << (32 - len));
  }
}

// Writes the bits of one record that fall in [lo, hi).
__device__ __forceinline__ void emit_record(uint32_t *buf, int64_t w0, int64_t lo, int64_t hi,
                                            const RecordMeta &M) {
  if (M.e <= lo || M.s >= hi) return;
  const int e1 = static_cast<int>(eg0_len(M.c));
  const uint64_t d = M.k - M.l;
  const int e2 = static_cast<int>(eg0_len(d));
  if (e1 + e2 <= 64) {  // both codes as one field: EG0(c) EG0(d) = (c+1, d+1) in e1 + e2 bits
    put_num_smem(buf, w0, lo, hi, M.s, e1 + e2, ((M.c + 1) << e2) | (d + 1));
  } else {
    put_num_smem(buf, w0, lo, hi, M.s, e1, M.c + 1);
    put_num_smem(buf, w0, lo, hi, M.s + e1, e2, d + 1);
  }
  const int64_t o3 = M.s + e1 + e2;
  put_arena_smem(buf, w0, lo, hi, o3, static_cast<int64_t>(d), M.key.arena, 8 * M.key.begin + M.l,
                 M.key.end);
  const int64_t o4 = o3 + static_cast<int64_t>(d);
  if (!M.tomb) {  // a tombstone is the single bit 0, already zero
    const uint64_t vb = M.val.end - M.val.begin;
    const int ev = static_cast<int>(eg0_len(vb));
    put_num_smem(buf, w0, lo, hi, o4, 1 + ev, (uint64_t(1) << ev) | (vb + 1));
    put_arena_smem(buf, w0, lo, hi, o4 + 1 + ev, static_cast<int64_t>(8 * vb), M.val.arena,
                   8 * M.val.begin, M.val.end);
  }
}

// ---- the same composition in run-relative 32-bit positions ----------------------
// For every record shorter than 2^30 bits (then all its positions fit in 32
// bits): p is a field's first bit relative to the run's first bit (it may
// be negative), the window is [0, H), and buf word j holds run bits
// [32 j, 32 j + 32). The steps are those of put_num_smem, put_arena_smem
// and emit_record, on 32-bit positions.
// A numeric field of 1 <= W <= 64 bits (MSB first) at p, ORed in: the
// value MSB-aligned in 64 bits, shifted into the (at most three) words it
// meets. The run's window starts on a word boundary and no field reaches
// past the stream's end, so keeping the words inside [0, (H + 31) / 32) is
// the whole clip.
__device__ __forceinline__ void put_num32(uint32_t *buf, int H, int p, int W, uint64_t V) {
  const int WN = (H + 31) >> 5;
  const uint64_t a = V << (64 - W);
  const int j = p >> 5;  // floor, p may be negative
  const int r = p & 31;
  if (j >= 0 && j < WN) atomicOr(&buf[j], static_cast<uint32_t>(a >> (32 + r)));
  if (W + r > 32 && j + 1 >= 0 && j + 1 < WN) atomicOr(&buf[j + 1], static_cast<uint32_t>(a >> r));
  if (W + r > 64 && j + 2 >= 0 && j + 2 < WN)
    atomicOr(&buf[j + 2], static_cast<uint32_t>(a << (32 - r)));
}

__device__ __forceinline__ void put_arena32(uint32_t *buf, int H, int p, int W,
                                            const uint8_t *arena, uint64_t src_bit) {
  int x = p > 0 ? p : 0;
  const int e = p + W < H ? p + W : H;
  if (x >= e) return;
  uint64_t sb = src_bit + static_cast<uint64_t>(x - p);
  if (x & 31) {  // partial first word
    const int wb = x & ~31;
    const int ce = e < wb + 32 ? e : wb + 32;
    const int len = ce - x;
    atomicOr(&buf[wb >> 5], arena_bits(arena, sb, len) << (wb + 32 - ce));
    sb += static_cast<uint64_t>(len);
    x = ce;
  }
  const int nfull = (e - x) >> 5;
  if (nfull > 0) {
    uint32_t *dst = &buf[x >> 5];
    const uint32_t *src = reinterpret_cast<const uint32_t *>(arena) + (sb >> 5);
    const int sh = static_cast<int>(sb & 31);
    const int extra = sh ? 1 : 0;  // a shifted word also takes bits of the next
    if (nfull <= 4) {
      uint32_t w[5];
#pragma unroll
      for (int u = 0; u < 5; ++u)
        w[u] = u < nfull + extra ? __byte_perm(__ldg(src + u), 0, 0x0123) : 0u;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (u < nfull) dst[u] = sh ? __funnelshift_l(w[u + 1], w[u], sh) : w[u];
    } else {
      for (int q0 = 0; q0 < nfull; q0 += 8) {
        const int cnt = nfull - q0 < 8 ? nfull - q0 : 8;
        uint32_t w[9];
#pragma unroll
        for (int u = 0; u < 9; ++u)
          w[u] = u < cnt + extra ? __byte_perm(__ldg(src + q0 + u), 0, 0x0123) : 0u;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (u < cnt) dst[q0 + u] = sh ? __funnelshift_l(w[u + 1], w[u], sh) : w[u];
      }
    }
    x += 32 * nfull;
    sb += uint64_t(32) * static_cast<uint64_t>(nfull);
  }
  if (x < e) {  // partial last word
    const int len = e - x;
    atomicOr(&buf[x >> 5], arena_bits(arena, sb, len) << (32 - len));
  }
}

__device__ __forceinline__ void emit_record32(uint32_t *buf, int H, int P, const RecordMeta &M) {
  const int e1 = static_cast<int>(eg0_len(M.c));
  const uint64_t d = M.k - M.l;
  const int e2 = static_cast<int>(eg0_len(d));
  if (e1 + e2 <= 64) {
    put_num32(buf, H, P, e1 + e2, ((M.c + 1) << e2) | (d + 1));
  } else {
    put_num32(buf, H, P, e1, M.c + 1);
    put_num32(buf, H, P + e1, e2, d + 1);
  }
  const int o3 = P + e1 + e2;
  put_arena32(buf, H, o3, static_cast<int>(d), M.key.arena, 8 * M.key.begin + M.l);
  if (!M.tomb) {  // a tombstone is the single bit 0, already zero
    const int o4 = o3 + static_cast<int>(d);
    const uint64_t vb = M.val.end - M.val.begin;
    const int ev = static_cast<int>(eg0_len(vb));
    put_num32(buf, H, o4, 1 + ev, (uint64_t(1) << ev) | (vb + 1));
    put_arena32(buf, H, o4 + 1 + ev, static_cast<int>(8 * vb), M.val.arena, 8 * M.val.begin);
  }
}

// Persistent: CTA c writes the contiguous runs [c R / P, (c + 1) R / P) of
// kEmitRun payload words each (R runs, P CTAs). Only its first run searches
// bit_off for the record holding the run's first bit; in every run each
// thread then loads the metadata of its records among the kEmitMaxRec from
// that record on (more chunks when the run needs more) and composes those
// that meet the run into a shared word buffer at once, with no staging
// arrays and no barrier between loads and composition (measured: 322 us
// against 334.5 us with the metadata staged in shared memory first); the
// record holding the next run's first bit is named by its own thread. Each
// run leaves by one bulk store. One record in flight per thread at five
// CTAs per SM (48 registers): 309-310 us, against 318-319 us for two records
// in flight at four (64 registers), 345 us for one record at six (40
// registers) and 367 us for two at five; then runs of 8192 words with 1024
// records a chunk 301.7 us, against 309.9 us for 4096 words and 512 records,
// 316 us for 8192 words and 512 records, 356 us for 2048 words.
#ifndef EMIT_MIN_BLOCKS
#define EMIT_MIN_BLOCKS 5
#endif
__global__ void __launch_bounds__(kEmitThreads, EMIT_MIN_BLOCKS) fc_emit_kernel(
    Source sa, Source sb, const uint32_t *__restrict__ refs, int64_t N,
    const uint32_t *__restrict__ lcp, const uint32_t *__restrict__ ctrl,
    const uint64_t *__restrict__ bit_off, uint32_t *__restrict__ payload, int64_t nwords) {
  pdl_begin();
  using L = EmitLayout;
  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t *sOut = reinterpret_cast<uint32_t *>(smem + L::kOut);
  __shared__ int64_t sNext2[2];  // record holding run r's first bit, in slot r & 1
  const int tid = threadIdx.x;
  const int64_t runs = (nwords + kEmitRun - 1) / kEmitRun;
  const int64_t P = gridDim.x;
  const int64_t ra = blockIdx.x * runs / P, rb = (blockIdx.x + 1) * runs / P;
  const int64_t total = N > 0 ? static_cast<int64_t>(__ldg(bit_off + N)) : 0;
  if (ra < rb && tid < 32) {
    const int64_t lo0 = ra * kEmitRun * 32;
    int64_t r = 0;
    if (lo0 < total) r = warp_record_at(bit_off, 0, N - 1, static_cast<uint64_t>(lo0));
    if (tid == 0) sNext2[0] = sNext2[1] = r;
  }
  for (int64_t run = ra; run < rb; ++run) {
    const int64_t w0 = run * kEmitRun;
    const int64_t wn = nwords - w0 < kEmitRun ? nwords - w0 : kEmitRun;
    const int64_t lo = w0 * 32;
    const int64_t hi = (w0 + wn) * 32 < total ? (w0 + wn) * 32 : total;
    for (int x = tid; x < kEmitRun; x += kEmitThreads) sOut[x] = 0u;
    __syncthreads();  // this run's first record is set and sOut is clear
    int64_t c0 = sNext2[run & 1];
    // each thread loads its records' metadata and composes them at once (no
    // staging arrays, no barrier between loads and composition); the record
    // holding bit hi names the next run's first record (in the other slot of
    // sNext2, which no thread still reads)
    while (lo < hi) {
      const int R = static_cast<int>(N - c0 < kEmitMaxRec ? N - c0 : kEmitMaxRec);
      bool more = false;
      for (int x = tid; x < R; x += kEmitThreads) {
        const int64_t r = c0 + x;
        const uint32_t ref = __ldg(refs + r);
        const int64_t rs = static_cast<int64_t>(__ldg(bit_off + r));
        const int64_t re = static_cast<int64_t>(__ldg(bit_off + r + 1));
        const uint32_t cc = __ldg(ctrl + r), ll = __ldg(lcp + r);
        const uint32_t idx = ref & ~LSM_REF_FROM_B;
        const Source &src = pick(sa, sb, ref);
        const uint64_t kb = __ldg(src.key.off + idx), ke = __ldg(src.key.off + idx + 1);
        const uint64_t vb = __ldg(src.val.off + idx), ve = __ldg(src.val.off + idx + 1);
        const uint32_t tw = src.tomb ? __ldg(src.tomb + (idx >> 5)) : 0u;
        if (rs <= hi && hi < re) sNext2[(run + 1) & 1] = r;
        if (x == R - 1 && re <= hi && r + 1 < N) {
          // the chunk ends at or before hi: the record after it starts the
          // next run, or the next chunk goes on with this run
          if (re == hi) sNext2[(run + 1) & 1] = r + 1;
          else more = true;
        }
        if (rs >= hi) continue;
        const bool tomb = (tw >> (idx & 31)) & 1u;
        RecordMeta M;
        M.s = rs;
        M.e = re;
        M.c = cc;
        M.l = ll;
        M.key = KeyRef{src.key.arena, kb, ke};
        M.k = 8 * (ke - kb);
        M.tomb = tomb;
        M.val = KeyRef{src.val.arena, tomb ? 0 : vb, tomb ? 0 : ve};
        if (M.e - M.s < (int64_t(1) << 30))
          emit_record32(sOut, static_cast<int>(hi - lo), static_cast<int>(M.s - lo), M);
        else
          emit_record(sOut, w0, lo, hi, M);
      }
      if (!__syncthreads_or(more)) break;
      c0 += R;
    }
    fence_proxy_async_smem();
    __syncthreads();
    const int bulk_words = static_cast<int>(wn) & ~3;
    if (tid == 0) {
      if (bulk_words) bulk_s2g(payload + w0, sOut, static_cast<uint32_t>(bulk_words) * 4);
      bulk_commit();
    }
    for (int x = bulk_words + tid; x < wn; x += kEmitThreads) payload[w0 + x] = sOut[x];
    if (tid == 0) bulk_wait_read_all();
    __syncthreads();  // the store has read sOut before the next run clears it
  }
}

Source make_source(const lsm_bytes &key, const lsm_bytes &val, const uint32_t *tomb,
                   const uint64_t *prefix = nullptr) {
  return Source{key, val, tomb, prefix};
}

}  // namespace

int64_t fc_scan_tiles(int64_t N) { return (N + kFcTile - 1) / kFcTile; }

size_t fc_scan_workspace_bytes(int64_t N) {
  return static_cast<size_t>(256 + align_up(fc_scan_tiles(N) * 8, 256));
}

extern int g_fc_lengths_flat;

cudaError_t launch_fc_lengths_scan(const lsm_fc_input &in, const uint32_t *refs, int64_t N,
                                   uint32_t *lcp, uint32_t *ctrl, uint32_t *rec_bits,
                                   uint64_t *bit_off, void *ws, int32_t *status, cudaStream_t s) {
  const int64_t tiles = fc_scan_tiles(N);
  uint64_t *tile_sum = static_cast<uint64_t *>(ws);  // tiles + 1 entries
  // prefix tables on both sides (an empty side needs none): the flat form
  const bool flat = (in.prefixA || in.m == 0) && (in.prefixB || in.n == 0) &&
                    (in.prefixA || in.prefixB) && g_fc_lengths_flat;
  cudaError_t err = cudaSuccess;
  if (!flat) {
    err = cudaFuncSetAttribute(fc_lengths_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(FcLayout::kBytes));
    if (err != cudaSuccess) return err;
  }
  profile_before(s);
  if (flat)
    err = launch_kernel(false, fc_lengths_flat_kernel, static_cast<unsigned>(tiles > 0 ? tiles : 1),
                        kFlatThreads, 0, s, make_source(in.keyA, in.valA, in.tombA, in.prefixA),
                        make_source(in.keyB, in.valB, in.tombB, in.prefixB), refs, N, lcp, ctrl,
                        rec_bits, bit_off, tile_sum, status);
  else
    err = launch_kernel(false, fc_lengths_kernel, static_cast<unsigned>(tiles > 0 ? tiles : 1),
                        kFcThreads, FcLayout::kBytes, s,
                        make_source(in.keyA, in.valA, in.tombA, in.prefixA),
                        make_source(in.keyB, in.valB, in.tombB, in.prefixB), refs, N, lcp, ctrl,
                        rec_bits, bit_off, tile_sum, status);
  if (err == cudaSuccess && N > 0)
    // the one-CTA scan and the offsets pass after it launch early (PDL): an
    // early-launched CTA here holds no room that a wave before it needs
    // (measured: lengths + scan 179.8 us against 184.5 us)
    err = launch_kernel(true, fc_tile_scan_kernel, 1u, kScanThreads, 0, s, tile_sum, tiles);
  if (err == cudaSuccess && N > 0)
    err = launch_kernel(true, fc_offsets_kernel, static_cast<unsigned>(tiles), kFcThreads, 0, s,
                        rec_bits, N, tile_sum, tiles, bit_off);
  profile_after(s);  // the profiled span covers all three launches
  return err;
}

int64_t fc_tile_records() { return kFcTile; }

// 1: the flat lengths kernel when prefix tables are given (the default);
// 0: always the staged one (for comparison).
#ifndef FC_LENGTHS_FLAT
#define FC_LENGTHS_FLAT 1
#endif
int g_fc_lengths_flat = FC_LENGTHS_FLAT;

cudaError_t launch_fc_offsets(const uint32_t *rec, int64_t N, uint64_t *tile_sum, uint64_t *off,
                              cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  const int64_t tiles = fc_scan_tiles(N);
  cudaError_t err = launch_kernel(true, fc_tile_scan_kernel, 1u, kScanThreads, 0, s, tile_sum, tiles);
  if (err == cudaSuccess)
    err = launch_kernel(true, fc_offsets_kernel, static_cast<unsigned>(tiles), kFcThreads, 0, s,
                        rec, N, static_cast<const uint64_t *>(tile_sum), tiles, off);
  return err;
}

cudaError_t launch_fc_emit(const lsm_fc_input &in, const uint32_t *refs, int64_t N,
                           const uint32_t *lcp, const uint32_t *ctrl, const uint64_t *bit_off,
                           uint32_t *payload, int64_t nwords, int32_t * /*status*/, cudaStream_t s) {
  if (nwords == 0) return cudaSuccess;
  const int64_t runs = (nwords + kEmitRun - 1) / kEmitRun;
  static bool configured = false;
  if (!configured) {
    cudaError_t err = cudaFuncSetAttribute(fc_emit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(EmitLayout::kBytes));
    if (err != cudaSuccess) return err;
    configured = true;
  }
  static int per_sm = 0;
  if (!per_sm) {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, fc_emit_kernel, kEmitThreads,
                                                      EmitLayout::kBytes) != cudaSuccess)
      v = 1;
    per_sm = v > 0 ? v : 1;
  }
  int64_t grid = static_cast<int64_t>(device_sm_count()) * per_sm;
  if (grid < 1) grid = 1;
  if (grid > runs) grid = runs;
  profile_before(s);
  const cudaError_t err = launch_kernel(false, fc_emit_kernel, static_cast<unsigned>(grid),
                                        kEmitThreads, EmitLayout::kBytes, s,
                                        make_source(in.keyA, in.valA, in.tombA),
                                        make_source(in.keyB, in.valB, in.tombB), refs, N, lcp, ctrl,
                                        bit_off, payload, nwords);
  profile_after(s);
  return err;
}

}  // namespace lsm
