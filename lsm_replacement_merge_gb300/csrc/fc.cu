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
//     no FC reset at a cut), and one invocation per final 32-bit word that
//     gathers its bits and writes the word once; unused final bits are zero.
// EG0(x) is the order-0 Exp-Golomb code word: floor(log2(x+1)) zero bits,
// then x+1 in binary; as a number of E(x) bits it is simply x + 1.
//
// fc_lengths_kernel: one CTA per tile of 2048 records (tile ids taken in
// launch order from a counter). Each thread computes eight consecutive
// records; a block scan and a decoupled lookback over the tiles turn the
// lengths into 64-bit offsets in a single pass. Each lookback wait is
// bounded in time; a tile that gives up records LSM_ERR_TIMEOUT and still
// publishes, so no other tile waits on it forever.
//
// fc_emit_kernel: one CTA per run of 256 x WPT payload words. One warp finds
// the first and last record overlapping the run (32-way probes over
// bit_off); each thread then owns WPT consecutive words, finds its first
// record by bisection inside that range, and composes each word from the
// fields of the records that overlap it. The run leaves through shared
// memory with one bulk store.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "strings.cuh"

namespace lsm {

namespace {

constexpr int kFcThreads = 256;
constexpr int kFcItems = 8;
constexpr int kFcTile = kFcThreads * kFcItems;
constexpr int kEmitThreads = 256;
constexpr int kEmitWords = 8;  // words per thread
constexpr int kEmitRun = kEmitThreads * kEmitWords;

__device__ __forceinline__ uint64_t eg0_len(uint64_t x) {
  return 2 * static_cast<uint64_t>(63 - __clzll(static_cast<long long>(x + 1))) + 1;
}

struct Source {
  lsm_bytes key, val;
  const uint32_t *tomb;
};

__device__ __forceinline__ const Source &pick(const Source &a, const Source &b, uint32_t ref) {
  return (ref & LSM_REF_FROM_B) ? b : a;
}

__device__ __forceinline__ bool is_tomb(const Source &s, uint32_t idx) {
  return s.tomb && ((__ldg(s.tomb + (idx >> 5)) >> (idx & 31)) & 1u);
}

// ---- lookback state ------------------------------------------------------------
constexpr uint64_t kFlagAgg = uint64_t(1) << 62;
constexpr uint64_t kFlagInc = uint64_t(2) << 62;
constexpr uint64_t kValMask = (uint64_t(1) << 62) - 1;


template <typename V>
__device__ __forceinline__ V warp_sum(V v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Called by warp 0 of tile t with the tile's aggregate; returns the sum of
// all earlier tiles (to every lane).
__device__ uint64_t lookback(uint64_t *state, uint32_t t, uint64_t agg, int32_t *status) {
  const int lane = threadIdx.x & 31;
  if (t == 0) {
    if (lane == 0) st_relaxed_u64(state, kFlagInc | agg);
    return 0;
  }
  if (lane == 0) st_relaxed_u64(state + t, kFlagAgg | agg);
  uint64_t prefix = 0;
  int64_t base = static_cast<int64_t>(t) - 1;
  const uint64_t t0 = globaltimer_ns();
  bool timed_out = false;
  for (;;) {
    const int64_t idx = base - lane;
    uint64_t v = idx >= 0 ? ld_relaxed_u64(state + idx) : kFlagInc;
    uint32_t polls = 0;
    while (!__all_sync(0xffffffffu, (v >> 62) != 0)) {
      if ((v >> 62) == 0) v = ld_relaxed_u64(state + idx);
      if ((++polls & 31) == 0) {
        const bool late = globaltimer_ns() - t0 > static_cast<uint64_t>(kWaitLimitNs);
        if (__any_sync(0xffffffffu, late)) {
          timed_out = true;
          if ((v >> 62) == 0) v = kFlagInc;  // give up: count the missing tile as zero
        }
      }
    }
    const uint32_t inc = __ballot_sync(0xffffffffu, (v >> 62) == 2);
    if (inc) {
      const int first = __ffs(inc) - 1;  // nearest tile that has its inclusive prefix
      prefix += warp_sum<uint64_t>(lane <= first ? (v & kValMask) : 0);
      break;
    }
    prefix += warp_sum<uint64_t>(v & kValMask);
    base -= 32;
  }
  if (lane == 0) {
    if (timed_out) report(status, LSM_ERR_TIMEOUT);
    st_relaxed_u64(state + t, kFlagInc | ((prefix + agg) & kValMask));
  }
  return prefix;
}

struct FcLayout {
  static constexpr int64_t kRefs = 0;                                   // u32[tile + 1]
  static constexpr int64_t kLcp = align_up((kFcTile + 1) * 4, 16);      // u32[tile]
  static constexpr int64_t kCtrl = kLcp + kFcTile * 4;
  static constexpr int64_t kRec = kCtrl + kFcTile * 4;
  static constexpr int64_t kOff = kRec + kFcTile * 4;                   // u64[tile]
  static constexpr int64_t kScan = kOff + kFcTile * 8;                  // u64[T/32 + 1]
  static constexpr int64_t kBytes = kScan + (kFcThreads / 32 + 2) * 8 + 16;
};

__global__ void __launch_bounds__(kFcThreads) fc_lengths_kernel(
    Source sa, Source sb, const uint32_t *__restrict__ refs, int64_t N, uint32_t *__restrict__ lcp,
    uint32_t *__restrict__ ctrl, uint32_t *__restrict__ rec_bits, uint64_t *__restrict__ bit_off,
    uint64_t *state, uint32_t *tile_counter, int32_t *status) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t *sRefs = reinterpret_cast<uint32_t *>(smem + FcLayout::kRefs);
  uint32_t *sLcp = reinterpret_cast<uint32_t *>(smem + FcLayout::kLcp);
  uint32_t *sCtrl = reinterpret_cast<uint32_t *>(smem + FcLayout::kCtrl);
  uint32_t *sRec = reinterpret_cast<uint32_t *>(smem + FcLayout::kRec);
  uint64_t *sOff = reinterpret_cast<uint64_t *>(smem + FcLayout::kOff);
  uint64_t *sScan = reinterpret_cast<uint64_t *>(smem + FcLayout::kScan);
  __shared__ uint32_t s_tile;
  __shared__ uint64_t s_prefix;
  const int tid = threadIdx.x;
  if (N == 0) {
    if (tid == 0) bit_off[0] = 0;
    return;
  }
  if (tid == 0) s_tile = atomicAdd(tile_counter, 1u);
  __syncthreads();
  const uint32_t t = s_tile;
  const int64_t start = static_cast<int64_t>(t) * kFcTile;
  const int cnt = static_cast<int>(N - start < kFcTile ? N - start : kFcTile);
  // sRefs[x] = refs[start - 1 + x]; sRefs[0] exists only after the first record
  for (int x = tid; x <= cnt; x += kFcThreads)
    if (start - 1 + x >= 0) sRefs[x] = refs[start - 1 + x];
  __syncthreads();

  const int b0 = tid * kFcItems;
  uint64_t sum = 0;
  bool overflow = false;
  if (b0 < cnt) {
    KeyRef prev{nullptr, 0, 0};
    uint64_t k_prev = 0;
    if (start + b0 > 0) {
      const uint32_t pr = sRefs[b0];
      prev = key_at(pick(sa, sb, pr).key, pr & ~LSM_REF_FROM_B);
      k_prev = 8 * (prev.end - prev.begin);
    }
    for (int s = 0; s < kFcItems && b0 + s < cnt; ++s) {
      const int64_t i = start + b0 + s;
      const uint32_t r = sRefs[b0 + s + 1];
      const uint32_t idx = r & ~LSM_REF_FROM_B;
      const Source &src = pick(sa, sb, r);
      const KeyRef cur = key_at(src.key, idx);
      const uint64_t k = 8 * (cur.end - cur.begin);
      const uint64_t l = i == 0 ? 0 : key_bit_lcp(prev, cur);
      const uint64_t c = (i % 15 == 0) ? 1 + l : k_prev - l;
      uint64_t v;
      if (is_tomb(src, idx)) {
        v = 1;
      } else {
        const uint64_t vb = __ldg(src.val.off + idx + 1) - __ldg(src.val.off + idx);
        v = 1 + eg0_len(vb) + 8 * vb;
      }
      const uint64_t L = eg0_len(c) + eg0_len(k - l) + (k - l) + v;
      overflow |= (L > 0xFFFFFFFFull) || (c > 0xFFFFFFFFull);
      sLcp[b0 + s] = static_cast<uint32_t>(l);
      sCtrl[b0 + s] = static_cast<uint32_t>(c);
      sRec[b0 + s] = static_cast<uint32_t>(L);
      sOff[b0 + s] = L;  // length for now, offset after the scan
      sum += L;
      prev = cur;
      k_prev = k;
    }
  }
  if (overflow) report(status, LSM_ERR_OVERFLOW);
  uint64_t agg;
  const uint64_t excl = block_exclusive_sum<kFcThreads, uint64_t>(sum, sScan, &agg);
  if (tid < 32) {
    const uint64_t p = lookback(state, t, agg, status);
    if (tid == 0) s_prefix = p;
  }
  __syncthreads();
  uint64_t run = s_prefix + excl;
  for (int s = 0; s < kFcItems && b0 + s < cnt; ++s) {
    const uint64_t L = sOff[b0 + s];
    sOff[b0 + s] = run;
    run += L;
  }
  __syncthreads();
  for (int x = tid; x < cnt; x += kFcThreads) {
    lcp[start + x] = sLcp[x];
    ctrl[start + x] = sCtrl[x];
    rec_bits[start + x] = sRec[x];
    bit_off[start + x] = sOff[x];
  }
  if (start + cnt == N && tid == 0) bit_off[N] = s_prefix + agg;
}

// ---- emit ------------------------------------------------------------------------
// Places bits [q0, q0 + len) of a W-bit numeric field (MSB first) that sits
// at stream bits [fstart, fstart + W) into the word covering [wb, wb + 32).
__device__ __forceinline__ void put_num(uint32_t &word, int64_t wb, int64_t fstart, int64_t W,
                                        uint64_t V) {
  const int64_t a = fstart > wb ? fstart : wb;
  const int64_t e = fstart + W < wb + 32 ? fstart + W : wb + 32;
  if (a >= e) return;
  const int64_t q0 = a - fstart;
  const int len = static_cast<int>(e - a);
  const uint64_t chunk = (V >> (W - q0 - len)) & ((uint64_t(1) << len) - 1);
  word |= static_cast<uint32_t>(chunk << (32 - (a - wb) - len));
}

// Same for a field whose bits come from an arena, starting at arena bit
// src_bit; the field's bytes end at byte src_end.
__device__ __forceinline__ void put_arena(uint32_t &word, int64_t wb, int64_t fstart, int64_t W,
                                          const uint8_t *arena, uint64_t src_bit, uint64_t src_end) {
  const int64_t a = fstart > wb ? fstart : wb;
  const int64_t e = fstart + W < wb + 32 ? fstart + W : wb + 32;
  if (a >= e) return;
  const uint64_t sbit = src_bit + static_cast<uint64_t>(a - fstart);
  const int len = static_cast<int>(e - a);
  const uint64_t be = load_be64(arena, sbit >> 3, src_end);
  const uint64_t chunk = (be << (sbit & 7)) >> (64 - len);
  word |= static_cast<uint32_t>(chunk << (32 - (a - wb) - len));
}

struct RecordMeta {
  int64_t s, e;        // stream bits [s, e)
  uint64_t c, l, k;    // control, LCP bits, key bits
  KeyRef key;
  bool tomb;
  KeyRef val;
};

__device__ __forceinline__ RecordMeta load_meta(const Source &sa, const Source &sb,
                                                const uint32_t *refs, const uint32_t *lcp,
                                                const uint32_t *ctrl, const uint64_t *bit_off,
                                                int64_t r) {
  RecordMeta M;
  M.s = static_cast<int64_t>(__ldg(bit_off + r));
  M.e = static_cast<int64_t>(__ldg(bit_off + r + 1));
  M.c = __ldg(ctrl + r);
  M.l = __ldg(lcp + r);
  const uint32_t ref = __ldg(refs + r);
  const uint32_t idx = ref & ~LSM_REF_FROM_B;
  const Source &src = pick(sa, sb, ref);
  M.key = key_at(src.key, idx);
  M.k = 8 * (M.key.end - M.key.begin);
  M.tomb = is_tomb(src, idx);
  M.val = M.tomb ? KeyRef{nullptr, 0, 0} : key_at(src.val, idx);
  return M;
}

__device__ __forceinline__ void compose(uint32_t &word, int64_t wb, const RecordMeta &M) {
  const int64_t e1 = static_cast<int64_t>(eg0_len(M.c));
  const uint64_t d = M.k - M.l;
  const int64_t e2 = static_cast<int64_t>(eg0_len(d));
  put_num(word, wb, M.s, e1, M.c + 1);
  put_num(word, wb, M.s + e1, e2, d + 1);
  const int64_t o3 = M.s + e1 + e2;
  put_arena(word, wb, o3, static_cast<int64_t>(d), M.key.arena, 8 * M.key.begin + M.l, M.key.end);
  const int64_t o4 = o3 + static_cast<int64_t>(d);
  if (!M.tomb) {  // a tombstone is the single bit 0, already zero
    const uint64_t vb = M.val.end - M.val.begin;
    const int64_t ev = static_cast<int64_t>(eg0_len(vb));
    put_num(word, wb, o4, 1 + ev, (uint64_t(1) << ev) | (vb + 1));
    put_arena(word, wb, o4 + 1 + ev, static_cast<int64_t>(8 * vb), M.val.arena, 8 * M.val.begin,
              M.val.end);
  }
}

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

__global__ void __launch_bounds__(kEmitThreads) fc_emit_kernel(
    Source sa, Source sb, const uint32_t *__restrict__ refs, int64_t N,
    const uint32_t *__restrict__ lcp, const uint32_t *__restrict__ ctrl,
    const uint64_t *__restrict__ bit_off, uint32_t *__restrict__ payload, int64_t nwords) {
  __shared__ __align__(16) uint32_t sOut[kEmitRun];
  __shared__ int64_t sRange[2];
  const int tid = threadIdx.x;
  const int64_t w0 = static_cast<int64_t>(blockIdx.x) * kEmitRun;
  const int64_t wn = nwords - w0 < kEmitRun ? nwords - w0 : kEmitRun;
  const uint64_t total = N > 0 ? __ldg(bit_off + N) : 0;
  const uint64_t b0 = static_cast<uint64_t>(w0) * 32;
  const bool any = b0 < total;
  if (any && tid < 64) {
    // warp 0: record holding the run's first bit; warp 1: its last bit
    const uint64_t bend = b0 + static_cast<uint64_t>(wn) * 32;
    const uint64_t bit = tid < 32 ? b0 : (bend < total ? bend : total) - 1;
    const int64_t r = warp_record_at(bit_off, 0, N - 1, bit);
    if ((tid & 31) == 0) sRange[tid >> 5] = r;
  }
  __syncthreads();
  const int64_t wfirst = w0 + static_cast<int64_t>(tid) * kEmitWords;
  uint32_t words[kEmitWords];
#pragma unroll
  for (int q = 0; q < kEmitWords; ++q) words[q] = 0u;
  if (any && wfirst < w0 + wn && static_cast<uint64_t>(wfirst) * 32 < total) {
    // this thread's first record, by bisection inside the run's record range
    int64_t lo = sRange[0], hi = sRange[1];
    const uint64_t bit = static_cast<uint64_t>(wfirst) * 32;
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) >> 1;
      if (__ldg(bit_off + mid) <= bit) lo = mid;
      else hi = mid - 1;
    }
    int64_t r = lo;
    RecordMeta M = load_meta(sa, sb, refs, lcp, ctrl, bit_off, r);
#pragma unroll 1
    for (int q = 0; q < kEmitWords; ++q) {
      const int64_t wb = (wfirst + q) * 32;
      if (wfirst + q >= w0 + wn || static_cast<uint64_t>(wb) >= total) break;
      uint32_t word = 0;
      for (;;) {
        compose(word, wb, M);
        if (M.e < wb + 32 && r + 1 < N) {  // the next record starts inside this word
          ++r;
          M = load_meta(sa, sb, refs, lcp, ctrl, bit_off, r);
          continue;
        }
        break;
      }
      words[q] = word;
    }
  }
#pragma unroll
  for (int q = 0; q < kEmitWords; ++q) sOut[tid * kEmitWords + q] = words[q];
  fence_proxy_async_smem();
  __syncthreads();
  const int bulk_words = static_cast<int>(wn) & ~3;
  if (tid == 0) {
    if (bulk_words) bulk_s2g(payload + w0, sOut, static_cast<uint32_t>(bulk_words) * 4);
    bulk_commit();
  }
  for (int x = bulk_words + tid; x < wn; x += kEmitThreads) payload[w0 + x] = sOut[x];
  if (tid == 0) bulk_wait_read_all();
}

Source make_source(const lsm_bytes &key, const lsm_bytes &val, const uint32_t *tomb) {
  return Source{key, val, tomb};
}

}  // namespace

int64_t fc_scan_tiles(int64_t N) { return (N + kFcTile - 1) / kFcTile; }

size_t fc_scan_workspace_bytes(int64_t N) {
  return static_cast<size_t>(256 + align_up(fc_scan_tiles(N) * 8, 256));
}

cudaError_t launch_fc_lengths_scan(const lsm_fc_input &in, const uint32_t *refs, int64_t N,
                                   uint32_t *lcp, uint32_t *ctrl, uint32_t *rec_bits,
                                   uint64_t *bit_off, void *ws, int32_t *status, cudaStream_t s) {
  const int64_t tiles = fc_scan_tiles(N);
  uint32_t *counter = static_cast<uint32_t *>(ws);
  uint64_t *state = reinterpret_cast<uint64_t *>(static_cast<uint8_t *>(ws) + 256);
  cudaError_t err = cudaMemsetAsync(ws, 0, fc_scan_workspace_bytes(N), s);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(fc_lengths_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(FcLayout::kBytes));
  if (err != cudaSuccess) return err;
  profile_before(s);
  fc_lengths_kernel<<<static_cast<unsigned>(tiles > 0 ? tiles : 1), kFcThreads, FcLayout::kBytes, s>>>(
      make_source(in.keyA, in.valA, in.tombA), make_source(in.keyB, in.valB, in.tombB), refs, N, lcp,
      ctrl, rec_bits, bit_off, state, counter, status);
  profile_after(s);
  return cudaGetLastError();
}

cudaError_t launch_fc_emit(const lsm_fc_input &in, const uint32_t *refs, int64_t N,
                           const uint32_t *lcp, const uint32_t *ctrl, const uint64_t *bit_off,
                           uint32_t *payload, int64_t nwords, int32_t * /*status*/, cudaStream_t s) {
  if (nwords == 0) return cudaSuccess;
  const int64_t runs = (nwords + kEmitRun - 1) / kEmitRun;
  profile_before(s);
  fc_emit_kernel<<<static_cast<unsigned>(runs), kEmitThreads, 0, s>>>(
      make_source(in.keyA, in.valA, in.tombA), make_source(in.keyB, in.valB, in.tombB), refs, N, lcp,
      ctrl, bit_off, payload, nwords);
  profile_after(s);
  return cudaGetLastError();
}

}  // namespace lsm
