// replace.cu -- collision bitmap, rank512 directory and the replacement merge
// of two strictly sorted unique-key inputs (uint64 keys).
//
// "Everett: collision bitmap and rank experiment":
//   - "Corrected record ordinals": C_i = 1 exactly when A_i's key is in B;
//     R(i) = sum_{t<i} C_t; a surviving A_i lands at i + lower_bound(B, A_i)
//     - R(i) and B_j, with lower bound i in A, at j + i - R(i).
//   - "Temporary rank layouts": per 512-bit block a 32-bit absolute prefix
//     and seven 9-bit prefixes at 64-bit granularity; a query reads the
//     directory, at most one preceding 32-bit word and the masked current
//     word.
//   - "The three experimental paths", third path: survivors of A and all of
//     B have disjoint keys and are merged by merge path.
//
// GPU design (both tile kernels run on the persistent, warp-specialized
// pipeline of pipeline.cuh: a producer warp stages each merge-path tile with
// bulk copies while the consumer warps work on the previous one):
//   collision_mark   partition (co-rank per tile, A first on ties; the same
//                    launch clears C), then per tile: the stage holds
//                    A[i0-1, i1) and B[j0, j1]; every B key of the tile takes
//                    its lower bound in the staged A span ([CB]: "for each B
//                    record, find its lower bound in A") by a two-level
//                    search (group heads of 32 keys over the whole span, then
//                    each key between its head's bound and the next); a
//                    match sets the collision bit. Each
//                    bit is set by the tile that owns its A index (the last A is
//                    checked against the first B after the tile), so bitmap
//                    words inside one tile take plain stores and only
//                    boundary words need atomicOr.
//   rank_build       one launch with a decoupled lookback over CTA totals
//                    when all CTAs fit on the device at once; otherwise
//                    count -> prefix -> finish in two launches ([CB]
//                    "Dispatch bindings"); at least one block for empty A.
//   compact          merge path over positions: B_j precedes A_i exactly when
//                    lb_B[j] <= i (this is B_j <= A_i, since lb_B[j] counts the
//                    A keys below B_j), so the merge of surviving A and B
//                    needs lb_B and C only, never the keys. In a tile with
//                    co-rank i0 at diagonal k0, B_j sits at slot
//                    (j - j0) + (lb_B[j] - i0); a bitmap of those slots and
//                    prefix popcounts over it and over C give every slot its
//                    element and its output position, k0 - R(i0) + slot -
//                    (dropped A records before the slot), where R(i0) is a
//                    rank query. Refs and ordinals leave by bulk stores.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "rank512.cuh"
#include "internal.h"
#include "lookback.cuh"
#include "pipeline.cuh"

namespace lsm {

namespace {

// ---- partition: co-rank per tile -----------------------------------------------
// uint64 keys, A first on ties.
struct U64AFirst {
  const uint64_t *A;
  const uint64_t *B;
  __device__ __forceinline__ bool too_small(int64_t i, int64_t k) const {
    return __ldg(A + i) <= __ldg(B + k - i - 1);
  }
};

// The co-rank of every tile boundary, each found by a group of
// kPartitionLanes lanes (group_corank); the launch also clears
// `clear_words`. With a few thousand boundaries the searches are bound by
// their dependent rounds of loads, and four lanes (five-way splits) cut the
// rounds from about 24 to 10 for fourfold the loads: the best measured.
#ifndef LSM_MARK_PARTITION_LANES
#define LSM_MARK_PARTITION_LANES 4
#endif
constexpr int kPartitionLanes = LSM_MARK_PARTITION_LANES;

template <class Pred>
__global__ void __launch_bounds__(256) partition_kernel(Pred pred, int64_t m, int64_t n, int64_t D,
                                                        int64_t G, int64_t *__restrict__ out_i,
                                                        uint32_t *__restrict__ clear_words,
                                                        int64_t nclear,
                                                        uint64_t *__restrict__ clear_states,
                                                        int64_t nstates) {
  pdl_begin();
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (clear_words) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t w = gtid; w < nclear; w += stride) clear_words[w] = 0u;
  }
  if (clear_states) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t w = gtid; w < nstates; w += stride) clear_states[w] = 0u;
  }
  const int64_t g = gtid / kPartitionLanes;
  const bool active = g <= G;
  const int64_t total = m + n;
  const int64_t k = active ? (g * D < total ? g * D : total) : 0;
  const int64_t i = group_corank<kPartitionLanes>(pred, k, m, n, active);
  if (active && (threadIdx.x & (kPartitionLanes - 1)) == 0) out_i[g] = i;
}

template <class Pred>
cudaError_t launch_partition(const Pred &pred, int64_t m, int64_t n, int64_t D, int64_t *out_i,
                             uint32_t *clear_words, int64_t nclear, cudaStream_t s,
                             uint64_t *clear_states = nullptr, int64_t nstates = 0) {
  const int64_t G = (m + n + D - 1) / D;
  int64_t threads = (G + 1) * kPartitionLanes;
  if (clear_words && threads < nclear / 4) threads = nclear / 4;
  const int64_t blocks = (threads + 255) / 256;
  return launch_kernel(true, partition_kernel<Pred>, static_cast<unsigned>(blocks), 256, 0, s, pred,
                       m, n, D, G, out_i, clear_words, nclear, clear_states, nstates);
}

// ---- rank512 --------------------------------------------------------------------
__device__ __forceinline__ void load_block_words(const uint32_t *__restrict__ C, int64_t nwords,
                                                 int64_t b, uint32_t w[16]) {
  const int64_t base = b * 16;
  if (base + 16 <= nwords) {
    const uint4 *p = reinterpret_cast<const uint4 *>(C + base);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = p[q];
      w[4 * q] = v.x;
      w[4 * q + 1] = v.y;
      w[4 * q + 2] = v.z;
      w[4 * q + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int t = 0; t < 16; ++t) w[t] = base + t < nwords ? C[base + t] : 0u;
  }
}

__global__ void __launch_bounds__(kRankThreads) rank_count_kernel(const uint32_t *__restrict__ C,
                                                                  int64_t m,
                                                                  uint32_t *__restrict__ cta_totals) {
  pdl_begin();
  __shared__ uint32_t scratch[kRankThreads / 32 + 1];
  const int64_t nwords = (m + 31) / 32;
  const int64_t nblk = m / 512 + 1;
  const int64_t b = static_cast<int64_t>(blockIdx.x) * kRankThreads + threadIdx.x;
  uint32_t pc = 0;
  if (b < nblk) {
    uint32_t w[16];
    load_block_words(C, nwords, b, w);
#pragma unroll
    for (int t = 0; t < 16; ++t) pc += __popc(w[t]);
  }
  const uint32_t total = block_sum<kRankThreads>(pc, scratch);
  if (threadIdx.x == 0) cta_totals[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kRankThreads) rank_finish_kernel(const uint32_t *__restrict__ C,
                                                                   int64_t m,
                                                                   const uint32_t *__restrict__ cta_totals,
                                                                   uint32_t *__restrict__ dir,
                                                                   int64_t *__restrict__ d_total) {
  pdl_begin();
  __shared__ uint32_t scratch[kRankThreads / 32 + 1];
  const int64_t nwords = (m + 31) / 32;
  const int64_t nblk = m / 512 + 1;
  // global prefix: the totals of every CTA before this one
  uint32_t acc = 0;
  for (int64_t x = threadIdx.x; x < blockIdx.x; x += kRankThreads) acc += cta_totals[x];
  const uint32_t prefix = block_sum<kRankThreads>(acc, scratch);

  const int64_t b = static_cast<int64_t>(blockIdx.x) * kRankThreads + threadIdx.x;
  uint32_t cum[8];
  uint32_t tot = 0;
  if (b < nblk) {
    uint32_t w[16];
    load_block_words(C, nwords, b, w);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      cum[s] = tot;  // popcount of the block's first s 64-bit words
      tot += __popc(w[2 * s]) + __popc(w[2 * s + 1]);
    }
  }
  uint32_t cta_sum;
  const uint32_t excl = block_exclusive_sum<kRankThreads>(b < nblk ? tot : 0u, scratch, &cta_sum);
  if (b < nblk) {
    uint64_t packed = 0;
#pragma unroll
    for (int s = 1; s < 8; ++s) packed |= static_cast<uint64_t>(cum[s]) << (9 * (s - 1));
    dir[3 * b] = prefix + excl;
    dir[3 * b + 1] = static_cast<uint32_t>(packed);
    dir[3 * b + 2] = static_cast<uint32_t>(packed >> 32);
  }
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) *d_total = static_cast<int64_t>(prefix) + cta_sum;
}

// The rank layout the earlier compaction reads R(i) from: the 512-bit
// directory above.
struct Rank512Dir {
  const uint32_t *dir;
  __device__ __forceinline__ uint64_t at(const uint32_t *__restrict__ C, int64_t p) const {
    return rank512_at(C, dir, p);
  }
};

// The compaction's partition, by a scan over lb_B instead of one search per
// boundary. With B first on ties, B_j sits at merged position
// p_j = j + lb_B[j] (strictly increasing, below 2^32), so the co-rank of
// diagonal k is i(k) = k - #{j : p_j < k}. A block takes the
// kPosPerBlock records [jb, je) and owns the boundaries whose diagonal lies
// in (p_{jb-1}, p_{je-1}] (the first block from k = 0, the last one up to
// k = m + n); for each it counts the positions below k by a bisection over
// the block's positions in shared memory. Results are clamped to the
// diagonal's valid range, so an lb_B that is not a lower-bound array cannot
// produce an out-of-range tile. Block 0 also writes the survivor count
// N = m + n - R(m).
constexpr int kPosThreads = 256;
constexpr int kPosItems = 8;
constexpr int kPosPerBlock = kPosThreads * kPosItems;

template <class RD>
__global__ void __launch_bounds__(kPosThreads) partition_positions_kernel(
    const uint32_t *__restrict__ lb_B, int64_t m, int64_t n, int64_t D, int64_t G,
    int64_t *__restrict__ out_i, const uint32_t *__restrict__ C, RD rank,
    int64_t *__restrict__ d_count) {
  pdl_begin();
  __shared__ uint32_t sp[kPosPerBlock];
  __shared__ int64_t sRange[2];
  const int t = threadIdx.x;
  const int64_t jb = static_cast<int64_t>(blockIdx.x) * kPosPerBlock;
  const int cnt = static_cast<int>(n - jb < kPosPerBlock ? n - jb : kPosPerBlock);
  if (blockIdx.x == 0 && t == 0 && d_count)
    *d_count = m + n - static_cast<int64_t>(rank.at(C, m));
  // kPosItems consecutive records per thread: two 16-byte loads when the
  // block is full (lb_B is 16-byte aligned and jb a multiple of 2048)
  const int x0 = t * kPosItems;
  if (cnt == kPosPerBlock) {
    const uint4 *q = reinterpret_cast<const uint4 *>(lb_B + jb + x0);
    const uint4 u = __ldg(q), v = __ldg(q + 1);
    const uint32_t lb[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < kPosItems; ++e) sp[x0 + e] = static_cast<uint32_t>(jb + x0 + e) + lb[e];
  } else {
#pragma unroll
    for (int e = 0; e < kPosItems; ++e)
      if (x0 + e < cnt) sp[x0 + e] = static_cast<uint32_t>(jb + x0 + e) + __ldg(lb_B + jb + x0 + e);
  }
  __syncthreads();
  if (t == 0) {
    // boundaries g with p_{jb-1} < g D <= p_{je-1}
    const bool last = jb + cnt >= n;
    int64_t g_lo = 0;
    if (jb > 0) g_lo = ((jb - 1) + static_cast<int64_t>(__ldg(lb_B + jb - 1))) / D + 1;
    int64_t g_hi = G;
    if (!last) {
      const int64_t q = static_cast<int64_t>(sp[cnt - 1]) / D;
      g_hi = q < G ? q : G;
    }
    sRange[0] = g_lo;
    sRange[1] = g_hi;
  }
  __syncthreads();
  const int64_t total = m + n;
  const int64_t g_hi = sRange[1];
  for (int64_t g = sRange[0] + t; g <= g_hi; g += kPosThreads) {
    const int64_t k = g * D < total ? g * D : total;
    int lo = 0, hi = cnt;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (static_cast<int64_t>(sp[mid]) < k) lo = mid + 1;
      else hi = mid;
    }
    int64_t i = k - (jb + lo);
    const int64_t ilo = k > n ? k - n : 0, ihi = k < m ? k : m;
    i = i < ilo ? ilo : (i > ihi ? ihi : i);
    out_i[g] = i;
  }
}

// Single-launch rank512 build: every CTA counts its 256 blocks, publishes
// its total, looks back over its predecessors for the prefix (decoupled
// lookback) and writes its entries. The state words are zero at launch (the
// launcher clears them, or a kernel earlier on the stream did). Used only
// when all CTAs are resident at once, so every CTA a lookback waits for is
// running; each wait is bounded in time.
__global__ void __launch_bounds__(kRankThreads) rank_single_kernel(const uint32_t *__restrict__ C,
                                                                   int64_t m,
                                                                   uint32_t *__restrict__ dir,
                                                                   int64_t *__restrict__ d_total,
                                                                   uint64_t *state,
                                                                   int32_t *status) {
  pdl_begin();
  __shared__ uint32_t scratch[kRankThreads / 32 + 1];
  __shared__ uint32_t s_prefix;
  const int64_t nwords = (m + 31) / 32;
  const int64_t nblk = m / 512 + 1;
  const uint32_t t = blockIdx.x;
  const int64_t b = static_cast<int64_t>(t) * kRankThreads + threadIdx.x;
  uint32_t cum[8];
  uint32_t tot = 0;
  if (b < nblk) {
    uint32_t w[16];
    load_block_words(C, nwords, b, w);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      cum[s] = tot;
      tot += __popc(w[2 * s]) + __popc(w[2 * s + 1]);
    }
  }
  uint32_t agg;
  const uint32_t excl = block_exclusive_sum<kRankThreads>(b < nblk ? tot : 0u, scratch, &agg);
  if (threadIdx.x < 32) {
    const uint32_t prefix = lookback_exclusive(state, t, agg, status);
    if (threadIdx.x == 0) s_prefix = prefix;
  }
  __syncthreads();
  const uint32_t prefix = s_prefix;
  if (b < nblk) {
    uint64_t packed = 0;
#pragma unroll
    for (int s = 1; s < 8; ++s) packed |= static_cast<uint64_t>(cum[s]) << (9 * (s - 1));
    dir[3 * b] = prefix + excl;
    dir[3 * b + 1] = static_cast<uint32_t>(packed);
    dir[3 * b + 2] = static_cast<uint32_t>(packed >> 32);
  }
  if (t == gridDim.x - 1 && threadIdx.x == 0) *d_total = static_cast<int64_t>(prefix) + agg;
}

__global__ void __launch_bounds__(256) rank_query_kernel(const uint32_t *__restrict__ C,
                                                         const uint32_t *__restrict__ dir, int64_t m,
                                                         const uint32_t *__restrict__ pos, int64_t q,
                                                         uint32_t *__restrict__ out, int32_t *status) {
  pdl_begin();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= q) return;
  const int64_t p = pos[t];
  if (p > m) {
    out[t] = 0xFFFFFFFFu;
    report(status, LSM_ERR_ARG);
    return;
  }
  out[t] = rank512_at(C, dir, p);
}

// ---- materialized survivors -------------------------------------------------------
// Four consecutive output records per thread (a warp covers 128), grid-stride
// over [0, N) with N = d_count[0] read on the device. Each lane copies its
// records' keys and values from the inputs their refs name, with 16-byte
// loads of refs and 16-byte stores of keys and values; its four tombstone
// flags form a nibble, and eight lanes' nibbles one word of the output
// bitmap. A count past m + n or a ref past its input records LSM_ERR_ARG
// and writes nothing for that record. refs, out_keys and out_vals are
// 16-byte aligned.
__global__ void __launch_bounds__(256) materialize_kernel(
    const uint64_t *__restrict__ A, const uint32_t *__restrict__ Aval,
    const uint32_t *__restrict__ tombA, int64_t m, const uint64_t *__restrict__ B,
    const uint32_t *__restrict__ Bval, const uint32_t *__restrict__ tombB, int64_t n,
    const uint32_t *__restrict__ refs, const int64_t *__restrict__ d_count,
    uint64_t *__restrict__ out_keys, uint32_t *__restrict__ out_vals,
    uint32_t *__restrict__ out_tomb, int32_t *status) {
  pdl_begin();
  const int64_t N = *d_count;
  if (N < 0 || N > m + n) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(status, LSM_ERR_ARG);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
       w * 128 < N; w += warps) {
    const int64_t t0 = w * 128 + 4 * lane;
    uint32_t r[4] = {0u, 0u, 0u, 0u};
    if (t0 + 4 <= N) {
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(refs + t0));
      r[0] = v.x;
      r[1] = v.y;
      r[2] = v.z;
      r[3] = v.w;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (t0 + q < N) r[q] = __ldg(refs + t0 + q);
    }
    uint64_t key[4] = {0, 0, 0, 0};
    uint32_t val[4] = {0u, 0u, 0u, 0u};
    uint32_t nib = 0;
    bool ok[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const bool from_b = (r[q] & LSM_REF_FROM_B) != 0;
      const int64_t idx = r[q] & ~LSM_REF_FROM_B;
      ok[q] = t0 + q < N && idx < (from_b ? n : m);
      if (t0 + q < N && !ok[q]) report(status, LSM_ERR_ARG);
      if (ok[q]) {
        key[q] = __ldg((from_b ? B : A) + idx);
        if (out_vals) val[q] = __ldg((from_b ? Bval : Aval) + idx);
        const uint32_t *tb = from_b ? tombB : tombA;
        if (tb && ((__ldg(tb + (idx >> 5)) >> (idx & 31)) & 1u)) nib |= 1u << q;
      }
    }
    if (ok[0] && ok[1] && ok[2] && ok[3]) {
      ulonglong2 *kd = reinterpret_cast<ulonglong2 *>(out_keys + t0);
      kd[0] = make_ulonglong2(key[0], key[1]);
      kd[1] = make_ulonglong2(key[2], key[3]);
      if (out_vals)
        *reinterpret_cast<uint4 *>(out_vals + t0) = make_uint4(val[0], val[1], val[2], val[3]);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (!ok[q]) continue;
        out_keys[t0 + q] = key[q];
        if (out_vals) out_vals[t0 + q] = val[q];
      }
    }
    // lanes 8k .. 8k+7 hold the 32 flags of bitmap word 4w + k
    uint32_t word = nib << (4 * (lane & 7));
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    word |= __shfl_xor_sync(0xffffffffu, word, 4);
    if (out_tomb && (lane & 7) == 0 && w * 128 + 4 * lane < N) out_tomb[4 * w + (lane >> 3)] = word;
  }
}

// ---- collision mark ------------------------------------------------------------
// One merge-path tile per pipeline step. The stage holds A[i0 - hp, i1) and
// B[j0, j1 + hn): one A key before the span (for the lower bounds of B's
// first keys) and one B key after it (for the collision bit of A's last key).
template <int T_, int E_, int S_>
struct MarkSpec {
  static constexpr int T = T_;
  static constexpr int E = E_;
  static constexpr int S = S_;
  static constexpr int D = T * E;
  static constexpr int64_t kStageBytes = align_up(int64_t(D + 4) * 8 + 160, 16);
  static constexpr int64_t kLB = 0;
  static constexpr int64_t kCw = align_up(int64_t(D + 8) * 4, 16);
  static constexpr int64_t kQ = kCw + align_up(int64_t(D / 32 + 4) * 4, 16);
  static constexpr int64_t kWorkBytes = kQ + align_up(int64_t(D / 32 + 2) * 4, 16);
  struct Params {
    const uint64_t *A, *B;
    int64_t m, n;
    const int64_t *part_i;
    uint32_t *C, *lb_B;
  };
  struct Desc {
    int64_t i0, j0;
    int32_t na, nb, hp, hn, offA, offB;
  };
  __device__ __forceinline__ static void init(uint8_t *work) {
    uint32_t *sCw = reinterpret_cast<uint32_t *>(work + kCw);
    for (int x = threadIdx.x; x < D / 32 + 4; x += T) sCw[x] = 0u;
  }
  __device__ __forceinline__ static void fetch(const Params &p, int64_t g, int64_t v[4]) {
    v[0] = __ldg(p.part_i + g);
    v[1] = __ldg(p.part_i + g + 1);
  }
  __device__ __forceinline__ static void produce(const Params &p, int64_t g, const int64_t v[4], uint8_t *stage,
                                 Desc &d, uint64_t *full) {
    const int64_t total = p.m + p.n;
    const int64_t i0 = v[0], i1 = v[1];
    const int64_t k0 = g * D, k1 = k0 + D < total ? k0 + D : total;
    const int64_t j0 = k0 - i0, j1 = k1 - i1;
    const int na = static_cast<int>(i1 - i0), nb = static_cast<int>(j1 - j0);
    const int hp = i0 > 0 ? 1 : 0, hn = j1 < p.n ? 1 : 0;
    const StagePlan pa = stage_plan_overfetch<8>(i0 - hp, na + hp, p.m);
    const StagePlan pb = stage_plan_overfetch<8>(j0, nb + hn, p.n);
    uint64_t *bufA = reinterpret_cast<uint64_t *>(stage);
    const int32_t offB = static_cast<int32_t>(stage_capacity_bytes<8>(pa.span) / 8);
    uint64_t *bufB = bufA + offB;
    for (int64_t x = pa.tail_from; x < i1; ++x) bufA[x - pa.first] = p.A[x];
    for (int64_t x = pb.tail_from; x < j1 + hn; ++x) bufB[x - pb.first] = p.B[x];
    d.i0 = i0;
    d.j0 = j0;
    d.na = na;
    d.nb = nb;
    d.hp = hp;
    d.hn = hn;
    d.offA = pa.lead + hp;
    d.offB = offB + pb.lead;
    mbar_arrive_expect_tx(full, pa.bulk + pb.bulk);
    stage_issue(bufA, p.A, pa, full);
    stage_issue(bufB, p.B, pb, full);
  }
  __device__ __forceinline__ static void consume(const Params &p, int64_t g, const Desc &dd, const uint8_t *stage,
                                 uint8_t *work, uint64_t *empty) {
    const int tid = threadIdx.x;
    const uint64_t *sA = reinterpret_cast<const uint64_t *>(stage) + dd.offA;  // sA[-1] = A[i0-1]
    const uint64_t *sB = reinterpret_cast<const uint64_t *>(stage) + dd.offB;  // sB[nb] = B[j1]
    uint32_t *sLBbuf = reinterpret_cast<uint32_t *>(work + kLB);
    uint32_t *sCw = reinterpret_cast<uint32_t *>(work + kCw);
    int *sQ = reinterpret_cast<int *>(work + kQ);
    const int na = dd.na, nb = dd.nb, hp = dd.hp, hn = dd.hn;
    const int64_t i0 = dd.i0, j0 = dd.j0, i1 = i0 + na;
    uint32_t *sLB = sLBbuf + (j0 & 3);  // global alignment of lb_B[j0] mirrored
    const int64_t w0 = i0 >> 5;
    const int wbit0 = static_cast<int>(i0 - (w0 << 5));  // bit of A[i0] in word w0
    // Every B key of the tile has its lower bound in the staged span
    // A[i0 - hp, i1] (A[i0-1] included when it exists). Two levels: one
    // thread per group of 32 consecutive B keys finds the group head's bound
    // over the whole span; then each B key searches only between its group
    // head's bound and the next head's. A warp's 32 lanes hold one group, so
    // they share the range and the number of steps.
    const uint64_t *sAx = sA - hp;
    const int lenx = na + hp;
    const uint32_t base = static_cast<uint32_t>(i0 - hp);
    const int ngroups = (nb + 31) >> 5;
    for (int q = tid; q < ngroups; q += T) {
      const uint64_t key = sB[q << 5];
      int lo = 0, hi = lenx;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (sAx[mid] < key) lo = mid + 1;
        else hi = mid;
      }
      sQ[q] = lo;
    }
    if (tid == 0) sQ[ngroups] = lenx;
    named_sync(1, T);
    for (int bi = tid; bi < nb; bi += T) {
      const uint64_t key = sB[bi];
      const int q = bi >> 5;
      int lo = sQ[q], hi = (bi & 31) ? sQ[q + 1] : lo;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (sAx[mid] < key) lo = mid + 1;
        else hi = mid;
      }
      sLB[bi] = base + static_cast<uint32_t>(lo);
      // A collision with A[i0-1] belongs to the previous tile, which finds it
      // by peeking at this B key.
      if (lo < lenx && lo >= hp && sAx[lo] == key) {
        const int x = wbit0 + (lo - hp);
        atomicOr(&sCw[x >> 5], 1u << (x & 31));
      }
    }
    // the tile's last A against the first B after the tile
    if (tid == 0 && hn && na > 0 && sA[na - 1] == sB[nb]) {
      const int x = wbit0 + na - 1;
      atomicOr(&sCw[x >> 5], 1u << (x & 31));
    }
    release_stage(empty);
    fence_proxy_async_smem();
    named_sync(1, T);
    store_u32_run<T>(p.lb_B, j0, nb, sLBbuf);
    if (tid == 0) bulk_commit();
    const int nw = na > 0 ? static_cast<int>(((i1 - 1) >> 5) - w0 + 1) : 0;
    for (int x = tid; x < nw; x += T) {
      const int64_t w = w0 + x;
      const uint32_t bits = sCw[x];
      sCw[x] = 0u;  // clean for the next tile
      if (w * 32 >= i0 && w * 32 + 32 <= i1) p.C[w] = bits;
      else if (bits) atomicOr(&p.C[w], bits);
    }
    if (tid == 0) bulk_wait_read_all();  // sLB is rewritten by the next tile
    named_sync(1, T);
  }
};

// ---- compact: merge path over positions ---------------------------------------------
// One tile of the merge of (A positions, lb_B) per pipeline step. The stage
// holds lb_B[j0, j1) and the collision words covering A[i0, i1); the
// producer lanes also look up R(i0), so the tile's first survivor lands at
// k0 - R(i0). In the tile's merged order (B first on ties) B_j sits at slot
// (j - j0) + (lb_B[j] - i0); a bitmap of those slots and prefix popcounts
// over it and over C give every slot its element and its output position
// directly, without walking the merge.
template <int T_, int E_, int S_, class RD = Rank512Dir>
struct CompactSpec {
  static constexpr int T = T_;
  static constexpr int E = E_;
  static constexpr int S = S_;
  static constexpr int D = T * E;
  static constexpr int NC = D / 32 + 4;  // collision words of one tile, at most
  static constexpr int64_t kLBBytes = align_up(int64_t(D) * 4 + 128, 16);
  static constexpr int64_t kStageBytes = kLBBytes + align_up(int64_t(NC + 4) * 4 + 64, 16);
  // ord_A and ord_B of a tile share one buffer (na + nb <= D), and the marks
  // (values <= D) are 16-bit: with 256 x 11 tiles four CTAs fit on an SM
  static constexpr int64_t kRefs = 0;
  static constexpr int64_t kOrd = align_up(int64_t(D + 8) * 4, 16);
  static constexpr int64_t kM = kOrd + align_up(int64_t(D + 16) * 4, 16);
  static constexpr int64_t kPC = kM + align_up(int64_t(D + 1) * 2, 16);
  static constexpr int64_t kScan = kPC + align_up(int64_t(NC + 1) * 4, 16);
  static constexpr int64_t kWorkBytes = kScan + align_up(int64_t(2 * (T / 32 + 1)) * 4, 16);
  static_assert(NC <= T, "one thread per collision word");
  static_assert(E <= 32, "a thread's collision bits fit one 64-bit window");
  static_assert(D < 65536, "16-bit marks");
  struct Params {
    int64_t m, n;
    const uint32_t *C;
    RD rank;
    const uint32_t *lb_B;
    const int64_t *part_i;
    uint32_t *refs, *ord_A, *ord_B;
    int32_t *status;
  };
  struct Desc {
    int64_t i0, j0, r0;
    int32_t na, nb, offLB, offC;
  };
  __device__ __forceinline__ static void init(uint8_t *work) {
    uint16_t *sM = reinterpret_cast<uint16_t *>(work + kM);
    for (int x = threadIdx.x; x < D + 1; x += T) sM[x] = 0;
  }
  // The co-ranks are clamped to their diagonals (and i1 - i0 to the tile's
  // length), so the staged ranges stay inside the arrays whatever lb_B held.
  __device__ __forceinline__ static void fetch(const Params &p, int64_t g, int64_t v[4]) {
    const int64_t total = p.m + p.n;
    const int64_t k0 = g * D, k1 = k0 + D < total ? k0 + D : total;
    int64_t i0 = __ldg(p.part_i + g), i1 = __ldg(p.part_i + g + 1);
    i0 = i0 < (k0 > p.n ? k0 - p.n : 0) ? (k0 > p.n ? k0 - p.n : 0) : i0;
    i0 = i0 > (k0 < p.m ? k0 : p.m) ? (k0 < p.m ? k0 : p.m) : i0;
    i1 = i1 < i0 ? i0 : i1;
    i1 = i1 > i0 + (k1 - k0) ? i0 + (k1 - k0) : i1;
    i1 = i1 > p.m ? p.m : i1;
    i1 = i1 < k1 - p.n ? k1 - p.n : i1;
    v[0] = i0;
    v[1] = i1;
    v[2] = static_cast<int64_t>(p.rank.at(p.C, i0));
  }
  __device__ __forceinline__ static void produce(const Params &p, int64_t g, const int64_t v[4], uint8_t *stage,
                                 Desc &d, uint64_t *full) {
    const int64_t total = p.m + p.n;
    const int64_t i0 = v[0], i1 = v[1];
    const int64_t k0 = g * D, k1 = k0 + D < total ? k0 + D : total;
    const int64_t j0 = k0 - i0, j1 = k1 - i1;
    const int na = static_cast<int>(i1 - i0), nb = static_cast<int>(j1 - j0);
    const int64_t nwords = (p.m + 31) / 32;
    const int64_t w0 = i0 >> 5;
    const int nw = na > 0 ? static_cast<int>(((i1 - 1) >> 5) - w0 + 1) : 0;
    const StagePlan pl = stage_plan_overfetch<4>(j0, nb, p.n);
    const StagePlan pc = stage_plan_overfetch<4>(w0, nw, nwords);
    uint32_t *bufLB = reinterpret_cast<uint32_t *>(stage);
    uint32_t *bufC = reinterpret_cast<uint32_t *>(stage + kLBBytes);
    for (int64_t x = pl.tail_from; x < j1; ++x) bufLB[x - pl.first] = p.lb_B[x];
    for (int64_t x = pc.tail_from; x < w0 + nw; ++x) bufC[x - pc.first] = p.C[x];
    d.i0 = i0;
    d.j0 = j0;
    d.r0 = v[2];
    d.na = na;
    d.nb = nb;
    d.offLB = pl.lead;
    d.offC = pc.lead;
    mbar_arrive_expect_tx(full, pl.bulk + pc.bulk);
    stage_issue(bufLB, p.lb_B, pl, full);
    stage_issue(bufC, p.C, pc, full);
  }
  __device__ __forceinline__ static void consume(const Params &p, int64_t g, const Desc &dd, const uint8_t *stage,
                                 uint8_t *work, uint64_t *empty) {
    const int tid = threadIdx.x;
    const uint32_t *sLB = reinterpret_cast<const uint32_t *>(stage) + dd.offLB;
    const uint32_t *sCw = reinterpret_cast<const uint32_t *>(stage + kLBBytes) + dd.offC;
    uint32_t *bufRefs = reinterpret_cast<uint32_t *>(work + kRefs);
    uint32_t *bufOrd = reinterpret_cast<uint32_t *>(work + kOrd);
    uint16_t *sM = reinterpret_cast<uint16_t *>(work + kM);
    uint32_t *sPC = reinterpret_cast<uint32_t *>(work + kPC);
    uint32_t *sScan = reinterpret_cast<uint32_t *>(work + kScan);
    const int na = dd.na, nb = dd.nb;
    const int64_t i0 = dd.i0, j0 = dd.j0;
    const int64_t out0 = g * D - dd.r0;
    const int64_t w0 = i0 >> 5;
    const int wbit0 = static_cast<int>(i0 - (w0 << 5));
    const int nwc = na > 0 ? static_cast<int>((((i0 + na - 1) >> 5) - w0) + 1) : 0;
    const uint32_t i0u = static_cast<uint32_t>(i0), j0u = static_cast<uint32_t>(j0);
    const uint32_t out0u = static_cast<uint32_t>(out0);
    const int cnt = na + nb;
    // ord_B's part of the shared buffer starts on a 16-byte boundary past ord_A's
    const int offB = (na + 3 + 4) & ~3;
    uint32_t *sRefs = bufRefs + (out0 & 3);
    uint32_t *sOrdA = bufOrd + (i0 & 3);
    uint32_t *sOrdB = bufOrd + offB + (j0 & 3);

    // 1. With B first on ties, B record bi precedes tile A record a exactly
    //    when L_bi = lb_B[j0 + bi] - i0 <= a, so the B records before A
    //    record a number max{bi + 1 : L_bi <= a}. The last B record of each
    //    run of equal L marks sM[L] = bi + 1; a prefix maximum over sM then
    //    gives every A record its count. An L outside [0, na] or a falling L
    //    means lb_B is not the lower-bound array of this merge: the tile is
    //    skipped and the call reports LSM_ERR_ARG.
    bool bad = false;
    for (int bi = tid; bi < nb; bi += T) {
      const uint32_t L = sLB[bi] - i0u;
      const uint32_t Ln = bi + 1 < nb ? sLB[bi + 1] - i0u : 0xFFFFFFFFu;
      if (L > static_cast<uint32_t>(na) || Ln < L) bad = true;
      else if (L < static_cast<uint32_t>(na) && Ln != L) sM[L] = static_cast<uint16_t>(bi + 1);
    }
    // collision words: bits of this tile's A records only (not those before
    // A[i0] in the first word, nor the next tile's in the last word)
    const uint32_t cmask0 = wbit0 ? (1u << wbit0) - 1u : 0u;  // bits before A[i0]
    uint32_t cw_own = tid < nwc ? sCw[tid] : 0u;
    if (tid == 0) cw_own &= ~cmask0;
    const int xend = wbit0 + na;
    if (tid == nwc - 1 && (xend & 31)) cw_own &= (1u << (xend & 31)) - 1u;
    if (named_sync_or(1, T, bad)) {
      if (tid == 0) report(p.status, LSM_ERR_ARG);
      release_stage(empty);
      for (int x = tid; x < na; x += T) sM[x] = 0;
      named_sync(1, T);
      return;
    }
    // 2. one scan: prefix popcounts of the collision words, and the prefix
    //    maximum of sM over each thread's E consecutive A records
    const int a0 = tid * E;
    uint32_t mv[E];
    uint32_t mloc = 0;
#pragma unroll
    for (int q = 0; q < E; ++q) {
      mv[q] = a0 + q < na ? sM[a0 + q] : 0u;
      mloc = mv[q] > mloc ? mv[q] : mloc;
    }
#pragma unroll
    for (int q = 0; q < E; ++q)
      if (a0 + q < na && mv[q]) sM[a0 + q] = 0;  // clean for the next tile
    uint32_t totC, mbefore;
    const uint32_t exC = consumer_exclusive_sum_max<T>(
        tid < nwc ? static_cast<uint32_t>(__popc(cw_own)) : 0u, mloc, sScan, &totC, &mbefore);
    if (tid < nwc) sPC[tid] = exC;
    named_sync(1, T);
    // collisions among tile A records [0, x), x in [0, na]
    auto dropped_before = [&](int x) -> int {
      if (x >= na) return static_cast<int>(totC);
      const int xa = wbit0 + x, wa = xa >> 5;
      const uint32_t cwa = sCw[wa];
      return static_cast<int>(sPC[wa]) + __popc(cwa & ((1u << (xa & 31)) - 1u)) -
             (wa == 0 ? __popc(cwa & cmask0) : 0);
    };
    // 3. A records: slot a + (B records before it), output slot minus the
    //    dropped A records before it
    if (a0 < na) {
      int drops = dropped_before(a0);
      uint32_t run = mbefore;
      // the collision bits of this thread's E records (E <= 32): one 64-bit
      // window over the two words they span; bit q belongs to record a0 + q
      const int xa0 = wbit0 + a0;
      const uint64_t win =
          ((static_cast<uint64_t>(sCw[(xa0 >> 5) + 1]) << 32) | sCw[xa0 >> 5]) >> (xa0 & 31);
      const int lim = na - a0 < E ? na - a0 : E;
#pragma unroll
      for (int q = 0; q < E; ++q) {
        if (q < lim) {
          run = mv[q] > run ? mv[q] : run;
          const bool dropped = (win >> q) & 1u;
          const int ol = a0 + q + static_cast<int>(run) - drops;
          if (!dropped) sRefs[ol] = i0u + static_cast<uint32_t>(a0 + q);
          sOrdA[a0 + q] = dropped ? LSM_ORD_DROPPED : out0u + static_cast<uint32_t>(ol);
          drops += dropped ? 1 : 0;
        }
      }
    }
    // 4. B records: slot bi + L_bi, output slot minus the dropped A records
    //    before it (those below L_bi)
    for (int bi = tid; bi < nb; bi += T) {
      const int L = static_cast<int>(sLB[bi] - i0u);
      const int ol = bi + L - dropped_before(L);
      sRefs[ol] = LSM_REF_FROM_B | (j0u + static_cast<uint32_t>(bi));
      sOrdB[bi] = out0u + static_cast<uint32_t>(ol);
    }
    release_stage(empty);
    const int kept_total = cnt - static_cast<int>(totC);
    fence_proxy_async_smem();
    named_sync(1, T);
    store_u32_run<T>(p.refs, out0, kept_total, bufRefs);
    store_u32_run<T>(p.ord_A, i0, na, bufOrd);
    store_u32_run<T>(p.ord_B, j0, nb, bufOrd + offB);
    if (tid == 0) {
      bulk_commit();
      bulk_wait_read_all();  // the buffers are rewritten by the next tile
    }
    named_sync(1, T);
  }
};

// ---- fused: collision bits, lower bounds, ordinals and refs in one pass -------------
// The three steps above in one pass over merge-path tiles of the keys (A
// first on ties), by the stable merge's own walk: each tile stages A[i0-1,
// i1) and B[j0, j1] (the keys on either side included where they exist);
// each of T threads bisects its diagonal d = tid E inside the staged spans
// and walks E merge steps, which give every record directly:
//   an A record is dropped exactly when the B head it is compared with (the
//     next B in merged order, B[j1] past the tile's end) has its key;
//   a B record's lb_B is i0 plus the tile A records taken before it, minus
//     one when the A record just before it has its key;
//   every record's merged slot is d + step.
// One scan of the threads' drop counts gives each slot its dropped A records
// before it, and R(i0), the collisions of all earlier tiles, comes from a
// decoupled lookback over the tiles' collision counts (every A record
// before i0 lies in an earlier tile), so a record lands at k0 + slot -
// (R(i0) + dropped before it in the tile): the ordinals of [CB] "Corrected
// record ordinals". Tile states are flag << 62 | value words (1 = aggregate,
// 2 = inclusive prefix), cleared by the partition launch; each lookback wait
// is bounded in time. All CTAs of the persistent grid are resident, and a
// tile waits only on earlier tiles, each of which its CTA reaches without
// waiting on a later one.
constexpr uint64_t kStateAgg = 1ull << 62, kStateInc = 2ull << 62;
constexpr uint64_t kStateVal = (1ull << 62) - 1;

template <int T_, int E_, int S_>
struct FusedSpec {
  static constexpr int T = T_;
  static constexpr int E = E_;
  static constexpr int S = S_;
  static constexpr int D = T * E;
  static constexpr int NC = D / 32 + 4;  // collision words of one tile, at most
  static constexpr int64_t kStageBytes = align_up(int64_t(D + 4) * 8 + 160, 16);
  static constexpr int64_t kLB = 0;
  static constexpr int64_t kRefs = kLB + align_up(int64_t(D + 8) * 4, 16);
  static constexpr int64_t kOrd = kRefs + align_up(int64_t(D + 8) * 4, 16);
  static constexpr int64_t kCw = kOrd + align_up(int64_t(D + 16) * 4, 16);
  static constexpr int64_t kScan = kCw + align_up(int64_t(NC) * 4, 16);
  static constexpr int64_t kBcast = kScan + align_up(int64_t(T / 32 + 1) * 4, 16);
  static constexpr int64_t kWorkBytes = kBcast + 16;
  static_assert(D < 32768, "15-bit tile indices");
  struct Params {
    const uint64_t *A, *B;
    int64_t m, n, G;
    const int64_t *part_i;
    uint32_t *C, *lb_B, *refs, *ord_A, *ord_B;
    int64_t *d_count;
    uint64_t *state;
    int32_t *status;
  };
  struct Desc {
    int64_t i0, j0;
    int32_t na, nb, hp, hn, offA, offB;
  };
  __device__ __forceinline__ static void init(uint8_t *work) {
    uint32_t *sCw = reinterpret_cast<uint32_t *>(work + kCw);
    for (int x = threadIdx.x; x < NC; x += T) sCw[x] = 0u;
  }
  __device__ __forceinline__ static void fetch(const Params &p, int64_t g, int64_t v[4]) {
    v[0] = __ldg(p.part_i + g);
    v[1] = __ldg(p.part_i + g + 1);
  }
  __device__ __forceinline__ static void produce(const Params &p, int64_t g, const int64_t v[4],
                                                 uint8_t *stage, Desc &d, uint64_t *full) {
    const int64_t total = p.m + p.n;
    const int64_t i0 = v[0], i1 = v[1];
    const int64_t k0 = g * D, k1 = k0 + D < total ? k0 + D : total;
    const int64_t j0 = k0 - i0, j1 = k1 - i1;
    const int na = static_cast<int>(i1 - i0), nb = static_cast<int>(j1 - j0);
    const int hp = i0 > 0 ? 1 : 0, hn = j1 < p.n ? 1 : 0;
    const StagePlan pa = stage_plan_overfetch<8>(i0 - hp, na + hp, p.m);
    const StagePlan pb = stage_plan_overfetch<8>(j0, nb + hn, p.n);
    uint64_t *bufA = reinterpret_cast<uint64_t *>(stage);
    const int32_t offB = static_cast<int32_t>(stage_capacity_bytes<8>(pa.span) / 8);
    uint64_t *bufB = bufA + offB;
    for (int64_t x = pa.tail_from; x < i1; ++x) bufA[x - pa.first] = p.A[x];
    for (int64_t x = pb.tail_from; x < j1 + hn; ++x) bufB[x - pb.first] = p.B[x];
    d.i0 = i0;
    d.j0 = j0;
    d.na = na;
    d.nb = nb;
    d.hp = hp;
    d.hn = hn;
    d.offA = pa.lead + hp;
    d.offB = offB + pb.lead;
    mbar_arrive_expect_tx(full, pa.bulk + pb.bulk);
    stage_issue(bufA, p.A, pa, full);
    stage_issue(bufB, p.B, pb, full);
  }

  // R(i0) for tile g: publish the tile's collision count, sum the earlier
  // tiles' published counts back to the first inclusive prefix (warp 0).
  __device__ __forceinline__ static uint32_t lookback(const Params &p, int64_t g, uint32_t totC,
                                                      uint32_t *bcast) {
    const int tid = threadIdx.x;
    if (tid < 32) {
      const int lane = tid;
      uint64_t prefix = 0;
      if (g == 0) {
        if (lane == 0) st_relaxed_u64(p.state, kStateInc | totC);
      } else {
        if (lane == 0) st_relaxed_u64(p.state + g, kStateAgg | totC);
        int64_t base = g - 1;
        const uint64_t t0 = globaltimer_ns();
        bool late = false;
        for (;;) {
          const int64_t idx = base - lane;
          uint64_t v = idx >= 0 ? ld_relaxed_u64(p.state + idx) : kStateInc;
          uint32_t polls = 0;
          while (!__all_sync(0xffffffffu, (v >> 62) != 0)) {
            if ((v >> 62) == 0) v = ld_relaxed_u64(p.state + idx);
            if ((++polls & 31) == 0 &&
                __any_sync(0xffffffffu, globaltimer_ns() - t0 > static_cast<uint64_t>(kWaitLimitNs))) {
              late = true;
              if ((v >> 62) == 0) v = kStateInc;  // give up: counted as zero
            }
          }
          const uint32_t inc = __ballot_sync(0xffffffffu, (v >> 62) == 2);
          uint64_t c = v & kStateVal;
          if (inc) {
            const int first = __ffs(inc) - 1;
            c = lane <= first ? c : 0;
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
          prefix += c;
          if (inc) break;
          base -= 32;
        }
        if (lane == 0) {
          if (late) report(p.status, LSM_ERR_TIMEOUT);
          st_relaxed_u64(p.state + g, kStateInc | ((prefix + totC) & kStateVal));
        }
      }
      if (lane == 0) *bcast = static_cast<uint32_t>(prefix);
    }
    named_sync(1, T);
    return *bcast;
  }

  __device__ __forceinline__ static void consume(const Params &p, int64_t g, const Desc &dd,
                                                 const uint8_t *stage, uint8_t *work,
                                                 uint64_t *empty) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t *sA = reinterpret_cast<const uint64_t *>(stage) + dd.offA;  // sA[-1] = A[i0-1]
    const uint64_t *sB = reinterpret_cast<const uint64_t *>(stage) + dd.offB;  // sB[nb] = B[j1]
    uint32_t *sLBbuf = reinterpret_cast<uint32_t *>(work + kLB);
    uint32_t *bufRefs = reinterpret_cast<uint32_t *>(work + kRefs);
    uint32_t *bufOrd = reinterpret_cast<uint32_t *>(work + kOrd);
    uint32_t *sCw = reinterpret_cast<uint32_t *>(work + kCw);
    uint32_t *sScan = reinterpret_cast<uint32_t *>(work + kScan);
    uint32_t *sBcast = reinterpret_cast<uint32_t *>(work + kBcast);
    const int na = dd.na, nb = dd.nb, hp = dd.hp, hn = dd.hn;
    const int64_t i0 = dd.i0, j0 = dd.j0, i1 = i0 + na;
    const int64_t k0 = g * D;
    const int cnt = na + nb;
    const int64_t w0 = i0 >> 5;
    const int wbit0 = static_cast<int>(i0 - (w0 << 5));  // bit of A[i0] in word w0
    const int nwc = na > 0 ? static_cast<int>(((i1 - 1) >> 5) - w0 + 1) : 0;

    // 1. this thread's diagonal, bisected in the staged spans (A first on
    //    ties), then E merge steps. Each record is kept as one word:
    //    bit 31 = from B, bit 30 = dropped A / B matching the A before it,
    //    bits 0..14 = its index in its tile span.
    const int d = tid * E < cnt ? tid * E : cnt;
    int lo = d > nb ? d - nb : 0, hi = d < na ? d : na;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sA[mid] <= sB[d - mid - 1]) lo = mid + 1;
      else hi = mid;
    }
    int ai = lo, bi = d - lo;
    const int nbx = nb + hn;  // B keys staged, the one after the tile included
    uint64_t a = ai < na ? sA[ai] : 0, b = bi < nbx ? sB[bi] : 0;
    // A B record matches an A record exactly when the last A record taken
    // before it has its key (with A first on ties the equal A comes right
    // before it: no other B fits between equal keys). The last A before the
    // thread's first record is A[i0 + ai - 1], or A[i0 - 1] when ai = 0.
    bool prevA = ai > 0 || hp;
    uint64_t prevkey = prevA ? sA[ai - 1] : 0;
    uint32_t rec[E];
    uint32_t drops = 0;
#pragma unroll
    for (int q = 0; q < E; ++q) {
      rec[q] = 0xFFFFFFFFu;
      if (d + q < cnt) {
        const bool takeA = bi >= nb || (ai < na && a <= b);
        if (takeA) {
          const bool dropped = bi < nbx && b == a;  // the next B has this key
          rec[q] = (dropped ? 0x40000000u : 0u) | static_cast<uint32_t>(ai);
          drops += dropped ? 1u : 0u;
          prevA = true;
          prevkey = a;
          ++ai;
          a = ai < na ? sA[ai] : 0;
        } else {
          const bool match = prevA && prevkey == b;
          rec[q] = 0x80000000u | (match ? 0x40000000u : 0u) | static_cast<uint32_t>(bi) |
                   (static_cast<uint32_t>(ai) << 15);
          ++bi;
          b = bi < nbx ? sB[bi] : 0;
        }
      }
    }
    release_stage(empty);  // the keys are not read again
    // 2. exclusive scan of the drop counts in merged order (thread order)
    uint32_t inc = drops;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) sScan[warp] = inc;
    named_sync(1, T);
    if (warp == 0) {
      const uint32_t w = lane < T / 32 ? sScan[lane] : 0u;
      uint32_t wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += t;
      }
      if (lane < T / 32) sScan[lane] = wi - w;
      if (lane == T / 32 - 1) sScan[T / 32] = wi;
    }
    named_sync(1, T);
    uint32_t before = sScan[warp] + inc - drops;  // dropped A records before slot d
    const uint32_t totC = sScan[T / 32];
    // 3. R(i0) from the earlier tiles (contains a barrier over the consumers)
    const uint32_t r0 = lookback(p, g, totC, sBcast);
    const int64_t out0 = k0 - r0;
    const uint32_t out0u = static_cast<uint32_t>(out0);
    const uint32_t i0u = static_cast<uint32_t>(i0), j0u = static_cast<uint32_t>(j0);
    const int offB = (na + 3 + 4) & ~3;  // ord_B's part starts past ord_A's, 16-byte aligned
    uint32_t *sRefs = bufRefs + (out0 & 3);
    uint32_t *sOrdA = bufOrd + (i0 & 3);
    uint32_t *sOrdB = bufOrd + offB + (j0 & 3);
    uint32_t *sLB = sLBbuf + (j0 & 3);
    // 4. every record to its output slot
#pragma unroll
    for (int q = 0; q < E; ++q) {
      const uint32_t r = rec[q];
      if (r != 0xFFFFFFFFu) {
        const int slot = d + q;
        const int ol = slot - static_cast<int>(before);
        const uint32_t idx = r & 0x7FFFu;
        if (r & 0x80000000u) {
          const uint32_t ai_at = (r >> 15) & 0x7FFFu;
          sLB[idx] = i0u + ai_at - ((r & 0x40000000u) ? 1u : 0u);
          sRefs[ol] = LSM_REF_FROM_B | (j0u + idx);
          sOrdB[idx] = out0u + static_cast<uint32_t>(ol);
        } else if (r & 0x40000000u) {
          sOrdA[idx] = LSM_ORD_DROPPED;
          const int x = wbit0 + static_cast<int>(idx);
          atomicOr(&sCw[x >> 5], 1u << (x & 31));
          ++before;
        } else {
          sRefs[ol] = i0u + idx;
          sOrdA[idx] = out0u + static_cast<uint32_t>(ol);
        }
      }
    }
    fence_proxy_async_smem();
    named_sync(1, T);
    store_u32_run<T>(p.lb_B, j0, nb, sLBbuf);
    store_u32_run<T>(p.refs, out0, cnt - static_cast<int>(totC), bufRefs);
    store_u32_run<T>(p.ord_A, i0, na, bufOrd);
    store_u32_run<T>(p.ord_B, j0, nb, bufOrd + offB);
    if (tid == 0) {
      bulk_commit();
      if (g == p.G - 1) *p.d_count = p.m + p.n - (static_cast<int64_t>(r0) + totC);
    }
    // collision words: whole words inside the tile's A range by plain
    // stores, the shared boundary words by atomicOr (C was cleared)
    for (int x = tid; x < nwc; x += T) {
      const int64_t w = w0 + x;
      const uint32_t bits = sCw[x];
      sCw[x] = 0u;  // clean for the next tile
      if (w * 32 >= i0 && w * 32 + 32 <= i1) p.C[w] = bits;
      else if (bits) atomicOr(&p.C[w], bits);
    }
    if (tid == 0) bulk_wait_read_all();  // the staging buffers are rewritten by the next tile
    named_sync(1, T);
  }
};

}  // namespace

// Tile variants of the two replacement pipelines: (consumer threads, items
// per thread, stages). Selected process-wide by lsm_tune_replace.
struct ReplaceVariant {
  int T, E, S;
};
constexpr ReplaceVariant kReplaceVariants[] = {{256, 11, 2}, {128, 23, 2}, {256, 23, 2}, {512, 11, 2}};
// -1 selects the warp pipelines of replacement.cu (the default); 0..3 the
// tile variants above (the earlier block-synchronous pipelines).
int g_mark_variant = -1, g_compact_variant = -1;

template <int V>
cudaError_t launch_mark_variant(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                uint32_t *C, uint32_t *lb_B, int64_t *part_i, int32_t *status,
                                cudaStream_t s) {
  constexpr ReplaceVariant v = kReplaceVariants[V];
  using Spec = MarkSpec<v.T, v.E, v.S>;
  constexpr int64_t D = Spec::D;
  const int64_t nwords = (m + 31) / 32;
  cudaError_t err = launch_partition(U64AFirst{A, B}, m, n, D, part_i, C, nwords, s);
  if (err != cudaSuccess) return err;
  const int64_t G = (m + n + D - 1) / D;
  if (G == 0) return cudaSuccess;
  typename Spec::Params p{A, B, m, n, part_i, C, lb_B};
  profile_before(s);
  err = launch_pipeline<Spec>(p, G, status, s, device_sm_count());
  profile_after(s);
  return err;
}

cudaError_t launch_collision_mark(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                  uint32_t *C, uint32_t *lb_B, int64_t *part_i, int32_t *status,
                                  cudaStream_t s) {
  if (g_mark_variant < 0)
    return launch_mark_tiles(A, m, B, n, C, lb_B, nullptr, part_i, nullptr, status, s);
  switch (g_mark_variant) {
    case 1: return launch_mark_variant<1>(A, m, B, n, C, lb_B, part_i, status, s);
    case 2: return launch_mark_variant<2>(A, m, B, n, C, lb_B, part_i, status, s);
    case 3: return launch_mark_variant<3>(A, m, B, n, C, lb_B, part_i, status, s);
    default: return launch_mark_variant<0>(A, m, B, n, C, lb_B, part_i, status, s);
  }
}

// ---- fused replacement ---------------------------------------------------------------
constexpr int kFusedT = 256, kFusedE = 11, kFusedS = 2;
using FusedDefault = FusedSpec<kFusedT, kFusedE, kFusedS>;

__global__ void set_count_kernel(int64_t *d_count, int64_t v) {
  pdl_begin();
  *d_count = v;
}

int64_t fused_tile() { return FusedDefault::D; }

cudaError_t launch_replacement_fused(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                     uint32_t *C, uint32_t *lb_B, uint32_t *refs, uint32_t *ord_A,
                                     uint32_t *ord_B, int64_t *d_count, int64_t *part_i,
                                     uint64_t *state, int32_t *status, cudaStream_t s) {
  using Spec = FusedDefault;
  constexpr int64_t D = Spec::D;
  const int64_t G = (m + n + D - 1) / D;
  if (G == 0) return launch_kernel(false, set_count_kernel, 1, 1, 0, s, d_count, int64_t(0));
  const int64_t nwords = (m + 31) / 32;
  cudaError_t err = launch_partition(U64AFirst{A, B}, m, n, D, part_i, C, nwords, s, state, G);
  if (err != cudaSuccess) return err;
  typename Spec::Params p{A, B, m, n, G, part_i, C, lb_B, refs, ord_A, ord_B, d_count, state, status};
  profile_before(s);
  err = launch_pipeline<Spec>(p, G, status, s, device_sm_count());
  profile_after(s);
  return err;
}

int64_t replace_min_tile() {
  int64_t d = INT64_MAX;
  for (const ReplaceVariant &v : kReplaceVariants) d = d < int64_t(v.T) * v.E ? d : int64_t(v.T) * v.E;
  return d;
}

int set_replace_variant(int kernel, int threads, int items) {
  if (threads == 0 && items == 0) {
    if (kernel == 0) g_mark_variant = -1;
    else if (kernel == 1) g_compact_variant = -1;
    else return LSM_ERR_ARG;
    return LSM_OK;
  }
  for (int i = 0; i < 4; ++i) {
    if (kReplaceVariants[i].T == threads && kReplaceVariants[i].E == items) {
      if (kernel == 0) g_mark_variant = i;
      else if (kernel == 1) g_compact_variant = i;
      else return LSM_ERR_ARG;
      return LSM_OK;
    }
  }
  return LSM_ERR_ARG;
}

int64_t rank_build_ctas(int64_t m) { return (m / 512 + 1 + kRankThreads - 1) / kRankThreads; }

cudaError_t launch_rank_build(const uint32_t *C, int64_t m, uint32_t *dir, int64_t *d_total,
                              uint32_t *cta_totals, cudaStream_t s) {
  const int64_t ctas = rank_build_ctas(m);
  profile_before(s);
  cudaError_t err = launch_kernel(true, rank_count_kernel, static_cast<unsigned>(ctas),
                                  kRankThreads, 0, s, C, m, cta_totals);
  if (err != cudaSuccess) return err;
  err = launch_kernel(true, rank_finish_kernel, static_cast<unsigned>(ctas), kRankThreads, 0, s, C,
                      m, cta_totals, dir, d_total);
  profile_after(s);
  return err;
}

cudaError_t launch_rank_build_ws(const uint32_t *C, int64_t m, uint32_t *dir, int64_t *d_total,
                                 void *ws, int32_t *status, cudaStream_t s, bool ws_clear) {
  static int per_sm = -1;  // CTAs of rank_single_kernel resident per SM
  if (per_sm < 0) {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, rank_single_kernel, kRankThreads, 0) !=
        cudaSuccess)
      v = 0;
    per_sm = v;
  }
  const int64_t ctas = rank_build_ctas(m);
  // one launch only while every CTA is resident at once, so each CTA a
  // lookback waits for is already running
  if (ctas <= static_cast<int64_t>(device_sm_count()) * per_sm) {
    if (!ws_clear) {
      const cudaError_t e = cudaMemsetAsync(ws, 0, static_cast<size_t>(ctas) * 8, s);
      if (e != cudaSuccess) return e;
    }
    profile_before(s);
    const cudaError_t err = launch_kernel(true, rank_single_kernel, static_cast<unsigned>(ctas),
                                          kRankThreads, 0, s, C, m, dir, d_total,
                                          static_cast<uint64_t *>(ws), status);
    profile_after(s);
    return err;
  }
  return launch_rank_build(C, m, dir, d_total, static_cast<uint32_t *>(ws), s);
}

// ---- allocation-free rank_build --------------------------------------------------
// Scratch for lsm_rank_build_noalloc: the per-CTA popcount totals live in this
// file-scope device array instead of a caller workspace. 4096 CTAs of 256
// 512-bit blocks cover m <= 2^29 - 1 bit positions; the array is 16 KB and every
// device that loads the library keeps it until the process exits. The count
// kernel overwrites every entry the finish kernel reads, so nothing in it has
// to start at zero.
constexpr int64_t kNoAllocRankCtas = 4096;
constexpr int64_t kNoAllocRankMaxM = (int64_t(1) << 29) - 1;
static __device__ __align__(256) uint32_t g_rank_noalloc_scratch[kNoAllocRankCtas];

namespace {
std::mutex g_noalloc_mu;
uint32_t *g_noalloc_ptr[64];

// Device address of the scratch array on the current device. In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
int noalloc_scratch(uint32_t **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LSM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    uint32_t *p = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_rank_noalloc_scratch) != cudaSuccess)
      return LSM_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return LSM_OK;
}
}  // namespace

cudaError_t launch_rank_query(const uint32_t *C, const uint32_t *dir, int64_t m,
                              const uint32_t *pos, int64_t q, uint32_t *out, int32_t *status,
                              cudaStream_t s) {
  if (q == 0) return cudaSuccess;
  return launch_kernel(true, rank_query_kernel, static_cast<unsigned>((q + 255) / 256), 256, 0, s,
                       C, dir, m, pos, q, out, status);
}

template <int V, class RD>
cudaError_t launch_compact_variant(int64_t m, int64_t n, const uint32_t *C, RD rank,
                                   const uint32_t *lb_B, uint32_t *refs, uint32_t *ord_A,
                                   uint32_t *ord_B, int64_t *d_count, int64_t *part_i,
                                   int32_t *status, cudaStream_t s) {
  constexpr ReplaceVariant v = kReplaceVariants[V];
  using Spec = CompactSpec<v.T, v.E, v.S, RD>;
  constexpr int64_t D = Spec::D;
  const int64_t G = (m + n + D - 1) / D;
  const int64_t blocks = n > 0 ? (n + kPosPerBlock - 1) / kPosPerBlock : 1;
  cudaError_t err = launch_kernel(true, partition_positions_kernel<RD>, static_cast<unsigned>(blocks),
                                  kPosThreads, 0, s, lb_B, m, n, D, G, part_i, C, rank, d_count);
  if (err != cudaSuccess) return err;
  if (G == 0) return cudaSuccess;
  typename Spec::Params p{m, n, C, rank, lb_B, part_i, refs, ord_A, ord_B, status};
  profile_before(s);
  err = launch_pipeline<Spec>(p, G, status, s, device_sm_count());
  profile_after(s);
  return err;
}

cudaError_t launch_materialize(const uint64_t *A, const uint32_t *Aval, const uint32_t *tombA,
                               int64_t m, const uint64_t *B, const uint32_t *Bval,
                               const uint32_t *tombB, int64_t n, const uint32_t *refs,
                               const int64_t *d_count, uint64_t *out_keys, uint32_t *out_vals,
                               uint32_t *out_tomb, int32_t *status, cudaStream_t s) {
  const int64_t need = (m + n + 1023) / 1024;  // four records per thread at most
  int64_t blocks = static_cast<int64_t>(device_sm_count()) * 8;
  if (blocks > need) blocks = need;
  if (blocks < 1) blocks = 1;
  // Plain stream order: launched early behind the persistent compaction
  // kernel, its waiting blocks cost the 12M + 4M step about 40 us
  // (238 us against 198 us, CUDA events over the whole step).
  profile_before(s);
  const cudaError_t err = launch_kernel(false, materialize_kernel, static_cast<unsigned>(blocks),
                                        256, 0, s, A, Aval, tombA, m, B, Bval, tombB, n, refs,
                                        d_count, out_keys, out_vals, out_tomb, status);
  profile_after(s);
  return err;
}

cudaError_t launch_compact(int64_t m, int64_t n, const uint32_t *C, const uint32_t *dir,
                           const uint32_t *lb_B, uint32_t *refs, uint32_t *ord_A,
                           uint32_t *ord_B, int64_t *d_count, int64_t *part_i,
                           uint32_t *mb_scratch, int32_t *status, cudaStream_t s) {
  if (g_compact_variant < 0)
    return launch_compact_tiles(m, n, C, dir, lb_B, mb_scratch, nullptr, part_i, refs, ord_A,
                                ord_B, d_count, status, s);
  const Rank512Dir rank{dir};
  switch (g_compact_variant) {
    case 1: return launch_compact_variant<1>(m, n, C, rank, lb_B, refs, ord_A, ord_B, d_count, part_i, status, s);
    case 2: return launch_compact_variant<2>(m, n, C, rank, lb_B, refs, ord_A, ord_B, d_count, part_i, status, s);
    case 3: return launch_compact_variant<3>(m, n, C, rank, lb_B, refs, ord_A, ord_B, d_count, part_i, status, s);
    default: return launch_compact_variant<0>(m, n, C, rank, lb_B, refs, ord_A, ord_B, d_count, part_i, status, s);
  }
}


}  // namespace lsm

// Allocation-free variant of lsm_rank_build (declared in include/lsmmerge.h).
extern "C" LSM_API int lsm_rank_build_noalloc(const uint32_t *C, int64_t m, uint32_t *dir,
                                              int64_t *d_total, void *stream) {
  using namespace lsm;
  if (m < 0 || !dir || !d_total || (m && !C)) return LSM_ERR_ARG;
  if (m > kNoAllocRankMaxM) return LSM_ERR_OVERFLOW;
  if (C && (reinterpret_cast<uintptr_t>(C) & 15u)) return LSM_ERR_ALIGN;
  uint32_t *scratch = nullptr;
  if (int r = noalloc_scratch(&scratch)) return r;
  const cudaError_t e = launch_rank_build(C, m, dir, d_total, scratch, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LSM_OK : LSM_ERR_CUDA;
}
