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
// GPU design:
//   collision_mark   partition (co-rank per tile, A first on ties; the same
//                    launch clears C) + one CTA per merge-path tile. The tile
//                    stages A[i0-1, i1) and B[j0, j1] in shared memory with
//                    bulk copies, walks its merge, and for each B element
//                    records lb = (A elements before it) - (1 if the element
//                    before it is an equal A). Each collision bit is set by
//                    the tile that owns the A index (it peeks at the B
//                    element after its span), so bitmap words that lie inside
//                    one tile take plain stores and only boundary words need
//                    atomicOr.
//   rank_build       count -> prefix -> finish in two launches: per-CTA
//                    popcount totals, then each CTA sums the totals before it
//                    and writes its directory entries ([CB] "Dispatch
//                    bindings": the constructor is count, global scan,
//                    finish; the finish runs at least one block for empty A).
//   compact          merge path over positions: B_j precedes A_i exactly when
//                    lb_B[j] <= i (this is B_j <= A_i, since lb_B[j] counts the
//                    A keys below B_j), so the merge of surviving A and B
//                    needs lb_B and C only, never the keys. A tile starting at
//                    diagonal k0 with co-rank i0 has R(i0) dropped records
//                    before it (a rank query), so its first survivor lands at
//                    k0 - R(i0); a block-wide exclusive scan of keep flags
//                    places the rest. Refs and ordinals leave through shared
//                    memory in coalesced runs.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace lsm {

namespace {

// ---- partition: co-rank per tile on uint64 keys, A first; clears C ----------
struct U64AFirst {
  const uint64_t *A;
  const uint64_t *B;
  __device__ __forceinline__ bool too_small(int64_t i, int64_t k) const {
    return __ldg(A + i) <= __ldg(B + k - i - 1);
  }
};

// B_j precedes A_i exactly when lb_B[j] <= i, so A_i precedes B_j when i < lb_B[j].
struct PositionsBFirst {
  const uint32_t *lb_B;
  __device__ __forceinline__ bool too_small(int64_t i, int64_t k) const {
    return i < static_cast<int64_t>(__ldg(lb_B + k - i - 1));
  }
};

template <class Pred>
__global__ void __launch_bounds__(256) partition_kernel(Pred pred, int64_t m, int64_t n, int64_t D,
                                                        int64_t G, int64_t *__restrict__ out_i,
                                                        uint32_t *__restrict__ clear_words,
                                                        int64_t nclear) {
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (clear_words) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t w = gtid; w < nclear; w += stride) clear_words[w] = 0u;
  }
  const int64_t g = gtid;
  if (g > G) return;
  const int64_t total = m + n;
  const int64_t k = g * D < total ? g * D : total;
  out_i[g] = thread_corank(pred, k, m, n);
}

template <class Pred>
cudaError_t launch_partition(const Pred &pred, int64_t m, int64_t n, int64_t D, int64_t *out_i,
                             uint32_t *clear_words, int64_t nclear, cudaStream_t s) {
  const int64_t G = (m + n + D - 1) / D;
  int64_t threads = G + 1;
  if (clear_words && threads < nclear / 4) threads = nclear / 4;
  const int64_t blocks = (threads + 255) / 256;
  partition_kernel<Pred><<<static_cast<unsigned>(blocks), 256, 0, s>>>(pred, m, n, D, G, out_i,
                                                                       clear_words, nclear);
  return cudaGetLastError();
}

// ---- collision mark ------------------------------------------------------------
template <int T, int E>
struct MarkLayout {
  static constexpr int D = T * E;
  static constexpr int64_t kBar = 0;
  static constexpr int64_t kKeys = 128;
  static constexpr int64_t kKeysBytes = align_up(int64_t(D + 2) * 8 + 128, 16);
  static constexpr int64_t kLB = kKeys + kKeysBytes;
  static constexpr int64_t kLBBytes = align_up(int64_t(D) * 4, 16);
  static constexpr int64_t kCw = kLB + kLBBytes;
  static constexpr int64_t kCwBytes = align_up(int64_t(D / 32 + 4) * 4, 16);
  static constexpr int64_t kBytes = kCw + kCwBytes;
};

template <int T, int E>
__global__ void __launch_bounds__(T) collision_mark_kernel(const uint64_t *__restrict__ A, int64_t m,
                                                           const uint64_t *__restrict__ B, int64_t n,
                                                           const int64_t *__restrict__ part_i,
                                                           uint32_t *__restrict__ C,
                                                           uint32_t *__restrict__ lb_B,
                                                           int32_t *status) {
  using L = MarkLayout<T, E>;
  constexpr int D = L::D;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::kBar);
  uint32_t *sLB = reinterpret_cast<uint32_t *>(smem + L::kLB);
  uint32_t *sCw = reinterpret_cast<uint32_t *>(smem + L::kCw);
  const int tid = threadIdx.x;

  const int64_t g = blockIdx.x;
  const int64_t total = m + n;
  const int64_t k0 = g * D;
  const int64_t k1 = k0 + D < total ? k0 + D : total;
  const int64_t i0 = part_i[g], i1 = part_i[g + 1];
  const int64_t j0 = k0 - i0, j1 = k1 - i1;
  const int na = static_cast<int>(i1 - i0), nb = static_cast<int>(j1 - j0);
  const int hp = i0 > 0 ? 1 : 0;   // A[i0-1] staged in front (for B's lower bounds)
  const int hn = j1 < n ? 1 : 0;   // B[j1] staged behind (for A's collision bits)

  const StagePlan pa = stage_plan<8>(i0 - hp, na + hp);
  const StagePlan pb = stage_plan<8>(j0, nb + hn);
  uint64_t *bufA = reinterpret_cast<uint64_t *>(smem + L::kKeys);
  uint64_t *bufB = reinterpret_cast<uint64_t *>(smem + L::kKeys + stage_capacity_bytes<8>(pa.span));

  const int64_t w0 = i0 >> 5;
  const int nw = na > 0 ? static_cast<int>(((i1 - 1) >> 5) - w0 + 1) : 0;
  for (int x = tid; x < nw; x += T) sCw[x] = 0u;

  if (tid == 0) mbar_init(bar, 1);
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, pa.bulk + pb.bulk);
    stage_issue(bufA, A, pa, bar);
    stage_issue(bufB, B, pb, bar);
  }
  stage_tail(bufA, A, pa, i0 - hp, na + hp, tid);
  stage_tail(bufB, B, pb, j0, nb + hn, tid);
  const bool ok = mbar_wait_bounded(bar, 0, kWaitLimitNs);
  if (__syncthreads_or(!ok)) {
    if (tid == 0) report(status, LSM_ERR_TIMEOUT);
    return;
  }

  const uint64_t *sA = bufA + pa.lead + hp;  // sA[-1] = A[i0-1] when hp
  const uint64_t *sB = bufB + pb.lead;       // sB[nb] = B[j1] when hn
  const int cnt = na + nb;
  const int d = tid * E < cnt ? tid * E : cnt;
  int lo = d > nb ? d - nb : 0, hi = d < na ? d : na;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (sA[mid] <= sB[d - mid - 1]) lo = mid + 1;
    else hi = mid;
  }
  int ai = lo, bi = d - lo;
#pragma unroll
  for (int s = 0; s < E; ++s) {
    if (d + s < cnt) {
      const bool takeA = (bi >= nb) || (ai < na && sA[ai] <= sB[bi]);
      if (takeA) {
        // A_i collides exactly when the B element at the head equals it.
        if ((bi < nb || hn) && sA[ai] == sB[bi]) {
          const int64_t gi = i0 + ai;
          atomicOr(&sCw[(gi >> 5) - w0], 1u << (gi & 31));
        }
        ++ai;
      } else {
        const uint64_t bk = sB[bi];
        const int hit = ((ai > 0 || hp) && sA[ai - 1] == bk) ? 1 : 0;
        sLB[bi] = static_cast<uint32_t>(i0 + ai - hit);
        ++bi;
      }
    }
  }
  __syncthreads();
  for (int x = tid; x < nb; x += T) lb_B[j0 + x] = sLB[x];
  for (int x = tid; x < nw; x += T) {
    const int64_t w = w0 + x;
    const uint32_t bits = sCw[x];
    const bool whole = (w * 32 >= i0) && (w * 32 + 32 <= i1);
    if (whole) C[w] = bits;
    else if (bits) atomicOr(&C[w], bits);
  }
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

__global__ void __launch_bounds__(256) rank_query_kernel(const uint32_t *__restrict__ C,
                                                         const uint32_t *__restrict__ dir, int64_t m,
                                                         const uint32_t *__restrict__ pos, int64_t q,
                                                         uint32_t *__restrict__ out, int32_t *status) {
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

// ---- compact: merge path over positions ---------------------------------------------
template <int T, int E>
struct CompactLayout {
  static constexpr int D = T * E;
  static constexpr int64_t kBar = 0;
  static constexpr int64_t kLB = 128;
  static constexpr int64_t kLBBytes = align_up(int64_t(D) * 4 + 128, 16);
  static constexpr int64_t kCw = kLB + kLBBytes;
  static constexpr int64_t kCwBytes = align_up(int64_t(D / 32 + 4) * 4, 16);
  static constexpr int64_t kRefs = kCw + kCwBytes;
  static constexpr int64_t kOrdA = kRefs + align_up(int64_t(D) * 4, 16);
  static constexpr int64_t kOrdB = kOrdA + align_up(int64_t(D) * 4, 16);
  static constexpr int64_t kScan = kOrdB + align_up(int64_t(D) * 4, 16);
  static constexpr int64_t kBytes = kScan + align_up(int64_t(T / 32 + 2) * 4, 16);
};

constexpr uint32_t kRecNone = 0u;
constexpr uint32_t kRecA = 1u << 30;      // A element kept
constexpr uint32_t kRecDrop = 2u << 30;   // A element dropped
constexpr uint32_t kRecB = 3u << 30;      // B element
constexpr uint32_t kRecIdx = (1u << 30) - 1u;

template <int T, int E>
__global__ void __launch_bounds__(T) compact_kernel(int64_t m, int64_t n, const uint32_t *__restrict__ C,
                                                    const uint32_t *__restrict__ dir,
                                                    const uint32_t *__restrict__ lb_B,
                                                    const int64_t *__restrict__ part_i,
                                                    uint32_t *__restrict__ refs,
                                                    uint32_t *__restrict__ ord_A,
                                                    uint32_t *__restrict__ ord_B,
                                                    int64_t *__restrict__ d_count, int32_t *status) {
  using L = CompactLayout<T, E>;
  constexpr int D = L::D;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::kBar);
  uint32_t *bufLB = reinterpret_cast<uint32_t *>(smem + L::kLB);
  uint32_t *sCw = reinterpret_cast<uint32_t *>(smem + L::kCw);
  uint32_t *sRefs = reinterpret_cast<uint32_t *>(smem + L::kRefs);
  uint32_t *sOrdA = reinterpret_cast<uint32_t *>(smem + L::kOrdA);
  uint32_t *sOrdB = reinterpret_cast<uint32_t *>(smem + L::kOrdB);
  uint32_t *sScan = reinterpret_cast<uint32_t *>(smem + L::kScan);
  __shared__ uint32_t sR0;
  const int tid = threadIdx.x;

  const int64_t g = blockIdx.x;
  const int64_t total = m + n;
  if (total == 0) {  // the single CTA launched for two empty inputs
    if (tid == 0) *d_count = 0;
    return;
  }
  const int64_t k0 = g * D;
  const int64_t k1 = k0 + D < total ? k0 + D : total;
  const int64_t i0 = part_i[g], i1 = part_i[g + 1];
  const int64_t j0 = k0 - i0, j1 = k1 - i1;
  const int na = static_cast<int>(i1 - i0), nb = static_cast<int>(j1 - j0);

  const StagePlan pl = stage_plan<4>(j0, nb);
  if (tid == 0) mbar_init(bar, 1);
  const int64_t w0 = i0 >> 5;
  const int nw = na > 0 ? static_cast<int>(((i1 - 1) >> 5) - w0 + 1) : 0;
  for (int x = tid; x < nw; x += T) sCw[x] = C[w0 + x];
  if (tid == 0) sR0 = rank512_at(C, dir, i0);
  if (g == 0 && tid == 0) *d_count = total - static_cast<int64_t>(rank512_at(C, dir, m));
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, pl.bulk);
    stage_issue(bufLB, lb_B, pl, bar);
  }
  stage_tail(bufLB, lb_B, pl, j0, nb, tid);
  const bool ok = mbar_wait_bounded(bar, 0, kWaitLimitNs);
  if (__syncthreads_or(!ok)) {
    if (tid == 0) report(status, LSM_ERR_TIMEOUT);
    return;
  }
  const uint32_t *sLB = bufLB + pl.lead;

  const int cnt = na + nb;
  const int d = tid * E < cnt ? tid * E : cnt;
  int lo = d > nb ? d - nb : 0, hi = d < na ? d : na;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (i0 + mid < static_cast<int64_t>(sLB[d - mid - 1])) lo = mid + 1;
    else hi = mid;
  }
  int ai = lo, bi = d - lo;
  uint32_t rec[E];
  uint32_t kept = 0;
#pragma unroll
  for (int s = 0; s < E; ++s) {
    rec[s] = kRecNone;
    if (d + s < cnt) {
      const bool takeA = (bi >= nb) || (ai < na && i0 + ai < static_cast<int64_t>(sLB[bi]));
      if (takeA) {
        const int64_t gi = i0 + ai;
        const uint32_t drop = (sCw[(gi >> 5) - w0] >> (gi & 31)) & 1u;
        rec[s] = (drop ? kRecDrop : kRecA) | static_cast<uint32_t>(ai);
        kept += 1u - drop;
        ++ai;
      } else {
        rec[s] = kRecB | static_cast<uint32_t>(bi);
        ++kept;
        ++bi;
      }
    }
  }
  uint32_t kept_total;
  uint32_t pos = block_exclusive_sum<T>(kept, sScan, &kept_total);
  const int64_t out0 = k0 - static_cast<int64_t>(sR0);
#pragma unroll
  for (int s = 0; s < E; ++s) {
    const uint32_t kind = rec[s] & ~kRecIdx, idx = rec[s] & kRecIdx;
    if (kind == kRecA) {
      sRefs[pos] = static_cast<uint32_t>(i0 + idx);
      sOrdA[idx] = static_cast<uint32_t>(out0 + pos);
      ++pos;
    } else if (kind == kRecDrop) {
      sOrdA[idx] = LSM_ORD_DROPPED;
    } else if (kind == kRecB) {
      sRefs[pos] = LSM_REF_FROM_B | static_cast<uint32_t>(j0 + idx);
      sOrdB[idx] = static_cast<uint32_t>(out0 + pos);
      ++pos;
    }
  }
  __syncthreads();
  for (uint32_t x = tid; x < kept_total; x += T) refs[out0 + x] = sRefs[x];
  for (int x = tid; x < na; x += T) ord_A[i0 + x] = sOrdA[x];
  for (int x = tid; x < nb; x += T) ord_B[j0 + x] = sOrdB[x];
}

}  // namespace

cudaError_t launch_collision_mark(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                  uint32_t *C, uint32_t *lb_B, int64_t *part_i, int32_t *status,
                                  cudaStream_t s) {
  using L = MarkLayout<kMarkThreads, kMarkItems>;
  const int64_t nwords = (m + 31) / 32;
  cudaError_t err = launch_partition(U64AFirst{A, B}, m, n, L::D, part_i, C, nwords, s);
  if (err != cudaSuccess) return err;
  const int64_t G = (m + n + L::D - 1) / L::D;
  if (G == 0) return cudaSuccess;
  auto kern = collision_mark_kernel<kMarkThreads, kMarkItems>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(L::kBytes));
  if (err != cudaSuccess) return err;
  profile_before(s);
  kern<<<static_cast<unsigned>(G), kMarkThreads, L::kBytes, s>>>(A, m, B, n, part_i, C, lb_B, status);
  profile_after(s);
  return cudaGetLastError();
}

int64_t rank_build_ctas(int64_t m) { return (m / 512 + 1 + kRankThreads - 1) / kRankThreads; }

cudaError_t launch_rank_build(const uint32_t *C, int64_t m, uint32_t *dir, int64_t *d_total,
                              uint32_t *cta_totals, cudaStream_t s) {
  const int64_t ctas = rank_build_ctas(m);
  profile_before(s);
  rank_count_kernel<<<static_cast<unsigned>(ctas), kRankThreads, 0, s>>>(C, m, cta_totals);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  rank_finish_kernel<<<static_cast<unsigned>(ctas), kRankThreads, 0, s>>>(C, m, cta_totals, dir, d_total);
  profile_after(s);
  return cudaGetLastError();
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
  rank_query_kernel<<<static_cast<unsigned>((q + 255) / 256), 256, 0, s>>>(C, dir, m, pos, q, out, status);
  return cudaGetLastError();
}

cudaError_t launch_compact(int64_t m, int64_t n, const uint32_t *C, const uint32_t *dir,
                           const uint32_t *lb_B, uint32_t *refs, uint32_t *ord_A,
                           uint32_t *ord_B, int64_t *d_count, int64_t *part_i, int32_t *status,
                           cudaStream_t s) {
  using L = CompactLayout<kCompactThreads, kCompactItems>;
  cudaError_t err = launch_partition(PositionsBFirst{lb_B}, m, n, L::D, part_i, nullptr, 0, s);
  if (err != cudaSuccess) return err;
  const int64_t G = (m + n + L::D - 1) / L::D;
  auto kern = compact_kernel<kCompactThreads, kCompactItems>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(L::kBytes));
  if (err != cudaSuccess) return err;
  // At least one CTA, so that d_count is written for two empty inputs.
  profile_before(s);
  kern<<<static_cast<unsigned>(G > 0 ? G : 1), kCompactThreads, L::kBytes, s>>>(
      m, n, C, dir, lb_B, part_i, refs, ord_A, ord_B, d_count, status);
  profile_after(s);
  return cudaGetLastError();
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
