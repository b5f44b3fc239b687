// replacement.cu -- the replacement merge of two strictly sorted unique-key
// inputs (uint64 keys) as two tile pipelines with warp-independent consumers.
//
// "Everett: collision bitmap and rank experiment":
//   - "Corrected record ordinals": C_i = 1 exactly when A_i's key is in B;
//     R(i) = sum_{t<i} C_t; a surviving A_i lands at i + lower_bound(B, A_i)
//     - R(i) and B_j, with lower bound i in A, at j + i - R(i).
//   - "The three experimental paths", third path: survivors of A and all of
//     B have disjoint keys and are merged by merge path.
//   - "Dispatch bindings": count, global scan, finish.
//
// The path: a co-rank partition of the keys (A first on ties; also clears C),
// the collision mark, the rank512 build and the compaction.
//
//   mark      per merge-path tile of D = T E keys the loader warp stages
//             A[i0-1, i1) and B[j0, j1 + 1) with bulk copies; once they land
//             every consumer thread finds the lower bound of one HG-th B key
//             (a group head) in the staged A span, and the last one writes
//             the compaction's co-rank at the tile start. After one consumer
//             barrier every lane searches two B keys between their groups'
//             heads (the two searches stepped together); lb_B goes to global
//             memory straight from the lanes when the caller wants it, a key
//             equal to its lower-bound A key sets that collision bit with an
//             atomic OR (C was cleared by the partition), and the key's
//             position in the merge with B first on ties, j + lb_B[j], sets a
//             bit of the tile's words of the merge bitmap MB in shared memory,
//             which the last warp writes out at the next tile's barrier.
//   compact   merge path over positions (B first on ties): position p of the
//             merge holds a B record exactly when MB bit p is set, so the
//             merge of A's survivors and B needs MB and C only. Its tiles have
//             the mark's diagonals: the co-rank at k0 in this order is the
//             mark's i0, less one when A[i0-1] = B[j0] (the one equal pair
//             that can straddle the cut). The loader stages the tile's MB
//             words and C words and fetches R(i0) from the rank directory.
//             Each consumer warp owns 32 E consecutive positions: popcounts
//             of the MB words and C words before them give its first B record
//             and its dropped A records before, two warp scans place every
//             lane, and each lane walks its E positions, writing refs and
//             ordinals into the warp's shared buffers, which the warp moves
//             out as three contiguous runs (bulk stores), with no barrier
//             between consumer warps.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "lookback.cuh"
#include "pipeline.cuh"
#include "rank2048.cuh"
#include "rank512.cuh"

// Minimum resident CTAs per SM the mark kernel is compiled for (register
// budget). Measured on the 12M + 4M step (whole path, L2 flushed by a write
// before each step, medians of 50): 3 CTAs (72 registers, no spills) 89.8
// us against 91.8 us for 2 (94 registers) and for the compiler's choice (96).
#ifndef MARK_MIN_BLOCKS
#define MARK_MIN_BLOCKS 3
#endif
// The same for the compaction kernel: 5 CTAs (72 registers, no spills)
// 87.7 us against 88.8 us before its walk lost its branches, 90.8 us for 4
// CTAs (94 registers) and 93.8 us for the compiler's choice (119, 3 CTAs).
#ifndef COMPACT_MIN_BLOCKS
#define COMPACT_MIN_BLOCKS 5
#endif

namespace lsm {

namespace {

// ---- co-rank partition ---------------------------------------------------------
struct KeysAFirst {
  const uint64_t *A;
  const uint64_t *B;
  __device__ __forceinline__ bool too_small(int64_t i, int64_t k) const {
    return __ldg(A + i) <= __ldg(B + k - i - 1);
  }
};

// The co-rank of every diagonal k_g = min(g D, m + n), g = 0..G, by a group
// of L lanes per diagonal (L + 1-way splits per round: about log_{L+1}(n)
// dependent rounds of loads); the same launch clears C and the lookback
// states of the kernels after it (Z0[0, n0), Z1[0, n1)).
template <int L>
__global__ void __launch_bounds__(256) corank_partition_kernel(KeysAFirst pred, int64_t m, int64_t n,
                                                               int64_t D, int64_t G,
                                                               int64_t *__restrict__ out_i,
                                                               uint32_t *__restrict__ C,
                                                               int64_t nwords,
                                                               uint64_t *__restrict__ Z0,
                                                               int64_t n0,
                                                               uint64_t *__restrict__ Z1,
                                                               int64_t n1) {
  pdl_begin();
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t w = gtid; w < nwords; w += stride) C[w] = 0u;
  for (int64_t w = gtid; w < n0; w += stride) Z0[w] = 0u;
  for (int64_t w = gtid; w < n1; w += stride) Z1[w] = 0u;
  const int64_t g = gtid / L;
  const bool active = g <= G;
  const int64_t total = m + n;
  const int64_t k = active ? (g * D < total ? g * D : total) : 0;
  const int64_t i = group_corank<L>(pred, k, m, n, active);
  if (active && (threadIdx.x & (L - 1)) == 0) out_i[g] = i;
}

// ---- waits that sleep ------------------------------------------------------------
// mbarrier.try_wait with a suspend-time hint: a thread whose phase is not yet
// complete is suspended until the phase completes (or the hint runs out)
// instead of returning at once, so that waiting warps do not take issue slots
// from the warps doing the work. Bounded like every wait here: past limit_ns
// of %globaltimer the wait gives up and returns false.
constexpr uint32_t kSuspendHintNs = 1000000;  // 1 ms per suspended try

__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

static __device__ __noinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, int64_t limit_ns) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 20); ++it) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (globaltimer_ns() - t0 > static_cast<uint64_t>(limit_ns)) return false;
  }
  return false;
}

// ---- the warp pipeline -----------------------------------------------------------
// One CTA per SM slot loops over tiles c, c + P, ... (P = gridDim.x). The
// last warp is the loader: its lanes fetch the per-tile prologue values of
// 32 tiles at a time and lane 0 stages each tile into one of S stages with
// bulk copies (Spec::produce, completing `full`) as soon as that stage's
// previous tile has been released. The consumer warps wait on `full`; each
// runs Spec::consume on its own share of the tile, with no barrier between
// consumer warps, and arrives on `empty` once it no longer reads the stage.
// Every wait is bounded in time.
template <class Spec>
struct WLayout {
  static constexpr int S = Spec::S;
  static constexpr int64_t kFull = 0, kEmpty = 8 * S, kDesc = 16 * S;
  static constexpr int64_t kStage0 = align_up(16 * S + 64 * S, 128);
  static constexpr int64_t kStageStride = align_up(Spec::kStageBytes, 128);
  static constexpr int64_t kWork = kStage0 + S * kStageStride;
  static constexpr int64_t kBytes = kWork + Spec::kWorkBytes;
};

template <class Spec>
__global__ void __launch_bounds__(Spec::T + 32, Spec::kMinBlocks) warp_pipeline_kernel(typename Spec::Params p,
                                                                     int64_t G, int32_t *status) {
  pdl_begin();
  using L = WLayout<Spec>;
  constexpr int S = Spec::S;
  constexpr int T = Spec::T;
  using Desc = typename Spec::Desc;
  static_assert(sizeof(Desc) <= 64, "descriptor slot");
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kFull);
  uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L::kEmpty);
  Desc *desc = reinterpret_cast<Desc *>(smem + L::kDesc);
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int64_t P = gridDim.x;
  const int64_t R = (G - blockIdx.x + P - 1) / P;  // tiles of this CTA (grid <= G)

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], T / 32);
    }
  }
  Spec::init(smem + L::kWork);
  __syncthreads();

  if (tid >= T) {
    int64_t v[4] = {0, 0, 0, 0};
    for (int64_t r = 0; r < R; ++r) {
      if ((r & 31) == 0) {
        const int64_t gl = blockIdx.x + (r + lane) * P;
        v[0] = v[1] = v[2] = v[3] = 0;
        if (gl < G) Spec::fetch(p, gl, v);
      }
      int64_t w[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) w[t] = __shfl_sync(0xffffffffu, v[t], static_cast<int>(r & 31));
      int failed = 0;
      if (lane == 0) {
        const int s = static_cast<int>(r % S);
        if (r >= S && !mbar_wait_sleep(&empty[s], static_cast<uint32_t>(((r / S) + 1) & 1),
                                       kWaitLimitNs)) {
          report(status, LSM_ERR_TIMEOUT);
          failed = 1;
        } else {
          Spec::produce(p, blockIdx.x + r * P, w, smem + L::kStage0 + s * L::kStageStride, desc[s],
                        &full[s]);
        }
      }
      if (__shfl_sync(0xffffffffu, failed, 0)) return;
    }
    return;
  }

  int64_t done = 0;
  for (int64_t r = 0; r < R; ++r) {
    const int s = static_cast<int>(r % S);
    const bool ok = mbar_wait_sleep(&full[s], static_cast<uint32_t>((r / S) & 1), kWaitLimitNs);
    // a private copy: once the stage is released the loader rewrites it
    const Desc d = desc[s];
    if (!Spec::consume(p, blockIdx.x + r * P, r, d, smem + L::kStage0 + s * L::kStageStride,
                       smem + L::kWork, &empty[s], ok, status))
      break;
    done = r + 1;
  }
  Spec::finish(p, smem + L::kWork, done);
}

// Launches the pipeline with as many CTAs as fit on the device (at most G).
template <class Spec>
cudaError_t launch_warp_pipeline(const typename Spec::Params &p, int64_t G, int32_t *status,
                                 cudaStream_t s) {
  using L = WLayout<Spec>;
  static_assert(L::kBytes <= 227 * 1024, "pipeline exceeds shared memory");
  auto kern = warp_pipeline_kernel<Spec>;
  static int per_sm = 0;
  if (!per_sm) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(L::kBytes));
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Spec::T + 32, L::kBytes);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
  }
  int64_t grid = static_cast<int64_t>(device_sm_count()) * per_sm;
  if (grid > G) grid = G;
  if (grid < 1) return cudaSuccess;
  return launch_kernel(true, kern, static_cast<unsigned>(grid), Spec::T + 32, L::kBytes, s, p, G,
                       status);
}

// Bulk copy global -> shared with an L2 evict-first policy: each staged key
// or lower bound is read once, so its lines go first when L2 needs room
// (rather than lines that other work still needs, or dirty lines that would
// have to be written back).
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
template <typename T>
__device__ __forceinline__ void stage_issue_ef(T *buf, const T *g, const StagePlan &pl,
                                               uint64_t *bar) {
  if (pl.bulk) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1], %2, [%3], %4;" ::"r"(smem_u32(buf)),
        "l"(g + pl.first), "r"(pl.bulk), "r"(smem_u32(bar)), "l"(evict_first_policy())
        : "memory");
  }
}

// Writes global uint32 elements [g0, g0 + count) of `gbase` from a warp's
// shared buffer that holds element g0 at sbuf[g0 & 3] (sbuf 16-byte aligned,
// gbase 16-byte aligned), so that shared and global addresses agree modulo
// 16: lane 0 moves the aligned body with one bulk store (committed by the
// caller), lanes 1-3 the head and lanes 8-10 the tail elements. The caller
// fences the shared writes for the async proxy and syncs the warp first.
__device__ __forceinline__ void warp_store_run(uint32_t *gbase, int64_t g0, int count,
                                               const uint32_t *sbuf) {
  if (count <= 0) return;
  const int lane = threadIdx.x & 31;
  const int shift = static_cast<int>(g0 & 3);
  const int head = count < ((4 - shift) & 3) ? count : ((4 - shift) & 3);
  const int body = (count - head) & ~3;
  const int tail = count - head - body;
  if (lane == 0 && body) bulk_s2g(gbase + g0 + head, sbuf + shift + head, static_cast<uint32_t>(body) * 4);
  const int t = lane - 1;
  if (t >= 0 && t < head) gbase[g0 + t] = sbuf[shift + t];
  if (t >= 7 && t < 7 + tail) gbase[g0 + head + body + (t - 7)] = sbuf[shift + head + body + (t - 7)];
}

// Count of x in [lo, hi) with a[x] < key (a sorted), by steps of the powers
// of two below `span` (the largest hi - lo over the warp, so that every lane
// takes the same number of steps): lo plus that count. Each step loads at a
// clamped index (inside [lo, hi)) and keeps the candidate only when it lies
// inside the range, so that the step needs no branch. Spans below 64 (the
// common case of a group of keys between two heads) run fully unrolled.
__device__ __forceinline__ int count_below_step(const uint64_t *a, int x, int hi, uint64_t key,
                                                int step) {
  const int c = x + step;
  const int ci = c < hi ? c : hi;  // >= x + 1 > lo whenever a step is taken
  const bool lt = a[ci - 1] < key;
  return (c <= hi && lt) ? c : x;
}

__device__ __forceinline__ int count_below(const uint64_t *a, int lo, int hi, uint64_t key,
                                           int span) {
  int x = lo;
  if (span < 64) {
    const int k = span ? 32 - __clz(span) : 0;  // steps: the bit length of span
    switch (k) {
      case 6: x = count_below_step(a, x, hi, key, 32); [[fallthrough]];
      case 5: x = count_below_step(a, x, hi, key, 16); [[fallthrough]];
      case 4: x = count_below_step(a, x, hi, key, 8); [[fallthrough]];
      case 3: x = count_below_step(a, x, hi, key, 4); [[fallthrough]];
      case 2: x = count_below_step(a, x, hi, key, 2); [[fallthrough]];
      case 1: x = count_below_step(a, x, hi, key, 1); [[fallthrough]];
      default: break;
    }
    return x;
  }
  for (int step = 1 << (31 - __clz(span)); step; step >>= 1) x = count_below_step(a, x, hi, key, step);
  return x;
}

// Two independent count_below searches stepped together (the same number of
// steps, from the larger span), so that each step's two shared loads and
// compares overlap instead of forming one chain per key.
__device__ __forceinline__ void count_below2(const uint64_t *a, int &x0, int hi0, uint64_t key0,
                                             int &x1, int hi1, uint64_t key1, int span) {
  if (span < 64) {
    const int k = span ? 32 - __clz(span) : 0;
    switch (k) {
#define LSM_CB2_STEP(s)                                  \
  x0 = count_below_step(a, x0, hi0, key0, s);            \
  x1 = count_below_step(a, x1, hi1, key1, s);
      case 6: LSM_CB2_STEP(32) [[fallthrough]];
      case 5: LSM_CB2_STEP(16) [[fallthrough]];
      case 4: LSM_CB2_STEP(8) [[fallthrough]];
      case 3: LSM_CB2_STEP(4) [[fallthrough]];
      case 2: LSM_CB2_STEP(2) [[fallthrough]];
      case 1: LSM_CB2_STEP(1) [[fallthrough]];
      default: break;
#undef LSM_CB2_STEP
    }
    return;
  }
  for (int step = 1 << (31 - __clz(span)); step; step >>= 1) {
    x0 = count_below_step(a, x0, hi0, key0, step);
    x1 = count_below_step(a, x1, hi1, key1, step);
  }
}

// The first x in [lo, hi] at which a monotone predicate (true, then false)
// turns false, found by 16 lanes together: each round the half-warp tests
// the 16 pivots lo + (l span) / 16 (l = 0..15) and keeps the gap between the
// last true and the first false, so the range shrinks about 16-fold per
// round. Lanes 0-15 and 16-31 search independently; every lane of the warp
// must call it.
template <class Pred>
__device__ __forceinline__ int half_warp_search(int lo, int hi, const Pred &pred) {
  const int lane = threadIdx.x & 31;
  const int l = lane & 15, sh = lane & 16;
  while (__any_sync(0xffffffffu, lo < hi)) {
    const int span = hi - lo;
    const bool t = span > 0 && pred(lo + ((l * span) >> 4));
    const int c = __popc((__ballot_sync(0xffffffffu, t) >> sh) & 0xFFFFu);
    if (span > 0) {
      // pivots 0..c-1 are true (below the answer), pivot c is the first false
      const int nlo = c > 0 ? lo + (((c - 1) * span) >> 4) + 1 : lo;
      const int nhi = c < 16 ? lo + ((c * span) >> 4) : hi;
      lo = nlo;
      hi = nhi;
    }
  }
  return lo;
}

// ---- collision mark ------------------------------------------------------------
// Stage: A[i0 - hp, i1) and B[j0, j1 + hn), hp = (i0 > 0), hn = (j1 < n): the
// A key before the tile bounds the lower bounds of its first B keys, and B[j0]
// is read for the compaction's co-rank even when the tile holds no B key.
// Every B key of the tile has its lower bound in [i0 - hp, i1] (merge path,
// A first on ties). Two phases per tile: every HG-th B key (a group head)
// takes its lower bound over the whole staged A span, one head per consumer
// thread; after a consumer barrier every B key searches only between its
// group's head and the next one. The heads live in two buffers (tile parity),
// so a warp may start the next tile's heads while others finish this one.
template <int T_, int E_, int S_, int HG_>
struct MarkTile {
  static constexpr int T = T_, E = E_, S = S_, HG = HG_;
  static constexpr int D = T * E, NW = T / 32;
  static constexpr int kMaxHeads = D / HG + 4;
  static constexpr int NMB = D / 32;  // merge bitmap words of one tile
  static constexpr int kMinBlocks = MARK_MIN_BLOCKS;
  static constexpr int64_t kStageBytes = align_up(int64_t(D + 4) * 8 + 160, 16);
  static constexpr int64_t kHeadsBytes = align_up(int64_t(kMaxHeads) * 4, 16);
  static constexpr int64_t kBitsBytes = align_up(int64_t(NMB) * 4, 16);
  static constexpr int64_t kWorkBytes = 2 * kHeadsBytes + 2 * kBitsBytes + 16;
  static_assert(D % 32 == 0, "a tile's merge bitmap is whole words");
  static_assert(32 % HG == 0, "group heads divide a warp's 32 keys");
  struct Params {
    const uint64_t *A, *B;
    int64_t m, n, G;
    const int64_t *part_i;
    uint32_t *C, *lb_B;
    int64_t *part_c;  // the compaction's co-ranks (G + 1), or null
    uint32_t *MB;     // the merge bitmap (cleared), or null
  };
  struct Desc {
    int64_t i0, j0;
    int32_t na, nb, hp, hn, offA, offB;
  };
  __device__ __forceinline__ static uint32_t *bits_buf(uint8_t *work, int64_t r) {
    return reinterpret_cast<uint32_t *>(work + 2 * kHeadsBytes + (r & 1) * kBitsBytes);
  }
  __device__ __forceinline__ static void init(uint8_t *work) {
    uint32_t *b = reinterpret_cast<uint32_t *>(work + 2 * kHeadsBytes);
    for (int x = threadIdx.x; x < 2 * NMB; x += blockDim.x) b[x] = 0u;
  }
  // The merge bitmap words of the tile consumed at step r, once every
  // consumer warp has passed the barrier of step r + 1 (or the final one):
  // written by the last warp and cleared for step r + 2.
  __device__ __forceinline__ static void flush_bits(const Params &p, int64_t g, uint8_t *work,
                                                    int64_t r) {
    if (!p.MB || threadIdx.x < T - 32) return;
    uint32_t *b = bits_buf(work, r);
    const int64_t total = p.m + p.n;
    const int64_t k0 = g * D;
    const int nw = static_cast<int>(((total - k0 < D ? total - k0 : D) + 31) / 32);
    for (int x = threadIdx.x & 31; x < NMB; x += 32) {
      if (x < nw) p.MB[g * NMB + x] = b[x];
      b[x] = 0u;
    }
    __syncwarp();
  }
  // After the last tile: one more consumer barrier, then its bitmap words.
  __device__ __forceinline__ static void finish(const Params &p, uint8_t *work, int64_t rdone) {
    if (!p.MB || rdone <= 0) return;
    named_sync(1, T);
    flush_bits(p, blockIdx.x + (rdone - 1) * static_cast<int64_t>(gridDim.x), work, rdone - 1);
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
    stage_issue_ef(bufA, p.A, pa, full);
    stage_issue_ef(bufB, p.B, pb, full);
  }
  __device__ __forceinline__ static bool consume(const Params &p, int64_t g, int64_t r,
                                                 const Desc &d, const uint8_t *stage, uint8_t *work,
                                                 uint64_t *empty, bool ok, int32_t *status) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t *sA = reinterpret_cast<const uint64_t *>(stage) + d.offA;
    const uint64_t *sAx = sA - d.hp;
    const uint64_t *sB = reinterpret_cast<const uint64_t *>(stage) + d.offB;
    const int nb = d.nb, lenx = d.na + d.hp;
    int *heads = reinterpret_cast<int *>(work + (r & 1) * align_up(int64_t(kMaxHeads) * 4, 16));
    const int nh = (nb + HG - 1) / HG;
    // 1. the group heads, one per thread, and the compaction's co-rank at
    //    this tile's diagonal (B first on ties: one less when the equal pair
    //    A[i0-1] = B[j0] straddles it)
    uint32_t *bits = bits_buf(work, r);
    const int64_t k0 = g * D;
    if (ok) {
      for (int h = tid; h < nh; h += T) heads[h] = count_below(sAx, 0, lenx, sB[h * HG], lenx);
      if (tid == T - 1) {
        heads[nh] = lenx;
        if (p.part_c) {
          const bool tie = d.hp && nb + d.hn > 0 && sA[-1] == sB[0];
          p.part_c[g] = d.i0 - (tie ? 1 : 0);
          if (g == p.G - 1) p.part_c[p.G] = p.m;
        }
        // B[j1] (after the tile) sits at this tile's last position of the
        // merge with B first on ties exactly when it equals the tile's last
        // A key, A[i1-1]
        if (p.MB && d.hn && d.na > 0 && sA[d.na - 1] == sB[nb]) {
          const int rp = (d.na + nb) - 1;
          atomicOr(bits + (rp >> 5), 1u << (rp & 31));
        }
      }
    }
    if (named_sync_or(1, T, !ok)) {
      if (tid == 0) report(status, LSM_ERR_TIMEOUT);
      release_stage(empty);
      return false;
    }
    if (r > 0) flush_bits(p, g - static_cast<int64_t>(gridDim.x), work, r - 1);
    // 2. every B key between its group's heads, two keys per lane (b and
    //    b + 32) searched together; lb_B straight to global memory (32
    //    consecutive words per warp and key slot) unless the caller wants
    //    none, collisions by atomic OR
    const uint32_t base = static_cast<uint32_t>(d.i0 - d.hp);
    const uint32_t jbase = static_cast<uint32_t>(d.j0);
    uint32_t *lbo = p.lb_B ? p.lb_B + d.j0 : nullptr;
    // the tile-relative position of B key bi with lower bound base + x in the
    // merge with B first on ties is jbase + bi + base + x - k0; this tile
    // owns positions [k0, k0 + D) (B[j0] falls at k0 - 1, in the previous
    // tile, when it equals A[i0-1])
    const uint32_t rbase = jbase + base - static_cast<uint32_t>(k0);
    for (int b0 = warp * 64; b0 < nb; b0 += NW * 64) {
      const int bi0 = b0 + lane, bi1 = bi0 + 32;
      const bool act0 = bi0 < nb, act1 = bi1 < nb;
      const uint64_t key0 = sB[act0 ? bi0 : nb - 1], key1 = sB[act1 ? bi1 : nb - 1];
      const int h0 = bi0 / HG, h1 = bi1 / HG;
      int x0 = act0 ? heads[h0] : 0, x1 = act1 ? heads[h1] : 0;
      const int hi0 = act0 ? heads[h0 + 1] : 0, hi1 = act1 ? heads[h1 + 1] : 0;
      const int sp = (hi0 - x0) > (hi1 - x1) ? (hi0 - x0) : (hi1 - x1);
      const int span = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(sp)));
      count_below2(sAx, x0, hi0, key0, x1, hi1, key1, span);
      const bool hit0 = act0 && x0 < lenx && sAx[x0] == key0;
      const bool hit1 = act1 && x1 < lenx && sAx[x1] == key1;
      if (lbo) {
        if (act0) lbo[bi0] = base + static_cast<uint32_t>(x0);
        if (act1) lbo[bi1] = base + static_cast<uint32_t>(x1);
      }
      if (hit0) {
        const uint32_t ia = base + static_cast<uint32_t>(x0);
        atomicOr(p.C + (ia >> 5), 1u << (ia & 31));
      }
      if (hit1) {
        const uint32_t ia = base + static_cast<uint32_t>(x1);
        atomicOr(p.C + (ia >> 5), 1u << (ia & 31));
      }
      if (p.MB) {
        const int rp0 = static_cast<int>(rbase + static_cast<uint32_t>(bi0 + x0));
        const int rp1 = static_cast<int>(rbase + static_cast<uint32_t>(bi1 + x1));
        if (act0 && rp0 >= 0) atomicOr(bits + (rp0 >> 5), 1u << (rp0 & 31));
        if (act1 && rp1 >= 0) atomicOr(bits + (rp1 >> 5), 1u << (rp1 & 31));
      }
    }
    release_stage(empty);
    return true;
  }
};

// ---- compaction ---------------------------------------------------------------
// The merge bitmap MB has bit p set exactly when position p of the merge of
// A's survivors-to-be and B (B first on ties) holds a B record: B_j sits at
// p_j = j + lb_B[j]. Tile g covers positions [g D, g D + D) (D a multiple of
// 32: whole MB words). Stage: the tile's MB words and the C words holding
// A[i0, i1) (tile A record a is bit x = (i0 mod 32) + a of the staged C
// words). Consumer warp w owns the W = 32 E positions [W w, W w + W): the
// popcount of the tile's MB words before them gives its first B record, a
// popcount of the staged C bits its dropped A records before its first A
// record; two warp scans over the lanes' E positions place every lane, and
// each lane writes its refs and ordinals into the warp's shared buffers,
// which the warp stores as three contiguous runs (an aligned bulk copy and
// a few plain stores each). A warp whose counts disagree with the tile's
// co-ranks (an MB that does not come from a lower-bound array of this
// merge) writes nothing and records LSM_ERR_ARG.
template <int T_, int E_, int S_, class RD>
struct CompactTile {
  static constexpr int T = T_, E = E_, S = S_;
  static constexpr int D = T * E, NW = T / 32, W = 32 * E;
  static constexpr int NMB = D / 32;       // merge bitmap words of one tile
  static constexpr int NCW = D / 32 + 4;   // C words of one tile, at most, and slack
  static constexpr int kMinBlocks = COMPACT_MIN_BLOCKS;
  static constexpr int64_t kMBBytes = align_up(int64_t(NMB) * 4 + 16, 16);
  static constexpr int64_t kStageBytes = kMBBytes + align_up(int64_t(NCW + 8) * 4, 16);
  // per warp: refs (W words + alignment lead), ordinals (ord_A then ord_B,
  // W words + two alignment leads and a gap)
  static constexpr int kRefsWords = (W + 8 + 3) & ~3;
  static constexpr int kOrdWords = (W + 12 + 3) & ~3;
  static constexpr int kWarpWords = kRefsWords + kOrdWords;
  static constexpr int64_t kWorkBytes = int64_t(NW) * kWarpWords * 4;
  static_assert(E < 32, "a lane's positions fit one 32-bit window");
  static_assert(D % 128 == 0, "a tile's merge bitmap words start on 16-byte boundaries");
  struct Params {
    int64_t m, n, G;
    const uint32_t *C;
    RD rank;
    const uint32_t *MB;
    const int64_t *part_i;
    uint32_t *refs, *ord_A, *ord_B;
    int64_t *d_count;
  };
  struct Desc {
    int64_t i0, j0, r0;
    int32_t na, nb, offC, pad;
  };
  __device__ __forceinline__ static void init(uint8_t *) {}
  // Bulk stores read shared memory asynchronously: each warp's lane 0 waits
  // for its own before the CTA exits.
  template <class PP>
  __device__ __forceinline__ static void finish(const PP &, uint8_t *, int64_t) {
    if ((threadIdx.x & 31) == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  // The co-ranks are clamped to their diagonals (and i1 - i0 to the tile's
  // length), so that staged ranges stay inside the arrays whatever part_i holds.
  __device__ __forceinline__ static void fetch(const Params &p, int64_t g, int64_t v[4]) {
    const int64_t total = p.m + p.n;
    const int64_t k0 = g * D, k1 = k0 + D < total ? k0 + D : total;
    int64_t i0 = __ldg(p.part_i + g), i1 = __ldg(p.part_i + g + 1);
    const int64_t lo0 = k0 > p.n ? k0 - p.n : 0, hi0 = k0 < p.m ? k0 : p.m;
    i0 = i0 < lo0 ? lo0 : (i0 > hi0 ? hi0 : i0);
    const int64_t lo1 = k1 > p.n ? k1 - p.n : 0, hi1 = k1 < p.m ? k1 : p.m;
    i1 = i1 < lo1 ? lo1 : (i1 > hi1 ? hi1 : i1);
    i1 = i1 < i0 ? i0 : (i1 > i0 + (k1 - k0) ? i0 + (k1 - k0) : i1);  // i1 >= i0, j1 >= j0
    v[0] = i0;
    v[1] = i1;
    v[2] = static_cast<int64_t>(p.rank.at(p.C, i0));
    if (g == 0 && p.d_count) *p.d_count = p.m + p.n - static_cast<int64_t>(p.rank.at(p.C, p.m));
  }
  __device__ __forceinline__ static void produce(const Params &p, int64_t g, const int64_t v[4],
                                                 uint8_t *stage, Desc &d, uint64_t *full) {
    const int64_t total = p.m + p.n;
    const int64_t i0 = v[0], i1 = v[1];
    const int64_t k0 = g * D, k1 = k0 + D < total ? k0 + D : total;
    const int na = static_cast<int>(i1 - i0), nb = static_cast<int>((k1 - i1) - (k0 - i0));
    const int64_t nwords = (p.m + 31) / 32;
    const int64_t w0 = i0 >> 5;
    const int nw = na > 0 ? static_cast<int>(((i1 - 1) >> 5) - w0 + 1) : 0;
    const StagePlan pc = stage_plan_overfetch<4>(w0, nw, nwords);
    uint32_t *bufMB = reinterpret_cast<uint32_t *>(stage);
    uint32_t *bufC = reinterpret_cast<uint32_t *>(stage + kMBBytes);
    for (int64_t x = pc.tail_from; x < w0 + nw; ++x) bufC[x - pc.first] = p.C[x];
    // the tile's merge bitmap words (the array is padded to whole 16-byte
    // groups past its last word)
    const uint32_t mbytes = static_cast<uint32_t>(align_up(((k1 - k0 + 31) / 32) * 4, 16));
    d.i0 = i0;
    d.j0 = k0 - i0;
    d.r0 = v[2];
    d.na = na;
    d.nb = nb;
    d.offC = pc.lead;
    mbar_arrive_expect_tx(full, mbytes + pc.bulk);
    StagePlan pm{};
    pm.first = g * NMB;
    pm.bulk = mbytes;
    stage_issue_ef(bufMB, p.MB, pm, full);
    stage_issue_ef(bufC, p.C, pc, full);
  }
  __device__ __forceinline__ static bool consume(const Params &p, int64_t g, int64_t,
                                                 const Desc &d, const uint8_t *stage, uint8_t *work,
                                                 uint64_t *empty, bool ok, int32_t *status) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int na = d.na, nb = d.nb, cnt = na + nb;
    const int s0 = warp * W;
    bool bad = false;
    if (ok && s0 < cnt) {
      const uint32_t *mb = reinterpret_cast<const uint32_t *>(stage);
      const uint32_t *cw = reinterpret_cast<const uint32_t *>(stage + kMBBytes) + d.offC;
      uint32_t *wRefs = reinterpret_cast<uint32_t *>(work) + warp * kWarpWords;
      uint32_t *wOrd = wRefs + kRefsWords;
      const uint32_t i0u = static_cast<uint32_t>(d.i0), j0u = static_cast<uint32_t>(d.j0);
      const int wbit0 = static_cast<int>(d.i0 & 31);
      const int s1 = cnt - s0 < W ? cnt : s0 + W;  // the warp's positions [s0, s1)
      // 1. B records before the warp's first position, and dropped A records
      //    before its first A record: two popcount sums over the warp
      int pb = 0;
      for (int x = lane; x < (s0 >> 5); x += 32) pb += __popc(mb[x]);
      int a_first_l = 0;  // known only after the B count; summed below
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) pb += __shfl_xor_sync(0xffffffffu, pb, o);
      const int bw0 = pb;
      int a_first = s0 - bw0;  // tile A records before the warp's first position
      bad = a_first < 0 || a_first > na;
      if (bad) a_first = 0;
      const int yend = wbit0 + a_first;
      int pcnt = 0;
      for (int x = lane; x < (yend >> 5); x += 32) pcnt += __popc(cw[x]);
      if (lane == 0) {
        if (yend & 31) pcnt += __popc(cw[yend >> 5] & ((1u << (yend & 31)) - 1u));
        pcnt -= __popc(cw[0] & ((1u << wbit0) - 1u));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) pcnt += __shfl_xor_sync(0xffffffffu, pcnt, o);
      const int drop0 = pcnt;
      (void)a_first_l;
      // 2. this lane's E positions: which hold B records, how many A records
      //    and how many of those are dropped
      const int y = lane * E;
      const int nvalid = (s1 - s0) - y < 0 ? 0 : ((s1 - s0) - y < E ? (s1 - s0) - y : E);
      const int sp = s0 + y;
      const uint32_t w_lo = mb[sp >> 5];
      const uint32_t w_hi = mb[(sp >> 5) + 1];
      uint32_t win = static_cast<uint32_t>(((static_cast<uint64_t>(w_hi) << 32) | w_lo) >> (sp & 31));
      win &= (1u << nvalid) - 1u;
      const int numB = __popc(win);
      const int numA = nvalid - numB;
      const int incB = warp_inclusive_sum(numB);
      const int nB_w = __shfl_sync(0xffffffffu, incB, 31);
      const int nA_w = (s1 - s0) - nB_w;
      bad = bad || a_first + nA_w > na || bw0 + nB_w > nb;
      int a_rel = y - (incB - numB);  // the warp's A records before this lane's first position
      int b_rel = incB - numB;
      const int xa = wbit0 + a_first + a_rel;
      uint32_t cwin = static_cast<uint32_t>(
          ((static_cast<uint64_t>(cw[(xa >> 5) + 1]) << 32) | cw[xa >> 5]) >> (xa & 31));
      cwin &= numA ? (0xFFFFFFFFu >> (32 - numA)) : 0u;
      const int drops = __popc(cwin);
      const int incD = warp_inclusive_sum(drops);
      const int kept_w = (s1 - s0) - __shfl_sync(0xffffffffu, incD, 31);
      int out_rel = y - (incD - drops);  // warp-relative output slot
      // 3. walk the lane's positions into the warp's buffers, laid out at the
      //    global runs' alignment (element t of a run at lead + t, lead = its
      //    first global index mod 4)
      const int64_t gr0 = g * D - d.r0 + s0 - drop0;  // refs run
      const int64_t ga0 = d.i0 + a_first;             // ord_A run
      const int64_t gb0 = d.j0 + bw0;                 // ord_B run
      const int offB = (nA_w + 7) & ~3;
      uint32_t *sR = wRefs + (gr0 & 3);
      uint32_t *sOA = wOrd + (ga0 & 3);
      uint32_t *sOB = wOrd + offB + (gb0 & 3);
      const uint32_t wout0 = static_cast<uint32_t>(gr0);
      const uint32_t ia0 = i0u + static_cast<uint32_t>(a_first), jb0 = j0u + static_cast<uint32_t>(bw0);
      if (lane == 0) bulk_wait_read_all();  // the previous tile's stores from these buffers
      __syncwarp();
      if (!bad && __all_sync(0xffffffffu, nvalid == E)) {
        // every lane holds E positions: a walk without branches. Running
        // shared addresses of the next ord_A, ord_B and refs slots and the
        // next ref values; a dropped A record's ref goes to a scratch word
        // past the refs run (kRefsWords - 1 > 3 + W), so every position
        // makes exactly two stores.
        uint32_t pA = smem_u32(sOA + a_rel), pB = smem_u32(sOB + b_rel);
        uint32_t pR = smem_u32(sR + out_rel);
        const uint32_t dummy = smem_u32(wRefs + kRefsWords - 1);
        uint32_t vA = ia0 + static_cast<uint32_t>(a_rel);
        uint32_t vB = LSM_REF_FROM_B | (jb0 + static_cast<uint32_t>(b_rel));
        uint32_t o = wout0 + static_cast<uint32_t>(out_rel);
        uint32_t cw2 = cwin;
#pragma unroll
        for (int q = 0; q < E; ++q) {
          const bool isB = (win >> q) & 1u;
          const bool dr = !isB && (cw2 & 1u);
          cw2 = isB ? cw2 : (cw2 >> 1);
          st_shared_u32(isB ? pB : pA, dr ? LSM_ORD_DROPPED : o);
          st_shared_u32(dr ? dummy : pR, isB ? vB : vA);
          pB += isB ? 4u : 0u;
          vB += isB ? 1u : 0u;
          pA += isB ? 0u : 4u;
          vA += isB ? 0u : 1u;
          pR += dr ? 0u : 4u;
          o += dr ? 0u : 1u;
        }
      } else if (!bad) {
#pragma unroll
        for (int q = 0; q < E; ++q) {
          const bool valid = q < nvalid;
          const bool isB = (win >> q) & 1u;
          const bool isA = valid && !isB;
          const bool dropped = isA && (cwin & 1u);
          cwin >>= isA ? 1 : 0;
          const uint32_t ref = isB ? (LSM_REF_FROM_B | (jb0 + static_cast<uint32_t>(b_rel)))
                                   : (ia0 + static_cast<uint32_t>(a_rel));
          const int oi = isB ? offB + static_cast<int>(gb0 & 3) + b_rel
                             : static_cast<int>(ga0 & 3) + a_rel;
          if (valid) wOrd[oi] = dropped ? LSM_ORD_DROPPED : wout0 + static_cast<uint32_t>(out_rel);
          if (valid && !dropped) sR[out_rel] = ref;
          out_rel += (valid && !dropped) ? 1 : 0;
          b_rel += isB ? 1 : 0;
          a_rel += isA ? 1 : 0;
        }
      }
      release_stage(empty);  // the stage is not read again
      fence_proxy_async_smem();
      __syncwarp();
      if (!bad) {
        // 4. three runs, each an aligned bulk body and at most three words
        //    at either end
        warp_store_run(p.refs, gr0, kept_w, wRefs);
        warp_store_run(p.ord_A, ga0, nA_w, wOrd);
        warp_store_run(p.ord_B, gb0, nB_w, wOrd + offB);
        if (lane == 0) bulk_commit();
      }
    } else {
      release_stage(empty);
    }
    if (lane == 0) {
      if (!ok) report(status, LSM_ERR_TIMEOUT);
      else if (bad) report(status, LSM_ERR_ARG);
    }
    return ok;
  }
};

// The merge bitmap from a lower-bound array (for a compaction called on its
// own): bit j + lb_B[j] for every B record, after a check that lb_B is a
// nondecreasing array of values <= m (else LSM_ERR_ARG and the record is
// skipped). The bitmap is cleared before.
__global__ void __launch_bounds__(256) merge_bitmap_kernel(const uint32_t *__restrict__ lb_B,
                                                           int64_t m, int64_t n,
                                                           uint32_t *__restrict__ MB,
                                                           int32_t *status) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t j0 = static_cast<int64_t>(blockIdx.x) * blockDim.x; j0 < n; j0 += stride) {
    const int64_t j = j0 + threadIdx.x;
    const bool in = j < n;
    const uint32_t lb = in ? __ldg(lb_B + j) : 0u;
    const uint32_t prev = in && j > 0 ? __ldg(lb_B + j - 1) : 0u;
    const bool act = in && lb <= static_cast<uint64_t>(m) && prev <= lb;
    if (in && !act) report(status, LSM_ERR_ARG);
    const uint64_t pos = static_cast<uint64_t>(j) + lb;
    const uint32_t word = act ? static_cast<uint32_t>(pos >> 5) : 0xFFFFFFFFu;
    const uint32_t peers = __match_any_sync(0xffffffffu, word);
    const uint32_t bits = __reduce_or_sync(peers, act ? 1u << (pos & 31) : 0u);
    if (act && lane == __ffs(peers) - 1) atomicOr(MB + word, bits);
  }
}

// ---- the compaction's co-ranks from lb_B (when the mark's are not at hand) -----------
// With B first on ties B_j sits at merged position p_j = j + lb_B[j] (strictly
// increasing), so the co-rank of diagonal k is k - #{j : p_j < k}: one thread
// per diagonal, a bisection over the positions. Results are clamped to the
// diagonal's valid range.
__global__ void __launch_bounds__(256) position_partition_kernel(const uint32_t *__restrict__ lb_B,
                                                                 int64_t m, int64_t n, int64_t D,
                                                                 int64_t G, int64_t *__restrict__ out_i) {
  pdl_begin();
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g > G) return;
  const int64_t total = m + n;
  const int64_t k = g * D < total ? g * D : total;
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (mid + static_cast<int64_t>(__ldg(lb_B + mid)) < k) lo = mid + 1;
    else hi = mid;
  }
  int64_t i = k - lo;
  const int64_t ilo = k > n ? k - n : 0, ihi = k < m ? k : m;
  out_i[g] = i < ilo ? ilo : (i > ihi ? ihi : i);
}

__global__ void set_count_kernel2(int64_t *d_count, int64_t v) {
  pdl_begin();
  *d_count = v;
}

struct Rank512At {
  const uint32_t *dir;
  __device__ __forceinline__ uint64_t at(const uint32_t *__restrict__ C, int64_t p) const {
    return rank512_at(C, dir, p);
  }
};
struct Rank2048At {
  const uint64_t *dir, *epochs;
  __device__ __forceinline__ uint64_t at(const uint32_t *__restrict__ C, int64_t p) const {
    return rank2048_at(C, dir, epochs, p);
  }
};

// Lanes per diagonal of the co-rank partition. Measured on the 12M + 4M
// step: 8 lanes 98.5 us, 16 lanes 100.5 us, 32 lanes 102.5 us (more lanes cut
// dependent rounds but multiply the scattered loads of each round).
#ifndef LSM_REPL_PART_LANES
#define LSM_REPL_PART_LANES 8
#endif
constexpr int kPartLanes = LSM_REPL_PART_LANES;
// Tile shapes, measured on the 12M + 4M step (CUDA events, L2 flushed by a
// write before each step): D = 3840 diagonals, the mark with 8 consumer warps
// (15 merge positions per thread) and two stages, the compaction with 4 warps
// of 30 positions per lane and four stages: 89.7 us, against 96.9 us for D =
// 2816 (8 x 11 / 4 x 22), 90.8 us for D = 5632 and 95.9 us for D = 7680;
// longer lane walks amortize each warp's popcounts and scans (4 x 30: 89.7
// us, 8 x 15: 98.0 us).
constexpr int kTileT = 256, kTileE = 15, kMarkS = 2, kMarkHG = 8;
constexpr int kCompactT = 128, kCompactE = 30, kCompactS = 4;
using MarkDefault = MarkTile<kTileT, kTileE, kMarkS, kMarkHG>;
using CompactDefault = CompactTile<kCompactT, kCompactE, kCompactS, Rank512At>;
using Compact2048 = CompactTile<kCompactT, kCompactE, kCompactS, Rank2048At>;
// The string keys' compaction: tiles of 4 x 896 positions, on every fourth
// tile boundary of the string mark (which writes those co-ranks and the
// merge bitmap)
constexpr int kStrCompactE = 28;
using CompactStr = CompactTile<kCompactT, kStrCompactE, kCompactS, Rank512At>;
static_assert(CompactStr::D % (kMarkStrThreads * kMarkStrItems) == 0,
              "string compaction tiles are whole string mark tiles");

// ---- the whole path in one persistent kernel ------------------------------------
// The mark and the compaction of each tile in one CTA, by warp roles: the
// loader warp stages tile g's keys as the mark pipeline does; eight mark
// warps find the tile's lower bounds and put its merge-bitmap words and its
// collision bits (indexed by staged A position) into a ring slot in shared
// memory, as well as the bits of C, and the last of them publishes the
// tile's collision count; the lookback warp adds the counts published since
// this CTA's previous tile to R there, which gives R at the tile's first A
// record ("Everett: collision bitmap and rank experiment", "Corrected
// record ordinals": R(i) counts the collisions before i); four compaction
// warps then place the tile's refs and ordinals
// from the ring slot as the compaction pipeline does. With two ring slots
// the mark warps run a tile ahead of the compaction warps, so that the
// lookback's wait is off their path. The grid is sized so that every CTA is
// resident, so every tile a lookback waits for is being worked on; every
// wait is bounded in time.
#ifndef FUSED_MARK_T
#define FUSED_MARK_T 256
#define FUSED_MARK_E 15
#endif
struct FusedMC {
  static constexpr int TM = FUSED_MARK_T, EM = FUSED_MARK_E, D = TM * EM, HG = 8, NWM = TM / 32;
  static constexpr int TC = 128, EC = 30, NWC = TC / 32, WC = 32 * EC;
#ifndef FUSED_RING
#define FUSED_RING 6
#endif
  static constexpr int S = 2, NB = FUSED_RING;
  static constexpr int kLookWarp = (TM + TC) / 32, kLoadWarp = kLookWarp + 1;
  static constexpr int kThreads = TM + TC + 64;
  // states per lane in one round of the lookback's loads: 32 x 10 covers
  // the P - 1 tiles between a CTA's consecutive tiles at two CTAs per SM
  static constexpr int kLookK = 10;
  static constexpr int NMB = D / 32 + 4;             // a tile's merge-bitmap words, window slack
  static constexpr int NCT = (D + 2 + 31) / 32 + 4;  // collision words by staged A position
  static constexpr int kRing = NMB + NCT;
  static constexpr int kRefsWords = (WC + 8 + 3) & ~3;
  static constexpr int kOrdWords = (WC + 12 + 3) & ~3;
  static constexpr int kWarpWords = kRefsWords + kOrdWords;
  static_assert(TC * EC == D, "the compaction covers the mark's tile");
  static_assert(EC < 32, "a lane's positions fit one 32-bit window");
  using Mark = MarkTile<TM, EM, S, HG>;
  using MDesc = Mark::Desc;
  struct TDesc {  // the compaction's view of a tile, written by the mark and the lookback
    int64_t i0, j0, r0;
    int32_t na, nb, wbit0, cnt, te, pad;
    uint32_t hits, warps_done;  // the tile's collisions, mark warps finished (shared atomics)
  };
  static constexpr int64_t kHeadsBytes = align_up(int64_t(Mark::kMaxHeads) * 4, 16);
  static constexpr int64_t kBars = 0;  // full[S], empty[S], markdone[NB], rdone[NB], cdone[NB]
  static constexpr int64_t kMDesc = align_up(8 * (2 * S + 3 * NB), 64);
  static constexpr int64_t kTDesc = kMDesc + 64 * S;
  static constexpr int64_t kStage0 = align_up(kTDesc + 64 * NB, 128);
  static constexpr int64_t kStageStride = align_up(Mark::kStageBytes, 128);
  static constexpr int64_t kHeads = kStage0 + S * kStageStride;
  static constexpr int64_t kRingOff = kHeads + 2 * kHeadsBytes;
  static constexpr int64_t kCBuf = align_up(kRingOff + int64_t(NB) * kRing * 4, 128);
  static constexpr int64_t kBytes = kCBuf + int64_t(NWC) * kWarpWords * 4;
  static_assert(kBytes <= 113 * 1024, "two CTAs per SM");
  static_assert(sizeof(TDesc) <= 64 && sizeof(MDesc) <= 64, "descriptor slots");
  struct Params {
    typename Mark::Params mp;  // keys, sizes, co-ranks, C, lb_B (MB and part_c unused)
    uint32_t *refs, *ord_A, *ord_B;
    int64_t *d_count;
    uint64_t *state;  // G lookback words
  };
};

__global__ void __launch_bounds__(FusedMC::kThreads, 2) fused_mc_kernel(FusedMC::Params p,
                                                                      int64_t G,
                                                                      int32_t *status) {
  pdl_begin();
  using F = FusedMC;
  constexpr int S = F::S, NB = F::NB, TM = F::TM, HG = F::HG, D = F::D;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + F::kBars);
  uint64_t *empty = full + S;
  uint64_t *markdone = empty + S;
  uint64_t *rdone = markdone + NB;
  uint64_t *cdone = rdone + NB;
  F::MDesc *mdesc = reinterpret_cast<F::MDesc *>(smem + F::kMDesc);
  F::TDesc *tdesc = reinterpret_cast<F::TDesc *>(smem + F::kTDesc);
  uint32_t *ring = reinterpret_cast<uint32_t *>(smem + F::kRingOff);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t P = gridDim.x;
  const int64_t R = (G - blockIdx.x + P - 1) / P;  // tiles of this CTA (grid <= G)
  const int64_t total = p.mp.m + p.mp.n;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], F::NWM);
    }
    for (int q = 0; q < NB; ++q) {
      mbar_init(&markdone[q], F::NWM);
      mbar_init(&rdone[q], 1);
      mbar_init(&cdone[q], F::NWC);
    }
  }
  __syncthreads();

  if (warp == F::kLoadWarp) {
    // the loader: co-ranks of 32 tiles at a time, then each tile's keys
    int64_t v[4] = {0, 0, 0, 0};
    for (int64_t r = 0; r < R; ++r) {
      if ((r & 31) == 0) {
        const int64_t gl = blockIdx.x + (r + lane) * P;
        v[0] = v[1] = v[2] = v[3] = 0;
        if (gl < G) F::Mark::fetch(p.mp, gl, v);
      }
      int64_t w[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) w[t] = __shfl_sync(0xffffffffu, v[t], static_cast<int>(r & 31));
      int failed = 0;
      if (lane == 0) {
        const int s = static_cast<int>(r % S);
        if (r >= S && !mbar_wait_sleep(&empty[s], static_cast<uint32_t>(((r / S) + 1) & 1),
                                       kWaitLimitNs)) {
          report(status, LSM_ERR_TIMEOUT);
          failed = 1;
        } else {
          F::Mark::produce(p.mp, blockIdx.x + r * P, w,
                           smem + F::kStage0 + s * F::kStageStride, mdesc[s], &full[s]);
        }
      }
      if (__shfl_sync(0xffffffffu, failed, 0)) return;
    }
    return;
  }

  if (warp < F::NWM) {
    // the mark warps
    for (int64_t r = 0; r < R; ++r) {
      const int s = static_cast<int>(r % S), q = static_cast<int>(r % NB);
      const int64_t g = blockIdx.x + r * P;
      bool ok = mbar_wait_sleep(&full[s], static_cast<uint32_t>((r / S) & 1), kWaitLimitNs);
      // the ring slot's previous tile has left the compaction warps
      if (ok && r >= NB)
        ok = mbar_wait_sleep(&cdone[q], static_cast<uint32_t>(((r / NB) - 1) & 1), kWaitLimitNs);
      const F::MDesc d = mdesc[s];
      const uint8_t *stage = smem + F::kStage0 + s * F::kStageStride;
      const uint64_t *sA = reinterpret_cast<const uint64_t *>(stage) + d.offA;
      const uint64_t *sAx = sA - d.hp;
      const uint64_t *sB = reinterpret_cast<const uint64_t *>(stage) + d.offB;
      const int nb = d.nb, lenx = d.na + d.hp;
      int *heads = reinterpret_cast<int *>(smem + F::kHeads + (r & 1) * F::kHeadsBytes);
      const int nh = (nb + HG - 1) / HG;
      uint32_t *mbt = ring + q * F::kRing;
      uint32_t *ct = mbt + F::NMB;
      const int64_t k0 = g * D;
      const int cnt = d.na + d.nb;
      if (ok) {
        for (int x = tid; x < F::kRing; x += TM) mbt[x] = 0u;
        if (tid == 0) {
          tdesc[q].hits = 0u;
          tdesc[q].warps_done = 0u;
        }
        for (int h = tid; h < nh; h += TM) heads[h] = count_below(sAx, 0, lenx, sB[h * HG], lenx);
        if (tid == TM - 1) {
          heads[nh] = lenx;
          // the equal pair A[i0-1] = B[j0] at the tile's start (B first on
          // ties: A[i0-1] is this tile's first A record) and A[i1-1] = B[j1]
          // at its end (A[i1-1] belongs to the next tile)
          const bool ts = d.hp && nb + d.hn > 0 && sA[-1] == sB[0];
          const bool te = d.hn && lenx > 0 && sAx[lenx - 1] == sB[nb];
          F::TDesc &t = tdesc[q];
          t.i0 = d.i0 - (ts ? 1 : 0);
          t.j0 = k0 - t.i0;
          t.na = d.na + (ts ? 1 : 0) - (te ? 1 : 0);
          t.nb = cnt - t.na;
          t.wbit0 = d.hp - (ts ? 1 : 0);
          t.cnt = cnt;
          t.te = te ? 1 : 0;
        }
      }
      if (named_sync_or(1, TM, !ok)) {
        if (tid == 0) report(status, LSM_ERR_TIMEOUT);
        break;
      }
      // B[j1] sits at the tile's last position when it equals A[i1-1]
      if (tid == TM - 1 && tdesc[q].te) atomicOr(mbt + ((cnt - 1) >> 5), 1u << ((cnt - 1) & 31));
      const uint32_t base = static_cast<uint32_t>(d.i0 - d.hp);
      uint32_t *lbo = p.mp.lb_B ? p.mp.lb_B + d.j0 : nullptr;
      uint32_t hits = 0;  // this warp's collisions (warp-uniform)
      for (int b0 = warp * 64; b0 < nb; b0 += F::NWM * 64) {
        const int bi0 = b0 + lane, bi1 = bi0 + 32;
        const bool act0 = bi0 < nb, act1 = bi1 < nb;
        const uint64_t key0 = sB[act0 ? bi0 : nb - 1], key1 = sB[act1 ? bi1 : nb - 1];
        const int h0 = bi0 / HG, h1 = bi1 / HG;
        int x0 = act0 ? heads[h0] : 0, x1 = act1 ? heads[h1] : 0;
        const int hi0 = act0 ? heads[h0 + 1] : 0, hi1 = act1 ? heads[h1 + 1] : 0;
        const int sp = (hi0 - x0) > (hi1 - x1) ? (hi0 - x0) : (hi1 - x1);
        const int span =
            static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(sp)));
        count_below2(sAx, x0, hi0, key0, x1, hi1, key1, span);
        const bool hit0 = act0 && x0 < lenx && sAx[x0] == key0;
        const bool hit1 = act1 && x1 < lenx && sAx[x1] == key1;
        hits += __popc(__ballot_sync(0xffffffffu, hit0)) + __popc(__ballot_sync(0xffffffffu, hit1));
        if (lbo) {
          if (act0) lbo[bi0] = base + static_cast<uint32_t>(x0);
          if (act1) lbo[bi1] = base + static_cast<uint32_t>(x1);
        }
        if (hit0) {
          const uint32_t ia = base + static_cast<uint32_t>(x0);
          atomicOr(p.mp.C + (ia >> 5), 1u << (ia & 31));
          atomicOr(ct + (x0 >> 5), 1u << (x0 & 31));
        }
        if (hit1) {
          const uint32_t ia = base + static_cast<uint32_t>(x1);
          atomicOr(p.mp.C + (ia >> 5), 1u << (ia & 31));
          atomicOr(ct + (x1 >> 5), 1u << (x1 & 31));
        }
        // B key bi sits at tile position bi + x - hp of the merge with B
        // first on ties (B[j0] falls before the tile when it equals A[i0-1])
        const int rp0 = bi0 + x0 - d.hp, rp1 = bi1 + x1 - d.hp;
        if (act0 && rp0 >= 0) atomicOr(mbt + (rp0 >> 5), 1u << (rp0 & 31));
        if (act1 && rp1 >= 0) atomicOr(mbt + (rp1 >> 5), 1u << (rp1 & 31));
      }
      release_stage(&empty[s]);  // also orders the warp's shared writes before its arrival
      if (lane == 0) {
        // the tile's collision count goes to the lookback as soon as the last
        // mark warp is done, so that no tile waits for another CTA's lookback
        // warp to publish it
        atomicAdd(&tdesc[q].hits, hits);
        __threadfence_block();
        if (atomicAdd(&tdesc[q].warps_done, 1u) == F::NWM - 1) {
          __threadfence_block();
          const uint32_t agg = atomicAdd(&tdesc[q].hits, 0u);
          st_relaxed_u64(p.state + g, kPublished | agg);
        }
        mbar_arrive(&markdone[q]);
      }
    }
    return;
  }

  if (warp == F::kLookWarp) {
    // the lookback warp: R at each tile's first A record. This CTA's
    // previous tile is g - P, so R(g) = R(g - P) plus the collision counts
    // of tiles g - P .. g - 1, which their mark warps publish as soon as they
    // are done: no tile waits for another tile's prefix.
    uint32_t rprev = 0;  // R at this CTA's previous tile
    for (int64_t r = 0; r < R; ++r) {
      const int q = static_cast<int>(r % NB);
      const int64_t g = blockIdx.x + r * P;
      // R(g) needs only earlier tiles' counts: it is summed while this
      // tile's own mark is still running
      const uint32_t prefix = (r == 0 ? 0u : rprev) +
                              window_sum<F::kLookK>(p.state, r == 0 ? 0 : g - P, g, status);
      rprev = prefix;
      // the ring slot holds this tile once its mark is done
      if (!mbar_wait_sleep(&markdone[q], static_cast<uint32_t>((r / NB) & 1), kWaitLimitNs)) {
        if (lane == 0) report(status, LSM_ERR_TIMEOUT);
        break;
      }
      if (lane == 0) {
        tdesc[q].r0 = prefix;
        if (g == G - 1 && p.d_count)
          *p.d_count = total - static_cast<int64_t>(prefix + tdesc[q].hits);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rdone[q]);
    }
    return;
  }

  // the compaction warps
  const int cwarp = warp - F::NWM;
  uint32_t *wRefs = reinterpret_cast<uint32_t *>(smem + F::kCBuf) + cwarp * F::kWarpWords;
  uint32_t *wOrd = wRefs + F::kRefsWords;
  constexpr int E = F::EC, W = F::WC;
  for (int64_t r = 0; r < R; ++r) {
    const int q = static_cast<int>(r % NB);
    const int64_t g = blockIdx.x + r * P;
    if (!mbar_wait_sleep(&rdone[q], static_cast<uint32_t>((r / NB) & 1), kWaitLimitNs)) {
      if (lane == 0) report(status, LSM_ERR_TIMEOUT);
      break;
    }
    const F::TDesc td = tdesc[q];
    const uint32_t *mb = ring + q * F::kRing;
    const uint32_t *cw = mb + F::NMB;
    const int na = td.na, nb = td.nb, cnt = td.cnt;
    const int s0 = cwarp * W;
    bool bad = false;
    if (s0 < cnt) {
      const uint32_t i0u = static_cast<uint32_t>(td.i0), j0u = static_cast<uint32_t>(td.j0);
      const int wbit0 = td.wbit0;
      const int s1 = cnt - s0 < W ? cnt : s0 + W;
      // B records before the warp's first position, dropped A records before
      // its first A record
      int pb = 0;
      for (int x = lane; x < (s0 >> 5); x += 32) pb += __popc(mb[x]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) pb += __shfl_xor_sync(0xffffffffu, pb, o);
      const int bw0 = pb;
      int a_first = s0 - bw0;
      // R(i0) <= i0 whatever the lookback returned, so that no run starts
      // before the output
      bad = a_first < 0 || a_first > na || td.r0 < 0 || td.r0 > td.i0;
      if (bad) a_first = 0;
      const int yend = wbit0 + a_first;
      int pcnt = 0;
      for (int x = lane; x < (yend >> 5); x += 32) pcnt += __popc(cw[x]);
      if (lane == 0) {
        if (yend & 31) pcnt += __popc(cw[yend >> 5] & ((1u << (yend & 31)) - 1u));
        pcnt -= __popc(cw[0] & ((1u << wbit0) - 1u));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) pcnt += __shfl_xor_sync(0xffffffffu, pcnt, o);
      const int drop0 = pcnt;
      const int y = lane * E;
      const int nvalid = (s1 - s0) - y < 0 ? 0 : ((s1 - s0) - y < E ? (s1 - s0) - y : E);
      const int sp = s0 + y;
      const uint32_t w_lo = mb[sp >> 5];
      const uint32_t w_hi = mb[(sp >> 5) + 1];
      uint32_t win = static_cast<uint32_t>(((static_cast<uint64_t>(w_hi) << 32) | w_lo) >> (sp & 31));
      win &= (1u << nvalid) - 1u;
      const int numB = __popc(win);
      const int numA = nvalid - numB;
      const int incB = warp_inclusive_sum(numB);
      const int nB_w = __shfl_sync(0xffffffffu, incB, 31);
      const int nA_w = (s1 - s0) - nB_w;
      bad = bad || a_first + nA_w > na || bw0 + nB_w > nb;
      int a_rel = y - (incB - numB);
      int b_rel = incB - numB;
      const int xa = wbit0 + a_first + a_rel;
      uint32_t cwin = static_cast<uint32_t>(
          ((static_cast<uint64_t>(cw[(xa >> 5) + 1]) << 32) | cw[xa >> 5]) >> (xa & 31));
      cwin &= numA ? (0xFFFFFFFFu >> (32 - numA)) : 0u;
      const int drops = __popc(cwin);
      const int incD = warp_inclusive_sum(drops);
      const int kept_w = (s1 - s0) - __shfl_sync(0xffffffffu, incD, 31);
      int out_rel = y - (incD - drops);
      const int64_t gr0 = g * D - td.r0 + s0 - drop0;  // refs run
      const int64_t ga0 = td.i0 + a_first;             // ord_A run
      const int64_t gb0 = td.j0 + bw0;                 // ord_B run
      const int offB = (nA_w + 7) & ~3;
      uint32_t *sR = wRefs + (gr0 & 3);
      uint32_t *sOA = wOrd + (ga0 & 3);
      uint32_t *sOB = wOrd + offB + (gb0 & 3);
      const uint32_t wout0 = static_cast<uint32_t>(gr0);
      const uint32_t ia0 = i0u + static_cast<uint32_t>(a_first);
      const uint32_t jb0 = j0u + static_cast<uint32_t>(bw0);
      if (lane == 0) bulk_wait_read_all();  // the previous tile's stores from these buffers
      __syncwarp();
      if (!bad && __all_sync(0xffffffffu, nvalid == E)) {
        uint32_t pA = smem_u32(sOA + a_rel), pB = smem_u32(sOB + b_rel);
        uint32_t pR = smem_u32(sR + out_rel);
        const uint32_t dummy = smem_u32(wRefs + F::kRefsWords - 1);
        uint32_t vA = ia0 + static_cast<uint32_t>(a_rel);
        uint32_t vB = LSM_REF_FROM_B | (jb0 + static_cast<uint32_t>(b_rel));
        uint32_t o = wout0 + static_cast<uint32_t>(out_rel);
        uint32_t cw2 = cwin;
#pragma unroll
        for (int qq = 0; qq < E; ++qq) {
          const bool isB = (win >> qq) & 1u;
          const bool dr = !isB && (cw2 & 1u);
          cw2 = isB ? cw2 : (cw2 >> 1);
          st_shared_u32(isB ? pB : pA, dr ? LSM_ORD_DROPPED : o);
          st_shared_u32(dr ? dummy : pR, isB ? vB : vA);
          pB += isB ? 4u : 0u;
          vB += isB ? 1u : 0u;
          pA += isB ? 0u : 4u;
          vA += isB ? 0u : 1u;
          pR += dr ? 0u : 4u;
          o += dr ? 0u : 1u;
        }
      } else if (!bad) {
#pragma unroll
        for (int qq = 0; qq < E; ++qq) {
          const bool valid = qq < nvalid;
          const bool isB = (win >> qq) & 1u;
          const bool isA = valid && !isB;
          const bool dropped = isA && (cwin & 1u);
          cwin >>= isA ? 1 : 0;
          const uint32_t ref = isB ? (LSM_REF_FROM_B | (jb0 + static_cast<uint32_t>(b_rel)))
                                   : (ia0 + static_cast<uint32_t>(a_rel));
          const int oi = isB ? offB + static_cast<int>(gb0 & 3) + b_rel
                             : static_cast<int>(ga0 & 3) + a_rel;
          if (valid) wOrd[oi] = dropped ? LSM_ORD_DROPPED : wout0 + static_cast<uint32_t>(out_rel);
          if (valid && !dropped) sR[out_rel] = ref;
          out_rel += (valid && !dropped) ? 1 : 0;
          b_rel += isB ? 1 : 0;
          a_rel += isA ? 1 : 0;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&cdone[q]);  // the ring slot is not read again
      fence_proxy_async_smem();
      __syncwarp();
      if (!bad) {
        warp_store_run(p.refs, gr0, kept_w, wRefs);
        warp_store_run(p.ord_A, ga0, nA_w, wOrd);
        warp_store_run(p.ord_B, gb0, nB_w, wOrd + offB);
        if (lane == 0) bulk_commit();
      }
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&cdone[q]);
    }
    if (lane == 0 && bad) report(status, LSM_ERR_ARG);
  }
  if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
static_assert(MarkDefault::D == CompactDefault::D, "the compaction reuses the mark's diagonals");

}  // namespace

int64_t replacement_tile() { return MarkDefault::D; }

int64_t merge_bitmap_words(int64_t total) { return align_up((total + 31) / 32, 4) + 4; }

cudaError_t launch_mark_tiles(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                              uint32_t *C, uint32_t *lb_B, uint32_t *MB, int64_t *part_m,
                              int64_t *part_c, int32_t *status, cudaStream_t s,
                              uint64_t *clear, int64_t nclear) {
  constexpr int64_t D = MarkDefault::D;
  const int64_t G = (m + n + D - 1) / D;
  const int64_t nwords = (m + 31) / 32;  // the mark writes every word of MB itself
  int64_t threads = (G + 1) * kPartLanes;
  if (threads < nwords / 4) threads = nwords / 4;
  const int64_t blocks = (threads + 255) / 256;
  cudaError_t err = launch_kernel(true, corank_partition_kernel<kPartLanes>,
                                  static_cast<unsigned>(blocks > 0 ? blocks : 1), 256, 0, s,
                                  KeysAFirst{A, B}, m, n, D, G, part_m, C, nwords, clear, nclear,
                                  static_cast<uint64_t *>(nullptr), int64_t(0));
  if (err != cudaSuccess || G == 0) return err;
  typename MarkDefault::Params p{A, B, m, n, G, part_m, C, lb_B, part_c, MB};
  profile_before(s);
  err = launch_warp_pipeline<MarkDefault>(p, G, status, s);
  profile_after(s);
  return err;
}

template <class Spec, class RD>
cudaError_t launch_compact_with(int64_t m, int64_t n, const uint32_t *C, RD rank,
                                const uint32_t *lb_B, uint32_t *MB, const int64_t *part_c,
                                int64_t *part_scratch, uint32_t *refs, uint32_t *ord_A,
                                uint32_t *ord_B, int64_t *d_count, int32_t *status,
                                cudaStream_t s) {
  constexpr int64_t D = Spec::D;
  const int64_t G = (m + n + D - 1) / D;
  if (G == 0) return launch_kernel(false, set_count_kernel2, 1, 1, 0, s, d_count, int64_t(0));
  if (!part_c) {
    // called on its own: the co-ranks and the merge bitmap from lb_B
    cudaError_t err = launch_kernel(true, position_partition_kernel,
                                    static_cast<unsigned>((G + 1 + 255) / 256), 256, 0, s, lb_B, m,
                                    n, D, G, part_scratch);
    if (err == cudaSuccess)
      err = cudaMemsetAsync(MB, 0, static_cast<size_t>(merge_bitmap_words(m + n)) * 4, s);
    if (err == cudaSuccess && n > 0) {
      int64_t blocks = (n + 255) / 256;
      const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
      if (blocks > cap) blocks = cap;
      err = launch_kernel(false, merge_bitmap_kernel, static_cast<unsigned>(blocks), 256, 0, s,
                          lb_B, m, n, MB, status);
    }
    if (err != cudaSuccess) return err;
    part_c = part_scratch;
  }
  typename Spec::Params p{m, n, G, C, rank, MB, part_c, refs, ord_A, ord_B, d_count};
  profile_before(s);
  const cudaError_t err = launch_warp_pipeline<Spec>(p, G, status, s);
  profile_after(s);
  return err;
}

cudaError_t launch_compact_tiles(int64_t m, int64_t n, const uint32_t *C, const uint32_t *dir,
                                 const uint32_t *lb_B, uint32_t *MB, const int64_t *part_c,
                                 int64_t *part_scratch, uint32_t *refs, uint32_t *ord_A,
                                 uint32_t *ord_B, int64_t *d_count, int32_t *status,
                                 cudaStream_t s) {
  return launch_compact_with<CompactDefault>(m, n, C, Rank512At{dir}, lb_B, MB, part_c,
                                             part_scratch, refs, ord_A, ord_B, d_count, status, s);
}

cudaError_t launch_compact_tiles_rank2048(int64_t m, int64_t n, const uint32_t *C,
                                          const uint64_t *dir, const uint64_t *epochs,
                                          const uint32_t *lb_B, uint32_t *MB, int64_t *part_scratch,
                                          uint32_t *refs, uint32_t *ord_A, uint32_t *ord_B,
                                          int64_t *d_count, int32_t *status, cudaStream_t s) {
  return launch_compact_with<Compact2048>(m, n, C, Rank2048At{dir, epochs}, lb_B, MB, nullptr,
                                          part_scratch, refs, ord_A, ord_B, d_count, status, s);
}

int64_t replacement_str_tile() { return CompactStr::D; }

// The whole path for string keys: the string partition and mark (which also
// writes the merge bitmap and the compaction's co-ranks at every fourth tile
// start), the rank512 build, the compaction over positions.
cudaError_t launch_replacement_merge_str(const lsm_bytes &A, int64_t m, const lsm_bytes &B,
                                         int64_t n, uint32_t *C, uint32_t *lb_B,
                                         uint64_t *prefixA, uint64_t *prefixB, uint32_t *dir,
                                         int64_t *d_total, uint32_t *refs, uint32_t *ord_A,
                                         uint32_t *ord_B, int64_t *d_count, int64_t *part_m,
                                         int64_t *part_c, uint32_t *MB, void *rank_ws,
                                         int32_t *status, cudaStream_t s) {
  constexpr int cstep = CompactStr::D / (kMarkStrThreads * kMarkStrItems);
  cudaError_t err = cudaSuccess;
  if (m + n > 0)
    err = launch_collision_mark_str_mb(A, m, B, n, C, lb_B, prefixA, prefixB, part_m, MB, part_c,
                                       cstep, status, s, static_cast<uint64_t *>(rank_ws),
                                       rank_build_ctas(m));
  if (err != cudaSuccess) return err;
  err = launch_rank_build_ws(C, m, dir, d_total, rank_ws, status, s, m + n > 0);
  if (err != cudaSuccess) return err;
  return launch_compact_with<CompactStr>(m, n, C, Rank512At{dir}, nullptr, MB, part_c, nullptr,
                                         refs, ord_A, ord_B, d_count, status, s);
}

// The whole path: partition + mark (which also writes the merge bitmap and
// the compaction's co-ranks), rank512 build, compaction.
int64_t replacement_fused_tile() { return FusedMC::D; }

// The whole path with the mark and the compaction in one kernel: the co-rank
// partition (which clears C), the fused kernel (refs, ordinals, C, the count;
// lb_B when asked for), then the rank512 directory from the finished C.
cudaError_t launch_replacement_merge_one(const uint64_t *A, int64_t m, const uint64_t *B,
                                        int64_t n, uint32_t *C, uint32_t *lb_B, uint32_t *dir,
                                        int64_t *d_total, uint32_t *refs, uint32_t *ord_A,
                                        uint32_t *ord_B, int64_t *d_count, int64_t *part_m,
                                        uint64_t *state, void *rank_ws, int32_t *status,
                                        cudaStream_t s) {
  constexpr int64_t D = FusedMC::D;
  const int64_t G = (m + n + D - 1) / D;
  cudaError_t err = cudaSuccess;
  if (G > 0) {
    const int64_t nwords = (m + 31) / 32;
    int64_t threads = (G + 1) * kPartLanes;
    if (threads < nwords / 4) threads = nwords / 4;
    const int64_t blocks = (threads + 255) / 256;
    // the partition also zeroes both lookback states: the tiles' and the
    // rank512 build's
    err = launch_kernel(true, corank_partition_kernel<kPartLanes>,
                        static_cast<unsigned>(blocks > 0 ? blocks : 1), 256, 0, s, KeysAFirst{A, B},
                        m, n, D, G, part_m, C, nwords, state, G,
                        static_cast<uint64_t *>(rank_ws), rank_build_ctas(m));
    if (err != cudaSuccess) return err;
    static int per_sm = 0;
    if (!per_sm) {
      err = cudaFuncSetAttribute(fused_mc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(FusedMC::kBytes));
      if (err != cudaSuccess) return err;
      err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_mc_kernel,
                                                          FusedMC::kThreads, FusedMC::kBytes);
      if (err != cudaSuccess) return err;
      if (per_sm < 1) return cudaErrorLaunchOutOfResources;
    }
    // every CTA resident at once: a tile's lookback waits only for tiles
    // that are being worked on
    int64_t grid = static_cast<int64_t>(device_sm_count()) * per_sm;
    if (grid > G) grid = G;
    FusedMC::Params p{};
    p.mp = FusedMC::Mark::Params{A, B, m, n, G, part_m, C, lb_B, nullptr, nullptr};
    p.refs = refs;
    p.ord_A = ord_A;
    p.ord_B = ord_B;
    p.d_count = d_count;
    p.state = state;
    profile_before(s);
    err = launch_kernel(true, fused_mc_kernel, static_cast<unsigned>(grid), FusedMC::kThreads,
                        FusedMC::kBytes, s, p, G, status);
    profile_after(s);
    if (err != cudaSuccess) return err;
  }
  err = launch_rank_build_ws(C, m, dir, d_total, rank_ws, status, s, G > 0);
  if (err != cudaSuccess || G > 0) return err;
  return launch_kernel(false, set_count_kernel2, 1, 1, 0, s, d_count, int64_t(0));
}

cudaError_t launch_replacement_merge(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                    uint32_t *C, uint32_t *lb_B, uint32_t *dir, int64_t *d_total,
                                    uint32_t *refs, uint32_t *ord_A, uint32_t *ord_B,
                                    int64_t *d_count, int64_t *part_m, int64_t *part_c,
                                    uint32_t *MB, void *rank_ws, int32_t *status, cudaStream_t s) {
  cudaError_t err = cudaSuccess;
  if (m + n > 0)
    err = launch_mark_tiles(A, m, B, n, C, lb_B, MB, part_m, part_c, status, s,
                            static_cast<uint64_t *>(rank_ws), rank_build_ctas(m));
  if (err != cudaSuccess) return err;
  err = launch_rank_build_ws(C, m, dir, d_total, rank_ws, status, s, m + n > 0);
  if (err != cudaSuccess) return err;
  return launch_compact_tiles(m, n, C, dir, lb_B, MB, part_c, nullptr, refs, ord_A, ord_B, d_count,
                              status, s);
}

}  // namespace lsm
