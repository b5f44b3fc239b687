// merge.cu -- merge path partition, the stable merge of two sorted arrays,
// and the bottom-up merge sort built from that merge.
//
// "Day 36: CUDA merge path", section "The merge matrix, and the diagonal
// that cuts it": the first k merge outputs are A[0, i) and B[0, k - i) for
// the co-rank i of k, found by bisection with two tests; ties go to A.
// The production form the page leaves undone ("Note." after the coRank
// listing, and "Go deeper") stages each block's spans in shared memory
// before any thread searches; that is the design here:
//
//   1. partition_keys_kernel: one thread per tile boundary finds the co-rank
//      of k_g = g * D in global memory, first on a sample grid shared by all
//      boundaries (L2-resident), then by bisection inside the bracket.
//   2. merge_tile_kernel: a persistent, warp-specialized kernel that loops
//      over tiles of D = 256 * E outputs. A producer warp keeps the bulk
//      copies of the next tiles' A and B spans (keys and payloads) in flight
//      through S shared-memory stages, each with a full and an empty
//      mbarrier; eight merging warps take a stage, each thread bisects its
//      own diagonal inside shared memory and walks E outputs into one of two
//      output tiles, and thread 0 writes the tile back with a bulk store
//      while the next tile merges. Global memory sees each input byte read
//      once and each output byte written once, in 16-byte aligned bulk
//      transfers.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace lsm {

namespace {

// Sampled co-rank (A_i precedes B_j in the stable merge exactly when
// A_i <= B_j: ties go to A). With tens of thousands of boundaries a plain bisection
// is bound by its scattered reads (two 32-byte sectors per level, ~27 levels
// for 2^27 elements), not by its rounds. Here the search first runs on the
// grid i = t s of A: at a grid point, B[k - i - 1] lies between the B grid
// elements B[u s] and B[(u + 1) s] (u = floor((k - i - 1) / s)), so
// A[i] <= B[u s] proves i too small and A[i] > B[(u + 1) s] proves it is
// not. The proven-too-small grid points form a prefix (found by bisection
// over t), and at most two grid points after it are undecided, so the
// co-rank lies in a bracket of at most 2 s positions; a plain bisection
// finishes inside it. Every search reads the same grid elements, which stay
// in L2, so only the last ~log2(2 s) levels read scattered sectors. Measured
// on 2^26 + 2^26 uint64 keys (47,663 boundaries): plain bisection 44 us;
// with L2 flushed first (as after the previous merge) 37.5 us at s = 512
// and 33.4 us from s = 2048 up.
constexpr int64_t kPartitionSample = 4096;

template <typename K>
__device__ __forceinline__ int64_t sampled_corank(const K *__restrict__ A, const K *__restrict__ B,
                                                  int64_t k, int64_t m, int64_t n) {
  constexpr int64_t s = kPartitionSample;
  const int64_t lo_k = k > n ? k - n : 0, hi_k = k < m ? k : m;
  int64_t lo = lo_k, hi = hi_k;
  const int64_t tmin = (lo_k + s - 1) / s, tmax = hi_k / s;
  if (hi_k > lo_k && tmin <= tmax) {
    int64_t a = tmin, b = tmax + 1;  // proven too small on [tmin, a)
    while (a < b) {
      const int64_t t = (a + b) >> 1;
      const int64_t i = t * s;
      bool small = false;
      if (i < hi_k) small = __ldg(A + i) <= __ldg(B + ((k - i - 1) / s) * s);
      if (small) a = t + 1;
      else b = t;
    }
    const int64_t t1 = a - 1;
    if (t1 >= tmin) lo = t1 * s + 1;
    // the first of the next three grid points proven not too small
    bool big[3];
    int64_t at[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int64_t i = (t1 + 1 + q) * s;
      at[q] = i;
      big[q] = false;
      if (t1 + 1 + q <= tmax) {
        if (i >= hi_k) {
          big[q] = true;
        } else {
          int64_t ub = ((k - i - 1) / s + 1) * s;
          if (ub > n - 1) ub = n - 1;
          big[q] = __ldg(A + i) > __ldg(B + ub);
        }
      }
    }
#pragma unroll
    for (int q = 2; q >= 0; --q)
      if (big[q] && at[q] < hi) hi = at[q];
  }
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (__ldg(A + mid) <= __ldg(B + k - mid - 1)) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

template <typename K>
__global__ void __launch_bounds__(256) partition_keys_kernel(const K *__restrict__ A, int64_t m,
                                                             const K *__restrict__ B, int64_t n,
                                                             int64_t D, int64_t G,
                                                             int64_t *__restrict__ out_i,
                                                             int64_t *__restrict__ out_ij) {
  pdl_begin();
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g > G) return;
  const int64_t total = m + n;
  const int64_t k = g * D < total ? g * D : total;
  const int64_t i = sampled_corank(A, B, k, m, n);
  if (out_i) out_i[g] = i;
  if (out_ij) {
    out_ij[2 * g] = i;
    out_ij[2 * g + 1] = k - i;
  }
}

// Shared-memory layout of one CTA: S input stages (keys region then payload
// region, each large enough for D elements plus the 16-byte alignment slack
// of two spans), NOUT output tiles, and per stage a full barrier, an empty
// barrier and a tile descriptor written by the producer.
template <typename K, bool PAY, int E, int S, int NOUT>
struct MergeLayout {
  static constexpr int D = kMergeThreads * E;
  static constexpr int SZ = sizeof(K);
  static constexpr int64_t kFull = 0;                                  // S x 8
  static constexpr int64_t kEmpty = 8 * S;                             // S x 8
  static constexpr int64_t kMeta = 16 * S;                             // S x 32
  static constexpr int64_t kStage0 = align_up(48 * S, 128);
  static constexpr int64_t kKeysBytes = align_up(int64_t(D) * SZ + 128, 16);
  static constexpr int64_t kPayBytes = PAY ? align_up(int64_t(D) * 4 + 128, 16) : 0;
  static constexpr int64_t kStageBytes = kKeysBytes + kPayBytes;
  static constexpr int64_t kOut0 = kStage0 + S * kStageBytes;
  static constexpr int64_t kOutKeysBytes = align_up(int64_t(D) * SZ, 16);
  static constexpr int64_t kOutBytes = kOutKeysBytes + (PAY ? align_up(int64_t(D) * 4, 16) : 0);
  static constexpr int64_t kBytes = kOut0 + NOUT * kOutBytes;
};

// A tile as the merging warps see it: counts and the element offsets of the
// four spans inside the stage buffer (computed once, by the producer).
struct TileDesc {
  int32_t na, nb;
  int32_t offA, offB;    // in keys, from the stage start
  int32_t offPA, offPB;  // in uint32 words, from the payload region start
  int32_t pad0, pad1;
};
static_assert(sizeof(TileDesc) == 32, "descriptor slot");

// Warp-specialized persistent kernel: warps 0..T/32-1 merge, the last warp
// stages tiles. CTA c handles tiles c, c + P, c + 2P, ... (P = gridDim.x).
// Stage s = r % S holds the r-th tile; full[s] completes when its bulk copies
// land, empty[s] when every merging warp has finished reading it.
//
// SEG selects one pass of the bottom-up merge sort instead of one merge: A
// and B are then the same array of m = n = N elements, made of sorted runs
// of w elements, and tile g (whose D outputs lie inside one pair of runs,
// since D divides 2w) merges its pair's left run (as A) with its right run
// (as B). part_i then holds co-ranks local to each boundary's pair.
template <typename K, bool PAY, int E, int S, int NOUT, bool SEG = false>
__global__ void __launch_bounds__(kMergeThreads + 32) merge_tile_kernel(
    const K *__restrict__ A, const uint32_t *__restrict__ Apay, int64_t m, const K *__restrict__ B,
    const uint32_t *__restrict__ Bpay, int64_t n, const int64_t *__restrict__ part_i, int64_t G,
    K *__restrict__ out, uint32_t *__restrict__ out_pay, int32_t *status, int64_t w) {
  pdl_begin();
  using L = MergeLayout<K, PAY, E, S, NOUT>;
  constexpr int D = L::D;
  constexpr int SZ = L::SZ;
  constexpr int T = kMergeThreads;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kFull);
  uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L::kEmpty);
  TileDesc *desc = reinterpret_cast<TileDesc *>(smem + L::kMeta);
  const int tid = threadIdx.x;
  const int64_t total = SEG ? m : m + n;
  const int64_t P = gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], T / 32);
    }
  }
  __syncthreads();

  if (tid >= T) {
    // ---------------- producer warp ----------------
    // The 32 lanes fetch the partition entries of 32 upcoming tiles at once;
    // lane 0 then stages those tiles one after the other as stages free up.
    const int lane = tid & 31;
    for (int64_t r0 = 0; blockIdx.x + r0 * P < G; r0 += 32) {
      const int64_t gl = blockIdx.x + (r0 + lane) * P;
      int64_t pi0 = 0, pi1 = 0;
      if (gl < G) {
        pi0 = __ldg(part_i + gl);
        pi1 = __ldg(part_i + gl + 1);
      }
      for (int q = 0; q < 32; ++q) {
        const int64_t r = r0 + q;
        const int64_t g = blockIdx.x + r * P;
        if (g >= G) break;
        const int64_t i0 = __shfl_sync(0xffffffffu, pi0, q);
        const int64_t i1 = __shfl_sync(0xffffffffu, pi1, q);
        int failed = 0;
        if (lane == 0) {
          const int s = static_cast<int>(r % S);
          if (r >= S && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>(((r / S) + 1) & 1),
                                           kWaitLimitNs)) {
            report(status, LSM_ERR_TIMEOUT);
            failed = 1;
          } else {
            const int64_t k0 = g * D, k1 = k0 + D < total ? k0 + D : total;
            // the tile's spans [a0, a1) of A and [j0, j1) of B
            int64_t a0 = i0, a1 = i1, j0 = k0 - i0, j1 = k1 - i1;
            if (SEG) {
              const int64_t ps = (k0 / (2 * w)) * (2 * w);  // the pair's first element
              const int64_t la = w < total - ps ? w : total - ps;
              const int64_t lab = 2 * w < total - ps ? 2 * w : total - ps;
              // the pair's last tile ends where the pair ends: all of its left run
              const int64_t e1 = k1 - ps == lab ? la : i1;
              a0 = ps + i0;
              a1 = ps + e1;
              j0 = ps + la + (k0 - ps - i0);
              j1 = ps + la + (k1 - ps - e1);
            }
            const int na = static_cast<int>(a1 - a0), nb = static_cast<int>(j1 - j0);
            uint8_t *stage = smem + L::kStage0 + s * L::kStageBytes;
            const StagePlan pa = stage_plan_overfetch<SZ>(a0, na, m);
            const StagePlan pb = stage_plan_overfetch<SZ>(j0, nb, n);
            K *bufA = reinterpret_cast<K *>(stage);
            const int32_t offB = static_cast<int32_t>(stage_capacity_bytes<SZ>(pa.span) / SZ);
            K *bufB = bufA + offB;
            TileDesc td;
            td.na = na;
            td.nb = nb;
            td.offA = pa.lead;
            td.offB = offB + pb.lead;
            td.offPA = td.offPB = 0;
            // ragged ends (only where a span touches the end of its array) by
            // plain loads, before the arrive so that the barrier covers them
            for (int64_t x = pa.tail_from; x < a1; ++x) bufA[x - pa.first] = A[x];
            for (int64_t x = pb.tail_from; x < j1; ++x) bufB[x - pb.first] = B[x];
            uint32_t tx = pa.bulk + pb.bulk;
            StagePlan qa{}, qb{};
            uint32_t *bufPA = nullptr, *bufPB = nullptr;
            if (PAY) {
              qa = stage_plan_overfetch<4>(a0, na, m);
              qb = stage_plan_overfetch<4>(j0, nb, n);
              bufPA = reinterpret_cast<uint32_t *>(stage + L::kKeysBytes);
              const int32_t offPB = static_cast<int32_t>(stage_capacity_bytes<4>(qa.span) / 4);
              bufPB = bufPA + offPB;
              td.offPA = qa.lead;
              td.offPB = offPB + qb.lead;
              for (int64_t x = qa.tail_from; x < a1; ++x) bufPA[x - qa.first] = Apay[x];
              for (int64_t x = qb.tail_from; x < j1; ++x) bufPB[x - qb.first] = Bpay[x];
              tx += qa.bulk + qb.bulk;
            }
            desc[s] = td;
            mbar_arrive_expect_tx(&full[s], tx);
            stage_issue(bufA, A, pa, &full[s]);
            stage_issue(bufB, B, pb, &full[s]);
            if (PAY) {
              stage_issue(bufPA, Apay, qa, &full[s]);
              stage_issue(bufPB, Bpay, qb, &full[s]);
            }
          }
        }
        if (__shfl_sync(0xffffffffu, failed, 0)) return;
      }
    }
    return;
  }

  // ---------------- merging warps ----------------
  const int lane = tid & 31;
  for (int64_t r = 0;; ++r) {
    const int64_t g = blockIdx.x + r * P;
    if (g >= G) break;
    const int s = static_cast<int>(r % S);
    // The output tile about to be written was last stored NOUT tiles ago;
    // wait until at most NOUT - 1 stores still read shared memory.
    if (tid == 0) {
      if (NOUT == 1) bulk_wait_read_all();
      else bulk_wait_read_allow1();
    }
    const bool ok = mbar_wait_bounded(&full[s], static_cast<uint32_t>((r / S) & 1), kWaitLimitNs);
    if (named_sync_or(1, T, !ok)) {
      if (tid == 0) report(status, LSM_ERR_TIMEOUT);
      break;
    }
    const TileDesc td = desc[s];
    const int na = td.na, nb = td.nb;
    const K *stageK = reinterpret_cast<const K *>(smem + L::kStage0 + s * L::kStageBytes);
    const K *sA = stageK + td.offA;
    const K *sB = stageK + td.offB;
    const uint32_t *stageP =
        reinterpret_cast<const uint32_t *>(smem + L::kStage0 + s * L::kStageBytes + L::kKeysBytes);
    const uint32_t *sPA = stageP + td.offPA;
    const uint32_t *sPB = stageP + td.offPB;
    uint8_t *obuf = smem + L::kOut0 + (NOUT == 1 ? 0 : (r & 1)) * L::kOutBytes;
    K *oK = reinterpret_cast<K *>(obuf);
    uint32_t *oP = reinterpret_cast<uint32_t *>(obuf + L::kOutKeysBytes);

    // This thread's diagonal inside the tile, bisected in shared memory with
    // the same A-first test as the partition, then E merge steps.
    const int cnt = na + nb;
    const int d = tid * E < cnt ? tid * E : cnt;
    int lo = d > nb ? d - nb : 0, hi = d < na ? d : na;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sA[mid] <= sB[d - mid - 1]) lo = mid + 1;
      else hi = mid;
    }
    int ai = lo, bi = d - lo;
    K a = ai < na ? sA[ai] : K(0);
    K b = bi < nb ? sB[bi] : K(0);
#pragma unroll
    for (int q = 0; q < E; ++q) {
      const int pos = d + q;
      if (pos < cnt) {
        const bool takeA = (bi >= nb) || (ai < na && a <= b);
        oK[pos] = takeA ? a : b;
        if (PAY) oP[pos] = takeA ? sPA[ai] : sPB[bi];
        if (takeA) {
          ++ai;
          if (ai < na) a = sA[ai];
        } else {
          ++bi;
          if (bi < nb) b = sB[bi];
        }
      }
    }
    // this warp is done reading the stage: hand it back to the producer
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    fence_proxy_async_smem();
    named_sync(1, T);

    const int64_t k0 = g * D;
    const int key_bulk = (cnt * SZ) & ~15;
    const int pay_bulk = (cnt * 4) & ~15;
    if (tid == 0) {
      if (key_bulk) bulk_s2g(out + k0, oK, key_bulk);
      if (PAY && pay_bulk) bulk_s2g(out_pay + k0, oP, pay_bulk);
      bulk_commit();
    }
    // ragged end of the last tile
    for (int x = key_bulk / SZ + tid; x < cnt; x += T) out[k0 + x] = oK[x];
    if (PAY)
      for (int x = pay_bulk / 4 + tid; x < cnt; x += T) out_pay[k0 + x] = oP[x];
    if (NOUT == 1) named_sync(1, T);  // the ragged-end reads precede the next tile's writes
  }
  if (tid == 0) bulk_wait_read_all();
}

// Tile configurations: items per thread E, input stages S, output tiles NOUT.
struct MergeConfig {
  int E, S, NOUT;
};
constexpr MergeConfig kMergeConfigs[] = {
    {5, 2, 1}, {7, 2, 1}, {11, 2, 1}, {15, 2, 1}, {7, 4, 2}, {11, 3, 2}, {15, 2, 2}, {7, 3, 1},
};
constexpr int kNumMergeConfigs = sizeof(kMergeConfigs) / sizeof(kMergeConfigs[0]);
int g_config[3] = {0, 2, 2};  // indexed by key type; (11, 2, 1)

template <typename K, bool PAY, int E, int S, int NOUT>
cudaError_t launch_merge_tiles(const K *A, const uint32_t *Apay, int64_t m, const K *B,
                               const uint32_t *Bpay, int64_t n, K *out, uint32_t *out_pay,
                               const int64_t *part_i, int32_t *status, cudaStream_t s) {
  using L = MergeLayout<K, PAY, E, S, NOUT>;
  static_assert(L::kBytes <= 225 * 1024, "tile configuration exceeds shared memory");
  auto kern = merge_tile_kernel<K, PAY, E, S, NOUT>;
  constexpr int threads = kMergeThreads + 32;
  static int per_sm = 0;  // resident CTAs per SM for this instantiation
  if (!per_sm) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(L::kBytes));
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, L::kBytes);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
  }
  const int64_t G = (m + n + L::D - 1) / L::D;
  int64_t grid = static_cast<int64_t>(device_sm_count()) * per_sm;
  if (grid < 1) grid = 1;
  if (grid > G) grid = G;
  profile_before(s);
  // launched early (PDL) behind the partition, whose few blocks per SM leave
  // the tile CTAs' room free (measured: step 0.5102 ms against 0.5114 ms)
  const cudaError_t err = launch_kernel(true, kern, static_cast<unsigned>(grid), threads,
                                        L::kBytes, s, A, Apay, m, B, Bpay, n, part_i, G, out,
                                        out_pay, status, int64_t(0));
  profile_after(s);
  return err;
}

template <typename K, bool PAY, int C>
cudaError_t launch_config(const K *A, const uint32_t *Apay, int64_t m, const K *B,
                          const uint32_t *Bpay, int64_t n, K *out, uint32_t *out_pay,
                          const int64_t *part_i, int32_t *status, cudaStream_t s) {
  constexpr MergeConfig c = kMergeConfigs[C];
  return launch_merge_tiles<K, PAY, c.E, c.S, c.NOUT>(A, Apay, m, B, Bpay, n, out, out_pay, part_i,
                                                      status, s);
}

template <typename K, bool PAY>
cudaError_t dispatch_merge(int cfg, const K *A, const uint32_t *Apay, int64_t m, const K *B,
                           const uint32_t *Bpay, int64_t n, K *out, uint32_t *out_pay,
                           const int64_t *part_i, int32_t *status, cudaStream_t s) {
#define LSM_MERGE_CASE(C) \
  case C:                 \
    return launch_config<K, PAY, C>(A, Apay, m, B, Bpay, n, out, out_pay, part_i, status, s);
  switch (cfg) {
    LSM_MERGE_CASE(0)
    LSM_MERGE_CASE(1)
    LSM_MERGE_CASE(2)
    LSM_MERGE_CASE(3)
    LSM_MERGE_CASE(4)
    LSM_MERGE_CASE(5)
    LSM_MERGE_CASE(6)
    LSM_MERGE_CASE(7)
    default:
      return cudaErrorInvalidValue;
  }
#undef LSM_MERGE_CASE
}
static_assert(kNumMergeConfigs == 8, "dispatch_merge lists every configuration");

template <typename K>
cudaError_t launch_partition_typed(const K *A, int64_t m, const K *B, int64_t n, int64_t D,
                                   int64_t *out_i, int64_t *out_ij, cudaStream_t s) {
  const int64_t G = (m + n + D - 1) / D;
  const int64_t blocks = (G + 1 + 255) / 256;
  return launch_kernel(false, partition_keys_kernel<K>, static_cast<unsigned>(blocks), 256, 0, s, A,
                       m, B, n, D, G, out_i, out_ij);
}

// ---- bottom-up merge sort ([CH14] section 14.2) ------------------------------------
// The sort runs the chapter's passes (runs of width w merged in pairs, w
// doubling) with two changes of where the passes run, not of what they
// compute: the passes of widths 1 .. D/2 happen inside one CTA's shared
// memory (block_sort_kernel leaves sorted runs of D elements), and each
// pass from w = D on is one segmented partition plus one launch of the
// persistent tile kernel, whose tiles never straddle a pair because D
// divides 2w.
constexpr int kSortE = 11;  // items per thread of the sort's tiles
constexpr int kSortS = 2;   // input stages of its tile kernel
constexpr int kSortD = kMergeThreads * kSortE;

template <typename K>
__device__ __forceinline__ K sort_key_max();
template <>
__device__ __forceinline__ int32_t sort_key_max<int32_t>() { return 0x7fffffff; }
template <>
__device__ __forceinline__ uint64_t sort_key_max<uint64_t>() { return ~0ull; }

// Sorts each tile of D = 256 E elements stably. Every thread sorts its E
// consecutive elements in registers (odd-even transposition: E rounds of
// compare-exchange that swaps only strictly greater pairs, so it is stable;
// positions past the tile's end hold the largest key and stay behind the
// real elements, equal or not), then the CTA runs the chapter's passes over
// shared memory with widths E, 2E, ..., each thread finding the pair of
// its E outputs from its output position, its co-rank inside that pair by
// bisection (ties to the left run), and merging E outputs.
template <typename K, bool PAY, int E>
__global__ void __launch_bounds__(kMergeThreads) block_sort_kernel(
    const K *__restrict__ in, const uint32_t *__restrict__ in_pay, int64_t N, K *__restrict__ out,
    uint32_t *__restrict__ out_pay) {
  pdl_begin();
  constexpr int T = kMergeThreads, D = T * E;
  extern __shared__ __align__(128) uint8_t smem[];
  // two buffers of D keys, then two of D payloads; buffer b starts at b * D
  K *const sk = reinterpret_cast<K *>(smem);
  uint32_t *const sp = reinterpret_cast<uint32_t *>(smem + 2 * D * sizeof(K));
  const int tid = threadIdx.x;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * D;
  const int cnt = static_cast<int>(N - base < D ? N - base : D);
  // coalesced loads, all E (and E payload) loads of a thread in flight at once
#pragma unroll
  for (int q = 0; q < E; ++q) {
    const int x = tid + q * T;
    if (x < cnt) {
      sk[x] = in[base + x];
      if (PAY) sp[x] = in_pay[base + x];
    }
  }
  __syncthreads();

  const int d = tid * E;
  K k[E];
  uint32_t p[E];
#pragma unroll
  for (int q = 0; q < E; ++q) {
    const bool v = d + q < cnt;
    k[q] = v ? sk[d + q] : sort_key_max<K>();
    p[q] = (PAY && v) ? sp[d + q] : 0u;
  }
#pragma unroll
  for (int r = 0; r < E; ++r) {
#pragma unroll
    for (int i = r & 1; i + 1 < E; i += 2) {
      if (k[i + 1] < k[i]) {
        const K tk = k[i];
        k[i] = k[i + 1];
        k[i + 1] = tk;
        if (PAY) {
          const uint32_t tp = p[i];
          p[i] = p[i + 1];
          p[i + 1] = tp;
        }
      }
    }
  }
  // each thread writes back exactly the positions it read
#pragma unroll
  for (int q = 0; q < E; ++q) {
    if (d + q < cnt) {
      sk[d + q] = k[q];
      if (PAY) sp[d + q] = p[q];
    }
  }
  // A pass whose pairs (2w elements) fit in one warp's 32 E elements reads
  // and writes only that warp's span, so the barrier before it can be the
  // warp's own: warps run the first passes (w = E .. 16 E) independently.
  __syncwarp();

  int src = 0;
  for (int w = E; w < cnt; w *= 2) {
    if (2 * w > 32 * E) __syncthreads();
    if (d < cnt) {
      const int ps = (d / (2 * w)) * (2 * w);
      const int la = w < cnt - ps ? w : cnt - ps;
      const int lb = w < cnt - ps - la ? w : cnt - ps - la;
      const K *a = sk + src * D + ps;
      const K *b = a + la;
      const int kd = d - ps;
      int lo = kd > lb ? kd - lb : 0, hi = kd < la ? kd : la;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= b[kd - mid - 1]) lo = mid + 1;
        else hi = mid;
      }
      // The pair's runs are adjacent: B's element bi sits at a[la + bi]. Each
      // step is branch-free (lanes of a warp take A or B independently): one
      // payload load and one head reload at a computed index, clamped into
      // the pair so that an exhausted run's reload stays in bounds (its value
      // is then never compared).
      int ai = lo, bi = kd - lo;
      const uint32_t *pp = sp + src * D + ps;
      K *ok = sk + (src ^ 1) * D + ps;
      uint32_t *op = sp + (src ^ 1) * D + ps;
      const int end = la + lb;
      K ha = a[ai < end ? ai : end - 1];
      K hb = a[la + bi < end ? la + bi : end - 1];
#pragma unroll
      for (int q = 0; q < E; ++q) {
        const int pos = kd + q;
        if (pos < end) {
          const bool takeA = bi >= lb || (ai < la && ha <= hb);
          const int from = takeA ? ai : la + bi;
          ok[pos] = takeA ? ha : hb;
          if (PAY) op[pos] = pp[from];
          ai += takeA ? 1 : 0;
          bi += takeA ? 0 : 1;
          const int nx = from + 1 < end ? from + 1 : end - 1;
          const K nv = a[nx];
          ha = takeA ? nv : ha;
          hb = takeA ? hb : nv;
        }
      }
    }
    __syncwarp();
    src ^= 1;
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < E; ++q) {
    const int x = tid + q * T;
    if (x < cnt) {
      out[base + x] = sk[src * D + x];
      if (PAY) out_pay[base + x] = sp[src * D + x];
    }
  }
}

// Co-ranks of one sort pass: boundary g sits at k = min(gD, N) inside the
// pair that starts at ps = floor(k / 2w) 2w; its entry is the co-rank of
// k - ps in the merge of the pair's runs [ps, ps + la) and [ps + la, ps + la + lb).
template <typename K>
__global__ void __launch_bounds__(256) partition_sort_kernel(const K *__restrict__ src, int64_t N,
                                                             int64_t w, int64_t D, int64_t G,
                                                             int64_t *__restrict__ out_i) {
  pdl_begin();
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g > G) return;
  const int64_t k = g * D < N ? g * D : N;
  const int64_t ps = (k / (2 * w)) * (2 * w);
  const int64_t la = w < N - ps ? w : N - ps;
  const int64_t lb = w < N - ps - la ? w : N - ps - la;
  out_i[g] = sampled_corank(src + ps, src + ps + la, k - ps, la, lb);
}

template <typename K, bool PAY>
cudaError_t launch_merge_sort_typed(const K *in, const uint32_t *in_pay, int64_t N, K *out,
                                    uint32_t *out_pay, K *tmp, uint32_t *tmp_pay, int64_t *part,
                                    int32_t *status, cudaStream_t s) {
  constexpr int D = kSortD;
  using L = MergeLayout<K, PAY, kSortE, kSortS, 1>;
  static_assert(L::D == D, "the pass tiles and the sorted runs have the same size");
  constexpr size_t kBlockSmem = 2 * size_t(D) * (sizeof(K) + (PAY ? 4 : 0));
  auto bkern = block_sort_kernel<K, PAY, kSortE>;
  auto mkern = merge_tile_kernel<K, PAY, kSortE, kSortS, 1, true>;
  constexpr int mthreads = kMergeThreads + 32;
  static int per_sm = 0;  // resident tile CTAs per SM
  if (!per_sm) {
    cudaError_t err = cudaFuncSetAttribute(bkern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kBlockSmem));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(mkern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(L::kBytes));
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mkern, mthreads, L::kBytes);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
  }
  const int64_t G = (N + D - 1) / D;
  int passes = 0;
  for (int64_t w = D; w < N; w *= 2) ++passes;
  // ping-pong so that the last pass lands in `out`
  K *kb[2] = {out, tmp};
  uint32_t *pb[2] = {out_pay, tmp_pay};
  int cur = passes & 1;
  // the profiling hook brackets the last launch that moves every element:
  // the last pass's tile kernel, or the block sort when it is the only one
  if (passes == 0) profile_before(s);
  cudaError_t err = launch_kernel(false, bkern, static_cast<unsigned>(G), kMergeThreads,
                                  kBlockSmem, s, in, in_pay, N, kb[cur], pb[cur]);
  if (passes == 0) profile_after(s);
  if (err != cudaSuccess) return err;
  int64_t grid = static_cast<int64_t>(device_sm_count()) * per_sm;
  if (grid < 1) grid = 1;
  if (grid > G) grid = G;
  for (int64_t w = D; w < N; w *= 2) {
    err = launch_kernel(false, partition_sort_kernel<K>, static_cast<unsigned>((G + 1 + 255) / 256),
                        256, 0, s, static_cast<const K *>(kb[cur]), N, w, int64_t(D), G, part);
    if (err != cudaSuccess) return err;
    const bool last = 2 * w >= N;
    if (last) profile_before(s);
    err = launch_kernel(true, mkern, static_cast<unsigned>(grid), mthreads, L::kBytes, s,
                        static_cast<const K *>(kb[cur]), static_cast<const uint32_t *>(pb[cur]), N,
                        static_cast<const K *>(kb[cur]), static_cast<const uint32_t *>(pb[cur]), N,
                        static_cast<const int64_t *>(part), G, kb[cur ^ 1], pb[cur ^ 1], status, w);
    if (last) profile_after(s);
    if (err != cudaSuccess) return err;
    cur ^= 1;
  }
  return cudaSuccess;
}

}  // namespace

int64_t merge_sort_tile() { return kSortD; }

cudaError_t launch_merge_sort(int key_type, const void *in, const uint32_t *in_pay, int64_t N,
                              void *out, uint32_t *out_pay, void *tmp, uint32_t *tmp_pay,
                              int64_t *part, int32_t *status, cudaStream_t s) {
  const bool pay = in_pay != nullptr;
  if (key_type == LSM_KEY_I32) {
    auto i = static_cast<const int32_t *>(in);
    auto o = static_cast<int32_t *>(out);
    auto t = static_cast<int32_t *>(tmp);
    return pay ? launch_merge_sort_typed<int32_t, true>(i, in_pay, N, o, out_pay, t, tmp_pay, part, status, s)
               : launch_merge_sort_typed<int32_t, false>(i, in_pay, N, o, out_pay, t, tmp_pay, part, status, s);
  }
  auto i = static_cast<const uint64_t *>(in);
  auto o = static_cast<uint64_t *>(out);
  auto t = static_cast<uint64_t *>(tmp);
  return pay ? launch_merge_sort_typed<uint64_t, true>(i, in_pay, N, o, out_pay, t, tmp_pay, part, status, s)
             : launch_merge_sort_typed<uint64_t, false>(i, in_pay, N, o, out_pay, t, tmp_pay, part, status, s);
}

int device_sm_count() {
  static std::mutex mu;
  static int cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev);
  return cache[dev];
}

int merge_items_per_thread(int key_type) {
  return (key_type == LSM_KEY_I32 || key_type == LSM_KEY_U64) ? kMergeConfigs[g_config[key_type]].E : 0;
}

int set_merge_config(int key_type, int items, int stages, int out_tiles) {
  if (key_type != LSM_KEY_I32 && key_type != LSM_KEY_U64) return LSM_ERR_DTYPE;
  for (int c = 0; c < kNumMergeConfigs; ++c) {
    if (kMergeConfigs[c].E == items && kMergeConfigs[c].S == stages &&
        kMergeConfigs[c].NOUT == out_tiles) {
      g_config[key_type] = c;
      return LSM_OK;
    }
  }
  return LSM_ERR_ARG;
}

cudaError_t launch_partition_keys(int key_type, const void *A, int64_t m, const void *B, int64_t n,
                                  int64_t D, int64_t *out_i, int64_t *out_ij, cudaStream_t s) {
  if (key_type == LSM_KEY_I32)
    return launch_partition_typed(static_cast<const int32_t *>(A), m,
                                  static_cast<const int32_t *>(B), n, D, out_i, out_ij, s);
  return launch_partition_typed(static_cast<const uint64_t *>(A), m,
                                static_cast<const uint64_t *>(B), n, D, out_i, out_ij, s);
}

cudaError_t launch_merge_stable(int key_type, const void *A, const uint32_t *Apay, int64_t m,
                                const void *B, const uint32_t *Bpay, int64_t n, void *out,
                                uint32_t *out_pay, int64_t *part_i, int32_t *status,
                                cudaStream_t s) {
  const int cfg = g_config[key_type];
  const int64_t D = int64_t(kMergeThreads) * kMergeConfigs[cfg].E;
  cudaError_t err = launch_partition_keys(key_type, A, m, B, n, D, part_i, nullptr, s);
  if (err != cudaSuccess) return err;
  const bool pay = Apay != nullptr;
  if (key_type == LSM_KEY_I32) {
    auto a = static_cast<const int32_t *>(A);
    auto b = static_cast<const int32_t *>(B);
    auto o = static_cast<int32_t *>(out);
    return pay ? dispatch_merge<int32_t, true>(cfg, a, Apay, m, b, Bpay, n, o, out_pay, part_i, status, s)
               : dispatch_merge<int32_t, false>(cfg, a, Apay, m, b, Bpay, n, o, out_pay, part_i, status, s);
  }
  auto a = static_cast<const uint64_t *>(A);
  auto b = static_cast<const uint64_t *>(B);
  auto o = static_cast<uint64_t *>(out);
  return pay ? dispatch_merge<uint64_t, true>(cfg, a, Apay, m, b, Bpay, n, o, out_pay, part_i, status, s)
             : dispatch_merge<uint64_t, false>(cfg, a, Apay, m, b, Bpay, n, o, out_pay, part_i, status, s);
}

}  // namespace lsm
