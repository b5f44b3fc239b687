// merge.cu -- merge path partition and the stable merge of two sorted arrays.
//
// "Day 36: CUDA merge path", section "The merge matrix, and the diagonal
// that cuts it": the first k merge outputs are A[0, i) and B[0, k - i) for
// the co-rank i of k, found by bisection with two tests; ties go to A.
// The production form the page leaves undone ("Note." after the coRank
// listing, and "Go deeper") stages each block's spans in shared memory
// before any thread searches; that is the design here:
//
//   1. partition_keys_kernel: one warp per tile boundary finds the co-rank
//      of k_g = g * D with a 32-way probe per round (six rounds for 2^26).
//   2. merge_tile_kernel: one CTA per tile of D = T * E outputs. Thread 0
//      issues bulk copies of the tile's A and B spans (keys and payloads)
//      into shared memory; each thread then bisects its own diagonal inside
//      shared memory and walks E outputs into an output tile in shared
//      memory; thread 0 writes the finished tile back with bulk stores.
//      Global memory sees each input byte read once and each output byte
//      written once, in 16-byte aligned bulk transfers.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace lsm {

namespace {

// A_i precedes B_j in the stable merge exactly when A_i <= B_j (ties to A).
template <typename K>
struct KeysAFirst {
  const K *A;
  const K *B;
  __device__ __forceinline__ bool too_small(int64_t i, int64_t k) const { return A[i] <= B[k - i - 1]; }
};

template <typename K>
__global__ void __launch_bounds__(256) partition_keys_kernel(const K *__restrict__ A, int64_t m,
                                                             const K *__restrict__ B, int64_t n,
                                                             int64_t D, int64_t G,
                                                             int64_t *__restrict__ out_i,
                                                             int64_t *__restrict__ out_ij) {
  const int64_t g = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (g > G) return;  // whole warps exit together: blockDim is a multiple of 32
  const int64_t total = m + n;
  const int64_t k = g * D < total ? g * D : total;
  KeysAFirst<K> pred{A, B};
  const int64_t i = warp_corank(pred, k, m, n);
  if ((threadIdx.x & 31) == 0) {
    if (out_i) out_i[g] = i;
    if (out_ij) {
      out_ij[2 * g] = i;
      out_ij[2 * g + 1] = k - i;
    }
  }
}

template <typename K, bool PAY, int T, int E>
struct MergeLayout {
  static constexpr int D = T * E;
  static constexpr int SZ = sizeof(K);
  static constexpr int64_t kBar = 0;
  static constexpr int64_t kInKeys = 128;
  static constexpr int64_t kInKeysBytes = align_up(int64_t(D) * SZ + 128, 16);
  static constexpr int64_t kInPay = kInKeys + kInKeysBytes;
  static constexpr int64_t kInPayBytes = PAY ? align_up(int64_t(D) * 4 + 128, 16) : 0;
  static constexpr int64_t kOutKeys = kInPay + kInPayBytes;
  static constexpr int64_t kOutPay = kOutKeys + align_up(int64_t(D) * SZ, 16);
  static constexpr int64_t kBytes = kOutPay + (PAY ? align_up(int64_t(D) * 4, 16) : 0);
};

template <typename K, bool PAY, int T, int E>
__global__ void __launch_bounds__(T) merge_tile_kernel(
    const K *__restrict__ A, const uint32_t *__restrict__ Apay, int64_t m, const K *__restrict__ B,
    const uint32_t *__restrict__ Bpay, int64_t n, const int64_t *__restrict__ part_i,
    K *__restrict__ out, uint32_t *__restrict__ out_pay, int32_t *status) {
  using L = MergeLayout<K, PAY, T, E>;
  constexpr int D = L::D;
  constexpr int SZ = L::SZ;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::kBar);
  const int tid = threadIdx.x;

  const int64_t g = blockIdx.x;
  const int64_t total = m + n;
  const int64_t k0 = g * D;
  const int64_t k1 = k0 + D < total ? k0 + D : total;
  const int64_t i0 = part_i[g], i1 = part_i[g + 1];
  const int64_t j0 = k0 - i0, j1 = k1 - i1;
  const int na = static_cast<int>(i1 - i0), nb = static_cast<int>(j1 - j0);

  // shared-memory placement of the four spans (A keys, B keys, payloads)
  const StagePlan pa = stage_plan<SZ>(i0, na), pb = stage_plan<SZ>(j0, nb);
  K *bufA = reinterpret_cast<K *>(smem + L::kInKeys);
  K *bufB = reinterpret_cast<K *>(smem + L::kInKeys + stage_capacity_bytes<SZ>(pa.span));
  StagePlan qa{}, qb{};
  uint32_t *bufPA = nullptr, *bufPB = nullptr;
  if (PAY) {
    qa = stage_plan<4>(i0, na);
    qb = stage_plan<4>(j0, nb);
    bufPA = reinterpret_cast<uint32_t *>(smem + L::kInPay);
    bufPB = reinterpret_cast<uint32_t *>(smem + L::kInPay + stage_capacity_bytes<4>(qa.span));
  }

  if (tid == 0) mbar_init(bar, 1);
  __syncthreads();
  if (tid == 0) {
    const uint32_t tx = pa.bulk + pb.bulk + (PAY ? qa.bulk + qb.bulk : 0u);
    mbar_arrive_expect_tx(bar, tx);
    stage_issue(bufA, A, pa, bar);
    stage_issue(bufB, B, pb, bar);
    if (PAY) {
      stage_issue(bufPA, Apay, qa, bar);
      stage_issue(bufPB, Bpay, qb, bar);
    }
  }
  stage_tail(bufA, A, pa, i0, na, tid);
  stage_tail(bufB, B, pb, j0, nb, tid);
  if (PAY) {
    stage_tail(bufPA, Apay, qa, i0, na, tid);
    stage_tail(bufPB, Bpay, qb, j0, nb, tid);
  }
  const bool ok = mbar_wait_bounded(bar, 0, kWaitLimitNs);
  if (__syncthreads_or(!ok)) {
    if (tid == 0) report(status, LSM_ERR_TIMEOUT);
    return;
  }

  const K *sA = bufA + pa.lead;
  const K *sB = bufB + pb.lead;
  const uint32_t *sPA = PAY ? bufPA + qa.lead : nullptr;
  const uint32_t *sPB = PAY ? bufPB + qb.lead : nullptr;
  K *oK = reinterpret_cast<K *>(smem + L::kOutKeys);
  uint32_t *oP = reinterpret_cast<uint32_t *>(smem + L::kOutPay);

  // This thread's diagonal inside the tile, bisected in shared memory with
  // the same A-first test as the partition.
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
  for (int s = 0; s < E; ++s) {
    const int pos = d + s;
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
  fence_proxy_async_smem();
  __syncthreads();

  // Write the tile back: bulk stores for the 16-byte multiple prefix, plain
  // stores for the ragged end of the last tile.
  const int key_bulk = (cnt * SZ) & ~15;
  const int pay_bulk = (cnt * 4) & ~15;
  if (tid == 0) {
    if (key_bulk) bulk_s2g(out + k0, oK, key_bulk);
    if (PAY && pay_bulk) bulk_s2g(out_pay + k0, oP, pay_bulk);
    bulk_commit();
  }
  for (int x = key_bulk / SZ + tid; x < cnt; x += T) out[k0 + x] = oK[x];
  if (PAY)
    for (int x = pay_bulk / 4 + tid; x < cnt; x += T) out_pay[k0 + x] = oP[x];
  if (tid == 0) bulk_wait_read_all();
}

int g_items[3] = {0, 15, 15};  // indexed by key type

template <typename K, bool PAY, int E>
cudaError_t launch_merge_tiles(const K *A, const uint32_t *Apay, int64_t m, const K *B,
                               const uint32_t *Bpay, int64_t n, K *out, uint32_t *out_pay,
                               const int64_t *part_i, int32_t *status, cudaStream_t s) {
  using L = MergeLayout<K, PAY, kMergeThreads, E>;
  auto kern = merge_tile_kernel<K, PAY, kMergeThreads, E>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::kBytes));
  if (err != cudaSuccess) return err;
  const int64_t G = (m + n + L::D - 1) / L::D;
  profile_before(s);
  kern<<<static_cast<unsigned>(G), kMergeThreads, L::kBytes, s>>>(A, Apay, m, B, Bpay, n, part_i,
                                                                  out, out_pay, status);
  profile_after(s);
  return cudaGetLastError();
}

template <typename K, bool PAY>
cudaError_t dispatch_merge(int E, const K *A, const uint32_t *Apay, int64_t m, const K *B,
                           const uint32_t *Bpay, int64_t n, K *out, uint32_t *out_pay,
                           const int64_t *part_i, int32_t *status, cudaStream_t s) {
  switch (E) {
    case 7:
      return launch_merge_tiles<K, PAY, 7>(A, Apay, m, B, Bpay, n, out, out_pay, part_i, status, s);
    case 11:
      return launch_merge_tiles<K, PAY, 11>(A, Apay, m, B, Bpay, n, out, out_pay, part_i, status, s);
    case 15:
      return launch_merge_tiles<K, PAY, 15>(A, Apay, m, B, Bpay, n, out, out_pay, part_i, status, s);
    case 23:
      return launch_merge_tiles<K, PAY, 23>(A, Apay, m, B, Bpay, n, out, out_pay, part_i, status, s);
    default:
      return cudaErrorInvalidValue;
  }
}

template <typename K>
cudaError_t launch_partition_typed(const K *A, int64_t m, const K *B, int64_t n, int64_t D,
                                   int64_t *out_i, int64_t *out_ij, cudaStream_t s) {
  const int64_t G = (m + n + D - 1) / D;
  const int64_t threads = (G + 1) * 32;
  const int64_t blocks = (threads + 255) / 256;
  partition_keys_kernel<K><<<static_cast<unsigned>(blocks), 256, 0, s>>>(A, m, B, n, D, G, out_i,
                                                                          out_ij);
  return cudaGetLastError();
}

}  // namespace

int merge_items_per_thread(int key_type) {
  return (key_type == LSM_KEY_I32 || key_type == LSM_KEY_U64) ? g_items[key_type] : 0;
}

int set_merge_items_per_thread(int key_type, int e) {
  if (key_type != LSM_KEY_I32 && key_type != LSM_KEY_U64) return LSM_ERR_DTYPE;
  if (e != 7 && e != 11 && e != 15 && e != 23) return LSM_ERR_ARG;
  g_items[key_type] = e;
  return LSM_OK;
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
  const int E = merge_items_per_thread(key_type);
  const int64_t D = int64_t(kMergeThreads) * E;
  cudaError_t err = launch_partition_keys(key_type, A, m, B, n, D, part_i, nullptr, s);
  if (err != cudaSuccess) return err;
  const bool pay = Apay != nullptr;
  if (key_type == LSM_KEY_I32) {
    auto a = static_cast<const int32_t *>(A);
    auto b = static_cast<const int32_t *>(B);
    auto o = static_cast<int32_t *>(out);
    return pay ? dispatch_merge<int32_t, true>(E, a, Apay, m, b, Bpay, n, o, out_pay, part_i, status, s)
               : dispatch_merge<int32_t, false>(E, a, Apay, m, b, Bpay, n, o, out_pay, part_i, status, s);
  }
  auto a = static_cast<const uint64_t *>(A);
  auto b = static_cast<const uint64_t *>(B);
  auto o = static_cast<uint64_t *>(out);
  return pay ? dispatch_merge<uint64_t, true>(E, a, Apay, m, b, Bpay, n, o, out_pay, part_i, status, s)
             : dispatch_merge<uint64_t, false>(E, a, Apay, m, b, Bpay, n, o, out_pay, part_i, status, s);
}

}  // namespace lsm
