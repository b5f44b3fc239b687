// strings.cu -- collision bitmap and lower bounds for byte-string keys.
//
// The same merge-path tiling as the uint64 collision mark ("Everett:
// collision bitmap and rank experiment", "Corrected record ordinals"),
// with keys compared in place in their arenas (strings.cuh). A partition
// warp finds the co-rank of each tile boundary (A first on ties); each
// thread bisects its own diagonal inside the tile and walks E merge steps,
// keeping one comparison per step. For each B element it records the lower
// bound (A elements before it, minus one when the element just before it
// is an equal A key); for each A element it sets C_i when the B key at the
// head equals it. Bits are gathered per tile in shared memory; words inside
// the tile's A range take plain stores, boundary words atomicOr into the
// bitmap the partition launch cleared.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "strings.cuh"

namespace lsm {

namespace {

struct StrAFirst {
  lsm_bytes A, B;
  __device__ __forceinline__ bool too_small(int64_t i, int64_t k) const {
    return key_cmp(key_at(A, i), key_at(B, k - i - 1)) <= 0;
  }
};

// Lanes per boundary search (group_corank): each round of a string search
// is two dependent loads (offsets, then key bytes), so the rounds dominate.
#ifndef LSM_STR_PARTITION_LANES
#define LSM_STR_PARTITION_LANES 4
#endif
constexpr int kStrPartitionLanes = LSM_STR_PARTITION_LANES;

__global__ void __launch_bounds__(256) partition_str_kernel(StrAFirst pred, int64_t m, int64_t n,
                                                            int64_t D, int64_t G,
                                                            int64_t *__restrict__ out_i,
                                                            uint32_t *__restrict__ clear_words,
                                                            int64_t nclear) {
  pdl_begin();
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t w = gtid; w < nclear; w += stride) clear_words[w] = 0u;
  const int64_t g = gtid / kStrPartitionLanes;
  const bool active = g <= G;
  const int64_t total = m + n;
  const int64_t k = active ? (g * D < total ? g * D : total) : 0;
  const int64_t i = group_corank<kStrPartitionLanes>(pred, k, m, n, active);
  if (active && (threadIdx.x & (kStrPartitionLanes - 1)) == 0) out_i[g] = i;
}

template <int T, int E>
__global__ void __launch_bounds__(T) collision_mark_str_kernel(lsm_bytes A, int64_t m, lsm_bytes B,
                                                               int64_t n,
                                                               const int64_t *__restrict__ part_i,
                                                               uint32_t *__restrict__ C,
                                                               uint32_t *__restrict__ lb_B) {
  pdl_begin();
  constexpr int D = T * E;
  __shared__ uint32_t sLB[D];
  __shared__ uint32_t sCw[D / 32 + 4];
  const int tid = threadIdx.x;
  const int64_t g = blockIdx.x;
  const int64_t total = m + n;
  const int64_t k0 = g * D;
  const int64_t k1 = k0 + D < total ? k0 + D : total;
  const int64_t i0 = part_i[g], i1 = part_i[g + 1];
  const int64_t j0 = k0 - i0, j1 = k1 - i1;
  const int na = static_cast<int>(i1 - i0), nb = static_cast<int>(j1 - j0);
  const int64_t w0 = i0 >> 5;
  const int nw = na > 0 ? static_cast<int>(((i1 - 1) >> 5) - w0 + 1) : 0;
  for (int x = tid; x < nw; x += T) sCw[x] = 0u;
  __syncthreads();

  const int cnt = na + nb;
  const int d = tid * E < cnt ? tid * E : cnt;
  int lo = d > nb ? d - nb : 0, hi = d < na ? d : na;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (key_cmp(key_at(A, i0 + mid), key_at(B, j0 + d - mid - 1)) <= 0) lo = mid + 1;
    else hi = mid;
  }
  int ai = lo, bi = d - lo;
  // prev_eq: the element just before B's head in the merge is an A key equal
  // to it (then that B's lower bound is one less than the A count).
  bool prev_eq = false;
  if (d < cnt && i0 + ai > 0 && j0 + bi < n)
    prev_eq = key_cmp(key_at(A, i0 + ai - 1), key_at(B, j0 + bi)) == 0;
  for (int s = 0; s < E && d + s < cnt; ++s) {
    // c = cmp(A head, B head); B head may be B[j1] (one past the tile) only
    // for the collision test of A's last element.
    int c = 0;
    const bool has_a = ai < na;
    const bool has_b = j0 + bi < n;
    if (has_a && has_b) c = key_cmp(key_at(A, i0 + ai), key_at(B, j0 + bi));
    const bool takeA = (bi >= nb) || (has_a && c <= 0);
    if (takeA) {
      if (has_b && c == 0) {
        const int64_t gi = i0 + ai;
        atomicOr(&sCw[(gi >> 5) - w0], 1u << (gi & 31));
      }
      prev_eq = has_b && c == 0;
      ++ai;
    } else {
      sLB[bi] = static_cast<uint32_t>(i0 + ai - (prev_eq ? 1 : 0));
      prev_eq = false;
      ++bi;
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

}  // namespace

cudaError_t launch_collision_mark_str(const lsm_bytes &A, int64_t m, const lsm_bytes &B, int64_t n,
                                      uint32_t *C, uint32_t *lb_B, int64_t *part_i,
                                      int32_t * /*status*/, cudaStream_t s) {
  constexpr int64_t D = int64_t(kMarkStrThreads) * kMarkStrItems;
  const int64_t G = (m + n + D - 1) / D;
  const int64_t nwords = (m + 31) / 32;
  int64_t threads = (G + 1) * kStrPartitionLanes;
  if (threads < nwords / 4) threads = nwords / 4;
  cudaError_t err = launch_kernel(false, partition_str_kernel,
                                  static_cast<unsigned>((threads + 255) / 256), 256, 0, s,
                                  StrAFirst{A, B}, m, n, D, G, part_i, C, nwords);
  if (err != cudaSuccess || G == 0) return err;
  profile_before(s);
  err = launch_kernel(false, collision_mark_str_kernel<kMarkStrThreads, kMarkStrItems>,
                      static_cast<unsigned>(G), kMarkStrThreads, 0, s, A, m, B, n, part_i, C, lb_B);
  profile_after(s);
  return err;
}

}  // namespace lsm
