// scatter.cu -- the replacement merge's "tiled direct scatter" path.
//
// "Everett: collision bitmap and rank experiment", "The three experimental
// paths", second path: a thread handles 32 consecutive A records, performs
// one lower-bound search into B, then advances the B cursor monotonically
// for the rest of its records; both inputs then scatter to their corrected
// positions ("Corrected record ordinals"):
//   surviving A_i:  i + lower_bound(B, A_i) - R(i)      (dropped: 0xFFFFFFFF)
//   B_j:            j + lb_B[j] - R(lb_B[j])
// and refs[ordinal] = the record's reference. The outputs equal the
// compaction's (the bitmap, compact-A, merge-path path), which reads no keys;
// this path reads A and B again. One launch: the first blocks take A in
// runs of 32 records per thread, the rest take one B record per thread.
// Bounds: a dropped or surviving A record's ordinal is < N = m + n - R(m),
// and so is every B record's, for sorted unique inputs with a valid C and
// lb_B; every scatter is checked against N regardless, and a record that
// would land outside records LSM_ERR_ARG instead of writing.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "rank512.cuh"

namespace lsm {

namespace {

constexpr int kScatterThreads = 256;
constexpr int kScatterRun = 32;  // A records per thread ([CB]: 32 consecutive records)

__global__ void __launch_bounds__(kScatterThreads) direct_scatter_kernel(
    const uint64_t *__restrict__ A, int64_t m, const uint64_t *__restrict__ B, int64_t n,
    const uint32_t *__restrict__ C, const uint32_t *__restrict__ dir,
    const uint32_t *__restrict__ lb_B, uint32_t *__restrict__ refs, uint32_t *__restrict__ ord_A,
    uint32_t *__restrict__ ord_B, int64_t *__restrict__ d_count, int64_t a_blocks,
    int32_t *status) {
  pdl_begin();
  const int64_t N = m + n - static_cast<int64_t>(m ? rank512_at(C, dir, m) : 0u);
  if (blockIdx.x == 0 && threadIdx.x == 0) *d_count = N;
  if (static_cast<int64_t>(blockIdx.x) < a_blocks) {
    // ---- A: 32 consecutive records, one lower-bound search, then a monotone cursor
    const int64_t i0 = (static_cast<int64_t>(blockIdx.x) * kScatterThreads + threadIdx.x) * kScatterRun;
    if (i0 >= m) return;
    const int cnt = m - i0 < kScatterRun ? static_cast<int>(m - i0) : kScatterRun;
    const uint64_t a0 = A[i0];
    int64_t lo = 0, hi = n;
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (__ldg(B + mid) < a0) lo = mid + 1;
      else hi = mid;
    }
    int64_t j = lo;
    uint64_t bj = j < n ? __ldg(B + j) : 0;
    const uint32_t cw = C[i0 >> 5];  // i0 is a multiple of 32: one bitmap word
    int64_t r = rank512_at(C, dir, i0);
    uint32_t ord[kScatterRun];
#pragma unroll
    for (int q = 0; q < kScatterRun; ++q) {
      ord[q] = LSM_ORD_DROPPED;
      if (q < cnt) {
        const uint64_t a = A[i0 + q];
        while (j < n && bj < a) {
          ++j;
          bj = j < n ? __ldg(B + j) : 0;
        }
        if ((cw >> q) & 1u) {
          ++r;  // replaced by B: dropped, and counted from the next record on
        } else {
          const int64_t o = i0 + q + j - r;
          if (o >= 0 && o < N) {
            ord[q] = static_cast<uint32_t>(o);
            refs[o] = static_cast<uint32_t>(i0 + q);
          } else {
            report(status, LSM_ERR_ARG);
          }
        }
      }
    }
    if (cnt == kScatterRun) {
      uint4 *dst = reinterpret_cast<uint4 *>(ord_A + i0);
#pragma unroll
      for (int q = 0; q < kScatterRun / 4; ++q)
        dst[q] = make_uint4(ord[4 * q], ord[4 * q + 1], ord[4 * q + 2], ord[4 * q + 3]);
    } else {
#pragma unroll
      for (int q = 0; q < kScatterRun; ++q)
        if (q < cnt) ord_A[i0 + q] = ord[q];
    }
    return;
  }
  // ---- B: one record per thread
  const int64_t jb = (static_cast<int64_t>(blockIdx.x) - a_blocks) * kScatterThreads + threadIdx.x;
  if (jb >= n) return;
  const uint32_t lb = lb_B[jb];
  if (lb > m) {
    report(status, LSM_ERR_ARG);
    ord_B[jb] = LSM_ORD_DROPPED;
    return;
  }
  const int64_t o = jb + lb - static_cast<int64_t>(m ? rank512_at(C, dir, lb) : 0u);
  if (o >= 0 && o < N) {
    ord_B[jb] = static_cast<uint32_t>(o);
    refs[o] = static_cast<uint32_t>(jb) | LSM_REF_FROM_B;
  } else {
    ord_B[jb] = LSM_ORD_DROPPED;
    report(status, LSM_ERR_ARG);
  }
}

}  // namespace

cudaError_t launch_direct_scatter(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                  const uint32_t *C, const uint32_t *dir, const uint32_t *lb_B,
                                  uint32_t *refs, uint32_t *ord_A, uint32_t *ord_B,
                                  int64_t *d_count, int32_t *status, cudaStream_t s) {
  const int64_t a_threads = (m + kScatterRun - 1) / kScatterRun;
  const int64_t a_blocks = (a_threads + kScatterThreads - 1) / kScatterThreads;
  const int64_t b_blocks = (n + kScatterThreads - 1) / kScatterThreads;
  const int64_t blocks = a_blocks + b_blocks > 0 ? a_blocks + b_blocks : 1;
  profile_before(s);
  const cudaError_t err = launch_kernel(true, direct_scatter_kernel, static_cast<unsigned>(blocks),
                                        kScatterThreads, 0, s, A, m, B, n, C, dir, lb_B, refs,
                                        ord_A, ord_B, d_count, a_blocks, status);
  profile_after(s);
  return err;
}

}  // namespace lsm
