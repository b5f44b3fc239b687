// rank2048.cu -- build and query of the 2048-bit rank directory.
//
// "Everett: collision bitmap and rank experiment", "Temporary rank layouts"
// (the COLLISION_RANK2048 variant) and "Scratch space and likely costs" (its
// storage, (1/8 + 8/2048)|A| bytes with the bitmap, and its smaller
// block-scan scratch). The build is the page's count -> global scan ->
// finish path in two launches:
//
//   rank2048_count_kernel   one thread per 2048-bit block (sixteen 16-byte
//                           loads), the CTA's population -> cta_totals
//   rank2048_finish_kernel  each CTA sums its predecessors' totals (the
//                           global scan, in 64 bits) and the totals before
//                           its epoch's first CTA, recounts its blocks and
//                           writes every entry; the CTA starting an epoch
//                           writes that epoch's absolute count, the last CTA
//                           the total R(m).
//
// A CTA covers 256 blocks = 2^19 bits, so every CTA lies inside one 2^32-bit
// epoch (8192 CTAs per epoch).
//
// When every CTA of the build is resident at once (and so m < 2^31, a single
// epoch), the build is one launch instead: rank2048_single_kernel counts,
// finds its prefix by a decoupled lookback over the CTAs' published totals
// and writes its entries, reading C once.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "lookback.cuh"
#include "rank2048.cuh"

namespace lsm {

namespace {

constexpr int64_t kCtasPerEpoch = (int64_t(1) << 32) / (2048 * kRank2048Threads);

// The four 512-bit run populations of block b (words past nwords read as 0).
__device__ __forceinline__ void block2048_pops(const uint32_t *__restrict__ C, int64_t nwords,
                                               int64_t b, uint32_t pop[4]) {
  const int64_t base = b * 64;
#pragma unroll
  for (int r = 0; r < 4; ++r) pop[r] = 0;
  if (base + 64 <= nwords) {
    const uint4 *p = reinterpret_cast<const uint4 *>(C + base);
    uint4 v[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = p[q];
#pragma unroll
    for (int q = 0; q < 16; ++q)
      pop[q >> 2] += __popc(v[q].x) + __popc(v[q].y) + __popc(v[q].z) + __popc(v[q].w);
  } else {
    for (int t = 0; t < 64; ++t)
      if (base + t < nwords) pop[t >> 4] += __popc(C[base + t]);
  }
}

__global__ void __launch_bounds__(kRank2048Threads) rank2048_count_kernel(
    const uint32_t *__restrict__ C, int64_t m, uint32_t *__restrict__ cta_totals) {
  pdl_begin();
  __shared__ uint32_t scratch[kRank2048Threads / 32 + 1];
  const int64_t nwords = (m + 31) / 32;
  const int64_t nblk = m / 2048 + 1;
  const int64_t b = static_cast<int64_t>(blockIdx.x) * kRank2048Threads + threadIdx.x;
  uint32_t tot = 0;
  if (b < nblk) {
    uint32_t pop[4];
    block2048_pops(C, nwords, b, pop);
    tot = pop[0] + pop[1] + pop[2] + pop[3];
  }
  const uint32_t total = block_sum<kRank2048Threads>(tot, scratch);
  if (threadIdx.x == 0) cta_totals[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kRank2048Threads) rank2048_finish_kernel(
    const uint32_t *__restrict__ C, int64_t m, const uint32_t *__restrict__ cta_totals,
    uint64_t *__restrict__ dir, uint64_t *__restrict__ epochs, int64_t *__restrict__ d_total) {
  pdl_begin();
  __shared__ uint64_t scratch[kRank2048Threads / 32 + 1];
  __shared__ uint32_t scratch32[kRank2048Threads / 32 + 1];
  const int64_t nwords = (m + 31) / 32;
  const int64_t nblk = m / 2048 + 1;
  const int64_t c = blockIdx.x;
  const int64_t epoch_first = (c / kCtasPerEpoch) * kCtasPerEpoch;
  // the global scan: totals of every CTA before this one, and of those
  // before this epoch's first CTA
  uint64_t acc = 0, acc_epoch = 0;
  for (int64_t x = threadIdx.x; x < c; x += kRank2048Threads) {
    const uint64_t t = cta_totals[x];
    acc += t;
    if (x < epoch_first) acc_epoch += t;
  }
  const uint64_t prefix = block_sum<kRank2048Threads>(acc, scratch);
  const uint64_t epoch_base = block_sum<kRank2048Threads>(acc_epoch, scratch);

  const int64_t b = c * kRank2048Threads + threadIdx.x;
  uint32_t pop[4] = {0, 0, 0, 0};
  if (b < nblk) block2048_pops(C, nwords, b, pop);
  const uint32_t tot = pop[0] + pop[1] + pop[2] + pop[3];
  uint32_t cta_sum;
  const uint32_t excl = block_exclusive_sum<kRank2048Threads>(b < nblk ? tot : 0u, scratch32, &cta_sum);
  if (b < nblk) {
    const uint64_t rel = prefix - epoch_base + excl;  // below 2^32 inside one epoch
    dir[b] = rel | (static_cast<uint64_t>(pop[0]) << 32) | (static_cast<uint64_t>(pop[1]) << 42) |
             (static_cast<uint64_t>(pop[2]) << 52);
  }
  if (c == epoch_first && threadIdx.x == 0) epochs[c / kCtasPerEpoch] = prefix;
  if (c == gridDim.x - 1 && threadIdx.x == 0) *d_total = static_cast<int64_t>(prefix + cta_sum);
}

__global__ void __launch_bounds__(kRank2048Threads) rank2048_single_kernel(
    const uint32_t *__restrict__ C, int64_t m, uint64_t *__restrict__ dir,
    uint64_t *__restrict__ epochs, int64_t *__restrict__ d_total, uint64_t *state,
    int32_t *status) {
  pdl_begin();
  __shared__ uint32_t scratch[kRank2048Threads / 32 + 1];
  __shared__ uint32_t s_prefix;
  const int64_t nwords = (m + 31) / 32;
  const int64_t nblk = m / 2048 + 1;
  const uint32_t t = blockIdx.x;
  const int64_t b = static_cast<int64_t>(t) * kRank2048Threads + threadIdx.x;
  uint32_t pop[4] = {0, 0, 0, 0};
  if (b < nblk) block2048_pops(C, nwords, b, pop);
  const uint32_t tot = pop[0] + pop[1] + pop[2] + pop[3];
  uint32_t agg;
  const uint32_t excl = block_exclusive_sum<kRank2048Threads>(b < nblk ? tot : 0u, scratch, &agg);
  if (threadIdx.x < 32) {
    const uint32_t prefix = lookback_exclusive(state, t, agg, status);
    if (threadIdx.x == 0) s_prefix = prefix;
  }
  __syncthreads();
  const uint32_t prefix = s_prefix;
  if (b < nblk)
    dir[b] = static_cast<uint64_t>(prefix + excl) | (static_cast<uint64_t>(pop[0]) << 32) |
             (static_cast<uint64_t>(pop[1]) << 42) | (static_cast<uint64_t>(pop[2]) << 52);
  if (t == 0 && threadIdx.x == 0) epochs[0] = 0;
  if (t == gridDim.x - 1 && threadIdx.x == 0) *d_total = static_cast<int64_t>(prefix) + agg;
}

__global__ void __launch_bounds__(256) rank2048_query_kernel(
    const uint32_t *__restrict__ C, const uint64_t *__restrict__ dir,
    const uint64_t *__restrict__ epochs, int64_t m, const uint64_t *__restrict__ pos, int64_t q,
    uint64_t *__restrict__ out, int32_t *status) {
  pdl_begin();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= q) return;
  const uint64_t p = pos[t];
  if (p > static_cast<uint64_t>(m)) {
    out[t] = ~0ull;
    report(status, LSM_ERR_ARG);
    return;
  }
  out[t] = rank2048_at(C, dir, epochs, static_cast<int64_t>(p));
}

}  // namespace

int64_t rank2048_build_ctas(int64_t m) {
  return (m / 2048 + 1 + kRank2048Threads - 1) / kRank2048Threads;
}

cudaError_t launch_rank2048_build(const uint32_t *C, int64_t m, uint64_t *dir, uint64_t *epochs,
                                  int64_t *d_total, uint64_t *ws, int32_t *status, cudaStream_t s) {
  static int per_sm = -1;  // CTAs of rank2048_single_kernel resident per SM
  if (per_sm < 0) {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, rank2048_single_kernel, kRank2048Threads,
                                                      0) != cudaSuccess)
      v = 0;
    per_sm = v;
  }
  const int64_t ctas = rank2048_build_ctas(m);
  if (m < (int64_t(1) << 31) && ctas <= static_cast<int64_t>(device_sm_count()) * per_sm) {
    // every CTA resident at once, so each CTA a lookback waits for is
    // running; the lookback states start from zero at every call
    cudaError_t err = cudaMemsetAsync(ws, 0, static_cast<size_t>(ctas) * 8, s);
    if (err != cudaSuccess) return err;
    profile_before(s);
    err = launch_kernel(true, rank2048_single_kernel, static_cast<unsigned>(ctas),
                        kRank2048Threads, 0, s, C, m, dir, epochs, d_total, ws, status);
    profile_after(s);
    return err;
  }
  uint32_t *cta_totals = reinterpret_cast<uint32_t *>(ws);
  profile_before(s);  // the profiling hook brackets both launches
  cudaError_t err = launch_kernel(true, rank2048_count_kernel, static_cast<unsigned>(ctas),
                                  kRank2048Threads, 0, s, C, m, cta_totals);
  if (err == cudaSuccess)
    err = launch_kernel(true, rank2048_finish_kernel, static_cast<unsigned>(ctas),
                        kRank2048Threads, 0, s, C, m, static_cast<const uint32_t *>(cta_totals),
                        dir, epochs, d_total);
  profile_after(s);
  return err;
}

cudaError_t launch_rank2048_query(const uint32_t *C, const uint64_t *dir, const uint64_t *epochs,
                                  int64_t m, const uint64_t *pos, int64_t q, uint64_t *out,
                                  int32_t *status, cudaStream_t s) {
  return launch_kernel(true, rank2048_query_kernel, static_cast<unsigned>((q + 255) / 256), 256, 0,
                       s, C, dir, epochs, m, pos, q, out, status);
}

}  // namespace lsm
