// ef.cu -- Elias-Fano navigation over the FC record offsets.
//
// "Everett: GPU construction experiment": physical record offsets are
// sampled at ordinals 0, 15, 30, ... and at EOF (the payload extent); with a
// common encoded value width w the sequence subtracts w times the sample's
// ordinal; the output EF kernels derive each entry from the record-offset
// scan, decide per 256-entry group whether its high-position span reaches
// 4096 bits, scan the sparse counts into exception ranges, and write lows,
// high bits, sample pairs and sparse positions, each word by one owner. The
// entries and layout (see include/lsmmerge.h):
//   x_s = bit_off[15 s] - 15 s w (s < n - 1), x_{n-1} = bit_off[N] - N w,
//   n = ceil(N/15) + 1, U = x_{n-1}, L = the largest L with n 2^L <= U;
//   lows: x_s mod 2^L at bits [sL, sL+L); highs: bit (x_s >> L) + s.
//
// Two launches:
//   ef_groups_kernel   one CTA: clears the highs words, finds every group's
//                      first and last high position (two gathers), its sparse
//                      flag, the exclusive scan of sparse entry counts, and
//                      writes the sample pairs and the exception total
//   ef_entries_kernel  one CTA per group of 256 entries: each thread gathers
//                      its entry, sets its highs bit (lanes sharing a word
//                      combine their bits first; words two CTAs share take
//                      atomicOr), ORs its low bits into the group's 4L lows
//                      words in shared memory (256 L bits = 4 L whole words,
//                      so a group owns its lows words) and stores them, and a
//                      sparse group writes its positions to the exceptions.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace lsm {

namespace {

constexpr int kEfGroup = 256;
constexpr int kEfScanThreads = 1024;

struct EfParams {
  const uint64_t *bit_off;
  int64_t N, n;
  uint64_t w;
  int L;
  int64_t nlows, nhighs, groups;  // words, words, groups
};

__device__ __forceinline__ uint64_t ef_entry(const EfParams &p, int64_t s) {
  const int64_t ord = s == p.n - 1 ? p.N : 15 * s;
  return __ldg(p.bit_off + ord) - static_cast<uint64_t>(ord) * p.w;
}

__device__ __forceinline__ uint64_t ef_high(const EfParams &p, int64_t s) {
  return (ef_entry(p, s) >> p.L) + static_cast<uint64_t>(s);
}

__global__ void __launch_bounds__(kEfScanThreads) ef_groups_kernel(EfParams p, uint64_t U,
                                                                   uint64_t *__restrict__ highs,
                                                                   uint64_t *__restrict__ samples,
                                                                   int64_t *__restrict__ d_nsparse,
                                                                   int32_t *status) {
  pdl_begin();
  __shared__ int64_t scratch[kEfScanThreads / 32 + 1];
  const int tid = threadIdx.x;
  if (tid == 0 && __ldg(p.bit_off + p.N) - static_cast<uint64_t>(p.N) * p.w != U)
    report(status, LSM_ERR_ARG);
  for (int64_t x = tid; x < p.nhighs; x += kEfScanThreads) highs[x] = 0;
  int64_t carry = 0;
  for (int64_t g0 = 0; g0 < p.groups; g0 += kEfScanThreads) {
    const int64_t g = g0 + tid;
    int64_t cnt = 0;
    uint64_t h0 = 0;
    bool sp = false;
    if (g < p.groups) {
      const int64_t first = g * kEfGroup;
      const int64_t last = first + kEfGroup - 1 < p.n - 1 ? first + kEfGroup - 1 : p.n - 1;
      h0 = ef_high(p, first);
      sp = ef_high(p, last) - h0 >= 4096;
      cnt = sp ? last - first + 1 : 0;
    }
    int64_t tot;
    const int64_t excl = block_exclusive_sum<kEfScanThreads>(cnt, scratch, &tot);
    if (g < p.groups) {
      samples[2 * g] = h0;
      samples[2 * g + 1] = (static_cast<uint64_t>(carry + excl) << 1) | (sp ? 1u : 0u);
    }
    carry += tot;
  }
  if (tid == 0) *d_nsparse = carry;
}

__global__ void __launch_bounds__(kEfGroup) ef_entries_kernel(EfParams p,
                                                              uint64_t *__restrict__ lows,
                                                              uint64_t *__restrict__ highs,
                                                              const uint64_t *__restrict__ samples,
                                                              uint64_t *__restrict__ sparse,
                                                              int32_t *status) {
  pdl_begin();
  __shared__ unsigned long long s_lows[4 * 63];
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t g = blockIdx.x;
  const int64_t s = g * kEfGroup + tid;
  const int L = p.L;
  for (int x = tid; x < 4 * L; x += kEfGroup) s_lows[x] = 0;
  __syncthreads();
  const bool valid = s < p.n;
  uint64_t x = 0, h = 0;
  if (valid) {
    x = ef_entry(p, s);
    h = (x >> L) + static_cast<uint64_t>(s);
  }
  // highs: lanes whose bits share a word OR them together; the first lane of
  // each run of equal words stores (atomically: a word may span two groups)
  const bool in_range = valid && (h >> 6) < static_cast<uint64_t>(p.nhighs);
  if (valid && !in_range) report(status, LSM_ERR_ARG);
  const uint64_t word = in_range ? (h >> 6) : ~0ull;
  unsigned long long bits = in_range ? (1ull << (h & 63)) : 0ull;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long b2 = __shfl_down_sync(0xffffffffu, bits, o);
    const uint64_t w2 = __shfl_down_sync(0xffffffffu, word, o);
    if (lane + o < 32 && w2 == word) bits |= b2;
  }
  const uint64_t wprev = __shfl_up_sync(0xffffffffu, word, 1);
  if (in_range && (lane == 0 || wprev != word))
    atomicOr(reinterpret_cast<unsigned long long *>(highs) + word, bits);
  // lows: bits [sL, sL + L) of this group's 4L words
  if (valid && L > 0) {
    const uint64_t lo = x & ((1ull << L) - 1);  // L <= 63
    const int bit = tid * L;  // relative to the group's first lows bit
    atomicOr(&s_lows[bit >> 6], static_cast<unsigned long long>(lo << (bit & 63)));
    if ((bit & 63) + L > 64)
      atomicOr(&s_lows[(bit >> 6) + 1], static_cast<unsigned long long>(lo >> (64 - (bit & 63))));
  }
  // sparse exceptions of this group
  if (valid) {
    const uint64_t meta = samples[2 * g + 1];
    if (meta & 1u) sparse[static_cast<int64_t>(meta >> 1) + tid] = h;
  }
  __syncthreads();
  const int64_t w0 = g * 4 * L;
  for (int q = tid; q < 4 * L; q += kEfGroup)
    if (w0 + q < p.nlows) lows[w0 + q] = s_lows[q];
}

EfParams ef_params(const uint64_t *bit_off, int64_t N, uint64_t w, uint64_t U) {
  int64_t sz[5];
  ef_layout(N, U, sz);
  EfParams p;
  p.bit_off = bit_off;
  p.N = N;
  p.n = sz[0];
  p.w = w;
  p.L = static_cast<int>(sz[1]);
  p.nlows = sz[2];
  p.nhighs = sz[3];
  p.groups = sz[4];
  return p;
}

}  // namespace

void ef_layout(int64_t N, uint64_t U, int64_t sizes[5]) {
  const int64_t n = (N + 14) / 15 + 1;
  int L = 0;
  // the largest L with n 2^L <= U (128-bit products: no overflow)
  while (L < 63 && (static_cast<unsigned __int128>(n) << (L + 1)) <= U) ++L;
  sizes[0] = n;
  sizes[1] = L;
  sizes[2] = (n * L + 63) / 64;
  sizes[3] = static_cast<int64_t>(((U >> L) + static_cast<uint64_t>(n) + 63) / 64);
  sizes[4] = (n + kEfGroup - 1) / kEfGroup;
}

cudaError_t launch_ef_build(const uint64_t *bit_off, int64_t N, uint64_t w, uint64_t U,
                            uint64_t *lows, uint64_t *highs, uint64_t *samples, uint64_t *sparse,
                            int64_t *d_nsparse, int32_t *status, cudaStream_t s) {
  const EfParams p = ef_params(bit_off, N, w, U);
  profile_before(s);
  cudaError_t err = launch_kernel(true, ef_groups_kernel, 1, kEfScanThreads, 0, s, p, U, highs,
                                  samples, d_nsparse, status);
  if (err == cudaSuccess)
    err = launch_kernel(true, ef_entries_kernel, static_cast<unsigned>(p.groups), kEfGroup, 0, s, p,
                        lows, highs, static_cast<const uint64_t *>(samples), sparse, status);
  profile_after(s);
  return err;
}

}  // namespace lsm
