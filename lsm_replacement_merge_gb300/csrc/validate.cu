// validate.cu -- optional sortedness validator for the inputs of the merge and
// replacement calls.
//
// The merge and replacement calls trust their inputs' order, as the pages'
// parser does ("Everett: byte-profile GPU merge", "Pipeline": framing, tags,
// offset bounds and retained lengths are checked, sorted order is not). A
// caller that cannot vouch for its inputs runs this pass first: one thread
// per adjacent pair (t, t+1), grid-stride, compares the two keys and lowers
// *d_first to the smallest violating t with atomicMin, and records
// LSM_ERR_UNSORTED in the sticky device status. Nothing traps or faults: a
// string pair whose offsets are out of order or past the arena is reported
// as a violation without reading its bytes.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "strings.cuh"

namespace lsm {

namespace {

constexpr int kValidateThreads = 256;

template <typename K>
__global__ void __launch_bounds__(kValidateThreads) validate_keys_kernel(
    const K *__restrict__ keys, int64_t count, int strict, unsigned long long *first,
    int32_t *status) {
  pdl_begin();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kValidateThreads;
  bool bad_any = false;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kValidateThreads + threadIdx.x; t + 1 < count;
       t += stride) {
    const K a = __ldg(keys + t), b = __ldg(keys + t + 1);
    const bool bad = strict ? !(a < b) : (b < a);
    if (bad) {
      atomicMin(first, static_cast<unsigned long long>(t));
      bad_any = true;
    }
  }
  if (__any_sync(0xffffffffu, bad_any) && (threadIdx.x & 31) == 0) report(status, LSM_ERR_UNSORTED);
}

// Byte-string keys in a CSR arena. Pair t is compared only when
// off[t] <= off[t+1] <= off[t+2] <= arena_bytes; otherwise the pair is a
// violation and its bytes are not read.
__global__ void __launch_bounds__(kValidateThreads) validate_str_kernel(
    lsm_bytes col, int64_t count, uint64_t arena_bytes, int strict, unsigned long long *first,
    int32_t *status) {
  pdl_begin();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kValidateThreads;
  bool bad_any = false;
  // the offsets of a single key must still be in order and inside the arena
  if (count == 1 && blockIdx.x == 0 && threadIdx.x == 0) {
    const uint64_t b0 = __ldg(col.off), b1 = __ldg(col.off + 1);
    if (b0 > b1 || b1 > arena_bytes) {
      atomicMin(first, 0ull);
      bad_any = true;
    }
  }
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kValidateThreads + threadIdx.x; t + 1 < count;
       t += stride) {
    const uint64_t o0 = __ldg(col.off + t), o1 = __ldg(col.off + t + 1), o2 = __ldg(col.off + t + 2);
    bool bad = !(o0 <= o1 && o1 <= o2 && o2 <= arena_bytes);
    if (!bad) {
      const int c = key_cmp(KeyRef{col.arena, o0, o1}, KeyRef{col.arena, o1, o2});
      bad = strict ? c >= 0 : c > 0;
    }
    if (bad) {
      atomicMin(first, static_cast<unsigned long long>(t));
      bad_any = true;
    }
  }
  if (__any_sync(0xffffffffu, bad_any) && (threadIdx.x & 31) == 0) report(status, LSM_ERR_UNSORTED);
}

unsigned validate_grid(int64_t pairs) {
  int64_t g = (pairs + kValidateThreads - 1) / kValidateThreads;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  if (g > cap) g = cap;
  return static_cast<unsigned>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_validate_sorted(int key_type, const void *keys, int64_t count, int strict,
                                   int64_t *d_first, int32_t *status, cudaStream_t s) {
  // -1 (all bits set) means "no violation"; atomicMin on the unsigned view
  // keeps the smallest violating index
  cudaError_t err = cudaMemsetAsync(d_first, 0xFF, sizeof(int64_t), s);
  if (err != cudaSuccess || count < 2) return err;
  auto *first = reinterpret_cast<unsigned long long *>(d_first);
  const unsigned grid = validate_grid(count - 1);
  if (key_type == LSM_KEY_I32)
    return launch_kernel(false, validate_keys_kernel<int32_t>, grid, kValidateThreads, 0, s,
                         static_cast<const int32_t *>(keys), count, strict, first, status);
  return launch_kernel(false, validate_keys_kernel<uint64_t>, grid, kValidateThreads, 0, s,
                       static_cast<const uint64_t *>(keys), count, strict, first, status);
}

cudaError_t launch_validate_sorted_str(const lsm_bytes &col, int64_t count, uint64_t arena_bytes,
                                       int strict, int64_t *d_first, int32_t *status,
                                       cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(d_first, 0xFF, sizeof(int64_t), s);
  if (err != cudaSuccess || count < 1) return err;
  auto *first = reinterpret_cast<unsigned long long *>(d_first);
  const unsigned grid = validate_grid(count > 1 ? count - 1 : 1);
  return launch_kernel(false, validate_str_kernel, grid, kValidateThreads, 0, s, col, count,
                       arena_bytes, strict, first, status);
}

}  // namespace lsm
