// common.cuh -- device helpers shared by the merge-path kernels (sm_103a).
//
// Bulk asynchronous copies (the TMA engine's 1-D form) stage each CTA's
// merge-path tile into shared memory and write finished tiles back; an
// mbarrier with a transaction count tracks the loads. Every wait is bounded
// in time: past the limit the kernel records LSM_ERR_TIMEOUT in the status
// word it was given and returns, so that a stuck wait cannot hang the GPU.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "lsmmerge.h"

namespace lsm {

constexpr int64_t kWaitLimitNs = 1000000000LL;  // one second

// Programmatic dependent launch. Every kernel of this library starts with
// pdl_begin(): it waits until the kernel before it on the stream has
// finished and its writes are visible, then lets the kernel after it launch.
// Launched with programmatic stream serialization (launch_kernel below), the
// next kernel's launch and prologue so overlap this one's run, while every
// kernel still sees all earlier work complete before it touches memory;
// launched without it, the wait returns at once.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__host__ __device__ constexpr int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Launches `kern` on stream s, with programmatic stream serialization when
// `pdl` is set (see pdl_begin). It pays where the kernel before leaves SM
// room free (a partition of a few blocks per SM, a one-CTA scan): measured on
// GB300, the replacement chain gains ~6 us and the merge's tile launch ~1 us.
// Where the kernel before runs in waves, an early-launched kernel holds room
// those waves need: the string + FC chain lost ~90 us with every launch
// early, so its wave-filling launches go without it.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool pdl, void (*kern)(KArgs...), unsigned grid, unsigned block,
                          size_t smem, cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// First error wins; later errors do not overwrite it.
__device__ __forceinline__ void report(int32_t *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// A 32-bit store to a shared-memory address (as smem_u32 gives it).
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t *p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// ---- mbarrier --------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete, for at most
// limit_ns nanoseconds (and a bounded number of polls). Returns false when
// the limit ran out.
static __device__ __noinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 63 && globaltimer_ns() - t0 > static_cast<uint64_t>(limit_ns)) return false;
  }
  return false;
}

// ---- bulk copies -------------------------------------------------------------
// global -> shared, completion counted on `bar` (bytes: multiple of 16,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void *sdst, const void *gsrc, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// shared -> global in the current bulk group.
__device__ __forceinline__ void bulk_s2g(void *gdst, const void *ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until the committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Waits until at most one committed bulk-store group still reads shared
// memory (the most recent one may continue).
__device__ __forceinline__ void bulk_wait_read_allow1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (a following bulk store reads them).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- staging a 1-D span into shared memory ----------------------------------
// Global elements [s, s + c) of size SZ (array base 16-byte aligned) land in
// a 16-byte aligned shared buffer so that element s + x sits at buf[lead + x].
// A 16-byte aligned range [alo, ahi) moves with one bulk copy; elements of
// the span past ahi (at most 16/SZ - 1, and only at the end of the array)
// move with plain loads, so nothing past the array's end is ever read.
struct StagePlan {
  int64_t first;      // global index of buf[0]
  int64_t tail_from;  // first global index loaded with plain loads
  int32_t lead;       // s - first
  uint32_t bulk;      // bytes of the bulk copy (multiple of 16, may be 0)
  int32_t span;       // lead + c: elements of buf in use
};

// The plan for [s, s + c) of an array of `limit` elements: the bulk copy
// runs from the 16-byte boundary at or below s up to the next 16-byte
// boundary past s + c whenever that stays inside the array, so that a span
// needs plain loads only at the very end of its array.
template <int SZ>
__device__ __forceinline__ StagePlan stage_plan_overfetch(int64_t s, int64_t c, int64_t limit) {
  const int64_t lo = s * SZ, hi = (s + c) * SZ;
  const int64_t alo = lo & ~int64_t(15);
  const int64_t up = (hi + 15) & ~int64_t(15);
  const int64_t ahi = up <= ((limit * SZ) & ~int64_t(15)) ? up : (hi & ~int64_t(15));
  StagePlan p;
  p.first = alo / SZ;
  p.lead = static_cast<int32_t>(s - p.first);
  p.bulk = static_cast<uint32_t>(ahi > alo ? ahi - alo : 0);
  p.tail_from = ahi / SZ > s ? ahi / SZ : s;
  p.span = static_cast<int32_t>(p.lead + c);
  return p;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Barrier over the first `nthreads` threads of the block (named barrier
// `id`), returning whether any of them passed a true predicate.
__device__ __forceinline__ bool named_sync_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int SZ>
__host__ __device__ constexpr int64_t stage_capacity_bytes(int64_t c) {
  return align_up(c * SZ + 16, 16);
}

// Issues a plan's bulk copy (if any) against mbarrier `bar`; the caller
// loads the elements from p.tail_from on with plain loads.
template <typename T>
__device__ __forceinline__ void stage_issue(T *buf, const T *g, const StagePlan &p, uint64_t *bar) {
  if (p.bulk) bulk_g2s(buf, g + p.first, p.bulk, bar);
}

// ---- scans ------------------------------------------------------------------
template <typename V>
__device__ __forceinline__ V warp_inclusive_sum(V v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    V u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// Block-wide exclusive sum for a block of NT threads (NT multiple of 32).
// `scratch` holds NT/32 + 1 values. Returns the exclusive prefix; *total
// receives the block sum. Contains __syncthreads().
template <int NT, typename V>
__device__ __forceinline__ V block_exclusive_sum(V v, V *scratch, V *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  V inc = warp_inclusive_sum(v);
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    V w = lane < NT / 32 ? scratch[lane] : V(0);
    V wi = warp_inclusive_sum(w);
    if (lane < NT / 32) scratch[lane] = wi - w;
    if (lane == NT / 32 - 1) scratch[NT / 32] = wi;
  }
  __syncthreads();
  V out = scratch[warp] + inc - v;
  *total = scratch[NT / 32];
  __syncthreads();
  return out;
}

template <int NT, typename V>
__device__ __forceinline__ V block_sum(V v, V *scratch) {
  V total;
  block_exclusive_sum<NT>(v, scratch, &total);
  return total;
}

// ---- merge-path co-rank searches ---------------------------------------------------
// The co-rank of diagonal k is the first i in [max(0, k-n), min(k, m)] for
// which pred.too_small(i, k) is false.
// That co-rank found by a group of L lanes (L a power of two <= 32,
// groups aligned within the warp). Each round the group tests L pivots
// spread evenly over the open range and keeps the interval between the last
// pivot that is too small and the first that is not, so the range shrinks
// (L + 1)-fold per round: fewer dependent rounds of loads than bisection,
// for L times the loads per round. [lo, hi] is a bracket known to hold the
// co-rank, inside [max(0, k - n), min(k, m)]. Every lane of the warp must
// call it (the ballots span the warp); a lane with active = false joins with
// an empty range and returns its lower end.
template <int L, class Pred>
__device__ __forceinline__ int64_t group_corank_in(const Pred &pred, int64_t k, int64_t lo,
                                                   int64_t hi, bool active) {
  static_assert(L >= 1 && L <= 32 && (L & (L - 1)) == 0, "group size");
  if (!active || hi < lo) hi = lo;
  const int lane = threadIdx.x & 31;
  const int l = lane & (L - 1);
  const int gbase = lane & ~(L - 1);
  const uint32_t gmask = L == 32 ? 0xffffffffu : ((1u << L) - 1u);
  while (__any_sync(0xffffffffu, lo < hi)) {
    const int64_t span = hi - lo;
    const bool open = span > 0;
    const bool t = open && pred.too_small(lo + ((l + 1) * span) / (L + 1), k);
    const int c = __popc((__ballot_sync(0xffffffffu, t) >> gbase) & gmask);
    if (open) {
      const int64_t nlo = c > 0 ? lo + (c * span) / (L + 1) + 1 : lo;
      const int64_t nhi = c < L ? lo + ((c + 1) * span) / (L + 1) : hi;
      lo = nlo;
      hi = nhi;
    }
  }
  return lo;
}

// group_corank_in over the diagonal's whole range [max(0, k - n), min(k, m)].
template <int L, class Pred>
__device__ __forceinline__ int64_t group_corank(const Pred &pred, int64_t k, int64_t m, int64_t n,
                                                bool active) {
  return group_corank_in<L>(pred, k, k > n ? k - n : 0, k < m ? k : m, active);
}

}  // namespace lsm
