// pipeline.cuh -- persistent, warp-specialized tile pipeline.
//
// One CTA per SM slot loops over merge-path tiles c, c + P, c + 2P, ...
// (P = gridDim.x). The last warp is the producer: its 32 lanes fetch the
// per-tile prologue values of 32 upcoming tiles at once (Spec::fetch, e.g.
// the tile's co-ranks), then lane 0 stages the tiles one by one into S
// shared-memory stages with bulk copies (Spec::produce), each stage guarded
// by a full and an empty mbarrier. The other T threads consume a stage
// (Spec::consume) and hand it back. Every wait is bounded in time.
//
// A Spec provides:
//   static constexpr int T, S;                 consumer threads, stages
//   static constexpr int64_t kStageBytes, kWorkBytes;
//   struct Params; struct Desc (<= 64 bytes);
//   __device__ static void init(uint8_t *work);   consumers, once, before tiles
//   __device__ static void fetch(const Params&, int64_t g, int64_t v[4]);
//   __device__ static void produce(const Params&, int64_t g, const int64_t v[4],
//                                  uint8_t *stage, Desc &d, uint64_t *full);
//       (must end with mbar_arrive_expect_tx on `full` and its bulk copies)
//   __device__ static void consume(const Params&, int64_t g, const Desc &d,
//                                  const uint8_t *stage, uint8_t *work,
//                                  uint64_t *empty);
//       (run by the T consumer threads; must arrive on `empty` once per
//        consumer warp after its last read of the stage; may use named
//        barrier 1 over the T consumer threads)
#pragma once

#include <cstdint>

#include "common.cuh"

namespace lsm {

template <class Spec>
struct PipelineLayout {
  static constexpr int S = Spec::S;
  static constexpr int64_t kFull = 0;
  static constexpr int64_t kEmpty = 8 * S;
  static constexpr int64_t kDesc = 16 * S;
  static constexpr int64_t kStage0 = align_up(16 * S + 64 * S, 128);
  static constexpr int64_t kWork = kStage0 + S * align_up(Spec::kStageBytes, 128);
  static constexpr int64_t kBytes = kWork + Spec::kWorkBytes;
  static constexpr int64_t kStageStride = align_up(Spec::kStageBytes, 128);
};

// Releases a stage: every consumer warp arrives once.
__device__ __forceinline__ void release_stage(uint64_t *empty) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(empty);
}

template <class Spec>
__global__ void __launch_bounds__(Spec::T + 32) tile_pipeline_kernel(typename Spec::Params p,
                                                                     int64_t G, int32_t *status) {
  pdl_begin();
  using L = PipelineLayout<Spec>;
  constexpr int S = Spec::S;
  constexpr int T = Spec::T;
  using Desc = typename Spec::Desc;
  static_assert(sizeof(Desc) <= 64, "descriptor slot");
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kFull);
  uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L::kEmpty);
  Desc *desc = reinterpret_cast<Desc *>(smem + L::kDesc);
  const int tid = threadIdx.x;
  const int64_t P = gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], T / 32);
    }
  }
  __syncthreads();

  if (tid >= T) {
    const int lane = tid & 31;
    for (int64_t r0 = 0; blockIdx.x + r0 * P < G; r0 += 32) {
      const int64_t gl = blockIdx.x + (r0 + lane) * P;
      int64_t v[4] = {0, 0, 0, 0};
      if (gl < G) Spec::fetch(p, gl, v);
      for (int q = 0; q < 32; ++q) {
        const int64_t r = r0 + q;
        const int64_t g = blockIdx.x + r * P;
        if (g >= G) break;
        int64_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) w[t] = __shfl_sync(0xffffffffu, v[t], q);
        int failed = 0;
        if (lane == 0) {
          const int s = static_cast<int>(r % S);
          if (r >= S && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>(((r / S) + 1) & 1),
                                           kWaitLimitNs)) {
            report(status, LSM_ERR_TIMEOUT);
            failed = 1;
          } else {
            Spec::produce(p, g, w, smem + L::kStage0 + s * L::kStageStride, desc[s], &full[s]);
          }
        }
        if (__shfl_sync(0xffffffffu, failed, 0)) return;
      }
    }
    return;
  }

  Spec::init(smem + L::kWork);
  named_sync(1, T);
  for (int64_t r = 0;; ++r) {
    const int64_t g = blockIdx.x + r * P;
    if (g >= G) break;
    const int s = static_cast<int>(r % S);
    const bool ok = mbar_wait_bounded(&full[s], static_cast<uint32_t>((r / S) & 1), kWaitLimitNs);
    if (named_sync_or(1, T, !ok)) {
      if (tid == 0) report(status, LSM_ERR_TIMEOUT);
      break;
    }
    // A private copy: once the consumers release the stage, the producer may
    // rewrite its descriptor for the next tile.
    const Desc d = desc[s];
    Spec::consume(p, g, d, smem + L::kStage0 + s * L::kStageStride, smem + L::kWork, &empty[s]);
  }
}

// Launches the pipeline with as many CTAs as fit on the device (at most G).
template <class Spec>
cudaError_t launch_pipeline(const typename Spec::Params &p, int64_t G, int32_t *status,
                            cudaStream_t s, int sms) {
  using L = PipelineLayout<Spec>;
  static_assert(L::kBytes <= 225 * 1024, "pipeline exceeds shared memory");
  auto kern = tile_pipeline_kernel<Spec>;
  static int per_sm = 0;
  if (!per_sm) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(L::kBytes));
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Spec::T + 32, L::kBytes);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
  }
  int64_t grid = static_cast<int64_t>(sms) * per_sm;
  if (grid < 1) grid = 1;
  if (grid > G) grid = G;
  return launch_kernel(true, kern, static_cast<unsigned>(grid), Spec::T + 32, L::kBytes, s, p, G,
                       status);
}

// Writes global uint32 elements [g0, g0 + count) from a shared buffer that
// holds element g0 at sbuf[g0 & 3] (sbuf 16-byte aligned, gbase 16-byte
// aligned), so that shared and global addresses agree modulo 16: thread 0
// moves the aligned body with one bulk store (committed by the caller), the
// other consumer threads the at most three head and three tail elements.
// The caller fences the shared writes for the async proxy and barriers before
// calling, and later waits for the bulk store to finish reading.
template <int NT>
__device__ __forceinline__ void store_u32_run(uint32_t *gbase, int64_t g0, int count,
                                              const uint32_t *sbuf) {
  if (count <= 0) return;
  const int shift = static_cast<int>(g0 & 3);
  const int head = count < ((4 - shift) & 3) ? count : ((4 - shift) & 3);
  const int body = (count - head) & ~3;
  const int tid = threadIdx.x;
  if (tid == 0 && body) bulk_s2g(gbase + g0 + head, sbuf + shift + head, static_cast<uint32_t>(body) * 4);
  // head elements and the ragged tail, by threads 1..
  const int tail = count - head - body;
  const int t = tid - 1;
  if (t >= 0 && t < head) gbase[g0 + t] = sbuf[shift + t];
  if (t >= 8 && t < 8 + tail) gbase[g0 + head + body + (t - 8)] = sbuf[shift + head + body + (t - 8)];
}

// Exclusive sum of `v` and exclusive maximum of `mx` over the T consumer
// threads in one pass (named barrier 1). `scratch` holds 2 * (T/32 + 1)
// values; *total is the sum over all threads and *mx_before the maximum of
// `mx` over the threads before this one (0 for the first). The caller's
// next barrier must come before scratch is written again.
template <int NT>
__device__ __forceinline__ uint32_t consumer_exclusive_sum_max(uint32_t v, uint32_t mx,
                                                               uint32_t *scratch, uint32_t *total,
                                                               uint32_t *mx_before) {
  constexpr int NWARP = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v, mi = mx;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, inc, off);
    const uint32_t u = __shfl_up_sync(0xffffffffu, mi, off);
    if (lane >= off) {
      inc += t;
      mi = u > mi ? u : mi;
    }
  }
  // maximum over the lanes before this one
  uint32_t mprev = __shfl_up_sync(0xffffffffu, mi, 1);
  if (lane == 0) mprev = 0;
  if (lane == 31) {
    scratch[warp] = inc;
    scratch[NWARP + 1 + warp] = mi;
  }
  named_sync(1, NT);
  if (warp == 0) {
    const uint32_t w = lane < NWARP ? scratch[lane] : 0u;
    const uint32_t wm = lane < NWARP ? scratch[NWARP + 1 + lane] : 0u;
    uint32_t wi = w, wmi = wm;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, wi, off);
      const uint32_t u = __shfl_up_sync(0xffffffffu, wmi, off);
      if (lane >= off) {
        wi += t;
        wmi = u > wmi ? u : wmi;
      }
    }
    uint32_t wmprev = __shfl_up_sync(0xffffffffu, wmi, 1);
    if (lane == 0) wmprev = 0;
    if (lane < NWARP) {
      scratch[lane] = wi - w;
      scratch[NWARP + 1 + lane] = wmprev;
    }
    if (lane == NWARP - 1) scratch[NWARP] = wi;
  }
  named_sync(1, NT);
  *total = scratch[NWARP];
  const uint32_t wmb = scratch[NWARP + 1 + warp];
  *mx_before = wmb > mprev ? wmb : mprev;
  return scratch[warp] + inc - v;
}

}  // namespace lsm
