// api.cu -- the extern "C" entry points declared in include/lsmmerge.h.
//
// Each entry point checks its arguments on the host (null pointers, sizes,
// the 64-bit bound checks that precede 32-bit index arithmetic, alignment,
// workspace size), carves its scratch out of the caller's workspace and
// enqueues its kernels on the caller's stream. Nothing here allocates or
// synchronizes, except lsm_get_device_status, which exists to read the
// sticky status word.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "lsmmerge.h"

namespace lsm {

namespace {

// Sticky error word written by kernels whose bounded waits run out.
__device__ int32_t g_device_status;

constexpr int kMaxDevices = 64;
int32_t *g_status_ptr[kMaxDevices];
std::mutex g_status_mu;

// Device address of g_device_status on the current device (looked up once
// per device).
int32_t *status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int32_t *>(p);
  }
  return g_status_ptr[dev];
}

__global__ void timeout_probe_kernel(const volatile int32_t *never_set, int64_t limit_ns,
                                     int32_t *status) {
  pdl_begin();
  // Waits for a flag that no one writes, with the same bounded-time rule as
  // every other wait in this library.
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (*never_set != 0) return;
    if (globaltimer_ns() - t0 > static_cast<uint64_t>(limit_ns)) {
      if (threadIdx.x == 0) report(status, LSM_ERR_TIMEOUT);
      return;
    }
  }
  if (threadIdx.x == 0) report(status, LSM_ERR_TIMEOUT);
}

__device__ int32_t g_never_set_flag;

std::mutex g_prof_mu;
cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;

// ---- workspace carving ----------------------------------------------------------
struct Carver {
  uint8_t *p;
  size_t used = 0;
  template <typename T>
  T *take(int64_t count) {
    used = static_cast<size_t>(align_up(static_cast<int64_t>(used), 256));
    T *out = reinterpret_cast<T *>(p ? p + used : nullptr);
    used += static_cast<size_t>(count) * sizeof(T);
    return out;
  }
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned8(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? LSM_OK : LSM_ERR_CUDA; }

int64_t merge_tiles_max(int64_t total) { return (total + kMinMergeTile - 1) / kMinMergeTile; }

// Scratch of lsm_merge_sort: the alternate key and payload buffers of its
// passes, then the partition array.
template <typename KP, typename PP, typename IP>
void carve_merge_sort(Carver &c, int key_type, int64_t N, KP *keys, PP *pay, IP *part) {
  const int64_t D = merge_sort_tile();
  void *k = c.take<uint8_t>(N * (key_type == LSM_KEY_I32 ? 4 : 8));
  uint32_t *p = c.take<uint32_t>(N);
  int64_t *q = c.take<int64_t>((N + D - 1) / D + 1);
  if (keys) *keys = k;
  if (pay) *pay = p;
  if (part) *part = q;
}

size_t ws_bytes_for(int op, int64_t m, int64_t n, int key_type = LSM_KEY_U64) {
  Carver c{nullptr};
  switch (op) {
    case LSM_OP_MERGE_SORT:
      carve_merge_sort<void *, uint32_t *, int64_t *>(c, key_type, m, nullptr, nullptr, nullptr);
      break;
    case LSM_OP_MERGE_STABLE:
      c.take<int64_t>(merge_tiles_max(m + n) + 1);
      break;
    case LSM_OP_COLLISION_MARK: {
      const int64_t D = replace_min_tile();
      c.take<int64_t>((m + n + D - 1) / D + 1);
      break;
    }
    case LSM_OP_COLLISION_MARK_STR: {
      const int64_t D = int64_t(kMarkStrThreads) * kMarkStrItems;
      c.take<int64_t>((m + n + D - 1) / D + 1);
      break;
    }
    case LSM_OP_RANK_BUILD:
      c.take<uint64_t>(rank_build_ctas(m));
      break;
    case LSM_OP_RANK2048_BUILD:
      c.take<uint64_t>(rank2048_build_ctas(m));
      break;
    case LSM_OP_REPLACEMENT_FUSED: {
      const int64_t G = (m + n + fused_tile() - 1) / fused_tile();
      c.take<int64_t>(G + 1);
      c.take<uint64_t>(G > 0 ? G : 1);
      c.take<uint64_t>(rank_build_ctas(m));
      break;
    }
    case LSM_OP_REPLACEMENT_MERGE: {
      const int64_t G = (m + n + replacement_tile() - 1) / replacement_tile();
      c.take<int64_t>(G + 1);
      c.take<int64_t>(G + 1);
      c.take<uint64_t>(rank_build_ctas(m));
      c.take<uint32_t>(merge_bitmap_words(m + n));
      break;
    }
    case LSM_OP_REPLACEMENT_MERGE_STR: {
      const int64_t D = int64_t(kMarkStrThreads) * kMarkStrItems;
      const int64_t Dc = replacement_str_tile();
      c.take<int64_t>((m + n + D - 1) / D + 1);
      c.take<int64_t>((m + n + Dc - 1) / Dc + 1);
      c.take<uint64_t>(rank_build_ctas(m));
      c.take<uint32_t>(merge_bitmap_words(m + n));
      break;
    }
    case LSM_OP_REPLACEMENT_COMPACT: {
      const int64_t D = replace_min_tile();
      c.take<int64_t>((m + n + D - 1) / D + 1);
      c.take<uint32_t>(merge_bitmap_words(m + n));
      break;
    }
    case LSM_OP_FC_LENGTHS_SCAN:
      c.used = fc_scan_workspace_bytes(m);
      break;
    default:
      return 0;
  }
  return static_cast<size_t>(align_up(static_cast<int64_t>(c.used), 256)) + 256;
}

int check_ws(int op, int64_t m, int64_t n, const void *ws, size_t ws_bytes,
             int key_type = LSM_KEY_U64) {
  if (!ws) return LSM_ERR_WORKSPACE;
  if (!aligned16(ws)) return LSM_ERR_ALIGN;
  if (ws_bytes < ws_bytes_for(op, m, n, key_type)) return LSM_ERR_WORKSPACE;
  return LSM_OK;
}

constexpr int64_t kMax31 = (int64_t(1) << 31) - 1;

}  // namespace
}  // namespace lsm

using namespace lsm;

extern "C" {

LSM_API const char *lsm_status_string(int status) {
  switch (status) {
    case LSM_OK: return "LSM_OK";
    case LSM_ERR_ARG: return "LSM_ERR_ARG: invalid argument";
    case LSM_ERR_DTYPE: return "LSM_ERR_DTYPE: unsupported key type";
    case LSM_ERR_OVERFLOW: return "LSM_ERR_OVERFLOW: sizes exceed the supported index range";
    case LSM_ERR_CUDA: return "LSM_ERR_CUDA: a CUDA launch or runtime call failed";
    case LSM_ERR_TIMEOUT: return "LSM_ERR_TIMEOUT: a bounded device wait ran out";
    case LSM_ERR_WORKSPACE: return "LSM_ERR_WORKSPACE: workspace missing or too small";
    case LSM_ERR_ALIGN: return "LSM_ERR_ALIGN: pointer alignment requirement not met";
    case LSM_ERR_UNSORTED: return "LSM_ERR_UNSORTED: an input breaks its sorted order";
    default: return "unknown lsm status";
  }
}

LSM_API int lsm_abi_version(void) { return 101; }

LSM_API int lsm_get_device_status(int32_t *host_status, int reset, void *stream) {
  if (!host_status) return LSM_ERR_ARG;
  int32_t *d = status_ptr();
  if (!d) return LSM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return LSM_ERR_CUDA;
  if (cudaMemcpy(host_status, d, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return LSM_ERR_CUDA;
  if (reset && cudaMemset(d, 0, sizeof(int32_t)) != cudaSuccess) return LSM_ERR_CUDA;
  return LSM_OK;
}

LSM_API int lsm_workspace_size(int op, int key_type, int64_t m, int64_t n, size_t *bytes) {
  if (!bytes || m < 0 || n < 0) return LSM_ERR_ARG;
  if ((op == LSM_OP_MERGE_STABLE || op == LSM_OP_MERGE_SORT) && key_type != LSM_KEY_I32 &&
      key_type != LSM_KEY_U64)
    return LSM_ERR_DTYPE;
  if (op < LSM_OP_MERGE_STABLE || op > LSM_OP_REPLACEMENT_MERGE_STR) return LSM_ERR_ARG;
  *bytes = ws_bytes_for(op, m, n, key_type);
  return LSM_OK;
}

LSM_API int lsm_merge_path_partition(int key_type, const void *A, int64_t m, const void *B,
                                     int64_t n, int64_t items_per_tile, int64_t *out_ij,
                                     void *stream) {
  if (key_type != LSM_KEY_I32 && key_type != LSM_KEY_U64) return LSM_ERR_DTYPE;
  if (m < 0 || n < 0 || items_per_tile < 1 || !out_ij) return LSM_ERR_ARG;
  if ((m && !A) || (n && !B)) return LSM_ERR_ARG;
  if (m > (int64_t(1) << 40) || n > (int64_t(1) << 40)) return LSM_ERR_OVERFLOW;
  return cuda_status(launch_partition_keys(key_type, A, m, B, n, items_per_tile, nullptr, out_ij,
                                           static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_merge_stable(int key_type, const void *A, const uint32_t *Apay, int64_t m,
                             const void *B, const uint32_t *Bpay, int64_t n, void *out_keys,
                             uint32_t *out_pay, void *ws, size_t ws_bytes, void *stream) {
  if (key_type != LSM_KEY_I32 && key_type != LSM_KEY_U64) return LSM_ERR_DTYPE;
  if (m < 0 || n < 0) return LSM_ERR_ARG;
  const bool pay = Apay || Bpay || out_pay;
  if (pay && !(out_pay && (Apay || m == 0) && (Bpay || n == 0))) return LSM_ERR_ARG;
  if ((m && !A) || (n && !B) || (m + n && !out_keys)) return LSM_ERR_ARG;
  if (m > (int64_t(1) << 40) || n > (int64_t(1) << 40)) return LSM_ERR_OVERFLOW;
  if (m + n == 0) return LSM_OK;
  for (const void *p : {A, static_cast<const void *>(B), static_cast<const void *>(out_keys)})
    if (p && !aligned16(p)) return LSM_ERR_ALIGN;
  if (pay)
    for (const void *p : {static_cast<const void *>(Apay), static_cast<const void *>(Bpay),
                          static_cast<const void *>(out_pay)})
      if (p && !aligned16(p)) return LSM_ERR_ALIGN;
  if (int r = check_ws(LSM_OP_MERGE_STABLE, m, n, ws, ws_bytes)) return r;
  Carver c{static_cast<uint8_t *>(ws)};
  int64_t *part = c.take<int64_t>(merge_tiles_max(m + n) + 1);
  // A payload pointer of an empty side may be NULL; the kernels never read it.
  const uint32_t *ap = pay ? (Apay ? Apay : Bpay) : nullptr;
  const uint32_t *bp = pay ? (Bpay ? Bpay : Apay) : nullptr;
  const void *a = A ? A : B, *b = B ? B : A;
  return cuda_status(launch_merge_stable(key_type, a, ap, m, b, bp, n, out_keys, pay ? out_pay : nullptr,
                                         part, status_ptr(), static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_ef_sizes(int64_t N, uint64_t U, int64_t *sizes) {
  if (N < 0 || !sizes) return LSM_ERR_ARG;
  if (N > kMax31) return LSM_ERR_OVERFLOW;
  ef_layout(N, U, sizes);
  return LSM_OK;
}

LSM_API int lsm_fc_ef_build(const uint64_t *bit_off, int64_t N, uint64_t w, uint64_t U,
                            uint64_t *lows, uint64_t *highs, uint64_t *samples, uint64_t *sparse,
                            int64_t *d_nsparse, void *stream) {
  if (N < 0 || !bit_off || !highs || !samples || !sparse || !d_nsparse) return LSM_ERR_ARG;
  if (N > kMax31) return LSM_ERR_OVERFLOW;
  int64_t sz[5];
  ef_layout(N, U, sz);
  if (sz[2] > 0 && !lows) return LSM_ERR_ARG;
  for (const void *p : {static_cast<const void *>(bit_off), static_cast<const void *>(lows),
                        static_cast<const void *>(highs), static_cast<const void *>(samples),
                        static_cast<const void *>(sparse)})
    if (p && !aligned8(p)) return LSM_ERR_ALIGN;
  return cuda_status(launch_ef_build(bit_off, N, w, U, lows, highs, samples, sparse, d_nsparse,
                                     status_ptr(), static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_merge_sort(int key_type, const void *keys, const uint32_t *pay, int64_t N,
                           void *out_keys, uint32_t *out_pay, void *ws, size_t ws_bytes,
                           void *stream) {
  if (key_type != LSM_KEY_I32 && key_type != LSM_KEY_U64) return LSM_ERR_DTYPE;
  if (N < 0) return LSM_ERR_ARG;
  if (!pay != !out_pay) return LSM_ERR_ARG;
  if (N && (!keys || !out_keys)) return LSM_ERR_ARG;
  if (N > (int64_t(1) << 40)) return LSM_ERR_OVERFLOW;
  if (N == 0) return LSM_OK;
  for (const void *p : {keys, static_cast<const void *>(out_keys), static_cast<const void *>(pay),
                        static_cast<const void *>(out_pay)})
    if (p && !aligned16(p)) return LSM_ERR_ALIGN;
  if (int r = check_ws(LSM_OP_MERGE_SORT, N, 0, ws, ws_bytes, key_type)) return r;
  Carver c{static_cast<uint8_t *>(ws)};
  void *tmp = nullptr;
  uint32_t *tmp_pay = nullptr;
  int64_t *part = nullptr;
  carve_merge_sort(c, key_type, N, &tmp, &tmp_pay, &part);
  return cuda_status(launch_merge_sort(key_type, keys, pay, N, out_keys, out_pay, tmp,
                                       pay ? tmp_pay : nullptr, part, status_ptr(),
                                       static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_validate_sorted(int key_type, const void *keys, int64_t count, int strict,
                                int64_t *d_first, void *stream) {
  if (key_type != LSM_KEY_I32 && key_type != LSM_KEY_U64) return LSM_ERR_DTYPE;
  if (count < 0 || !d_first || (count && !keys) || (strict != 0 && strict != 1)) return LSM_ERR_ARG;
  if (count > (int64_t(1) << 40)) return LSM_ERR_OVERFLOW;
  const uintptr_t esz = key_type == LSM_KEY_I32 ? 4 : 8;
  if ((keys && (reinterpret_cast<uintptr_t>(keys) & (esz - 1))) || !aligned8(d_first))
    return LSM_ERR_ALIGN;
  return cuda_status(launch_validate_sorted(key_type, keys, count, strict, d_first, status_ptr(),
                                            static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_validate_sorted_str(const lsm_bytes *keys, int64_t count, uint64_t arena_bytes,
                                    int strict, int64_t *d_first, void *stream) {
  if (!keys || count < 0 || !d_first || (strict != 0 && strict != 1)) return LSM_ERR_ARG;
  if (count && (!keys->off || (arena_bytes && !keys->arena))) return LSM_ERR_ARG;
  if (count > kMax31) return LSM_ERR_OVERFLOW;
  if ((keys->arena && !aligned8(keys->arena)) || (keys->off && !aligned8(keys->off)) ||
      !aligned8(d_first))
    return LSM_ERR_ALIGN;
  return cuda_status(launch_validate_sorted_str(*keys, count, arena_bytes, strict, d_first,
                                                status_ptr(), static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_collision_mark(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                               uint32_t *C, uint32_t *lb_B, void *ws, size_t ws_bytes,
                               void *stream) {
  if (m < 0 || n < 0) return LSM_ERR_ARG;
  if ((m && (!A || !C)) || (n && (!B || !lb_B))) return LSM_ERR_ARG;
  if (m > kMax31 || n > kMax31) return LSM_ERR_OVERFLOW;
  if (m + n == 0) return LSM_OK;
  if ((A && !aligned16(A)) || (B && !aligned16(B)) || (lb_B && !aligned16(lb_B)))
    return LSM_ERR_ALIGN;
  if (int r = check_ws(LSM_OP_COLLISION_MARK, m, n, ws, ws_bytes)) return r;
  Carver c{static_cast<uint8_t *>(ws)};
  const int64_t D = replace_min_tile();
  int64_t *part = c.take<int64_t>((m + n + D - 1) / D + 1);
  return cuda_status(launch_collision_mark(A ? A : B, m, B ? B : A, n, C, lb_B, part, status_ptr(),
                                           static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_collision_mark_str(const lsm_bytes *A, int64_t m, const lsm_bytes *B, int64_t n,
                                   uint32_t *C, uint32_t *lb_B, void *ws, size_t ws_bytes,
                                   void *stream) {
  return lsm_collision_mark_str_prefix(A, m, B, n, C, lb_B, nullptr, nullptr, ws, ws_bytes,
                                       stream);
}

LSM_API int lsm_collision_mark_str_prefix(const lsm_bytes *A, int64_t m, const lsm_bytes *B,
                                          int64_t n, uint32_t *C, uint32_t *lb_B,
                                          uint64_t *prefixA, uint64_t *prefixB, void *ws,
                                          size_t ws_bytes, void *stream) {
  if (m < 0 || n < 0 || !A || !B) return LSM_ERR_ARG;
  if ((m && (!A->arena || !A->off || !C)) || (n && (!B->arena || !B->off || !lb_B)))
    return LSM_ERR_ARG;
  if (m > kMax31 || n > kMax31) return LSM_ERR_OVERFLOW;
  if (m + n == 0) return LSM_OK;
  if ((m && !aligned8(A->arena)) || (n && !aligned8(B->arena))) return LSM_ERR_ALIGN;
  if ((prefixA && !aligned16(prefixA)) || (prefixB && !aligned16(prefixB))) return LSM_ERR_ALIGN;
  if (int r = check_ws(LSM_OP_COLLISION_MARK_STR, m, n, ws, ws_bytes)) return r;
  Carver c{static_cast<uint8_t *>(ws)};
  const int64_t D = int64_t(kMarkStrThreads) * kMarkStrItems;
  int64_t *part = c.take<int64_t>((m + n + D - 1) / D + 1);
  return cuda_status(launch_collision_mark_str(*A, m, *B, n, C, lb_B, m ? prefixA : nullptr,
                                               n ? prefixB : nullptr, part, status_ptr(),
                                               static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_rank_build(const uint32_t *C, int64_t m, uint32_t *dir, int64_t *d_total,
                           void *ws, size_t ws_bytes, void *stream) {
  if (m < 0 || !dir || !d_total || (m && !C)) return LSM_ERR_ARG;
  if (m > kMax31) return LSM_ERR_OVERFLOW;
  if (C && !aligned16(C)) return LSM_ERR_ALIGN;
  if (int r = check_ws(LSM_OP_RANK_BUILD, m, 0, ws, ws_bytes)) return r;
  Carver c{static_cast<uint8_t *>(ws)};
  uint64_t *state = c.take<uint64_t>(rank_build_ctas(m));
  return cuda_status(launch_rank_build_ws(C, m, dir, d_total, state, status_ptr(),
                                          static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_rank_query(const uint32_t *C, const uint32_t *dir, int64_t m,
                           const uint32_t *pos, int64_t q, uint32_t *out, void *stream) {
  if (m < 0 || q < 0 || !dir || (m && !C) || (q && (!pos || !out))) return LSM_ERR_ARG;
  if (m > kMax31 || q > kMax31) return LSM_ERR_OVERFLOW;
  return cuda_status(launch_rank_query(C, dir, m, pos, q, out, status_ptr(),
                                       static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_rank2048_build(const uint32_t *C, int64_t m, uint64_t *dir, uint64_t *epochs,
                               int64_t *d_total, void *ws, size_t ws_bytes, void *stream) {
  if (m < 0 || !dir || !epochs || !d_total || (m && !C)) return LSM_ERR_ARG;
  if (m >= (int64_t(1) << 36)) return LSM_ERR_OVERFLOW;
  if ((C && !aligned16(C)) || !aligned8(dir) || !aligned8(epochs)) return LSM_ERR_ALIGN;
  if (int r = check_ws(LSM_OP_RANK2048_BUILD, m, 0, ws, ws_bytes)) return r;
  Carver c{static_cast<uint8_t *>(ws)};
  uint64_t *scratch = c.take<uint64_t>(rank2048_build_ctas(m));
  return cuda_status(launch_rank2048_build(C, m, dir, epochs, d_total, scratch, status_ptr(),
                                           static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_rank2048_query(const uint32_t *C, const uint64_t *dir, const uint64_t *epochs,
                               int64_t m, const uint64_t *pos, int64_t q, uint64_t *out,
                               void *stream) {
  if (m < 0 || q < 0 || !dir || !epochs || (m && !C) || (q && (!pos || !out))) return LSM_ERR_ARG;
  if (m >= (int64_t(1) << 36) || q > kMax31) return LSM_ERR_OVERFLOW;
  if (C && !aligned16(C)) return LSM_ERR_ALIGN;
  if (q == 0) return LSM_OK;
  return cuda_status(launch_rank2048_query(C, dir, epochs, m, pos, q, out, status_ptr(),
                                           static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_replacement_merge_compact(int64_t m, int64_t n, const uint32_t *C,
                                          const uint32_t *dir, const uint32_t *lb_B,
                                          uint32_t *out_refs, uint32_t *ord_A, uint32_t *ord_B,
                                          int64_t *d_count, void *ws, size_t ws_bytes,
                                          void *stream) {
  if (m < 0 || n < 0 || !dir || !d_count) return LSM_ERR_ARG;
  if ((m && (!C || !ord_A)) || (n && (!lb_B || !ord_B)) || (m + n && !out_refs)) return LSM_ERR_ARG;
  if (m > kMax31 || n > kMax31) return LSM_ERR_OVERFLOW;
  if ((lb_B && !aligned16(lb_B)) || (C && !aligned16(C)) || !aligned16(out_refs) ||
      (ord_A && !aligned16(ord_A)) || (ord_B && !aligned16(ord_B)))
    return LSM_ERR_ALIGN;
  if (int r = check_ws(LSM_OP_REPLACEMENT_COMPACT, m, n, ws, ws_bytes)) return r;
  Carver c{static_cast<uint8_t *>(ws)};
  const int64_t D = replace_min_tile();
  int64_t *part = c.take<int64_t>((m + n + D - 1) / D + 1);
  uint32_t *mb = c.take<uint32_t>(merge_bitmap_words(m + n));
  return cuda_status(launch_compact(m, n, C, dir, lb_B, out_refs, ord_A, ord_B, d_count, part, mb,
                                    status_ptr(), static_cast<cudaStream_t>(stream)));
}

// lsm_replacement_merge's form: 0 = two pipelines (the default, measured
// faster), 1 = the mark and the compaction in one kernel
// (lsm_tune_replacement_merge).
static int g_replacement_merge_mode = 0;

LSM_API int lsm_replacement_merge(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                  uint32_t *C, uint32_t *lb_B, uint32_t *dir, int64_t *d_total,
                                  uint32_t *out_refs, uint32_t *ord_A, uint32_t *ord_B,
                                  int64_t *d_count, void *ws, size_t ws_bytes, void *stream) {
  if (m < 0 || n < 0 || !dir || !d_total || !d_count) return LSM_ERR_ARG;
  // lb_B may be null here: the compaction reads the merge bitmap, not lb_B
  if ((m && (!A || !C || !ord_A)) || (n && (!B || !ord_B)) || (m + n && !out_refs))
    return LSM_ERR_ARG;
  if (m > kMax31 || n > kMax31) return LSM_ERR_OVERFLOW;
  for (const void *p : {static_cast<const void *>(A), static_cast<const void *>(B),
                        static_cast<const void *>(C), static_cast<const void *>(lb_B),
                        static_cast<const void *>(out_refs), static_cast<const void *>(ord_A),
                        static_cast<const void *>(ord_B)})
    if (p && !aligned16(p)) return LSM_ERR_ALIGN;
  if (int r = check_ws(LSM_OP_REPLACEMENT_MERGE, m, n, ws, ws_bytes)) return r;
  Carver c{static_cast<uint8_t *>(ws)};
  const int64_t G = (m + n + replacement_tile() - 1) / replacement_tile();
  int64_t *part_m = c.take<int64_t>(G + 1);
  int64_t *part_c = c.take<int64_t>(G + 1);
  uint64_t *rank_ws = c.take<uint64_t>(rank_build_ctas(m));
  uint32_t *mb = c.take<uint32_t>(merge_bitmap_words(m + n));
  if (g_replacement_merge_mode == 1)
    // one kernel for the mark and the compaction: part_c's words hold the
    // tiles' lookback states instead (G <= G + 1 words), the merge bitmap
    // stays in shared memory
    return cuda_status(launch_replacement_merge_one(
        A ? A : B, m, B ? B : A, n, C, lb_B, dir, d_total, out_refs, ord_A, ord_B, d_count, part_m,
        reinterpret_cast<uint64_t *>(part_c), rank_ws, status_ptr(),
        static_cast<cudaStream_t>(stream)));
  return cuda_status(launch_replacement_merge(A ? A : B, m, B ? B : A, n, C, lb_B, dir, d_total,
                                              out_refs, ord_A, ord_B, d_count, part_m, part_c, mb,
                                              rank_ws, status_ptr(),
                                              static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_replacement_merge_str(const lsm_bytes *A, int64_t m, const lsm_bytes *B, int64_t n,
                                      uint32_t *C, uint32_t *lb_B, uint64_t *prefixA,
                                      uint64_t *prefixB, uint32_t *dir, int64_t *d_total,
                                      uint32_t *out_refs, uint32_t *ord_A, uint32_t *ord_B,
                                      int64_t *d_count, void *ws, size_t ws_bytes, void *stream) {
  if (m < 0 || n < 0 || !A || !B || !dir || !d_total || !d_count) return LSM_ERR_ARG;
  if ((m && (!A->arena || !A->off || !C || !ord_A)) || (n && (!B->arena || !B->off || !ord_B)) ||
      (m + n && !out_refs))
    return LSM_ERR_ARG;
  if (m > kMax31 || n > kMax31) return LSM_ERR_OVERFLOW;
  if ((m && !aligned8(A->arena)) || (n && !aligned8(B->arena))) return LSM_ERR_ALIGN;
  for (const void *p : {static_cast<const void *>(C), static_cast<const void *>(lb_B),
                        static_cast<const void *>(prefixA), static_cast<const void *>(prefixB),
                        static_cast<const void *>(out_refs), static_cast<const void *>(ord_A),
                        static_cast<const void *>(ord_B)})
    if (p && !aligned16(p)) return LSM_ERR_ALIGN;
  if (int r = check_ws(LSM_OP_REPLACEMENT_MERGE_STR, m, n, ws, ws_bytes)) return r;
  Carver c{static_cast<uint8_t *>(ws)};
  const int64_t D = int64_t(kMarkStrThreads) * kMarkStrItems;
  const int64_t Dc = replacement_str_tile();
  int64_t *part_m = c.take<int64_t>((m + n + D - 1) / D + 1);
  int64_t *part_c = c.take<int64_t>((m + n + Dc - 1) / Dc + 1);
  uint64_t *rank_ws = c.take<uint64_t>(rank_build_ctas(m));
  uint32_t *mb = c.take<uint32_t>(merge_bitmap_words(m + n));
  return cuda_status(launch_replacement_merge_str(
      *A, m, *B, n, C, n ? lb_B : nullptr, m ? prefixA : nullptr, n ? prefixB : nullptr, dir,
      d_total, out_refs, ord_A, ord_B, d_count, part_m, part_c, mb, rank_ws, status_ptr(),
      static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_tune_replacement_merge(int mode) {
  if (mode != 0 && mode != 1) return LSM_ERR_ARG;
  g_replacement_merge_mode = mode;
  return LSM_OK;
}

LSM_API int lsm_replacement_merge_fused(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                        uint32_t *C, uint32_t *lb_B, uint32_t *dir,
                                        int64_t *d_total, uint32_t *out_refs, uint32_t *ord_A,
                                        uint32_t *ord_B, int64_t *d_count, void *ws,
                                        size_t ws_bytes, void *stream) {
  if (m < 0 || n < 0 || !dir || !d_total || !d_count) return LSM_ERR_ARG;
  if ((m && (!A || !C || !ord_A)) || (n && (!B || !lb_B || !ord_B)) || (m + n && !out_refs))
    return LSM_ERR_ARG;
  if (m > kMax31 || n > kMax31) return LSM_ERR_OVERFLOW;
  for (const void *p : {static_cast<const void *>(A), static_cast<const void *>(B),
                        static_cast<const void *>(C), static_cast<const void *>(lb_B),
                        static_cast<const void *>(out_refs), static_cast<const void *>(ord_A),
                        static_cast<const void *>(ord_B)})
    if (p && !aligned16(p)) return LSM_ERR_ALIGN;
  if (int r = check_ws(LSM_OP_REPLACEMENT_FUSED, m, n, ws, ws_bytes)) return r;
  Carver c{static_cast<uint8_t *>(ws)};
  const int64_t G = (m + n + fused_tile() - 1) / fused_tile();
  int64_t *part = c.take<int64_t>(G + 1);
  uint64_t *state = c.take<uint64_t>(G > 0 ? G : 1);
  uint64_t *rank_ws = c.take<uint64_t>(rank_build_ctas(m));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_replacement_fused(A ? A : B, m, B ? B : A, n, C, lb_B, out_refs, ord_A,
                                           ord_B, d_count, part, state, status_ptr(), s);
  if (e == cudaSuccess) e = launch_rank_build_ws(C, m, dir, d_total, rank_ws, status_ptr(), s);
  return cuda_status(e);
}

LSM_API int lsm_replacement_direct_scatter(const uint64_t *A, int64_t m, const uint64_t *B,
                                           int64_t n, const uint32_t *C, const uint32_t *dir,
                                           const uint32_t *lb_B, uint32_t *out_refs,
                                           uint32_t *ord_A, uint32_t *ord_B, int64_t *d_count,
                                           void *stream) {
  if (m < 0 || n < 0 || !dir || !d_count) return LSM_ERR_ARG;
  if ((m && (!A || !C || !ord_A)) || (n && (!B || !lb_B || !ord_B)) || (m + n && !out_refs))
    return LSM_ERR_ARG;
  if (m > kMax31 || n > kMax31) return LSM_ERR_OVERFLOW;
  for (const void *p : {static_cast<const void *>(A), static_cast<const void *>(B),
                        static_cast<const void *>(C), static_cast<const void *>(lb_B),
                        static_cast<const void *>(out_refs), static_cast<const void *>(ord_A),
                        static_cast<const void *>(ord_B)})
    if (p && !aligned16(p)) return LSM_ERR_ALIGN;
  return cuda_status(launch_direct_scatter(A, m, B, n, C, dir, lb_B, out_refs, ord_A, ord_B,
                                           d_count, status_ptr(),
                                           static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_replacement_merge_compact_rank2048(int64_t m, int64_t n, const uint32_t *C,
                                                   const uint64_t *dir, const uint64_t *epochs,
                                                   const uint32_t *lb_B, uint32_t *out_refs,
                                                   uint32_t *ord_A, uint32_t *ord_B,
                                                   int64_t *d_count, void *ws, size_t ws_bytes,
                                                   void *stream) {
  if (m < 0 || n < 0 || !dir || !epochs || !d_count) return LSM_ERR_ARG;
  if ((m && (!C || !ord_A)) || (n && (!lb_B || !ord_B)) || (m + n && !out_refs)) return LSM_ERR_ARG;
  if (m > kMax31 || n > kMax31) return LSM_ERR_OVERFLOW;
  if ((lb_B && !aligned16(lb_B)) || (C && !aligned16(C)) || !aligned16(out_refs) ||
      (ord_A && !aligned16(ord_A)) || (ord_B && !aligned16(ord_B)))
    return LSM_ERR_ALIGN;
  if (int r = check_ws(LSM_OP_REPLACEMENT_COMPACT, m, n, ws, ws_bytes)) return r;
  Carver c{static_cast<uint8_t *>(ws)};
  const int64_t D = replace_min_tile();
  int64_t *part = c.take<int64_t>((m + n + D - 1) / D + 1);
  uint32_t *mb = c.take<uint32_t>(merge_bitmap_words(m + n));
  return cuda_status(launch_compact_tiles_rank2048(m, n, C, dir, epochs, lb_B, mb, part, out_refs,
                                                   ord_A, ord_B, d_count, status_ptr(),
                                                   static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_replacement_materialize(const uint64_t *A, const uint32_t *Aval,
                                        const uint32_t *tombA, int64_t m, const uint64_t *B,
                                        const uint32_t *Bval, const uint32_t *tombB, int64_t n,
                                        const uint32_t *refs, const int64_t *d_count,
                                        uint64_t *out_keys, uint32_t *out_vals,
                                        uint32_t *out_tomb, void *stream) {
  if (m < 0 || n < 0 || !d_count) return LSM_ERR_ARG;
  if (m > kMax31 || n > kMax31) return LSM_ERR_OVERFLOW;
  if (m + n == 0) return LSM_OK;
  if ((m && !A) || (n && !B) || !refs || !out_keys) return LSM_ERR_ARG;
  if (out_vals && ((m && !Aval) || (n && !Bval))) return LSM_ERR_ARG;
  for (const void *p : {static_cast<const void *>(A), static_cast<const void *>(B),
                        static_cast<const void *>(out_keys), static_cast<const void *>(refs),
                        static_cast<const void *>(out_vals)})
    if (p && !aligned16(p)) return LSM_ERR_ALIGN;
  return cuda_status(launch_materialize(A, Aval, tombA, m, B, Bval, tombB, n, refs, d_count,
                                        out_keys, out_vals, out_tomb, status_ptr(),
                                        static_cast<cudaStream_t>(stream)));
}

static int check_fc_input(const lsm_fc_input *in) {
  if (!in || in->m < 0 || in->n < 0) return LSM_ERR_ARG;
  if (in->m > kMax31 || in->n > kMax31) return LSM_ERR_OVERFLOW;
  if (in->m && (!in->keyA.arena || !in->keyA.off || !in->valA.arena || !in->valA.off))
    return LSM_ERR_ARG;
  if (in->n && (!in->keyB.arena || !in->keyB.off || !in->valB.arena || !in->valB.off))
    return LSM_ERR_ARG;
  for (const void *p : {static_cast<const void *>(in->keyA.arena), static_cast<const void *>(in->valA.arena),
                        static_cast<const void *>(in->keyB.arena), static_cast<const void *>(in->valB.arena)})
    if (p && !aligned8(p)) return LSM_ERR_ALIGN;
  // prefix tables: both or neither (an empty side needs none)
  if ((in->prefixA || in->prefixB) &&
      ((in->m && !in->prefixA) || (in->n && !in->prefixB)))
    return LSM_ERR_ARG;
  if ((in->prefixA && !aligned16(in->prefixA)) || (in->prefixB && !aligned16(in->prefixB)))
    return LSM_ERR_ALIGN;
  return LSM_OK;
}

LSM_API int lsm_bytefc_lengths_scan(const lsm_fc_input *in, const uint32_t *refs, int64_t N,
                                    uint64_t W, uint32_t *lcp, uint32_t *ctrl,
                                    uint32_t *rec_bytes, uint64_t *byte_off, void *ws,
                                    size_t ws_bytes, void *stream) {
  if (int r = check_fc_input(in)) return r;
  if (N < 0 || !byte_off || (N && (!refs || !lcp || !ctrl || !rec_bytes))) return LSM_ERR_ARG;
  if (N > kMax31 || N > in->m + in->n) return LSM_ERR_OVERFLOW;
  if (!aligned16(rec_bytes) || !aligned16(byte_off)) return LSM_ERR_ALIGN;
  if (int r = check_ws(LSM_OP_FC_LENGTHS_SCAN, N, 0, ws, ws_bytes)) return r;
  return cuda_status(launch_bytefc_lengths_scan(*in, refs, N, W, lcp, ctrl, rec_bytes, byte_off,
                                                ws, status_ptr(),
                                                static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_bytefc_value_width(const lsm_fc_input *in, const uint32_t *refs, int64_t N,
                                   uint64_t *d_width, void *stream) {
  if (int r = check_fc_input(in)) return r;
  if (N < 0 || !d_width || (N && !refs)) return LSM_ERR_ARG;
  if (N > kMax31 || N > in->m + in->n) return LSM_ERR_OVERFLOW;
  if (!aligned8(d_width)) return LSM_ERR_ALIGN;
  return cuda_status(launch_bytefc_value_width(*in, refs, N, d_width,
                                               static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_bytefc_emit(const lsm_fc_input *in, const uint32_t *refs, int64_t N, uint64_t W,
                            const uint32_t *lcp, const uint32_t *ctrl, const uint64_t *byte_off,
                            uint8_t *payload, int64_t nbytes, void *stream) {
  if (int r = check_fc_input(in)) return r;
  if (N < 0 || nbytes < 0 || (N && (!refs || !lcp || !ctrl || !byte_off || !payload)))
    return LSM_ERR_ARG;
  if (N > kMax31 || N > in->m + in->n) return LSM_ERR_OVERFLOW;
  return cuda_status(launch_bytefc_emit(*in, refs, N, W, lcp, ctrl, byte_off, payload, nbytes,
                                        status_ptr(), static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_fc_lengths_scan(const lsm_fc_input *in, const uint32_t *refs, int64_t N,
                                uint32_t *lcp, uint32_t *ctrl, uint32_t *rec_bits,
                                uint64_t *bit_off, void *ws, size_t ws_bytes, void *stream) {
  if (int r = check_fc_input(in)) return r;
  if (N < 0 || !bit_off || (N && (!refs || !lcp || !ctrl || !rec_bits))) return LSM_ERR_ARG;
  if (N > kMax31 || N > in->m + in->n) return LSM_ERR_OVERFLOW;
  if (int r = check_ws(LSM_OP_FC_LENGTHS_SCAN, N, 0, ws, ws_bytes)) return r;
  return cuda_status(launch_fc_lengths_scan(*in, refs, N, lcp, ctrl, rec_bits, bit_off, ws,
                                            status_ptr(), static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_fc_emit(const lsm_fc_input *in, const uint32_t *refs, int64_t N,
                        const uint32_t *lcp, const uint32_t *ctrl, const uint64_t *bit_off,
                        uint32_t *payload, int64_t nwords, void *stream) {
  if (int r = check_fc_input(in)) return r;
  if (N < 0 || nwords < 0 || !bit_off || (N && (!refs || !lcp || !ctrl)) || (nwords && !payload))
    return LSM_ERR_ARG;
  if (N > kMax31 || N > in->m + in->n || nwords > (int64_t(1) << 40)) return LSM_ERR_OVERFLOW;
  if (payload && !aligned16(payload)) return LSM_ERR_ALIGN;
  return cuda_status(launch_fc_emit(*in, refs, N, lcp, ctrl, bit_off, payload, nwords,
                                    status_ptr(), static_cast<cudaStream_t>(stream)));
}

LSM_API int lsm_set_profile_events(void *start_event, void *stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return LSM_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_start = static_cast<cudaEvent_t>(start_event);
  g_prof_stop = static_cast<cudaEvent_t>(stop_event);
  return LSM_OK;
}

LSM_API int lsm_tune_replace(int kernel, int threads, int items_per_thread) {
  return set_replace_variant(kernel, threads, items_per_thread);
}

LSM_API int lsm_tune_merge(int key_type, int items_per_thread, int stages, int out_tiles) {
  return set_merge_config(key_type, items_per_thread, stages, out_tiles);
}

LSM_API int lsm_debug_timeout_probe(int64_t limit_ns, void *stream) {
  if (limit_ns < 1000) limit_ns = 1000;
  if (limit_ns > kWaitLimitNs) limit_ns = kWaitLimitNs;
  return cuda_status(launch_timeout_probe(limit_ns, status_ptr(), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace lsm {
void profile_before(cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (g_prof_start) {
    cudaEventRecord(g_prof_start, s);
    g_prof_start = nullptr;
  }
}

void profile_after(cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (g_prof_stop && !g_prof_start) {
    cudaEventRecord(g_prof_stop, s);
    g_prof_stop = nullptr;
  }
}

cudaError_t launch_timeout_probe(int64_t limit_ns, int32_t *status, cudaStream_t s) {
  void *flag = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&flag, g_never_set_flag);
  if (e != cudaSuccess) return e;
  return launch_kernel(true, timeout_probe_kernel, 1, 32, 0, s,
                       static_cast<const volatile int32_t *>(flag), limit_ns, status);
}
}  // namespace lsm
