// internal.h -- launchers shared between the kernel files and the C ABI layer.
// Host-side only; every launcher enqueues on `stream` and returns the CUDA
// launch status. Argument checking happens in api.cu before these run.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "lsmmerge.h"

namespace lsm {

// Tile geometry. Items per thread are odd so that per-thread output runs in
// shared memory fall on distinct banks.
constexpr int kMergeThreads = 256;
constexpr int kRankThreads = 256;

int merge_items_per_thread(int key_type);  // current setting (tunable)
// Selects the tile configuration (items per thread, input stages, output
// tiles) of lsm_merge_stable; returns LSM_OK or LSM_ERR_ARG.
int set_merge_config(int key_type, int items, int stages, int out_tiles);
// Smallest tile (elements) over the replacement pipelines' variants: sizes
// the partition arrays in their workspaces.
int64_t replace_min_tile();
// Selects the tile variant of collision_mark (kernel 0) or
// replacement_merge_compact (kernel 1); LSM_OK or LSM_ERR_ARG.
int set_replace_variant(int kernel, int threads, int items);
constexpr int64_t kMinMergeTile = kMergeThreads * 5;

// --- merge.cu ---
cudaError_t launch_partition_keys(int key_type, const void *A, int64_t m, const void *B, int64_t n,
                                  int64_t D, int64_t *out_i, int64_t *out_ij, cudaStream_t s);
cudaError_t launch_merge_stable(int key_type, const void *A, const uint32_t *Apay, int64_t m,
                                const void *B, const uint32_t *Bpay, int64_t n, void *out,
                                uint32_t *out_pay, int64_t *part_i, int32_t *status,
                                cudaStream_t s);
// Bottom-up merge sort: block sort to runs of merge_sort_tile() elements,
// then one partition + tile-kernel launch per pass. tmp / tmp_pay: N
// elements each (tmp_pay only with a payload); part: ceil(N / tile) + 1.
int64_t merge_sort_tile();
cudaError_t launch_merge_sort(int key_type, const void *in, const uint32_t *in_pay, int64_t N,
                              void *out, uint32_t *out_pay, void *tmp, uint32_t *tmp_pay,
                              int64_t *part, int32_t *status, cudaStream_t s);

// --- replacement.cu ---
// Tile of the warp pipelines (mark and compaction share their diagonals).
int64_t replacement_tile();
// Words of the merge bitmap for m + n positions (padded for whole-tile copies).
int64_t merge_bitmap_words(int64_t total);
// Partition (clears C) + mark; part_m: G + 1 co-ranks (A first on
// ties); part_c: G + 1 co-ranks of the compaction (B first on ties), or
// null; MB: the merge bitmap (merge_bitmap_words(m + n)), or null.
// clear[0, nclear): words (lookback states of a later kernel) the partition
// zeroes too.
cudaError_t launch_mark_tiles(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                              uint32_t *C, uint32_t *lb_B, uint32_t *MB, int64_t *part_m,
                              int64_t *part_c, int32_t *status, cudaStream_t s,
                              uint64_t *clear = nullptr, int64_t nclear = 0);
// Compaction; part_c: the mark's co-ranks (then MB is the mark's merge
// bitmap), or null to compute both from lb_B (co-ranks into part_scratch,
// G + 1; MB rebuilt).
cudaError_t launch_compact_tiles(int64_t m, int64_t n, const uint32_t *C, const uint32_t *dir,
                                 const uint32_t *lb_B, uint32_t *MB, const int64_t *part_c,
                                 int64_t *part_scratch, uint32_t *refs, uint32_t *ord_A,
                                 uint32_t *ord_B, int64_t *d_count, int32_t *status,
                                 cudaStream_t s);
// The same compaction reading R(i) from the rank2048 directory (co-ranks
// and merge bitmap from lb_B; part_scratch G + 1, MB merge_bitmap_words).
cudaError_t launch_compact_tiles_rank2048(int64_t m, int64_t n, const uint32_t *C,
                                          const uint64_t *dir, const uint64_t *epochs,
                                          const uint32_t *lb_B, uint32_t *MB, int64_t *part_scratch,
                                          uint32_t *refs, uint32_t *ord_A, uint32_t *ord_B,
                                          int64_t *d_count, int32_t *status, cudaStream_t s);
// The whole path (mark, rank512 build, compaction). part_m, part_c: G + 1
// each; MB: merge_bitmap_words(m + n); rank_ws: rank_build_ctas(m) uint64.
cudaError_t launch_replacement_merge_str(const lsm_bytes &A, int64_t m, const lsm_bytes &B,
                                         int64_t n, uint32_t *C, uint32_t *lb_B,
                                         uint64_t *prefixA, uint64_t *prefixB, uint32_t *dir,
                                         int64_t *d_total, uint32_t *refs, uint32_t *ord_A,
                                         uint32_t *ord_B, int64_t *d_count, int64_t *part_m,
                                         int64_t *part_c, uint32_t *MB, void *rank_ws,
                                         int32_t *status, cudaStream_t s);
int64_t replacement_str_tile();
cudaError_t launch_replacement_merge_one(const uint64_t *A, int64_t m, const uint64_t *B,
                                        int64_t n, uint32_t *C, uint32_t *lb_B, uint32_t *dir,
                                        int64_t *d_total, uint32_t *refs, uint32_t *ord_A,
                                        uint32_t *ord_B, int64_t *d_count, int64_t *part_m,
                                        uint64_t *state, void *rank_ws, int32_t *status,
                                        cudaStream_t s);
int64_t replacement_fused_tile();
cudaError_t launch_replacement_merge(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                    uint32_t *C, uint32_t *lb_B, uint32_t *dir, int64_t *d_total,
                                    uint32_t *refs, uint32_t *ord_A, uint32_t *ord_B,
                                    int64_t *d_count, int64_t *part_m, int64_t *part_c,
                                    uint32_t *MB, void *rank_ws, int32_t *status, cudaStream_t s);

// --- replace.cu ---
cudaError_t launch_collision_mark(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                  uint32_t *C, uint32_t *lb_B, int64_t *part_i, int32_t *status,
                                  cudaStream_t s);
cudaError_t launch_rank_build(const uint32_t *C, int64_t m, uint32_t *dir, int64_t *d_total,
                              uint32_t *cta_totals, cudaStream_t s);
// Workspace version: one launch (decoupled lookback) when the CTAs fit on
// the device at once, else count + finish. ws: rank_build_ctas(m) uint64;
// ws_clear: an earlier kernel on s has zeroed them for this call (else a
// memset node does).
cudaError_t launch_rank_build_ws(const uint32_t *C, int64_t m, uint32_t *dir, int64_t *d_total,
                                 void *ws, int32_t *status, cudaStream_t s, bool ws_clear = false);
cudaError_t launch_rank_query(const uint32_t *C, const uint32_t *dir, int64_t m,
                              const uint32_t *pos, int64_t q, uint32_t *out, int32_t *status,
                              cudaStream_t s);
cudaError_t launch_materialize(const uint64_t *A, const uint32_t *Aval, const uint32_t *tombA,
                               int64_t m, const uint64_t *B, const uint32_t *Bval,
                               const uint32_t *tombB, int64_t n, const uint32_t *refs,
                               const int64_t *d_count, uint64_t *out_keys, uint32_t *out_vals,
                               uint32_t *out_tomb, int32_t *status, cudaStream_t s);
// mb_scratch: merge_bitmap_words(m + n) uint32 (used by the default path).
cudaError_t launch_compact(int64_t m, int64_t n, const uint32_t *C, const uint32_t *dir,
                           const uint32_t *lb_B, uint32_t *refs, uint32_t *ord_A,
                           uint32_t *ord_B, int64_t *d_count, int64_t *part_i,
                           uint32_t *mb_scratch, int32_t *status, cudaStream_t s);
int64_t rank_build_ctas(int64_t m);
// The fused pass: collision bits, lb_B, ordinals, refs and the count in one
// tile pipeline. part_i: ceil((m+n)/fused_tile()) + 1 int64; state: as many
// uint64 tile states as tiles.
int64_t fused_tile();
cudaError_t launch_replacement_fused(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                     uint32_t *C, uint32_t *lb_B, uint32_t *refs, uint32_t *ord_A,
                                     uint32_t *ord_B, int64_t *d_count, int64_t *part_i,
                                     uint64_t *state, int32_t *status, cudaStream_t s);

// --- rank2048.cu ---
int64_t rank2048_build_ctas(int64_t m);
// ws: rank2048_build_ctas(m) uint64 of scratch (lookback states, or the
// per-CTA totals of the two-launch form).
cudaError_t launch_rank2048_build(const uint32_t *C, int64_t m, uint64_t *dir, uint64_t *epochs,
                                  int64_t *d_total, uint64_t *ws, int32_t *status, cudaStream_t s);
cudaError_t launch_rank2048_query(const uint32_t *C, const uint64_t *dir, const uint64_t *epochs,
                                  int64_t m, const uint64_t *pos, int64_t q, uint64_t *out,
                                  int32_t *status, cudaStream_t s);

// --- strings.cu ---
// prefixA / prefixB: optional key prefix tables (2 words per key), or NULL.
// The string mark that also writes the merge bitmap MB (bit p set when
// position p of the merge with B first on ties holds a B record) and the
// compaction's co-ranks at every cstep-th tile start (part_c, one more at the
// end); lb_B may be null. The partition also zeroes clear[0, nclear) (a
// later kernel's lookback states).
cudaError_t launch_collision_mark_str_mb(const lsm_bytes &A, int64_t m, const lsm_bytes &B,
                                         int64_t n, uint32_t *C, uint32_t *lb_B, uint64_t *prefixA,
                                         uint64_t *prefixB, int64_t *part_i, uint32_t *MB,
                                         int64_t *part_c, int cstep, int32_t *status,
                                         cudaStream_t s, uint64_t *clear = nullptr,
                                         int64_t nclear = 0);
cudaError_t launch_collision_mark_str(const lsm_bytes &A, int64_t m, const lsm_bytes &B, int64_t n,
                                      uint32_t *C, uint32_t *lb_B, uint64_t *prefixA,
                                      uint64_t *prefixB, int64_t *part_i, int32_t *status,
                                      cudaStream_t s);
constexpr int kMarkStrThreads = 128;
constexpr int kMarkStrItems = 7;

// --- fc.cu ---
int64_t fc_scan_tiles(int64_t N);
size_t fc_scan_workspace_bytes(int64_t N);
cudaError_t launch_fc_lengths_scan(const lsm_fc_input &in, const uint32_t *refs, int64_t N,
                                   uint32_t *lcp, uint32_t *ctrl, uint32_t *rec_bits,
                                   uint64_t *bit_off, void *ws, int32_t *status, cudaStream_t s);
cudaError_t launch_fc_emit(const lsm_fc_input &in, const uint32_t *refs, int64_t N,
                           const uint32_t *lcp, const uint32_t *ctrl, const uint64_t *bit_off,
                           uint32_t *payload, int64_t nwords, int32_t *status, cudaStream_t s);

// Offsets from per-record lengths: tile_sum[t] holds the total of records
// [t T, (t+1) T) (T = fc_tile_records()) on entry; the one-CTA tile scan and
// the offsets pass write off[0..N] (off[N] = the total).
int64_t fc_tile_records();
cudaError_t launch_fc_offsets(const uint32_t *rec, int64_t N, uint64_t *tile_sum, uint64_t *off,
                              cudaStream_t s);

// --- bytefc.cu ---
cudaError_t launch_bytefc_lengths_scan(const lsm_fc_input &in, const uint32_t *refs, int64_t N,
                                       uint64_t W, uint32_t *lcp, uint32_t *ctrl,
                                       uint32_t *rec_bytes, uint64_t *byte_off, void *ws,
                                       int32_t *status, cudaStream_t s);
// d_width: device uint64[4]; [0] receives the common width, [1..3] scratch.
cudaError_t launch_bytefc_value_width(const lsm_fc_input &in, const uint32_t *refs, int64_t N,
                                      uint64_t *d_width, cudaStream_t s);
cudaError_t launch_bytefc_emit(const lsm_fc_input &in, const uint32_t *refs, int64_t N, uint64_t W,
                               const uint32_t *lcp, const uint32_t *ctrl, const uint64_t *byte_off,
                               uint8_t *payload, int64_t nbytes, int32_t *status, cudaStream_t s);

// --- scatter.cu ---
cudaError_t launch_direct_scatter(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                  const uint32_t *C, const uint32_t *dir, const uint32_t *lb_B,
                                  uint32_t *refs, uint32_t *ord_A, uint32_t *ord_B,
                                  int64_t *d_count, int32_t *status, cudaStream_t s);

// --- ef.cu ---
// sizes: n entries, L, lows words, highs words, groups (host-only).
void ef_layout(int64_t N, uint64_t U, int64_t sizes[5]);
cudaError_t launch_ef_build(const uint64_t *bit_off, int64_t N, uint64_t w, uint64_t U,
                            uint64_t *lows, uint64_t *highs, uint64_t *samples, uint64_t *sparse,
                            int64_t *d_nsparse, int32_t *status, cudaStream_t s);

// --- validate.cu ---
// Sets *d_first to -1, then to the smallest t whose pair (t, t+1) breaks the
// order (strict: keys[t] < keys[t+1]; else keys[t] <= keys[t+1]); records
// LSM_ERR_UNSORTED in `status` when one does.
cudaError_t launch_validate_sorted(int key_type, const void *keys, int64_t count, int strict,
                                   int64_t *d_first, int32_t *status, cudaStream_t s);
cudaError_t launch_validate_sorted_str(const lsm_bytes &col, int64_t count, uint64_t arena_bytes,
                                       int strict, int64_t *d_first, int32_t *status,
                                       cudaStream_t s);

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// --- api.cu ---
cudaError_t launch_timeout_probe(int64_t limit_ns, int32_t *status, cudaStream_t s);
// Profiling hook (lsm_set_profile_events): record the pending start/stop
// events around a call's main kernel. No-ops when none are pending.
void profile_before(cudaStream_t s);
void profile_after(cudaStream_t s);

}  // namespace lsm
