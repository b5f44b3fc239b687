/*
 * lsmmerge.h -- C ABI of the GB300 merge-path replacement merge library.
 *
 * One shared library (liblsmmerge.so), hand-written CUDA kernels for sm_103a.
 * The operations follow these pages:
 *   [MP]   "Day 36: CUDA merge path: merging sorted arrays in parallel"
 *   [CH14] "Chapter 14: Merge Sort and Sample Sort", sections 14.1, 14.2
 *   [CB]   "Everett: collision bitmap and rank experiment"
 *   [GC]   "Everett: GPU construction experiment"
 *   [BP]   "Everett: byte-profile GPU merge"
 *
 * Conventions for every call
 *   - A is the older sorted input, B the newer one. Equal keys put A first
 *     ([GC], merge paragraph; [MP] "Exercise").
 *   - Pointers named d_* or described as device memory are CUDA device
 *     pointers owned by the caller; the library never allocates, frees or
 *     keeps them. Scratch comes from a caller workspace sized by
 *     lsm_workspace_size() ([CB] "Scratch space and likely costs": report the
 *     actual temporary capacities).
 *   - Sizes are int64_t element counts. Arrays of 8-byte keys, 4-byte
 *     payloads and workspaces must start on a 16-byte boundary (the kernels
 *     stage tiles with bulk asynchronous copies). Byte arenas must start on an
 *     8-byte boundary and stay readable up to the next multiple of 8 bytes
 *     past their last byte (keys are read in aligned 8-byte words; bytes past
 *     a key's end are masked off).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *     call is asynchronous on that stream and returns after launching.
 *   - Every call returns an lsm_status. Arguments are checked on the host
 *     before any launch; a call that returns an error launched nothing,
 *     except LSM_ERR_CUDA, which reports a failed launch.
 *   - Inputs are trusted to be sorted (and unique where stated), as the
 *     pages' parser trusts its accepted inputs ([BP] "Pipeline").
 *   - Bounded device waits: a kernel that waits (for a bulk copy or for a
 *     predecessor tile) gives up after about one second, records
 *     LSM_ERR_TIMEOUT in a sticky device status word and returns;
 *     lsm_get_device_status() reads it.
 *   - Stream capture: every call except lsm_get_device_status (which
 *     synchronizes) issues only kernel launches and memsets on `stream` and
 *     keeps no per-call host state, so a call captured into a CUDA graph can
 *     be replayed on new contents of the same buffers. Make one uncaptured
 *     call of each entry point first (it sets kernel attributes and looks up
 *     the device status word's address). Calls that find a
 *     prefix by a decoupled lookback over per-CTA state words in the
 *     workspace zero those words at every call, before the kernel that reads
 *     them, so the workspace rule below holds for them too.
 *   - Bitmaps hold bit t in 32-bit word t/32 at bit position t%32.
 *   - A reference is src<<31 | index with src 0 = A and src 1 = B.
 */
#ifndef LSMMERGE_H
#define LSMMERGE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define LSM_API __attribute__((visibility("default")))
#else
#define LSM_API
#endif

/* ---- status codes ------------------------------------------------------- */
enum {
  LSM_OK = 0,
  LSM_ERR_ARG = 1,       /* null pointer where data is needed, negative size */
  LSM_ERR_DTYPE = 2,     /* key type not supported by this call */
  LSM_ERR_OVERFLOW = 3,  /* sizes beyond the call's index range ([GC]: a 64-bit
                            bound check precedes every 32-bit scan) */
  LSM_ERR_CUDA = 4,      /* a CUDA launch or runtime call failed */
  LSM_ERR_TIMEOUT = 5,   /* a bounded device wait ran out (device status) */
  LSM_ERR_WORKSPACE = 6, /* workspace missing or smaller than required */
  LSM_ERR_ALIGN = 7,     /* a pointer misses its required alignment */
  LSM_ERR_UNSORTED = 8   /* only from the validators: an input breaks its order
                            (device status) */
};

/* Key types. */
enum { LSM_KEY_I32 = 1, LSM_KEY_U64 = 2 };

/* Operations, for lsm_workspace_size(). */
enum {
  LSM_OP_MERGE_STABLE = 1,
  LSM_OP_COLLISION_MARK = 2,
  LSM_OP_COLLISION_MARK_STR = 3,
  LSM_OP_RANK_BUILD = 4,
  LSM_OP_REPLACEMENT_COMPACT = 5,
  LSM_OP_FC_LENGTHS_SCAN = 6,
  LSM_OP_MERGE_SORT = 7,
  LSM_OP_RANK2048_BUILD = 8,
  LSM_OP_REPLACEMENT_FUSED = 9,
  LSM_OP_REPLACEMENT_MERGE = 10,
  LSM_OP_REPLACEMENT_MERGE_STR = 11
};

#define LSM_REF_FROM_B 0x80000000u
#define LSM_ORD_DROPPED 0xFFFFFFFFu

/* A byte-string column in CSR form: record t occupies
 * arena[off[t], off[t+1]). `off` holds count + 1 uint64 offsets. */
typedef struct {
  const uint8_t *arena;  /* device */
  const uint64_t *off;   /* device, count + 1 entries */
} lsm_bytes;

/* Inputs of the front-compression passes. Keys and values of both sources;
 * tombstone bitmaps may be NULL (no tombstones in that source). A value's
 * bytes are ignored when its record is a tombstone. prefixA and prefixB
 * are optional (both or neither): the key prefix tables that
 * lsm_collision_mark_str_prefix writes; with them lsm_fc_lengths_scan takes
 * each key's first 16 bytes from the table instead of the arena. */
typedef struct {
  lsm_bytes keyA, valA;
  const uint32_t *tombA; /* device bitmap, ceil(m/32) words, or NULL */
  int64_t m;
  lsm_bytes keyB, valB;
  const uint32_t *tombB; /* device bitmap, ceil(n/32) words, or NULL */
  int64_t n;
  const uint64_t *prefixA; /* device, 2 * m words, 16-byte aligned, or NULL */
  const uint64_t *prefixB; /* device, 2 * n words, 16-byte aligned, or NULL */
} lsm_fc_input;

/* ---- utilities ---------------------------------------------------------- */

/* Human-readable name of a status code (static string). */
LSM_API const char *lsm_status_string(int status);

/* Version of this ABI (major * 100 + minor). */
LSM_API int lsm_abi_version(void);

/* Reads the sticky device status word of the current device into
 * *host_status after synchronizing `stream`; resets it to LSM_OK when
 * `reset` is nonzero. Blocks the calling host thread. */
LSM_API int lsm_get_device_status(int32_t *host_status, int reset, void *stream);

/* Bytes of workspace that `op` needs for the given sizes (and key type for
 * LSM_OP_MERGE_STABLE). Host-only, never fails for valid sizes. The
 * workspace is scratch: its contents on entry are ignored and on exit are
 * unspecified. */
LSM_API int lsm_workspace_size(int op, int key_type, int64_t m, int64_t n, size_t *bytes);

/* ---- a1: merge path partition ------------------------------------------- */
/* [MP] "The merge matrix, and the diagonal that cuts it"; [CH14] "The
 * Concept, In Detail". For g = 0..G with G = ceil((m+n)/items_per_tile) and
 * k_g = min(g * items_per_tile, m + n), writes the co-rank of k_g:
 *   out_ij[2g]   = i, the number of A elements among the first k_g outputs
 *                  of the stable merge with A first on ties;
 *   out_ij[2g+1] = j = k_g - i.
 * A, B: device, sorted ascending, key_type elements (int32 compares signed).
 * out_ij: device, 2 * (G + 1) int64. items_per_tile >= 1. */
LSM_API int lsm_merge_path_partition(int key_type, const void *A, int64_t m, const void *B,
                                     int64_t n, int64_t items_per_tile, int64_t *out_ij,
                                     void *stream);

/* ---- a2: stable merge ---------------------------------------------------- */
/* [CH14] "The Sequential (CPU) Baseline" defines the result; [MP] the
 * partitioned form. Writes the m + n keys of A and B in ascending order,
 * A's element first when keys are equal, and, when Apay/Bpay/out_pay are all
 * non-NULL, each element's 32-bit payload beside it (payloads never take
 * part in comparisons). Apay/Bpay/out_pay must be all NULL or all non-NULL.
 * key_type: LSM_KEY_I32 or LSM_KEY_U64. out_keys must not alias the inputs.
 * ws: at least lsm_workspace_size(LSM_OP_MERGE_STABLE, key_type, m, n). */
LSM_API int lsm_merge_stable(int key_type, const void *A, const uint32_t *Apay, int64_t m,
                             const void *B, const uint32_t *Bpay, int64_t n, void *out_keys,
                             uint32_t *out_pay, void *ws, size_t ws_bytes, void *stream);

/* ---- f1: bottom-up merge sort -------------------------------------------- */
/* [CH14] section 14.2 "From Merge to Merge Sort: Repeated Pairwise Merging":
 * sorts N keys by passes of the stable merge above over adjacent runs whose
 * width doubles each pass (1, 2, 4, ...), the left run first on ties, so the
 * result is the stable sort: out_keys ascending, equal keys in input order,
 * and, when pay and out_pay are both non-NULL, each key's 32-bit payload
 * beside it (payloads never take part in comparisons; both NULL or both
 * non-NULL).
 * keys: device, N elements of key_type (LSM_KEY_I32 compares signed); pay:
 * device uint32[N] or NULL; out_keys / out_pay: device, N elements, must not
 * alias the inputs. All 16-byte aligned. N < 2^40. The input is not
 * modified. ws: at least lsm_workspace_size(LSM_OP_MERGE_SORT, key_type, N,
 * 0) bytes (one N-element copy of keys and payloads for the passes to
 * alternate with, plus the partition array). N = 0 returns LSM_OK. */
LSM_API int lsm_merge_sort(int key_type, const void *keys, const uint32_t *pay, int64_t N,
                           void *out_keys, uint32_t *out_pay, void *ws, size_t ws_bytes,
                           void *stream);

/* ---- a3: collision bitmap ------------------------------------------------- */
/* [CB] "Corrected record ordinals": for every B_j, lb_B[j] = lower_bound(A,
 * B_j), the number of A keys strictly less than B_j, and bit C_i is set
 * exactly when A_i == B_j for some j. The call clears C itself; bits at
 * positions >= m stay zero. A and B strictly increasing (unique keys).
 * A: device uint64[m]; B: device uint64[n]; C: device uint32[ceil(m/32)];
 * lb_B: device uint32[n]. A, B and lb_B 16-byte aligned. m, n < 2^31. */
LSM_API int lsm_collision_mark(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                               uint32_t *C, uint32_t *lb_B, void *ws, size_t ws_bytes,
                               void *stream);

/* Same for byte-string keys in unsigned lexicographic order, a proper prefix
 * first ([GC], prefix-cache paragraph). A and B are CSR columns of m and n
 * strictly increasing keys. */
LSM_API int lsm_collision_mark_str(const lsm_bytes *A, int64_t m, const lsm_bytes *B, int64_t n,
                                   uint32_t *C, uint32_t *lb_B, void *ws, size_t ws_bytes,
                                   void *stream);

/* lsm_collision_mark_str, and also the key prefix tables the call holds
 * anyway: for key t of A, prefixA[2t] and prefixA[2t+1] are its bytes 0..7
 * and 8..15 read as big-endian words, zero past the key's end (likewise
 * prefixB for B). They serve lsm_fc_lengths_scan through lsm_fc_input
 * (the LCP of two keys then needs no key bytes unless their first 16 bytes
 * agree). prefixA: device uint64[2m], prefixB: device uint64[2n], both
 * 16-byte aligned; either may be NULL (that table is not written). */
LSM_API int lsm_collision_mark_str_prefix(const lsm_bytes *A, int64_t m, const lsm_bytes *B,
                                          int64_t n, uint32_t *C, uint32_t *lb_B,
                                          uint64_t *prefixA, uint64_t *prefixB, void *ws,
                                          size_t ws_bytes, void *stream);

/* ---- a4: rank512 directory ------------------------------------------------ */
/* [CB] "Temporary rank layouts" and "Corrected record ordinals". Over the
 * bitmap C of m bits (tail bits zero) builds floor(m/512) + 1 entries of
 * three uint32 each:
 *   dir[3b]                       R(512 b), R(i) = sum_{t<i} C_t
 *   dir[3b+1] | dir[3b+2] << 32   sub-prefix s = 1..7 in bits [9(s-1), 9s):
 *                                 R(512 b + 64 s) - R(512 b)
 * (positions past m count as m), and d_total[0] = R(m).
 * C: device uint32[ceil(m/32)]; dir: device uint32[3 * (m/512 + 1)];
 * d_total: device int64[1]. m < 2^31. At least one block is always built, so
 * an empty A yields dir = {0,0,0} and R(0) = 0 ([CB] "Dispatch bindings"). */
LSM_API int lsm_rank_build(const uint32_t *C, int64_t m, uint32_t *dir, int64_t *d_total,
                           void *ws, size_t ws_bytes, void *stream);

/* Allocation-free variant of lsm_rank_build, for callers that cannot call
 * cudaMalloc or hand the library a workspace: code on a latency-critical path
 * where a device allocation (which may block and synchronize the device) is
 * not allowed after start-up, or a plug-in whose host program owns every
 * device buffer through its own pool. The pages have no counterpart; this is
 * a property of this library's interface, not of the method.
 * Same arguments and results as lsm_rank_build without the workspace: the
 * per-CTA totals live in a 16 KB static device array inside the library, so
 * the call allocates nothing. Limits and rules:
 *   - m <= 2^29 - 1 (536,870,911 bit positions); larger m returns
 *     LSM_ERR_OVERFLOW before anything is launched.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture. The address is kept for the life of the
 *     process: after cudaDeviceReset (or anything else that destroys the
 *     device's primary context) it is stale, so do not call this entry point
 *     on that device again after a reset.
 *   - Every call on a device shares the one array: calls that may overlap on
 *     the GPU (different streams, or different host threads) race and must be
 *     ordered by the caller. Each call rewrites every entry it reads, so the
 *     contents left by an earlier call never matter. */
LSM_API int lsm_rank_build_noalloc(const uint32_t *C, int64_t m, uint32_t *dir, int64_t *d_total,
                                   void *stream);

/* Rank queries: out[t] = R(pos[t]) for pos[t] in [0, m], using the directory,
 * at most one preceding 32-bit word and the masked current word ([CB]
 * "Temporary rank layouts"). A position above m yields 0xFFFFFFFF and
 * records LSM_ERR_ARG in the device status. pos, out: device uint32[q]. */
LSM_API int lsm_rank_query(const uint32_t *C, const uint32_t *dir, int64_t m,
                           const uint32_t *pos, int64_t q, uint32_t *out, void *stream);

/* ---- f3: rank2048 directory ---------------------------------------------- */
/* [CB] "Temporary rank layouts": the other temporary layout, one 8-byte
 * entry per 2048 bits with three packed populations of its 512-bit runs and
 * absolute counts at epochs of 2^32 bits; [CB] "Scratch space and likely
 * costs": (1/8 + 8/2048)|A| bytes with the bitmap. Layout (the pages give the
 * contents, this packing is a reading):
 *   epochs[e], e = 0..floor(m/2^32):  R(2^32 e)
 *   dir[b],    b = 0..floor(m/2048):  bits 0..31 = R(2048 b) - epochs[2048 b
 *     >> 32]; bits 32+10r..41+10r = population of bits [2048b + 512r,
 *     2048b + 512(r+1)) for r = 0, 1, 2; bits 62..63 zero.
 * R(i) = number of set bits of C below i. *d_total = R(m).
 * C: device uint32[ceil(m/32)], 16-byte aligned, bits at positions >= m zero.
 * dir: device uint64[floor(m/2048)+1]; epochs: device uint64[floor(m/2^32)+1];
 * d_total: device int64. m < 2^36. ws: at least
 * lsm_workspace_size(LSM_OP_RANK2048_BUILD, 0, m, 0) bytes. */
LSM_API int lsm_rank2048_build(const uint32_t *C, int64_t m, uint64_t *dir, uint64_t *epochs,
                               int64_t *d_total, void *ws, size_t ws_bytes, void *stream);

/* out[t] = R(pos[t]) from the rank2048 directory: the epoch, the entry's
 * count, the earlier runs' populations, then popcounts of the current run's
 * words before pos[t] and of the masked word holding it. pos[t] in [0, m]
 * (EOF allowed); a position past m yields UINT64_MAX and records LSM_ERR_ARG
 * in the device status word. pos, out: device uint64[q]. */
LSM_API int lsm_rank2048_query(const uint32_t *C, const uint64_t *dir, const uint64_t *epochs,
                               int64_t m, const uint64_t *pos, int64_t q, uint64_t *out,
                               void *stream);

/* ---- a5: replacement merge by bitmap, rank and merge path ----------------- */
/* [CB] "The three experimental paths" (bitmap, compact A, then Merge Path)
 * and "Corrected record ordinals"; [GC] merge paragraph (keep the newer
 * record; a newer tombstone remains a record). From the outputs of
 * lsm_collision_mark (C, lb_B) and lsm_rank_build (dir) writes
 *   out_refs[0..N)  the surviving records in merged order, N = m + n - R(m)
 *   ord_A[i]        i + lower_bound(B, A_i) - R(i) for a surviving A_i,
 *                   LSM_ORD_DROPPED when C_i = 1
 *   ord_B[j]        j + lb_B[j] - R(lb_B[j])
 *   d_count[0]      N
 * The keys themselves are not read: B_j precedes A_i in the merge exactly
 * when lb_B[j] <= i, so the merge path runs over positions: B_j sits at
 * position j + lb_B[j] of the merge with B first on ties, and the call marks
 * those positions in a bitmap in its workspace (a lb_B that is not
 * nondecreasing with values <= m records LSM_ERR_ARG) before the tiles read
 * it.
 * out_refs: device uint32[m + n] capacity; ord_A: uint32[m]; ord_B:
 * uint32[n]; d_count: int64[1]; C, lb_B, out_refs, ord_A and ord_B 16-byte
 * aligned. m, n < 2^31. */
LSM_API int lsm_replacement_merge_compact(int64_t m, int64_t n, const uint32_t *C,
                                          const uint32_t *dir, const uint32_t *lb_B,
                                          uint32_t *out_refs, uint32_t *ord_A, uint32_t *ord_B,
                                          int64_t *d_count, void *ws, size_t ws_bytes,
                                          void *stream);

/* The whole replacement merge, a3 + a4 + a5, in one call: the outputs of
 * lsm_collision_mark, lsm_rank_build and lsm_replacement_merge_compact in
 * turn (C, lb_B, dir, *d_total = R(m), out_refs, ord_A, ord_B, *d_count = m
 * + n - R(m)), by the same steps: the collision mark over merge-path tiles of
 * the keys ([CB] "Corrected record ordinals"), the rank512 build ([CB]
 * "Temporary rank layouts") and the compaction by merge path over positions
 * ([CB] "The three experimental paths", third path), with the compaction's
 * tiles on the mark's diagonals, so that the mark hands the compaction its
 * co-ranks and no second partition is needed. Arguments, alignment and
 * limits as those three calls; C needs no clearing. lb_B may be null: the
 * lower bounds are scratch on this path (the compaction reads the merge
 * bitmap), and a null lb_B leaves them unwritten. ws: at least
 * lsm_workspace_size(LSM_OP_REPLACEMENT_MERGE, 0, m, n) bytes. */
LSM_API int lsm_replacement_merge(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                  uint32_t *C, uint32_t *lb_B, uint32_t *dir, int64_t *d_total,
                                  uint32_t *out_refs, uint32_t *ord_A, uint32_t *ord_B,
                                  int64_t *d_count, void *ws, size_t ws_bytes, void *stream);

/* a3 + a4 + a5 in one call: the same outputs as lsm_collision_mark,
 * lsm_rank_build and lsm_replacement_merge_compact in turn (C, lb_B, dir,
 * *d_total = R(m), out_refs, ord_A, ord_B, *d_count = m + n - R(m)), from
 * one pass over merge-path tiles of the keys ([GC] merge paragraph: a
 * partitioned merge whose neighbouring-key comparison and scan keep the
 * newer record of each equal-key run) plus the rank512 build over C. Each
 * tile finds its lower bounds and collision bits on staged keys and places
 * its records at the ordinals of [CB] "Corrected record ordinals", taking
 * R of its first A record from a decoupled lookback over the tiles'
 * collision counts. Arguments, alignment and limits as those three calls;
 * C needs no clearing. ws: at least
 * lsm_workspace_size(LSM_OP_REPLACEMENT_FUSED, 0, m, n) bytes. */
LSM_API int lsm_replacement_merge_fused(const uint64_t *A, int64_t m, const uint64_t *B, int64_t n,
                                        uint32_t *C, uint32_t *lb_B, uint32_t *dir,
                                        int64_t *d_total, uint32_t *out_refs, uint32_t *ord_A,
                                        uint32_t *ord_B, int64_t *d_count, void *ws,
                                        size_t ws_bytes, void *stream);

/* The same compaction, reading R(i) from the rank2048 directory
 * (lsm_rank2048_build) instead of the rank512 one: [CB] "Suggested separate
 * modes" (collision512 against collision2048) compares the two layouts
 * inside the whole pipeline. Every output equals lsm_replacement_merge_compact's.
 * dir, epochs: device, as lsm_rank2048_build wrote them for this C and m.
 * Other arguments, limits and the workspace as lsm_replacement_merge_compact
 * (ws sized by LSM_OP_REPLACEMENT_COMPACT). */
LSM_API int lsm_replacement_merge_compact_rank2048(int64_t m, int64_t n, const uint32_t *C,
                                                   const uint64_t *dir, const uint64_t *epochs,
                                                   const uint32_t *lb_B, uint32_t *out_refs,
                                                   uint32_t *ord_A, uint32_t *ord_B,
                                                   int64_t *d_count, void *ws, size_t ws_bytes,
                                                   void *stream);

/* [CB] "The three experimental paths", the tiled direct scatter: each thread
 * takes 32 consecutive A records, finds lower_bound(B, A_i) for the first by
 * one binary search and for the rest by advancing a cursor through B, and
 * every record scatters to its corrected ordinal ([CB] "Corrected record
 * ordinals": i + lower_bound(B, A_i) - R(i) for a surviving A_i, j + lb_B[j]
 * - R(lb_B[j]) for B_j): ord_A[i] (0xFFFFFFFF when dropped), ord_B[j] and
 * out_refs[ordinal] = the record's reference. *d_count = m + n - R(m). Every
 * output equals lsm_replacement_merge_compact's; this path reads the keys
 * again where the compaction reads only lb_B and C. A, B: the keys given to
 * lsm_collision_mark; C, lb_B: its outputs; dir: lsm_rank_build's. A record
 * whose ordinal would fall outside [0, N) (inputs that break the contract)
 * records LSM_ERR_ARG in the device status word and writes no ref. All
 * arrays 16-byte aligned; m, n < 2^31. One launch; no workspace. */
LSM_API int lsm_replacement_direct_scatter(const uint64_t *A, int64_t m, const uint64_t *B,
                                           int64_t n, const uint32_t *C, const uint32_t *dir,
                                           const uint32_t *lb_B, uint32_t *out_refs,
                                           uint32_t *ord_A, uint32_t *ord_B, int64_t *d_count,
                                           void *stream);

/* Materialized survivors of the replacement merge ([GC] merge paragraph: of
 * each equal-key run the newer record is kept, and a newer tombstone stays a
 * record). For t < N = d_count[0] (the count lsm_replacement_merge_compact
 * wrote), record t is the source record out_refs[t] names:
 *   out_keys[t]   its key
 *   out_vals[t]   its 32-bit value (when Aval, Bval and out_vals are given)
 *   out_tomb      bit t (bit t%32 of word t/32) = its tombstone flag; the
 *                 words covering [0, N) are written, bits past N zero.
 * tombA / tombB: tombstone bitmaps of the inputs (bit i of word i/32), each
 * may be NULL (no tombstones in that input); out_tomb may be NULL. Records
 * t >= N are not touched. All pointers are device pointers; A, B, refs,
 * out_keys and out_vals 16-byte aligned; out_keys and out_vals hold m + n
 * entries, out_tomb ceil((m + n) / 32) words. m, n < 2^31. No workspace. */
LSM_API int lsm_replacement_materialize(const uint64_t *A, const uint32_t *Aval,
                                        const uint32_t *tombA, int64_t m, const uint64_t *B,
                                        const uint32_t *Bval, const uint32_t *tombB, int64_t n,
                                        const uint32_t *refs, const int64_t *d_count,
                                        uint64_t *out_keys, uint32_t *out_vals,
                                        uint32_t *out_tomb, void *stream);

/* ---- a6: front-compression lengths and bit offsets ----------------------- */
/* [GC], the control-argument equation and the record-length formula. For
 * output record i (refs[i] names its key and value):
 *   lcp[i]      l_i, exact bit LCP with record i-1's key, l_0 = 0, clamped
 *               to the shorter key
 *   ctrl[i]     c_i = 1 + l_i when i mod 15 = 0, else k_{i-1} - l_i
 *   rec_bits[i] E(c_i) + E(k_i - l_i) + (k_i - l_i) + v_i, E(x) =
 *               2 floor(log2(x+1)) + 1, v_i = 1 for a tombstone, else
 *               1 + E(byte length) + 8 * byte length
 *   bit_off[i]  sum_{t<i} rec_bits[t], for i = 0..N (bit_off[N] = total)
 * Keys are byte strings; k_i = 8 * byte length. refs: device uint32[N];
 * lcp, ctrl, rec_bits: device uint32[N]; bit_off: device uint64[N + 1].
 * N < 2^31. A record whose fields exceed 32 bits records LSM_ERR_OVERFLOW in
 * the device status. */
LSM_API int lsm_fc_lengths_scan(const lsm_fc_input *in, const uint32_t *refs, int64_t N,
                                uint32_t *lcp, uint32_t *ctrl, uint32_t *rec_bits,
                                uint64_t *bit_off, void *ws, size_t ws_bytes, void *stream);

/* ---- a7: word-owned payload emit ------------------------------------------ */
/* [GC], the paragraphs on exact lengths and on the record layout, and the
 * word-owned emit: each final 32-bit payload word is written to global
 * memory exactly once, by its owner. The owner is a CTA rather than a
 * thread: each CTA owns contiguous runs of 8192 payload words, composes a
 * run in shared memory with one thread per record (fields written into the
 * run's words, words that two fields or records share combined with a
 * shared-memory OR) and moves the finished run to global memory with one
 * bulk store. Measured on the 4M + 4M string workload: one thread per
 * output word gathering its bits took 1130 us, this form 302 us. Record i
 * occupies bits [bit_off[i],
 * bit_off[i+1]) as EG0(c_i) EG0(k_i - l_i) key bits [l_i, k_i) value, value
 * = 0 for a tombstone, else 1 EG0(byte length) bytes; EG0(x) is
 * floor(log2(x+1)) zero bits followed by x+1 in binary. Stream bit t is bit
 * 31 - t%32 of payload[t/32] (MSB first). All nwords words are written;
 * bits past bit_off[N] are zero. nwords must be >= ceil(bit_off[N] / 32)
 * (the host reads bit_off[N] once to size the payload); payload: device
 * uint32[nwords], 16-byte aligned. */
LSM_API int lsm_fc_emit(const lsm_fc_input *in, const uint32_t *refs, int64_t N,
                        const uint32_t *lcp, const uint32_t *ctrl, const uint64_t *bit_off,
                        uint32_t *payload, int64_t nwords, void *stream);

/* ---- f4: byte-profile front compression ---------------------------------- */
/* [BP] "Pipeline": the byte profile's records carry byte LEB128 counts, FC
 * literals and optional-value tags, with 15-record blocks, and a common
 * encoded value width leaves the value length out ("width seventeen means a
 * one-byte presence tag and sixteen payload bytes"). The pages do not print
 * the record grammar; this library reads it as the bit profile's record
 * ([GC] control-argument equation) in bytes, with LEB128 in place of EG0:
 *   p_i = byte LCP with record i-1's key (p_0 = 0), K_i = key length;
 *   b_i = 1 + p_i when i mod 15 = 0, else K_{i-1} - p_i;
 *   record = LEB128(b_i) LEB128(K_i - p_i) key bytes [p_i, K_i), then tag
 *   byte 0 for a tombstone, or tag 1, LEB128(value length) and the value
 *   bytes; under a common width W > 0 every record must be present with a
 *   (W - 1)-byte value and the length is left out.
 * LEB128 is unsigned: seven bits per byte, low group first, the top bit set
 * on every byte but the last. Records follow each other with no padding.
 * Inputs as lsm_fc_lengths_scan's; with the prefix tables, p_i comes from
 * the keys' first 16 bytes there (their first differing byte, clamped to the
 * shorter key), the arenas being read only when both keys are longer than
 * 16 bytes and those agree.
 * lsm_bytefc_lengths_scan writes lcp[i] = p_i, ctrl[i] = b_i, rec_bytes[i]
 * (the record's bytes) and byte_off[0..N] (exclusive scan, byte_off[N] =
 * the payload's bytes); rec_bytes and byte_off 16-byte aligned; ws sized by
 * LSM_OP_FC_LENGTHS_SCAN for N. A tombstone or a value of another length
 * under W > 0 records LSM_ERR_ARG, a record past 2^32 bytes
 * LSM_ERR_OVERFLOW, in the device status word. */
LSM_API int lsm_bytefc_lengths_scan(const lsm_fc_input *in, const uint32_t *refs, int64_t N,
                                    uint64_t W, uint32_t *lcp, uint32_t *ctrl,
                                    uint32_t *rec_bytes, uint64_t *byte_off, void *ws,
                                    size_t ws_bytes, void *stream);

/* The common encoded value width of the merged records, detected before they
 * are sized ([BP] "Pipeline"; "seventeen" there is a one-byte presence tag
 * and sixteen payload bytes): d_width[0] = 1 + L when every record that refs
 * names (N of them) is present, not a tombstone, and every one of their
 * values has L bytes; otherwise 0, and 0 for N = 0. Inputs that vary (other
 * lengths, tombstones) can merge into an output of one width when the newer
 * records replace the odd ones. d_width: device uint64[4], 8-byte aligned;
 * elements 1..3 are scratch. The caller reads d_width[0] (one host read, as
 * for the payload size) and passes it as W to lsm_bytefc_lengths_scan and
 * lsm_bytefc_emit. */
LSM_API int lsm_bytefc_value_width(const lsm_fc_input *in, const uint32_t *refs, int64_t N,
                                   uint64_t *d_width, void *stream);

/* Writes the payload: record i's bytes at [byte_off[i], byte_off[i+1]) of
 * payload (device, nbytes >= byte_off[N], any alignment); bytes past
 * byte_off[N] are not written. lcp, ctrl, byte_off: lsm_bytefc_lengths_scan's
 * outputs for the same inputs and W. Each CTA takes 256 consecutive records,
 * whose bytes form one contiguous span: one thread per record composes it in
 * shared memory (records never share a byte) and the span leaves with one
 * bulk store plus at most 15 plain bytes at either end. A record whose
 * offsets, lcp or control do not give exactly its own length records
 * LSM_ERR_ARG; its bytes read as zero. */
LSM_API int lsm_bytefc_emit(const lsm_fc_input *in, const uint32_t *refs, int64_t N, uint64_t W,
                            const uint32_t *lcp, const uint32_t *ctrl, const uint64_t *byte_off,
                            uint8_t *payload, int64_t nbytes, void *stream);

/* ---- f2: Elias-Fano navigation over the record offsets ------------------- */
/* [GC] "GPU construction experiment": physical offsets sampled at ordinals
 * 0, 15, 30, ... plus EOF; with a common encoded value width w every entry
 * subtracts w times its ordinal; the sections are EF lows, highs, select
 * samples and sparse exceptions, a 256-entry group being sparse when its
 * high-position span is at least 4096 bits. The pages fix these contents;
 * the bit layout is this library's reading (textbook Elias-Fano):
 *   entries  x_s = bit_off[15 s] - 15 s w for s < n - 1, and
 *            x_{n-1} = bit_off[N] - N w;  n = ceil(N/15) + 1;  U = x_{n-1}
 *   L        the largest L with n 2^L <= U (0 when U < n)
 *   lows     x_s mod 2^L at bits [sL, sL+L) (bit t = bit t%64 of word t/64)
 *   highs    bit (x_s >> L) + s set for every s, (U >> L) + n bits
 *   samples  per group g of entries [256g, min(256g+256, n)):
 *            samples[2g] = high position of entry 256g; samples[2g+1] =
 *            e_g << 1 | sparse_g, e_g = entries of sparse groups before g
 *   sparse   the high position of every entry of each sparse group, in order
 * Every unused bit of every word is zero. */

/* Host-only sizes for N records and U = bit_off[N] - N w: sizes[0] = n,
 * [1] = L, [2] = lows uint64 words, [3] = highs uint64 words, [4] = groups
 * (samples take 2 * groups uint64; sparse at most n uint64). */
LSM_API int lsm_ef_sizes(int64_t N, uint64_t U, int64_t *sizes);

/* Builds the four sections from bit_off (device uint64[N+1], nondecreasing,
 * as lsm_fc_lengths_scan wrote it) and writes the number of sparse entries
 * to *d_nsparse (device int64). w: the common value width in bits (0 when
 * widths differ); every record must be at least w bits long. U must equal
 * bit_off[N] - N w (the host reads bit_off[N] to size the sections); when
 * it does not, LSM_ERR_ARG is recorded in the device status word and no
 * write leaves the sections. lows, highs, samples: device, sized by
 * lsm_ef_sizes (lows may be NULL when it has no words); sparse: device,
 * n uint64. All 8-byte aligned. N < 2^31. Two launches. */
LSM_API int lsm_fc_ef_build(const uint64_t *bit_off, int64_t N, uint64_t w, uint64_t U,
                            uint64_t *lows, uint64_t *highs, uint64_t *samples, uint64_t *sparse,
                            int64_t *d_nsparse, void *stream);

/* ---- input validation ----------------------------------------------------- */
/* The merge and replacement calls trust their inputs' order, as the pages'
 * parser trusts its accepted inputs ([BP] "Pipeline": it checks framing,
 * tags, offset bounds and retained lengths, not order). A caller that cannot
 * vouch for an input runs one of these first. Each sets *d_first to -1 and
 * then, on the device, to the smallest t whose pair (t, t+1) breaks the
 * order, and records LSM_ERR_UNSORTED in the sticky device status word
 * (lsm_get_device_status) when one does; nothing traps or faults.
 *   strict = 1: strictly increasing (the unique-key inputs of the
 *               replacement calls); strict = 0: nondecreasing (the inputs of
 *               lsm_merge_stable).
 * keys: device, count elements of key_type (int32 compares signed), aligned
 * to the element size. d_first: device int64[1]. count < 2 leaves -1. */
LSM_API int lsm_validate_sorted(int key_type, const void *keys, int64_t count, int strict,
                                int64_t *d_first, void *stream);

/* The same for a byte-string column (unsigned lexicographic order, a proper
 * prefix first). arena_bytes is the arena's length: a pair whose offsets are
 * out of order or past arena_bytes counts as a violation and its bytes are
 * not read, so malformed offsets cannot cause an out-of-bounds access. With
 * count = 1 the key's two offsets are checked. keys: as in lsm_bytes (arena
 * 8-byte aligned and readable up to the next multiple of 8 bytes). */
LSM_API int lsm_validate_sorted_str(const lsm_bytes *keys, int64_t count, uint64_t arena_bytes,
                                    int strict, int64_t *d_first, void *stream);

/* ---- tuning ----------------------------------------------------------------- */
/* Selects the tile configuration of lsm_merge_stable for a key type:
 * items_per_thread E (a tile is 256 E outputs), `stages` input tiles kept in
 * flight per CTA, `out_tiles` output tiles (1 or 2). Compiled configurations
 * (E, stages, out_tiles): (5,2,1) (7,2,1) (11,2,1) (15,2,1) (7,4,2) (11,3,2)
 * (15,2,2) (7,3,1); any other returns LSM_ERR_ARG. Process-wide, read at each
 * call; the default is (11,2,1). E is the slice-size knob of [MP] "Measuring
 * it against one thread" and "Results". */
LSM_API int lsm_tune_merge(int key_type, int items_per_thread, int stages, int out_tiles);

/* Profiling hook: the next call that launches a tile kernel (merge_stable,
 * collision_mark, collision_mark_str, rank_build, replacement_merge_compact,
 * fc_lengths_scan, fc_emit) records the CUDA event `start_event` on its
 * stream just before its main kernel and `stop_event` just after it (for
 * rank_build: around both of its kernels), then forgets both events.
 * Process-wide, one-shot; pass NULL, NULL to cancel. The events are
 * cudaEvent_t handles owned by the caller. */
LSM_API int lsm_set_profile_events(void *start_event, void *stop_event);

/* Selects how lsm_collision_mark (kernel 0) or
 * lsm_replacement_merge_compact (kernel 1) run: (0, 0) selects the warp
 * pipelines that lsm_replacement_merge also uses (the default); threads per
 * CTA and items per thread from the set (256,11) (128,23) (256,23) (512,11)
 * select the earlier block-synchronous tile pipelines, kept for comparison.
 * Process-wide. */
LSM_API int lsm_tune_replace(int kernel, int threads, int items_per_thread);

/* Selects the form of lsm_replacement_merge: mode 0 (the default) runs the
 * mark and the compaction as two tile pipelines with the rank512 build
 * between them; mode 1 runs the mark and the compaction of each tile in one
 * persistent kernel (warp roles: a loader, mark warps, a lookback warp that
 * finds R at the tile's first A record from the collision counts the mark
 * warps publish, compaction warps), the tile's merge bitmap and collision
 * bits handed over in shared memory, then the rank512 build. Both give the
 * same outputs; mode 1 measured slower on the 12M + 4M workload (95.9 us
 * against 87.7 us per step). Process-wide; other modes return
 * LSM_ERR_ARG. */
LSM_API int lsm_tune_replacement_merge(int mode);

/* The whole replacement merge for byte-string keys in one call: the outputs
 * of lsm_collision_mark_str_prefix, lsm_rank_build and
 * lsm_replacement_merge_compact in turn (C, lb_B and the prefix tables when
 * given, dir, *d_total = R(m), out_refs, ord_A, ord_B, *d_count = m + n -
 * R(m)), by the same steps; the string mark also records the merge with B
 * first on ties as a bitmap and the compaction's co-ranks at every fourth of
 * its tile boundaries, so that the compaction needs no partition and no
 * lower bounds ([CB] "The three experimental paths", third path). Arguments,
 * alignment and limits as those calls; C needs no clearing; lb_B, prefixA
 * and prefixB may be NULL (then not written). ws: at least
 * lsm_workspace_size(LSM_OP_REPLACEMENT_MERGE_STR, 0, m, n) bytes. */
LSM_API int lsm_replacement_merge_str(const lsm_bytes *A, int64_t m, const lsm_bytes *B, int64_t n,
                                      uint32_t *C, uint32_t *lb_B, uint64_t *prefixA,
                                      uint64_t *prefixB, uint32_t *dir, int64_t *d_total,
                                      uint32_t *out_refs, uint32_t *ord_A, uint32_t *ord_B,
                                      int64_t *d_count, void *ws, size_t ws_bytes, void *stream);

/* ---- test hook ------------------------------------------------------------ */
/* Launches one block that waits, with the same bounded wait the kernels
 * use, on a device flag that nothing ever sets, and gives up after
 * limit_ns nanoseconds (clamped to [1 us, 1 s]). The wait runs out by
 * design: LSM_ERR_TIMEOUT is recorded in the device status word, the kernel
 * returns and the CUDA context stays usable. Exists so that tests can check
 * the timeout path without faulting or hanging a GPU. */
LSM_API int lsm_debug_timeout_probe(int64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LSMMERGE_H */
