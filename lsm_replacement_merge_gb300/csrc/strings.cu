// strings.cu -- collision bitmap and lower bounds for byte-string keys.
//
// The same merge-path tiling as the uint64 collision mark ("Everett:
// collision bitmap and rank experiment", "Corrected record ordinals"). A
// partition launch finds the co-rank of each tile boundary (A first on
// ties), comparing keys in place in their arenas (strings.cuh). Each tile
// then stages its keys' prefix caches ("Everett: GPU construction
// experiment", prefix-cache paragraph: the first 16 bytes, zero-padded, and
// the length) in shared memory; each thread bisects its own diagonal and
// walks E merge steps, one comparison per step, on the cached prefixes. For
// each B element it records the lower bound (A elements before it, minus
// one when the element just before it is an equal A key); for each A
// element it sets C_i when the B key at the head equals it. Bits are
// gathered per tile in shared memory; words inside the tile's A range take
// plain stores, boundary words atomicOr into the bitmap the partition
// launch cleared. The tile can also write its keys' cached prefixes out (the
// key prefix tables of the front-compression lengths pass).
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
    return key_cmp_prefix16(key_at(A, i), key_at(B, k - i - 1)) <= 0;
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
                                                            int64_t nclear,
                                                            uint64_t *__restrict__ clear_states,
                                                            int64_t nstates) {
  pdl_begin();
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t w = gtid; w < nclear; w += stride) clear_words[w] = 0u;
  for (int64_t w = gtid; w < nstates; w += stride) clear_states[w] = 0u;
  const int64_t g = gtid / kStrPartitionLanes;
  const bool active = g <= G;
  const int64_t total = m + n;
  const int64_t k = active ? (g * D < total ? g * D : total) : 0;
  const int64_t i = group_corank<kStrPartitionLanes>(pred, k, m, n, active);
  if (active && (threadIdx.x & (kStrPartitionLanes - 1)) == 0) out_i[g] = i;
}

// Bytes [16, len) of two keys that agree on their first 16 bytes and are
// both longer than 16, by one lane: 32 bytes a round with the eight
// windows' loads issued together, so keys up to 48 bytes take one round.
__device__ __forceinline__ int key_cmp_tail16(const uint8_t *pa, uint64_t ba, uint64_t la,
                                              const uint8_t *pb, uint64_t bb, uint64_t lb) {
  const uint64_t l = la < lb ? la : lb;
  for (uint64_t t = 16; t < l; t += 32) {
    uint64_t x[4], y[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint64_t p = t + 8 * q;
      x[q] = p < l ? load_be64(pa, ba + p, ba + l) : 0;
      y[q] = p < l ? load_be64(pb, bb + p, bb + l) : 0;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (x[q] != y[q]) return x[q] < y[q] ? -1 : 1;
  }
  return la == lb ? 0 : (la < lb ? -1 : 1);
}

// Settles the order of two keys that agree on their first 16 bytes and are
// both longer than 16, for every lane of the warp with `tail` set; `c` is
// returned unchanged on the other lanes. All 32 lanes call it together. The
// warp takes up to four such pairs a round, eight lanes a pair and one
// 8-byte window a lane, so a pair whose shorter key ends within 80 bytes
// costs one round of loads, and no lane compares alone.
__device__ __forceinline__ int warp_tail_cmp(bool tail, int c, const uint8_t *arenaA, uint64_t ba,
                                             uint64_t la, const uint8_t *arenaB, uint64_t bb,
                                             uint64_t lb) {
  constexpr unsigned kAll = 0xffffffffu;
  unsigned pend = __ballot_sync(kAll, tail);
  const int lane = threadIdx.x & 31, grp = lane >> 3, sub = lane & 7;
  while (pend) {
    int src = -1;  // the lane whose pair this lane's group settles
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (pend) {
        if (q == grp) src = __ffs(pend) - 1;
        pend &= pend - 1;
      }
    }
    const int from = src < 0 ? lane : src;
    const uint64_t gba = __shfl_sync(kAll, ba, from), gla = __shfl_sync(kAll, la, from);
    const uint64_t gbb = __shfl_sync(kAll, bb, from), glb = __shfl_sync(kAll, lb, from);
    const uint64_t l = gla < glb ? gla : glb;
    bool done = src < 0;
    int res = 0;
    for (uint64_t t = 16; !__all_sync(kAll, done); t += 64) {
      const uint64_t p = t + 8 * sub;
      const bool in = !done && p < l;
      uint64_t x = 0, y = 0;
      if (in) {
        x = load_be64(arenaA, gba + p, gba + l);
        y = load_be64(arenaB, gbb + p, gbb + l);
      }
      const unsigned gdiff = (__ballot_sync(kAll, in && x != y) >> (8 * grp)) & 0xFFu;
      const int first = 8 * grp + (gdiff ? __ffs(gdiff) - 1 : 0);
      const uint64_t xs = __shfl_sync(kAll, x, first), ys = __shfl_sync(kAll, y, first);
      if (!done) {
        if (gdiff) {
          res = xs < ys ? -1 : 1;
          done = true;
        } else if (t + 64 >= l) {
          res = gla == glb ? 0 : (gla < glb ? -1 : 1);
          done = true;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = __shfl_sync(kAll, res, 8 * q), s = __shfl_sync(kAll, src, 8 * q);
      if (lane == s) c = r;
    }
  }
  return c;
}

// A tile's staged keys. Each key keeps a prefix cache: the big-endian words
// of bytes 0..7 and 8..15 (zero past its end) in k0/k1; A slot x starts at
// begA[x] and ends at begA[x + 1], B slot y likewise in begB. Differing
// words order two keys. With equal words and one length at most 16, the
// shorter key is a proper prefix of the other (its missing bytes are the
// other's zero bytes), or the keys are equal. Two keys longer than 16 bytes
// with equal first 16 bytes need their further bytes: in exact mode from
// warp_tail_cmp; otherwise, when their lengths agree too, they are taken as
// equal and the pair is listed in `vlist` (`vn` counts the entries, also
// past `vcap`) for the caller to check.
struct TileKeys {
  const uint64_t *k0A, *k1A, *k0B, *k1B, *begA, *begB;
  const uint8_t *arenaA, *arenaB;
  uint32_t *vlist;
  int *vn;
  int vcap;
  // Order of A slot sa against B slot y; all 32 lanes call it, `open` says
  // whether this lane has a pair (the result is 0 when it has none).
  __device__ __forceinline__ int cmp(bool open, int sa, int y, bool exact) const {
    int c = 0;
    bool tail = false;
    uint64_t ba = 0, la = 0, bb = 0, lb = 0;
    if (open) {
      const uint64_t a0 = k0A[sa], b0 = k0B[y];
      const uint64_t a1 = k1A[sa], b1 = k1B[y];
      if (a0 != b0) {
        c = a0 < b0 ? -1 : 1;
      } else if (a1 != b1) {
        c = a1 < b1 ? -1 : 1;
      } else {
        ba = begA[sa];
        la = begA[sa + 1] - ba;
        bb = begB[y];
        lb = begB[y + 1] - bb;
        if (la <= 16 || lb <= 16) {
          c = la == lb ? 0 : (la < lb ? -1 : 1);
        } else if (!exact && la == lb) {
          const int v = atomicAdd(vn, 1);
          if (v < vcap) vlist[v] = (static_cast<uint32_t>(sa) << 16) | static_cast<uint32_t>(y);
        } else {
          tail = true;
        }
      }
    }
    return warp_tail_cmp(tail, c, arenaA, ba, la, arenaB, bb, lb);
  }
};

// One tile of T * E merged keys per CTA (T a multiple of 32). The tile's
// keys (and A[i0 - 1], B[j1] where they exist) are staged once in shared
// memory; each thread then finds its diagonal's co-rank by bisection and
// walks E merge steps, every comparison on the staged prefixes, the warp's
// lanes in step. A B key's lower bound is the A count before it in the
// A-first merge, one less when the A key just before it is equal; an A key
// equal to the B head it is taken before sets its collision bit. The first
// pass takes long keys with equal 16-byte prefixes and equal lengths as
// equal (in the common case these are the colliding keys) and the CTA then
// checks every such pair at once; if one differs, or the list overflowed,
// the tile runs again with exact comparisons.
template <int T, int E>
__global__ void __launch_bounds__(T) collision_mark_str_kernel(lsm_bytes A, int64_t m, lsm_bytes B,
                                                               int64_t n,
                                                               const int64_t *__restrict__ part_i,
                                                               uint32_t *__restrict__ C,
                                                               uint32_t *__restrict__ lb_B,
                                                               uint64_t *__restrict__ prefixA,
                                                               uint64_t *__restrict__ prefixB,
                                                               uint32_t *__restrict__ MB,
                                                               int64_t *__restrict__ part_c,
                                                               int64_t G, int cstep) {
  static_assert(T % 32 == 0, "whole warps");
  pdl_begin();
  constexpr int D = T * E;
  constexpr int NK = D + 2;             // staged keys at most
  constexpr int NQ = (NK + T - 1) / T;  // staged keys per thread at most
  __shared__ uint64_t sK0[NK], sK1[NK], sBeg[NK + 2];
  constexpr int kVCap = D / 2;           // pairs taken as equal, checked after
  __shared__ uint32_t sLB[D];
  __shared__ uint32_t sCw[D / 32 + 4];
  static_assert(D % 32 == 0, "a tile's merge bitmap is whole words");
  __shared__ uint32_t sMB[D / 32];  // the tile's merge bitmap words (when MB is given)
  __shared__ uint32_t sV[kVCap];
  __shared__ int sVn;
  const int tid = threadIdx.x;
  if (tid == 0) sVn = 0;
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
  for (int x = tid; x < D / 32; x += T) sMB[x] = 0u;

  // A slots [A[i0-1]] A[i0..i1), then B slots B[j0..j1) [B[j1]]; start
  // offsets in sBeg with one end offset after each side's run
  const int hp = i0 > 0 ? 1 : 0, hn = j1 < n ? 1 : 0;
  const int nA = hp + na, nB = nb + hn, nst = nA + nB;
  {
    uint64_t kb[NQ], ke[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int x = tid + q * T;
      kb[q] = ke[q] = 0;
      if (x < nst) {
        const uint64_t *off = x < nA ? A.off + (i0 - hp + x) : B.off + (j0 + (x - nA));
        kb[q] = __ldg(off);
        ke[q] = __ldg(off + 1);
      }
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int x = tid + q * T;
      if (x < nst) {
        const uint8_t *arena = x < nA ? A.arena : B.arena;
        uint64_t w0, w1;
        load_prefix16(arena, kb[q], ke[q], w0, w1);
        sK0[x] = w0;
        sK1[x] = w1;
        const int xb = x < nA ? x : x + 1;  // B's starts follow A's end offset
        sBeg[xb] = kb[q];
        if (x == nA - 1 || x == nst - 1) sBeg[xb + 1] = ke[q];
        // the prefix tables: every key of the tile once (not A[i0-1], B[j1])
        if (x < nA) {
          if (prefixA && x >= hp)
            reinterpret_cast<ulonglong2 *>(prefixA)[i0 - hp + x] = make_ulonglong2(w0, w1);
        } else if (prefixB && x - nA < nb) {
          reinterpret_cast<ulonglong2 *>(prefixB)[j0 + (x - nA)] = make_ulonglong2(w0, w1);
        }
      }
    }
  }
  __syncthreads();
  const TileKeys keys{sK0, sK1, sK0 + nA, sK1 + nA, sBeg, sBeg + nA + 1,
                      A.arena, B.arena, sV, &sVn, kVCap};
  // A[i0 + a] is A slot hp + a; B[j0 + b] is B slot b

  const int cnt = na + nb;
  const int d = tid * E < cnt ? tid * E : cnt;
  // 32-bit forms of the walk's index tests: B[j0 + b] exists for b < nbh;
  // A[i0 + a] for a >= 1 - hp; A index i0 + a is bit wb0 + a of the tile's
  // first collision word; lower bounds are below 2^31 (checked on the host)
  const int nbh = static_cast<int>(n - j0 < D + 1 ? n - j0 : D + 1);
  const int wb0 = static_cast<int>(i0 - (w0 << 5));
  const uint32_t i0u = static_cast<uint32_t>(i0);
  bool tie0 = false;  // thread 0: A[i0-1] = B[j0], the pair that straddles the tile's start
  for (int pass = 0;; ++pass) {
    const bool exact = pass > 0;
    int lo = d > nb ? d - nb : 0, hi = d < na ? d : na;
    while (__any_sync(0xffffffffu, lo < hi)) {
      const bool open = lo < hi;
      const int mid = (lo + hi) >> 1;
      const int c = keys.cmp(open, hp + mid, d - mid - 1, exact);
      if (open) {
        if (c <= 0) lo = mid + 1;
        else hi = mid;
      }
    }
    int ai = lo, bi = d - lo;
    // prev_eq: the element just before B's head in the merge is an A key
    // equal to it (then that B's lower bound is one less than the A count).
    const bool pq = d < cnt && ai + hp > 0 && bi < nbh;
    bool prev_eq = keys.cmp(pq, hp + ai - 1, bi, exact) == 0 && pq;
    if (tid == 0) tie0 = prev_eq;
    for (int s = 0; s < E; ++s) {
      // c = cmp(A head, B head); B head may be B[j1] (one past the tile)
      // only for the collision test of A's last element.
      const bool live = d + s < cnt;
      const bool has_a = ai < na;
      const bool has_b = bi < nbh;
      const int c = keys.cmp(live && has_a && has_b, hp + ai, bi, exact);
      if (!live) continue;
      const bool takeA = (bi >= nb) || (has_a && c <= 0);
      if (takeA) {
        if (has_b && c == 0) {
          const int x = wb0 + ai;
          atomicOr(&sCw[x >> 5], 1u << (x & 31));
          // B[j1] equal to the tile's last A key sits at the tile's last
          // position of the merge with B first on ties
          if (MB && bi == nb) atomicOr(&sMB[(cnt - 1) >> 5], 1u << ((cnt - 1) & 31));
        }
        prev_eq = has_b && c == 0;
        ++ai;
      } else {
        sLB[bi] = i0u + static_cast<uint32_t>(ai) - (prev_eq ? 1u : 0u);
        // its position in the merge with B first on ties; one before the
        // tile (in the previous tile) for B[j0] equal to A[i0-1]
        const int rp = ai + bi - (prev_eq ? 1 : 0);
        if (MB && rp >= 0) atomicOr(&sMB[rp >> 5], 1u << (rp & 31));
        prev_eq = false;
        ++bi;
      }
    }
    __syncthreads();
    if (exact) break;
    const int nv = sVn;
    bool wrong = nv > kVCap;
    for (int x = tid; x < nv && x < kVCap; x += T) {
      const int sa = static_cast<int>(sV[x] >> 16), y = static_cast<int>(sV[x] & 0xFFFFu);
      const uint64_t ba = keys.begA[sa], bb = keys.begB[y], l = keys.begA[sa + 1] - ba;
      if (key_cmp_tail16(A.arena, ba, l, B.arena, bb, l) != 0) wrong = true;
    }
    if (!__syncthreads_or(wrong)) break;
    for (int x = tid; x < nw; x += T) sCw[x] = 0u;
    for (int x = tid; x < D / 32; x += T) sMB[x] = 0u;
    __syncthreads();
  }
  if (lb_B)
    for (int x = tid; x < nb; x += T) lb_B[j0 + x] = sLB[x];
  if (MB) {
    // the tile's merge bitmap words (tile-owned: D is whole words), and the
    // compaction's co-rank at every cstep-th tile start (B first on ties)
    const int nmw = (cnt + 31) / 32;
    for (int x = tid; x < nmw; x += T) MB[g * (D / 32) + x] = sMB[x];
    if (tid == 0 && g % cstep == 0) part_c[g / cstep] = i0 - (tie0 ? 1 : 0);
    if (tid == 0 && g == G - 1) part_c[(G + cstep - 1) / cstep] = m;
  }
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
                                      uint32_t *C, uint32_t *lb_B, uint64_t *prefixA,
                                      uint64_t *prefixB, int64_t *part_i, int32_t *status,
                                      cudaStream_t s) {
  return launch_collision_mark_str_mb(A, m, B, n, C, lb_B, prefixA, prefixB, part_i, nullptr,
                                      nullptr, 1, status, s);
}

cudaError_t launch_collision_mark_str_mb(const lsm_bytes &A, int64_t m, const lsm_bytes &B,
                                         int64_t n, uint32_t *C, uint32_t *lb_B, uint64_t *prefixA,
                                         uint64_t *prefixB, int64_t *part_i, uint32_t *MB,
                                         int64_t *part_c, int cstep, int32_t * /*status*/,
                                         cudaStream_t s, uint64_t *clear, int64_t nclear) {
  constexpr int64_t D = int64_t(kMarkStrThreads) * kMarkStrItems;
  const int64_t G = (m + n + D - 1) / D;
  const int64_t nwords = (m + 31) / 32;
  int64_t threads = (G + 1) * kStrPartitionLanes;
  if (threads < nwords / 4) threads = nwords / 4;
  cudaError_t err = launch_kernel(false, partition_str_kernel,
                                  static_cast<unsigned>((threads + 255) / 256), 256, 0, s,
                                  StrAFirst{A, B}, m, n, D, G, part_i, C, nwords, clear, nclear);
  if (err != cudaSuccess || G == 0) return err;
  profile_before(s);
  // launched early behind the partition (PDL), whose fewer than one CTA per
  // SM leave the room free (measured: partition + mark 206 us against 209.5)
  err = launch_kernel(true, collision_mark_str_kernel<kMarkStrThreads, kMarkStrItems>,
                      static_cast<unsigned>(G), kMarkStrThreads, 0, s, A, m, B, n, part_i, C, lb_B,
                      prefixA, prefixB, MB, part_c, G, cstep);
  profile_after(s);
  return err;
}

}  // namespace lsm
