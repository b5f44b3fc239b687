/*
 * oracle.c -- plain CPU oracle for the merge-path replacement merge.
 *
 * TEST INFRASTRUCTURE. This is the slow, sequential, obviously correct
 * definition that the GPU library is checked against. Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg load it; the product
 * path never does. It shares no source, header, table or helper with the
 * CUDA library, and it does not know how the GPU partitions work.
 *
 * Every function follows the definition it cites:
 *   [MP]  "Day 36: CUDA merge path: merging sorted arrays in parallel"
 *         (gpu-preview.ayushworks.com/days/36-merge-path)
 *   [CH14] "Chapter 14: Merge Sort and Sample Sort", sections 14.1 and 14.2
 *         (maximumbeings.github.io/dsa_cuda_from_first_principles)
 *   [CB]  "Everett: collision bitmap and rank experiment"
 *         (ekmett.github.io/everett/collision-bitmap-and-rank-experiment.html)
 *   [GC]  "Everett: GPU construction experiment"
 *         (ekmett.github.io/everett/gpu-construction-experiment.html)
 *   [BP]  "Everett: byte-profile GPU merge"
 *         (ekmett.github.io/everett/byte-profile-gpu-merge.html)
 *
 * Conventions (readings of the pages where they are silent):
 *   - A is the older input, B the newer one. Equal keys put A first.
 *   - A reference is src<<31 | index, src 0 = A, src 1 = B.
 *   - Bitmaps (collision bits, tombstones) hold bit t in word t/32 at bit
 *     position t%32 (least significant first).
 *   - A dropped A record has ordinal 0xFFFFFFFF.
 *   - FC payload bit t is bit (31 - t%32) of 32-bit word t/32.
 *
 * Parity of the exact Exp-Golomb bit pattern and of the payload word layout
 * is pinned only by hand-derived fixtures (the pages give the lengths, not
 * the bit strings); the bit packing of the rank2048 entries and the layout
 * of the Elias-Fano sections are readings too (their contents, every R(p)
 * and every sampled offset, are pinned, their bit positions are not);
 * everything else is pinned by page examples, closed forms and brute force
 * in the tests.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define REF_FROM_B 0x80000000u
#define ORD_DROPPED 0xFFFFFFFFu

/* ------------------------------------------------------------------------ */
/* Stable merge. [CH14] "The Sequential (CPU) Baseline": walk two pointers,  */
/* take A while A[i] <= B[j] so that ties go to A, then copy what is left.  */
/* prov (optional) records which input each output came from: i for A[i],   */
/* m + j for B[j] ([MP] "Exercise", the provenance check).                  */
/* ------------------------------------------------------------------------ */
#define ORACLE_DEFINE_MERGE(NAME, KEY)                                        \
    void NAME(const KEY *A, const uint32_t *Apay, int64_t m, const KEY *B,    \
              const uint32_t *Bpay, int64_t n, KEY *out, uint32_t *out_pay,   \
              int64_t *prov) {                                                \
        int64_t i = 0, j = 0, k = 0;                                          \
        while (i < m && j < n) {                                              \
            if (A[i] <= B[j]) {                                               \
                out[k] = A[i];                                                \
                if (out_pay) out_pay[k] = Apay[i];                            \
                if (prov) prov[k] = i;                                        \
                i++;                                                          \
            } else {                                                          \
                out[k] = B[j];                                                \
                if (out_pay) out_pay[k] = Bpay[j];                            \
                if (prov) prov[k] = m + j;                                    \
                j++;                                                          \
            }                                                                 \
            k++;                                                              \
        }                                                                     \
        for (; i < m; i++, k++) {                                             \
            out[k] = A[i];                                                    \
            if (out_pay) out_pay[k] = Apay[i];                                \
            if (prov) prov[k] = i;                                            \
        }                                                                     \
        for (; j < n; j++, k++) {                                             \
            out[k] = B[j];                                                    \
            if (out_pay) out_pay[k] = Bpay[j];                                \
            if (prov) prov[k] = m + j;                                        \
        }                                                                     \
    }

ORACLE_DEFINE_MERGE(oracle_merge_i32, int32_t)
ORACLE_DEFINE_MERGE(oracle_merge_u64, uint64_t)

/* ------------------------------------------------------------------------ */
/* Co-rank by its definition. [MP] "The merge matrix, and the diagonal that  */
/* cuts it" and [CH14] "The Concept, In Detail": the co-rank of k is the    */
/* number of A elements among the first k outputs of the stable merge. The  */
/* oracle walks the merge itself; it does no bisection.                     */
/* Partition entries g = 0..G, G = ceil((m+n)/D), sit at k_g = min(gD, m+n) */
/* and hold (i, j) with i + j = k_g: out_ij[2g] = i, out_ij[2g+1] = j.      */
/* ------------------------------------------------------------------------ */
#define ORACLE_DEFINE_PARTITION(NAME, KEY)                                    \
    void NAME(const KEY *A, int64_t m, const KEY *B, int64_t n, int64_t D,    \
              int64_t *out_ij) {                                              \
        int64_t total = m + n;                                                \
        int64_t G = (total + D - 1) / D;                                      \
        int64_t i = 0, j = 0, g = 0;                                          \
        for (g = 0; g <= G; g++) {                                            \
            int64_t kg = g * D < total ? g * D : total;                       \
            while (i + j < kg) {                                              \
                if (j >= n || (i < m && A[i] <= B[j])) i++;                   \
                else j++;                                                     \
            }                                                                 \
            out_ij[2 * g] = i;                                                \
            out_ij[2 * g + 1] = j;                                            \
        }                                                                     \
    }

ORACLE_DEFINE_PARTITION(oracle_partition_i32, int32_t)
ORACLE_DEFINE_PARTITION(oracle_partition_u64, uint64_t)

/* ------------------------------------------------------------------------ */
/* Bottom-up merge sort. [CH14] section 14.2 "From Merge to Merge Sort":    */
/* every element starts as a sorted run of length 1; one pass merges each   */
/* pair of adjacent runs of the current width with the stable merge above   */
/* (the left run plays A, so equal keys keep their input order), and the    */
/* width doubles until a single run covers the array. A run with no right   */
/* partner at the end of a pass is copied through unchanged (the stable     */
/* merge with an empty B). The pair offset is added back before the merge   */
/* ("COMMON TRAP" of that section): pair p covers [2pw, min(2pw+2w, n)).     */
/* ------------------------------------------------------------------------ */
#define ORACLE_DEFINE_SORT(PASS, SORT, MERGE, KEY)                            \
    void PASS(const KEY *in, const uint32_t *pay, int64_t n, int64_t width,   \
              KEY *out, uint32_t *out_pay) {                                  \
        int64_t start;                                                        \
        for (start = 0; start < n; start += 2 * width) {                      \
            int64_t mid = start + width < n ? start + width : n;              \
            int64_t end = start + 2 * width < n ? start + 2 * width : n;      \
            MERGE(in + start, pay ? pay + start : NULL, mid - start,          \
                  in + mid, pay ? pay + mid : NULL, end - mid, out + start,   \
                  out_pay ? out_pay + start : NULL, NULL);                    \
        }                                                                     \
    }                                                                         \
    /* Returns the number of passes, or -1 if scratch could not be had. */    \
    int64_t SORT(const KEY *in, const uint32_t *pay, int64_t n, KEY *out,     \
                 uint32_t *out_pay) {                                         \
        KEY *tk = (KEY *)malloc((size_t)(n > 0 ? n : 1) * sizeof(KEY));       \
        uint32_t *tp = pay ? (uint32_t *)malloc((size_t)(n > 0 ? n : 1) * 4)  \
                           : NULL;                                            \
        int64_t width, passes = 0;                                            \
        if (!tk || (pay && !tp)) {                                            \
            free(tk);                                                         \
            free(tp);                                                         \
            return -1;                                                        \
        }                                                                     \
        memcpy(out, in, (size_t)n * sizeof(KEY));                             \
        if (pay) memcpy(out_pay, pay, (size_t)n * 4);                         \
        for (width = 1; width < n; width *= 2) {                              \
            PASS(out, pay ? out_pay : NULL, n, width, tk, tp);                \
            memcpy(out, tk, (size_t)n * sizeof(KEY));                         \
            if (pay) memcpy(out_pay, tp, (size_t)n * 4);                      \
            passes++;                                                         \
        }                                                                     \
        free(tk);                                                             \
        free(tp);                                                             \
        return passes;                                                        \
    }

ORACLE_DEFINE_SORT(oracle_mergesort_pass_i32, oracle_merge_sort_i32, oracle_merge_i32, int32_t)
ORACLE_DEFINE_SORT(oracle_mergesort_pass_u64, oracle_merge_sort_u64, oracle_merge_u64, uint64_t)

/* ------------------------------------------------------------------------ */
/* Byte-string order: unsigned lexicographic bytes, a proper prefix sorts   */
/* first ([GC], the prefix-cache paragraph: zero padding plus the length    */
/* keeps proper-prefix order exact).                                        */
/* ------------------------------------------------------------------------ */
static int str_cmp(const uint8_t *a, uint64_t la, const uint8_t *b, uint64_t lb) {
    uint64_t t, lmin = la < lb ? la : lb;
    for (t = 0; t < lmin; t++) {
        if (a[t] != b[t]) return a[t] < b[t] ? -1 : 1;
    }
    if (la == lb) return 0;
    return la < lb ? -1 : 1;
}

/* ------------------------------------------------------------------------ */
/* Replacement merge by sequential dedup. [GC] third paragraph: the stable  */
/* merge puts the older equal key first and only the newer record of each  */
/* equal-key run is kept; a newer tombstone stays a record. [CB] "Corrected */
/* record ordinals": C_i = 1 exactly when B holds A_i's key; lb_B[j] is the */
/* lower bound of B_j in A. Outputs:                                        */
/*   refs[0..count)       survivors in merged order                         */
/*   C[ceil(m/32)]        collision bitmap (tail bits zero)                 */
/*   lb_B[n]              lower bound of each B record in A                 */
/*   ord_A[m], ord_B[n]   output position of each record (dropped: ~0)      */
/* Any output pointer may be NULL. Returns count = m + n - popcount(C).     */
/* ------------------------------------------------------------------------ */
#define ORACLE_REPLACEMENT_BODY(A_LT_B, A_EQ_B, PREV_A_EQ_B)                  \
    int64_t i = 0, j = 0, k = 0;                                              \
    if (C) memset(C, 0, sizeof(uint32_t) * (size_t)((m + 31) / 32));          \
    while (i < m || j < n) {                                                  \
        int a_next = (j >= n) || (i < m && (A_LT_B || A_EQ_B));               \
        if (a_next) {                                                         \
            if (j < n && A_EQ_B) {                                            \
                if (C) C[i / 32] |= 1u << (i % 32);                           \
                if (ord_A) ord_A[i] = ORD_DROPPED;                            \
                i++;                                                          \
                continue;                                                     \
            }                                                                 \
            if (refs) refs[k] = (uint32_t)i;                                  \
            if (ord_A) ord_A[i] = (uint32_t)k;                                \
            i++;                                                              \
        } else {                                                              \
            int64_t hit = (i > 0 && PREV_A_EQ_B) ? 1 : 0;                     \
            if (refs) refs[k] = REF_FROM_B | (uint32_t)j;                     \
            if (lb_B) lb_B[j] = (uint32_t)(i - hit);                          \
            if (ord_B) ord_B[j] = (uint32_t)k;                                \
            j++;                                                              \
        }                                                                     \
        k++;                                                                  \
    }                                                                         \
    return k;

int64_t oracle_replacement_u64(const uint64_t *A, int64_t m, const uint64_t *B,
                               int64_t n, uint32_t *refs, uint32_t *C,
                               uint32_t *lb_B, uint32_t *ord_A, uint32_t *ord_B) {
    ORACLE_REPLACEMENT_BODY(A[i] < B[j], A[i] == B[j], A[i - 1] == B[j])
}

int64_t oracle_replacement_str(const uint8_t *Aar, const uint64_t *Aoff, int64_t m,
                               const uint8_t *Bar, const uint64_t *Boff, int64_t n,
                               uint32_t *refs, uint32_t *C, uint32_t *lb_B,
                               uint32_t *ord_A, uint32_t *ord_B) {
#define SA(x) (Aar + Aoff[(x)]), (Aoff[(x) + 1] - Aoff[(x)])
#define SB(x) (Bar + Boff[(x)]), (Boff[(x) + 1] - Boff[(x)])
    ORACLE_REPLACEMENT_BODY(str_cmp(SA(i), SB(j)) < 0, str_cmp(SA(i), SB(j)) == 0,
                            str_cmp(SA(i - 1), SB(j)) == 0)
#undef SA
#undef SB
}

/* ------------------------------------------------------------------------ */
/* Materialized survivors. [GC] merge paragraph: of each equal-key run the  */
/* newer record is kept, and a newer tombstone stays a record. Output       */
/* record t is the source record refs[t] names: its key, its 32-bit value   */
/* (when value arrays are given) and its tombstone flag, bit t of out_tomb  */
/* (bit t%32 of word t/32; bits past N zero). A tombstone bitmap may be     */
/* NULL (no tombstones in that input).                                      */
/* ------------------------------------------------------------------------ */
static int bit_at(const uint32_t *bits, int64_t i) {
    return bits ? (int)((bits[i / 32] >> (i % 32)) & 1u) : 0;
}

void oracle_materialize_u64(const uint64_t *A, const uint32_t *Aval, const uint32_t *tombA,
                            int64_t m, const uint64_t *B, const uint32_t *Bval,
                            const uint32_t *tombB, int64_t n, const uint32_t *refs, int64_t N,
                            uint64_t *out_keys, uint32_t *out_vals, uint32_t *out_tomb) {
    int64_t t;
    (void)m;
    (void)n;
    if (out_tomb) memset(out_tomb, 0, sizeof(uint32_t) * (size_t)((N + 31) / 32));
    for (t = 0; t < N; t++) {
        const int from_b = (refs[t] & REF_FROM_B) != 0;
        const int64_t idx = (int64_t)(refs[t] & ~REF_FROM_B);
        if (out_keys) out_keys[t] = from_b ? B[idx] : A[idx];
        if (out_vals) out_vals[t] = from_b ? Bval[idx] : Aval[idx];
        if (out_tomb && (from_b ? bit_at(tombB, idx) : bit_at(tombA, idx)))
            out_tomb[t / 32] |= 1u << (t % 32);
    }
}

/* ------------------------------------------------------------------------ */
/* Exclusive collision rank. [CB] "Corrected record ordinals":              */
/* R(i) = sum_{t<i} C_t for i = 0..m, endpoint included. Bit by bit.        */
/* ------------------------------------------------------------------------ */
void oracle_rank_prefix(const uint32_t *C, int64_t m, uint32_t *R) {
    int64_t t;
    R[0] = 0;
    for (t = 0; t < m; t++) R[t + 1] = R[t] + ((C[t / 32] >> (t % 32)) & 1u);
}

/* ------------------------------------------------------------------------ */
/* rank512 directory. [CB] "Temporary rank layouts": every 512-bit block    */
/* has a 32-bit absolute prefix and seven 9-bit prefixes, one at each later */
/* 64-bit word of the block. Layout (three u32 per block, floor(m/512)+1    */
/* blocks so that R(m) is answerable at EOF):                               */
/*   dir[3b]                 R(512 b)                                       */
/*   dir[3b+1] | dir[3b+2]<<32   sum over s=1..7 of                         */
/*                              (R(512b+64s) - R(512b)) << 9(s-1)           */
/* Positions past m count as m (bits beyond A's length are zero).           */
/* ------------------------------------------------------------------------ */
void oracle_rank512_dir(const uint32_t *C, int64_t m, uint32_t *dir) {
    uint32_t *R = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(m + 1));
    int64_t b, nb = m / 512 + 1;
    int s;
    oracle_rank_prefix(C, m, R);
    for (b = 0; b < nb; b++) {
        int64_t base = 512 * b;
        uint64_t packed = 0;
        for (s = 1; s <= 7; s++) {
            int64_t p = base + 64 * s;
            if (p > m) p = m;
            packed |= (uint64_t)(R[p] - R[base]) << (9 * (s - 1));
        }
        dir[3 * b] = R[base];
        dir[3 * b + 1] = (uint32_t)(packed & 0xFFFFFFFFu);
        dir[3 * b + 2] = (uint32_t)(packed >> 32);
    }
    free(R);
}

/* Rank queries R(pos[t]) for pos in [0, m], by the prefix definition. */
void oracle_rank_query(const uint32_t *C, int64_t m, const uint32_t *pos, int64_t q,
                       uint32_t *out) {
    uint32_t *R = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(m + 1));
    int64_t t;
    oracle_rank_prefix(C, m, R);
    for (t = 0; t < q; t++) out[t] = R[pos[t]];
    free(R);
}

/* ------------------------------------------------------------------------ */
/* rank2048 directory. [CB] "Temporary rank layouts": Everett's other layout */
/* keeps one 8-byte entry per 2048 bits holding three packed populations of */
/* its 512-bit runs, with absolute counts at epochs of 2^32 bits; its       */
/* storage is (1/8 + 8/2048)|A| bytes with the bitmap ("Scratch space and  */
/* likely costs"). The page fixes the contents, not the bit packing; the    */
/* reading taken here:                                                      */
/*   epochs[e], e = 0..floor(m/2^32):  R(2^32 e), a full 64-bit count       */
/*   dir[b],    b = 0..floor(m/2048):                                       */
/*     bits  0..31  R(2048 b) - epochs[floor(2048 b / 2^32)]                */
/*     bits 32..41  population of bits [2048b, 2048b+512)                   */
/*     bits 42..51  population of bits [2048b+512, 2048b+1024)              */
/*     bits 52..61  population of bits [2048b+1024, 2048b+1536)             */
/* (a population is at most 512, ten bits). Built by one sequential walk    */
/* over the bits with a running count; positions past m count as zero.      */
/* ------------------------------------------------------------------------ */
void oracle_rank2048_dir(const uint32_t *C, int64_t m, uint64_t *dir, uint64_t *epochs) {
    int64_t nb = m / 2048 + 1, b, t;
    uint64_t R = 0;
    for (b = 0; b < nb; b++) {
        int64_t base = 2048 * b;
        int r;
        uint64_t entry;
        if ((base & ((INT64_C(1) << 32) - 1)) == 0) epochs[base >> 32] = R;
        entry = R - epochs[base >> 32];
        for (r = 0; r < 4; r++) {
            uint64_t pop = 0;
            for (t = base + 512 * r; t < base + 512 * (r + 1) && t < m; t++)
                pop += (C[t / 32] >> (t % 32)) & 1u;
            if (r < 3) entry |= pop << (32 + 10 * r);
            R += pop;
        }
        dir[b] = entry;
    }
    /* an epoch that starts inside the last block's span past m (m >= 2^32 e
       > 2048 floor(m/2048)) cannot exist: 2^32 is a multiple of 2048 */
}

/* R(pos[t]) by the rank2048 layout's query procedure: the epoch, the       */
/* entry's relative count, the populations of the earlier 512-bit runs of   */
/* its 2048-bit block, then the whole 32-bit words of the current run      */
/* before pos and the masked word holding pos. pos in [0, m].              */
void oracle_rank2048_query(const uint32_t *C, const uint64_t *dir, const uint64_t *epochs,
                           const uint64_t *pos, int64_t q, uint64_t *out) {
    int64_t t;
    for (t = 0; t < q; t++) {
        uint64_t p = pos[t], w;
        uint64_t e = dir[p >> 11];
        uint64_t R = epochs[p >> 32] + (e & 0xFFFFFFFFu);
        int r, runs = (int)((p >> 9) & 3);
        for (r = 0; r < runs; r++) R += (e >> (32 + 10 * r)) & 0x3FFu;
        for (w = (p >> 9) * 16; w < (p >> 5); w++) {
            uint32_t x = C[w];
            while (x) { R += x & 1u; x >>= 1; }
        }
        if (p & 31) {
            uint32_t x = C[p >> 5] & ((1u << (p & 31)) - 1u);
            while (x) { R += x & 1u; x >>= 1; }
        }
        out[t] = R;
    }
}

/* ------------------------------------------------------------------------ */
/* Corrected ordinals by the closed forms, [CB] "Corrected record ordinals" */
/* and "The three experimental paths" (independent lower bounds, the        */
/* simplest oracle for the formulas):                                       */
/*   surviving A_i : i + lower_bound(B, A_i) - R(i)                         */
/*   B_j, lb = lower_bound(A, B_j) : j + lb - R(lb)                         */
/* C is recomputed here from the lower bounds, independently of the walk.  */
/* ------------------------------------------------------------------------ */
static int64_t lower_bound_u64(const uint64_t *X, int64_t len, uint64_t key) {
    int64_t lo = 0, hi = len;
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        if (X[mid] < key) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

void oracle_ordinals_formula_u64(const uint64_t *A, int64_t m, const uint64_t *B,
                                 int64_t n, uint32_t *C, uint32_t *lb_B,
                                 uint32_t *ord_A, uint32_t *ord_B) {
    uint32_t *R = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(m + 1));
    int64_t i, j;
    memset(C, 0, sizeof(uint32_t) * (size_t)((m + 31) / 32));
    for (j = 0; j < n; j++) {
        int64_t lb = lower_bound_u64(A, m, B[j]);
        lb_B[j] = (uint32_t)lb;
        if (lb < m && A[lb] == B[j]) C[lb / 32] |= 1u << (lb % 32);
    }
    oracle_rank_prefix(C, m, R);
    for (i = 0; i < m; i++) {
        if ((C[i / 32] >> (i % 32)) & 1u) ord_A[i] = ORD_DROPPED;
        else ord_A[i] = (uint32_t)(i + lower_bound_u64(B, n, A[i]) - R[i]);
    }
    for (j = 0; j < n; j++) ord_B[j] = (uint32_t)(j + lb_B[j] - R[lb_B[j]]);
    free(R);
}

/* ------------------------------------------------------------------------ */
/* Front-compressed record lengths and payload, [GC] the paragraphs on the  */
/* control argument and the record length:                                  */
/*   k_i  key length in bits, l_i exact bit LCP with the preceding surviving */
/*        key (l_0 = 0, clamped to the shorter key)                         */
/*   c_i  = 1 + l_i when i mod 15 = 0, else k_{i-1} - l_i                   */
/*   record = EG0(c_i) EG0(k_i - l_i) key bits [l_i, k_i) value             */
/*   value  = 0 for a tombstone, else 1 EG0(byte length) bytes              */
/*   E(x)   = 2 floor(log2(x+1)) + 1                                        */
/* EG0 is written as the textbook order-0 Exp-Golomb code: floor(log2(x+1)) */
/* zero bits, then x+1 in binary. Bits are written MSB first with no        */
/* padding between records; unused tail bits of the last word are zero.     */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint8_t *arena;
    const uint64_t *off; /* count + 1 offsets */
} oracle_bytes;

static uint64_t key_len(const oracle_bytes *K, uint32_t idx) {
    return K->off[idx + 1] - K->off[idx];
}

static int key_bit(const oracle_bytes *K, uint32_t idx, uint64_t p) {
    uint8_t byte = K->arena[K->off[idx] + p / 8];
    return (byte >> (7 - (p % 8))) & 1;
}

static int floor_log2_u64(uint64_t x) { /* x >= 1 */
    int r = 0;
    while (x > 1) {
        x >>= 1;
        r++;
    }
    return r;
}

static uint64_t eg0_len(uint64_t x) { return 2 * (uint64_t)floor_log2_u64(x + 1) + 1; }

/* E(x), exported so that the tests can pin it to the textbook code length. */
uint64_t oracle_eg0_len(uint64_t x) { return eg0_len(x); }


static void put_bit(uint32_t *payload, uint64_t *pos, int bit) {
    if (payload && bit) payload[*pos / 32] |= 1u << (31 - (*pos % 32));
    (*pos)++;
}

static void put_eg0(uint32_t *payload, uint64_t *pos, uint64_t x) {
    int z = floor_log2_u64(x + 1), b;
    for (b = 0; b < z; b++) put_bit(payload, pos, 0);
    for (b = z; b >= 0; b--) put_bit(payload, pos, (int)(((x + 1) >> b) & 1u));
}


/* ------------------------------------------------------------------------ */
/* Elias-Fano navigation over the record offsets. [GC] "GPU construction    */
/* experiment": physical offsets are sampled at ordinals 0, 15, 30, ... and */
/* at EOF (the payload extent); when every encoded value has the same width */
/* w, the sequence subtracts w times the sample's ordinal; the EF sections   */
/* are lows, highs, select samples and sparse exceptions, a 256-entry group */
/* being sparse when its high-position span is at least 4096 bits. The rest */
/* is textbook Elias-Fano; the layout is this library's reading:           */
/*   entries  x_s = bit_off[15 s] - 15 s w for s = 0..ceil(N/15)-1, then     */
/*            x_{n-1} = bit_off[N] - N w; n = ceil(N/15) + 1, U = x_{n-1}    */
/*   L        the largest L with n 2^L <= U (0 when U < n)                  */
/*   lows     x_s mod 2^L at bit positions [sL, sL + L) of a uint64 array    */
/*            (bit t in word t/64 at position t%64), ceil(nL/64) words      */
/*   highs    bit (x_s >> L) + s set for every s; (U >> L) + n bits, in      */
/*            ceil(((U >> L) + n)/64) uint64 words, same bit order          */
/*   samples  group g = entries [256 g, min(256 g + 256, n)):               */
/*            samples[2g] = the high position of entry 256 g;              */
/*            samples[2g+1] = e_g << 1 | sparse_g, where sparse_g = (high   */
/*            position of the group's last entry - that of its first >= 4096) */
/*            and e_g = the number of entries in sparse groups before g     */
/*   sparse   the high position of every entry of every sparse group, in   */
/*            entry order (group g's at [e_g, e_g + its entry count))       */
/* Unused bits of every word are zero. Returns the number of sparse entries. */
/* ------------------------------------------------------------------------ */
static uint64_t ef_entry(const uint64_t *bit_off, int64_t N, uint64_t w, int64_t n, int64_t s) {
    int64_t ord = s == n - 1 ? N : 15 * s;
    return bit_off[ord] - (uint64_t)ord * w;
}

/* sizes[0] = n, [1] = L, [2] = lows words, [3] = highs words, [4] = groups */
void oracle_ef_sizes(int64_t N, uint64_t U, int64_t *sizes) {
    int64_t n = (N + 14) / 15 + 1;
    int L = 0;
    while (L < 63 && ((unsigned __int128)n << (L + 1)) <= U) L++;
    sizes[0] = n;
    sizes[1] = L;
    sizes[2] = (n * L + 63) / 64;
    sizes[3] = (int64_t)(((U >> L) + (uint64_t)n + 63) / 64);
    sizes[4] = (n + 255) / 256;
}

int64_t oracle_ef_build(const uint64_t *bit_off, int64_t N, uint64_t w, uint64_t *lows,
                        uint64_t *highs, uint64_t *samples, uint64_t *sparse) {
    int64_t sz[5], n, L, s, g, e = 0;
    uint64_t U;
    n = (N + 14) / 15 + 1;
    U = ef_entry(bit_off, N, w, n, n - 1);
    oracle_ef_sizes(N, U, sz);
    L = sz[1];
    memset(lows, 0, (size_t)sz[2] * 8);
    memset(highs, 0, (size_t)sz[3] * 8);
    for (s = 0; s < n; s++) {
        uint64_t x = ef_entry(bit_off, N, w, n, s);
        uint64_t h = (x >> L) + (uint64_t)s;
        int64_t b;
        for (b = 0; b < L; b++)
            if ((x >> b) & 1u) lows[(s * L + b) / 64] |= (uint64_t)1 << ((s * L + b) % 64);
        highs[h / 64] |= (uint64_t)1 << (h % 64);
    }
    for (g = 0; g < sz[4]; g++) {
        int64_t first = 256 * g, last = 256 * g + 255 < n - 1 ? 256 * g + 255 : n - 1;
        uint64_t h0 = (ef_entry(bit_off, N, w, n, first) >> L) + (uint64_t)first;
        uint64_t h1 = (ef_entry(bit_off, N, w, n, last) >> L) + (uint64_t)last;
        int sp = h1 - h0 >= 4096;
        samples[2 * g] = h0;
        samples[2 * g + 1] = ((uint64_t)e << 1) | (uint64_t)sp;
        if (sp) {
            for (s = first; s <= last; s++)
                sparse[e++] = (ef_entry(bit_off, N, w, n, s) >> L) + (uint64_t)s;
        }
    }
    return e;
}

/* Writes EG0(x) into a zeroed word buffer; returns the bits written. */
uint64_t oracle_eg0_bits(uint64_t x, uint32_t *words) {
    uint64_t pos = 0;
    put_eg0(words, &pos, x);
    return pos;
}

/* Returns the total number of payload bits, or -1 if a per-record field
 * does not fit in 32 bits or the payload buffer is too small. payload may
 * be NULL (lengths only); it is zeroed before writing when given. */
int64_t oracle_fc_encode(const uint8_t *keyA_ar, const uint64_t *keyA_off,
                         const uint8_t *valA_ar, const uint64_t *valA_off,
                         const uint32_t *tombA, const uint8_t *keyB_ar,
                         const uint64_t *keyB_off, const uint8_t *valB_ar,
                         const uint64_t *valB_off, const uint32_t *tombB,
                         const uint32_t *refs, int64_t N, uint32_t *lcp,
                         uint32_t *ctrl, uint32_t *rec_bits, uint64_t *bit_off,
                         uint32_t *payload, int64_t nwords) {
    oracle_bytes KA = {keyA_ar, keyA_off}, KB = {keyB_ar, keyB_off};
    oracle_bytes VA = {valA_ar, valA_off}, VB = {valB_ar, valB_off};
    uint64_t pos = 0, k_prev = 0;
    int64_t i;
    if (payload) memset(payload, 0, sizeof(uint32_t) * (size_t)nwords);
    for (i = 0; i < N; i++) {
        uint32_t r = refs[i], idx = r & 0x7FFFFFFFu;
        const oracle_bytes *K = (r & REF_FROM_B) ? &KB : &KA;
        const oracle_bytes *V = (r & REF_FROM_B) ? &VB : &VA;
        const uint32_t *T = (r & REF_FROM_B) ? tombB : tombA;
        uint64_t k = 8 * key_len(K, idx), l = 0, c, v, L, p, start = pos;
        int tomb = T ? (int)((T[idx / 32] >> (idx % 32)) & 1u) : 0;
        if (i > 0) {
            uint32_t pr = refs[i - 1], pidx = pr & 0x7FFFFFFFu;
            const oracle_bytes *PK = (pr & REF_FROM_B) ? &KB : &KA;
            uint64_t kmin = 8 * key_len(PK, pidx);
            if (k < kmin) kmin = k;
            while (l < kmin && key_bit(PK, pidx, l) == key_bit(K, idx, l)) l++;
        }
        c = (i % 15 == 0) ? 1 + l : k_prev - l;
        if (tomb) v = 1;
        else {
            uint64_t vb = key_len(V, idx);
            v = 1 + eg0_len(vb) + 8 * vb;
        }
        L = eg0_len(c) + eg0_len(k - l) + (k - l) + v;
        if (l > 0xFFFFFFFFu || c > 0xFFFFFFFFu || L > 0xFFFFFFFFu) return -1;
        if (lcp) lcp[i] = (uint32_t)l;
        if (ctrl) ctrl[i] = (uint32_t)c;
        if (rec_bits) rec_bits[i] = (uint32_t)L;
        if (bit_off) bit_off[i] = start;
        if (payload && (uint64_t)nwords * 32 < start + L) return -1;
        put_eg0(payload, &pos, c);
        put_eg0(payload, &pos, k - l);
        for (p = l; p < k; p++) put_bit(payload, &pos, key_bit(K, idx, p));
        if (tomb) put_bit(payload, &pos, 0);
        else {
            uint64_t vb = key_len(V, idx);
            put_bit(payload, &pos, 1);
            put_eg0(payload, &pos, vb);
            for (p = 0; p < 8 * vb; p++) put_bit(payload, &pos, key_bit(V, idx, p));
        }
        if (pos != start + L) return -1; /* the length formula and the writer agree */
        k_prev = k;
    }
    if (bit_off) bit_off[N] = pos;
    return (int64_t)pos;
}


/* ------------------------------------------------------------------------ */
/* Byte-profile front compression. [BP] "Pipeline": the byte profile's      */
/* records carry byte LEB128 counts, FC literals and optional-value tags;   */
/* a common encoded value width is detected ("width seventeen means a      */
/* one-byte presence tag and sixteen payload bytes"); blocks and sampling   */
/* stay at 15 records; records are sized, scanned and emitted in order.     */
/* The pages do not print the record grammar. Reading: the bit profile's    */
/* record ([GC] control-argument equation and record-length formula) with   */
/* bytes for bits and LEB128 for Exp-Golomb:                                */
/*   p_i = byte LCP with the previous record's key (p_0 = 0), K_i = key    */
/*   length in bytes; control b_i = 1 + p_i when i mod 15 = 0, else         */
/*   K_{i-1} - p_i; record = LEB128(b_i) LEB128(K_i - p_i) key bytes        */
/*   [p_i, K_i) then the value: tag byte 0 for a tombstone, else tag 1,     */
/*   LEB128(value length) and the value bytes; with a common width W > 0    */
/*   (every record present, every value W - 1 bytes) the length is left     */
/*   out. LEB128 is the textbook unsigned form: seven bits per byte, low    */
/*   group first, the top bit set on every byte but the last.               */
/* Returns the payload bytes, or -1 (a field past 32 bits, a record that    */
/* breaks the common width, or a payload buffer too small).                 */
/* ------------------------------------------------------------------------ */
static uint64_t leb_len(uint64_t x) {
    uint64_t n = 1;
    while (x >= 128) { x >>= 7; n++; }
    return n;
}

uint64_t oracle_leb128(uint64_t x, uint8_t *out) {
    uint64_t n = 0;
    do {
        uint8_t b = (uint8_t)(x & 0x7F);
        x >>= 7;
        if (x) b |= 0x80;
        out[n++] = b;
    } while (x);
    return n;
}

int64_t oracle_bytefc_encode(const uint8_t *keyA_ar, const uint64_t *keyA_off,
                             const uint8_t *valA_ar, const uint64_t *valA_off,
                             const uint32_t *tombA, const uint8_t *keyB_ar,
                             const uint64_t *keyB_off, const uint8_t *valB_ar,
                             const uint64_t *valB_off, const uint32_t *tombB,
                             const uint32_t *refs, int64_t N, uint64_t W, uint32_t *lcp,
                             uint32_t *ctrl, uint32_t *rec_bytes, uint64_t *byte_off,
                             uint8_t *payload, int64_t cap) {
    oracle_bytes KA = {keyA_ar, keyA_off}, KB = {keyB_ar, keyB_off};
    oracle_bytes VA = {valA_ar, valA_off}, VB = {valB_ar, valB_off};
    uint64_t pos = 0, k_prev = 0;
    int64_t i;
    for (i = 0; i < N; i++) {
        uint32_t r = refs[i], idx = r & 0x7FFFFFFFu;
        const oracle_bytes *K = (r & REF_FROM_B) ? &KB : &KA;
        const oracle_bytes *V = (r & REF_FROM_B) ? &VB : &VA;
        const uint32_t *T = (r & REF_FROM_B) ? tombB : tombA;
        uint64_t k = key_len(K, idx), l = 0, c, v, L, q, start = pos;
        int tomb = T ? (int)((T[idx / 32] >> (idx % 32)) & 1u) : 0;
        if (i > 0) {
            uint32_t pr = refs[i - 1], pidx = pr & 0x7FFFFFFFu;
            const oracle_bytes *PK = (pr & REF_FROM_B) ? &KB : &KA;
            uint64_t kmin = key_len(PK, pidx);
            if (k < kmin) kmin = k;
            while (l < kmin && PK->arena[PK->off[pidx] + l] == K->arena[K->off[idx] + l]) l++;
        }
        c = (i % 15 == 0) ? 1 + l : k_prev - l;
        if (tomb) {
            if (W) return -1;
            v = 1;
        } else {
            uint64_t vb = key_len(V, idx);
            if (W && vb + 1 != W) return -1;
            v = W ? W : 1 + leb_len(vb) + vb;
        }
        L = leb_len(c) + leb_len(k - l) + (k - l) + v;
        if (l > 0xFFFFFFFFu || c > 0xFFFFFFFFu || L > 0xFFFFFFFFu) return -1;
        if (lcp) lcp[i] = (uint32_t)l;
        if (ctrl) ctrl[i] = (uint32_t)c;
        if (rec_bytes) rec_bytes[i] = (uint32_t)L;
        if (byte_off) byte_off[i] = start;
        if (payload) {
            if ((uint64_t)cap < start + L) return -1;
            pos += oracle_leb128(c, payload + pos);
            pos += oracle_leb128(k - l, payload + pos);
            for (q = l; q < k; q++) payload[pos++] = K->arena[K->off[idx] + q];
            if (tomb) payload[pos++] = 0;
            else {
                uint64_t vb = key_len(V, idx);
                payload[pos++] = 1;
                if (!W) pos += oracle_leb128(vb, payload + pos);
                for (q = 0; q < vb; q++) payload[pos++] = V->arena[V->off[idx] + q];
            }
            if (pos != start + L) return -1; /* the length formula and the writer agree */
        } else {
            pos += L;
        }
        k_prev = k;
    }
    if (byte_off) byte_off[N] = pos;
    return (int64_t)pos;
}

/* Independent byte-profile decoder: reads the records back in the same     */
/* grammar. Returns the bytes consumed or a negative code on a malformed    */
/* payload. Output capacities as oracle_fc_decode's.                        */
static int get_leb(const uint8_t *payload, uint64_t total, uint64_t *pos, uint64_t *x) {
    uint64_t v = 0;
    int shift = 0;
    for (;;) {
        uint8_t b;
        if (*pos >= total || shift > 63) return -1;
        b = payload[(*pos)++];
        v |= (uint64_t)(b & 0x7F) << shift;
        shift += 7;
        if (!(b & 0x80)) break;
    }
    *x = v;
    return 0;
}

int64_t oracle_bytefc_decode(const uint8_t *payload, uint64_t total, int64_t N, uint64_t W,
                             uint8_t *key_ar, uint64_t key_cap, uint64_t *key_off,
                             uint8_t *val_ar, uint64_t val_cap, uint64_t *val_off,
                             uint32_t *tomb) {
    uint64_t pos = 0, kpos = 0, vpos = 0, prev_len = 0;
    int64_t i;
    key_off[0] = 0;
    val_off[0] = 0;
    for (i = 0; i < N; i++) {
        uint64_t c, s, l, t, vb;
        uint8_t tag;
        if (get_leb(payload, total, &pos, &c) || get_leb(payload, total, &pos, &s)) return -1;
        if (i % 15 == 0) {
            if (c < 1) return -2;
            l = c - 1;
        } else {
            if (c > prev_len) return -2;
            l = prev_len - c;
        }
        if (i == 0 && l) return -2;
        if (l > prev_len || kpos + l + s > key_cap || pos + s > total) return -3;
        for (t = 0; t < l; t++) key_ar[kpos + t] = key_ar[key_off[i - (i > 0)] + t];
        for (t = 0; t < s; t++) key_ar[kpos + l + t] = payload[pos + t];
        pos += s;
        kpos += l + s;
        key_off[i + 1] = kpos;
        prev_len = l + s;
        if (pos >= total) return -4;
        tag = payload[pos++];
        if (tag == 0) {
            tomb[i / 32] |= 1u << (i % 32);
        } else if (tag == 1) {
            if (W) vb = W - 1;
            else if (get_leb(payload, total, &pos, &vb)) return -4;
            if (vpos + vb > val_cap || pos + vb > total) return -4;
            for (t = 0; t < vb; t++) val_ar[vpos + t] = payload[pos + t];
            pos += vb;
            vpos += vb;
        } else {
            return -5;
        }
        val_off[i + 1] = vpos;
    }
    return (int64_t)pos;
}

/* ------------------------------------------------------------------------ */
/* Independent FC decoder: parses a payload back into keys, values and      */
/* tombstones, following the same record grammar in the reading direction. */
/* Keys are rebuilt from the previous key's first l bits plus the literal   */
/* suffix, where l = c - 1 at a 15-record restart and k_{i-1} - c elsewhere. */
/* Outputs are caller-sized: key_ar/val_ar capacities in bytes, offsets     */
/* N + 1 entries, tomb ceil(N/32) words. Returns bits consumed or a         */
/* negative code on a malformed payload.                                    */
/* ------------------------------------------------------------------------ */
static int get_bit(const uint32_t *payload, uint64_t total, uint64_t *pos, int *bit) {
    if (*pos >= total) return -1;
    *bit = (int)((payload[*pos / 32] >> (31 - (*pos % 32))) & 1u);
    (*pos)++;
    return 0;
}

static int get_eg0(const uint32_t *payload, uint64_t total, uint64_t *pos, uint64_t *x) {
    int z = 0, bit = 0, b;
    uint64_t v = 1;
    for (;;) {
        if (get_bit(payload, total, pos, &bit)) return -1;
        if (bit) break;
        if (++z > 62) return -1;
    }
    for (b = 0; b < z; b++) {
        if (get_bit(payload, total, pos, &bit)) return -1;
        v = (v << 1) | (uint64_t)bit;
    }
    *x = v - 1;
    return 0;
}

int64_t oracle_fc_decode(const uint32_t *payload, uint64_t total_bits, int64_t N,
                         uint8_t *key_ar, uint64_t key_cap, uint64_t *key_off,
                         uint8_t *val_ar, uint64_t val_cap, uint64_t *val_off,
                         uint32_t *tomb) {
    uint64_t pos = 0, kpos = 0, vpos = 0, prev_start = 0, k_prev = 0, t;
    int64_t i;
    int bit;
    memset(tomb, 0, sizeof(uint32_t) * (size_t)((N + 31) / 32));
    key_off[0] = 0;
    val_off[0] = 0;
    for (i = 0; i < N; i++) {
        uint64_t c, d, l, k;
        if (get_eg0(payload, total_bits, &pos, &c)) return -2;
        if (get_eg0(payload, total_bits, &pos, &d)) return -2;
        if (i % 15 == 0) {
            if (c < 1) return -3;
            l = c - 1;
        } else {
            if (c > k_prev) return -3;
            l = k_prev - c;
        }
        if (l > k_prev) return -3;
        k = l + d;
        if (k % 8 != 0) return -4;
        if (kpos + k / 8 > key_cap) return -5;
        /* inherited prefix bits from the previous key, then the literal */
        memset(key_ar + kpos, 0, (size_t)(k / 8));
        for (t = 0; t < k; t++) {
            int b;
            if (t < l) {
                b = (key_ar[prev_start + t / 8] >> (7 - t % 8)) & 1;
            } else {
                if (get_bit(payload, total_bits, &pos, &b)) return -2;
            }
            if (b) key_ar[kpos + t / 8] |= (uint8_t)(1u << (7 - t % 8));
        }
        prev_start = kpos;
        kpos += k / 8;
        key_off[i + 1] = kpos;
        k_prev = k;
        if (get_bit(payload, total_bits, &pos, &bit)) return -2;
        if (!bit) {
            tomb[i / 32] |= 1u << (i % 32);
        } else {
            uint64_t vb;
            if (get_eg0(payload, total_bits, &pos, &vb)) return -2;
            if (vpos + vb > val_cap) return -5;
            for (t = 0; t < vb; t++) {
                int b, q;
                uint8_t byte = 0;
                for (q = 0; q < 8; q++) {
                    if (get_bit(payload, total_bits, &pos, &b)) return -2;
                    byte = (uint8_t)((byte << 1) | b);
                }
                val_ar[vpos + t] = byte;
            }
            vpos += vb;
        }
        val_off[i + 1] = vpos;
    }
    return (int64_t)pos;
}
