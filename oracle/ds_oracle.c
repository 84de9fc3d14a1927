/*
 * ds_oracle.c -- CPU oracle for DeepSelect top-k.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that the tests, the smoke check and the CPU
 * baseline leg of the benchmark have an independent, obviously correct answer
 * to compare the CUDA library against.  It shares no code, header or table
 * with the CUDA side.
 *
 * Sources (page titles as given on the pages; sections in brackets):
 *   [DS]  PFCCLab/DeepSelect "DeepSelect-deep-dive" -- sections "算法"
 *         (algorithm: scan / filter / compact loop, pseudocode, notes on the
 *         buffer bound) and "RadixSelectTopK 总处理元素数的期望上界"
 *         (expected-work bound: A, R, W, W = A + kR, R*B2 <= A).
 *   [OPS] milkfeng.top "CUDA 算子笔记 4" -- section "Top K Selection"
 *         (problem statement and worked example) and its sub-section
 *         "改造 Radix Sort" (order-preserving float -> unsigned key map; the
 *         same construction serves fp32, bf16 and IEEE binary16).
 *   [PHX] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 *         1, 2, 3", SC'11 -- definition of Philox4x32-10.
 *
 * Three things live here:
 *   1. ds_oracle_topk   -- the plain definition: sort every valid element of
 *      a row by (value descending, index ascending) and keep the first k.
 *   2. ds_oracle_model  -- the DeepSelect loop of [DS] "算法" step by step,
 *      with the counters A, R, W and the peak buffer length of [DS]'s
 *      expected-work section.  Used to pin the algorithm's invariants and to
 *      check the GPU's instrumented counters.
 *   3. Philox4x32-10 and the block permutation derived from it.
 *
 * Readings taken where the pages are silent (each also listed in the
 * project's design notes):
 *   - Total order.  NaN (any payload) is above +inf and all NaNs are equal;
 *     -0.0 and +0.0 are equal; otherwise the numeric order.  Equal values are
 *     ordered by lower index first.  The pages assume distinct elements
 *     ([DS] expected-work section); this order makes every element distinct.
 *   - The filter "x[j] > threshold" ([DS] pseudocode) compares the pair
 *     (value, index) in that total order, the threshold being the smallest
 *     pair kept by the last compaction.  The initial threshold "-inf" admits
 *     every element.
 *   - RadixSelectTopK "or another TopK algorithm" ([DS] "算法", step 3): the
 *     model compacts with a full sort, which is an exact TopK.
 *   - random_permutation: block b of (row r, slice c) gets the first output
 *     word of Philox4x32-10 with counter (b, r, c, 0) and key (seed low 32
 *     bits, seed high 32 bits); blocks are visited in ascending (word, b).
 *   - Split rows ([DS] "实现", last paragraph): the m blocks of a row are cut
 *     into S contiguous slices of ceil(m/S) blocks; each slice runs the loop
 *     on its own; the union of the slice results is reduced to the top k.
 *   - Rows with fewer than k valid elements return all of them, then pad
 *     with index -1 and value -inf.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define DS_ORACLE_FP32 0
#define DS_ORACLE_BF16 1
#define DS_ORACLE_FP16 2

/* ------------------------------------------------------------------------ */
/* Total order: unsigned key whose order is the value order.                 */
/* [OPS] "改造 Radix Sort": flip the sign bit of non-negative floats and all  */
/* bits of negative ones, so that unsigned comparison follows float order.   */
/* NaN and -0.0 are canonicalised first (reading above).                     */
/* ------------------------------------------------------------------------ */

uint32_t ds_oracle_key_f32(uint32_t bits)
{
    uint32_t magnitude = bits & 0x7FFFFFFFu;
    if (magnitude > 0x7F800000u)      /* NaN, any sign or payload */
        return 0xFFFFFFFFu;
    if (magnitude == 0u)              /* -0.0 and +0.0 */
        return 0x80000000u;
    if (bits & 0x80000000u)           /* negative: larger magnitude is smaller */
        return ~bits;
    return bits | 0x80000000u;        /* positive: above every negative */
}

uint32_t ds_oracle_key_bf16(uint32_t bits16)
{
    uint32_t bits = bits16 & 0xFFFFu;
    uint32_t magnitude = bits & 0x7FFFu;
    if (magnitude > 0x7F80u)
        return 0xFFFFu;
    if (magnitude == 0u)
        return 0x8000u;
    if (bits & 0x8000u)
        return (~bits) & 0xFFFFu;
    return bits | 0x8000u;
}

/* IEEE binary16: 5 exponent bits, 10 mantissa bits; the infinity pattern
 * is 0x7C00 and every larger magnitude is a NaN. */
uint32_t ds_oracle_key_f16(uint32_t bits16)
{
    uint32_t bits = bits16 & 0xFFFFu;
    uint32_t magnitude = bits & 0x7FFFu;
    if (magnitude > 0x7C00u)
        return 0xFFFFu;
    if (magnitude == 0u)
        return 0x8000u;
    if (bits & 0x8000u)
        return (~bits) & 0xFFFFu;
    return bits | 0x8000u;
}

/* Exhaustive check of ds_oracle_key_f32 over all 2^32 bit patterns against
 * C's own float comparison (IEEE 754, no fast-math): every non-NaN pattern is
 * visited in increasing numeric order -- negative patterns from -inf
 * (0xFF800000) down to -0 (0x80000000), then positive ones from +0 up to
 * +inf (0x7F800000) -- and each step must be numerically increasing as C
 * floats (or -0 to +0, which compare equal) with the key increasing in the
 * same way (equal exactly at -0 -> +0); every NaN pattern must map to the
 * largest key, above the key of +inf.  Returns the number of violations. */
int64_t ds_oracle_sweep_f32(void)
{
    int64_t bad = 0;
    uint32_t prev_bits = 0xFF800000u, prev_key = ds_oracle_key_f32(prev_bits);
    float prev_f;
    memcpy(&prev_f, &prev_bits, 4);
    uint32_t bits = 0xFF800000u;
    for (int half = 0; half < 2; ++half) {
        for (;;) {
            if (half == 0) {
                if (bits == 0x80000000u)
                    break;
                --bits;                       /* next negative pattern toward -0 */
            } else {
                bits = bits == 0x80000000u ? 0u : bits + 1u;
            }
            float f;
            memcpy(&f, &bits, 4);
            const uint32_t key = ds_oracle_key_f32(bits);
            const int same = prev_bits == 0x80000000u && bits == 0u;  /* -0 -> +0 */
            if (same) {
                if (!(f == prev_f) || key != prev_key)
                    ++bad;
            } else if (!(prev_f < f) || !(prev_key < key)) {
                ++bad;
            }
            prev_bits = bits;
            prev_key = key;
            prev_f = f;
            if (half == 1 && bits == 0x7F800000u)
                break;
        }
    }
    const uint32_t inf_key = ds_oracle_key_f32(0x7F800000u);
    for (uint32_t m = 0x7F800001u; m <= 0x7FFFFFFFu; ++m) {
        float f;
        memcpy(&f, &m, 4);
        if (f == f)                           /* C must agree that it is a NaN */
            ++bad;
        if (ds_oracle_key_f32(m) != 0xFFFFFFFFu || ds_oracle_key_f32(m | 0x80000000u) != 0xFFFFFFFFu)
            ++bad;
    }
    if (!(inf_key < 0xFFFFFFFFu))
        ++bad;
    return bad;
}

static int dtype_known(int dtype)
{
    return dtype == DS_ORACLE_FP32 || dtype == DS_ORACLE_BF16 || dtype == DS_ORACLE_FP16;
}

static uint32_t element_bits(const void *x, int dtype, int64_t pos)
{
    if (dtype == DS_ORACLE_FP32)
        return ((const uint32_t *)x)[pos];
    return ((const uint16_t *)x)[pos];
}

static uint32_t element_key(const void *x, int dtype, int64_t pos)
{
    uint32_t bits = element_bits(x, dtype, pos);
    if (dtype == DS_ORACLE_FP32)
        return ds_oracle_key_f32(bits);
    return dtype == DS_ORACLE_BF16 ? ds_oracle_key_bf16(bits) : ds_oracle_key_f16(bits);
}

/* Keys of n elements, for the tests. */
void ds_oracle_keys(const void *x, int dtype, int64_t n, uint32_t *keys)
{
    for (int64_t i = 0; i < n; ++i)
        keys[i] = element_key(x, dtype, i);
}

typedef struct {
    uint32_t key;
    int32_t idx;
} pair_t;

/* a before b  <=>  a.key > b.key, or equal keys and a.idx < b.idx */
static int pair_before(pair_t a, pair_t b)
{
    if (a.key != b.key)
        return a.key > b.key;
    return a.idx < b.idx;
}

static int pair_cmp(const void *pa, const void *pb)
{
    pair_t a = *(const pair_t *)pa, b = *(const pair_t *)pb;
    if (pair_before(a, b))
        return -1;
    if (pair_before(b, a))
        return 1;
    return 0;
}

static int64_t valid_length(const int32_t *row_len, int r, int64_t N)
{
    int64_t len = row_len ? (int64_t)row_len[r] : N;
    if (len < 0)
        len = 0;
    if (len > N)
        len = N;
    return len;
}

static void write_output(const void *x, int dtype, int64_t row_base, const pair_t *sorted,
                         int64_t count, int k, int32_t *out_idx, void *out_val, int64_t out_base)
{
    for (int64_t i = 0; i < k; ++i) {
        int32_t idx = -1;
        uint32_t bits = dtype == DS_ORACLE_FP32 ? 0xFF800000u
                      : dtype == DS_ORACLE_BF16 ? 0xFF80u : 0xFC00u; /* -inf */
        if (i < count) {
            idx = sorted[i].idx;
            bits = element_bits(x, dtype, row_base + idx);
        }
        out_idx[out_base + i] = idx;
        if (dtype == DS_ORACLE_FP32)
            ((uint32_t *)out_val)[out_base + i] = bits;
        else
            ((uint16_t *)out_val)[out_base + i] = (uint16_t)bits;
    }
}

/* ------------------------------------------------------------------------ */
/* 1. The definition.  [OPS] "Top K Selection": output the k largest.        */
/* Every valid element of the row is sorted by the total order; the first k  */
/* are the answer, already in (value desc, index asc) order.                 */
/* Returns 0, or -1 on bad arguments / allocation failure.                   */
/* ------------------------------------------------------------------------ */
int ds_oracle_topk(const void *x, int dtype, int rows, const int32_t *row_len, int64_t N,
                   int k, int32_t *out_idx, void *out_val)
{
    if (rows < 0 || N < 1 || k < 1 || !dtype_known(dtype))
        return -1;
    pair_t *pairs = (pair_t *)malloc((size_t)N * sizeof(pair_t));
    if (!pairs)
        return -1;
    for (int r = 0; r < rows; ++r) {
        int64_t len = valid_length(row_len, r, N);
        int64_t base = (int64_t)r * N;
        for (int64_t j = 0; j < len; ++j) {
            pairs[j].key = element_key(x, dtype, base + j);
            pairs[j].idx = (int32_t)j;
        }
        qsort(pairs, (size_t)len, sizeof(pair_t), pair_cmp);
        write_output(x, dtype, base, pairs, len < k ? len : k, k, out_idx, out_val, (int64_t)r * k);
    }
    free(pairs);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* 3. Philox4x32-10 [PHX].  One round: two 32x32->64 products of counter    */
/* words 0 and 2 with the round multipliers; the high halves are xored with */
/* the other two counter words and the round key; the key is bumped by the  */
/* Weyl constants between rounds.                                           */
/* ------------------------------------------------------------------------ */
void ds_oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += W0;
            k1 += W1;
        }
        uint64_t p0 = (uint64_t)M0 * c0;
        uint64_t p1 = (uint64_t)M1 * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

typedef struct {
    uint32_t word;
    uint32_t block;
} perm_key_t;

static int perm_key_cmp(const void *pa, const void *pb)
{
    perm_key_t a = *(const perm_key_t *)pa, b = *(const perm_key_t *)pb;
    if (a.word != b.word)
        return a.word < b.word ? -1 : 1;
    if (a.block != b.block)
        return a.block < b.block ? -1 : 1;
    return 0;
}

/* random_permutation of [DS] pseudocode, for blocks first .. first+m-1 of
 * (row, slice): visit order = ascending (Philox word 0, block id). */
int ds_oracle_permutation(uint32_t m, uint64_t seed, uint32_t row, uint32_t slice,
                          uint32_t first_block, uint32_t *perm)
{
    perm_key_t *keys = (perm_key_t *)malloc((size_t)(m ? m : 1) * sizeof(perm_key_t));
    if (!keys)
        return -1;
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    for (uint32_t i = 0; i < m; ++i) {
        uint32_t ctr[4] = {first_block + i, row, slice, 0u};
        uint32_t out[4];
        ds_oracle_philox4x32_10(ctr, key, out);
        keys[i].word = out[0];
        keys[i].block = first_block + i;
    }
    qsort(keys, m, sizeof(perm_key_t), perm_key_cmp);
    for (uint32_t i = 0; i < m; ++i)
        perm[i] = keys[i].block;
    free(keys);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* 2. The algorithm, step by step ([DS] "算法", pseudocode).                  */
/*                                                                          */
/* For every row and slice:                                                 */
/*   candidates = [], threshold = -inf (admit all)                          */
/*   for block in random_permutation(blocks of the slice):                  */
/*       append every (x[j], j) of the block that is above the threshold    */
/*       if len(candidates) >= k + B2:                                      */
/*           candidates = TopK(candidates, k); threshold = smallest kept    */
/*   result = TopK(candidates, k)                                           */
/* then the union of the slice results is reduced to the top k.            */
/*                                                                          */
/* Counters per (row, slice), [DS] expected-work section:                   */
/*   A    = elements appended,                                              */
/*   R    = compactions inside the loop,                                    */
/*   W    = total input length of all TopK calls, the final one included,  */
/*   peak = largest candidate-buffer length reached.                        */
/* stats (may be NULL) is int64 [rows][splits][4] = {A, R, W, peak}.        */
/* identity_order != 0 visits blocks in index order (diagnostic only).      */
/* ------------------------------------------------------------------------ */

/* TopK by full sort: keep the first k of the sorted candidates. */
static int64_t topk_by_sort(pair_t *cand, int64_t len, int k)
{
    qsort(cand, (size_t)len, sizeof(pair_t), pair_cmp);
    return len < k ? len : k;
}

int ds_oracle_model(const void *x, int dtype, int rows, const int32_t *row_len, int64_t N,
                    int k, int B, int B2, uint64_t seed, int splits, int identity_order,
                    int32_t *out_idx, void *out_val, int64_t *stats)
{
    if (rows < 0 || N < 1 || k < 1 || B < 1 || B2 < 1 || splits < 1 ||
        !dtype_known(dtype))
        return -1;
    int64_t m_max = (N + B - 1) / B;
    pair_t *cand = (pair_t *)malloc((size_t)(N + 1) * sizeof(pair_t));
    pair_t *merged = (pair_t *)malloc((size_t)splits * (size_t)k * sizeof(pair_t));
    uint32_t *perm = (uint32_t *)malloc((size_t)(m_max + 1) * sizeof(uint32_t));
    if (!cand || !merged || !perm) {
        free(cand);
        free(merged);
        free(perm);
        return -1;
    }
    for (int r = 0; r < rows; ++r) {
        int64_t len = valid_length(row_len, r, N);
        int64_t base = (int64_t)r * N;
        int64_t m = (len + B - 1) / B;
        int64_t per_slice = (m + splits - 1) / splits;
        int64_t merged_len = 0;
        for (int c = 0; c < splits; ++c) {
            int64_t first = (int64_t)c * per_slice;
            int64_t last = first + per_slice < m ? first + per_slice : m;
            int64_t ms = last > first ? last - first : 0;
            if (identity_order) {
                for (int64_t i = 0; i < ms; ++i)
                    perm[i] = (uint32_t)(first + i);
            } else if (ds_oracle_permutation((uint32_t)ms, seed, (uint32_t)r, (uint32_t)c,
                                             (uint32_t)first, perm) != 0) {
                free(cand);
                free(merged);
                free(perm);
                return -1;
            }
            int64_t n = 0;                 /* len(topk_candidate) */
            int have_threshold = 0;        /* threshold still -inf */
            pair_t threshold = {0u, 0};
            int64_t A = 0, R = 0, W = 0, peak = 0;
            for (int64_t i = 0; i < ms; ++i) {
                int64_t block = perm[i];
                int64_t lo = block * B;
                int64_t hi = lo + B < len ? lo + B : len;
                for (int64_t j = lo; j < hi; ++j) {
                    pair_t p = {element_key(x, dtype, base + j), (int32_t)j};
                    if (!have_threshold || pair_before(p, threshold)) {
                        cand[n++] = p;
                        ++A;
                    }
                }
                if (n > peak)
                    peak = n;
                if (n >= (int64_t)k + B2) {
                    W += n;
                    n = topk_by_sort(cand, n, k);
                    ++R;
                    threshold = cand[n - 1];   /* smallest kept pair */
                    have_threshold = 1;
                }
            }
            W += n;                            /* the final TopK call */
            n = topk_by_sort(cand, n, k);
            memcpy(merged + merged_len, cand, (size_t)n * sizeof(pair_t));
            merged_len += n;
            if (stats) {
                int64_t *s = stats + ((int64_t)r * splits + c) * 4;
                s[0] = A;
                s[1] = R;
                s[2] = W;
                s[3] = peak;
            }
        }
        int64_t count = topk_by_sort(merged, merged_len, k);
        write_output(x, dtype, base, merged, count, k, out_idx, out_val, (int64_t)r * k);
    }
    free(cand);
    free(merged);
    free(perm);
    return 0;
}
