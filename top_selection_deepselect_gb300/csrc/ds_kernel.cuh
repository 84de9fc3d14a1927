// ds_kernel.cuh -- the DeepSelect top-k kernel for sm_103a (device code).
//
// One CTA (256 threads) scans one row, or one slice of a row when the row is
// split across the CTAs of a thread-block cluster.  The loop is the one of
// PFCCLab/DeepSelect "DeepSelect-deep-dive", section "算法":
//   * the row's B-blocks are visited in a random order drawn from Philox
//     (independent of the data), each one read from HBM exactly once;
//   * every element above the running threshold T is appended to a
//     candidate buffer in shared memory;
//   * after a block, if the buffer holds k + B2 or more entries, a radix
//     select shrinks it to k and T becomes the smallest kept element.
// GB300 mapping:
//   * blocks are staged into a ring of shared-memory stages several stages
//     ahead of the filter by 16-byte asynchronous copies (cp.async): each
//     lane copies exactly the chunks it will filter and waits only on its
//     own copy groups, so the ring needs no barrier of its own;
//   * a stage holds one B-block per `warps_per_block` warps; each lane folds
//     its chunks into one NaN-propagating maximum and compares it once with
//     an unordered test (fp32, or packed bf16x2 / f16x2); only lanes whose
//     maximum passes build exact bit masks (packed compare, prmt, dp4a),
//     which are walked with __ffs (section "实现": one-pass mask + __ffs
//     placement) at slots from a warp scan of lane counts;
//   * the blocks of a stage are filtered in parallel against the same T; a
//     stage is cut at the first block after which the buffer would reach
//     k + B2, the buffer is compacted, and the rest of the stage is filtered
//     again with the new T -- exactly the block-by-block semantics, so the
//     counters A, R, W and the peak length equal the step-by-step model's;
//   * split rows (section "实现", last paragraph): each CTA of the cluster
//     selects the top k of its contiguous slice; the lists meet in CTA 0's
//     shared memory (distributed shared memory), which selects and orders
//     the union -- pruned to the entries at or above the largest slice
//     threshold when the union is large -- or, for the largest unions,
//     merges the slices' sorted lists.
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ds_device.cuh"

namespace cg = cooperative_groups;

namespace ds {

struct Params {
    const void *x;
    const int32_t *row_len;
    int32_t *out_idx;
    void *out_val;
    long long *stats;     // counters {A, R, W, peak} per (row, slice), or null
    long long N;
    long long total;      // elements in x: without row_len, row r holds min(N, total - r*N)
    int k, B, B2;
    unsigned int *check;  // bounds-checked builds: violation bits (null otherwise)
    uint32_t seed_lo, seed_hi;
    int splits;          // CTAs per row
    int wpb;             // warps per B-block (a power of two)
    int wpb_shift;       // log2(wpb)
    int bps;             // B-blocks per stage (kWarps / wpb)
    int stages;          // ring slots (1 for the plain-load path)
    int slot_bytes;      // bytes of one staged block (B * size rounded up to 16)
    int cpw;             // 16-byte chunks per warp of a block
    int cap;             // candidate-buffer entries (free-running scan: overflow bound)
    int identity;        // block-by-block kernel: visit blocks in index order (diagnostic)
    int pairs;           // free-running kernel: the instance that consumes pieces in pairs (capacity sized for it)
    int hist_words;      // histogram region: 3 x 256 words, or kHistWords when a select can exceed 6144 entries
    int off_cand, off_perm, off_hist, off_holes, off_misc;
};

// ---------------------------------------------------------------------------
// Filter of one warp's part of a block.
// ---------------------------------------------------------------------------
struct BlockView {
    const unsigned char *slot;  // shared-memory copy of the block
    int lo, hi;                 // row-local element range [lo, hi)
    int c0, c1;                 // this warp's 16-byte chunks [c0, c1)
    uint32_t t;                 // prefilter operand
    bool refine;                // resolve survivors exactly by composite
    bool plain;                 // no refinement and no partial chunk
};

// Packed unordered a >= t per 16-bit half (0xFFFF where it holds): bf16x2
// for DT = 1, f16x2 for DT = 2.
template <int DT>
__device__ __forceinline__ uint32_t geu2_mask(uint32_t a, uint32_t t)
{
    if (DT == 1)
        return __hgeu2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&a),
                            *reinterpret_cast<const __nv_bfloat162 *>(&t));
    return __hgeu2_mask(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&t));
}

// Prefilter bits of one 16-byte chunk, bit e = element e: !(v < t).
// bf16 / fp16: the packed unordered compare gives 0xFFFF per passing half;
// prmt gathers one byte per element and dp4a folds four 0/1 bytes into four bits
// (section "实现": set.bf16x2 / prmt / dp4a mask generation).
template <int DT>
__device__ __forceinline__ uint32_t prefilter_bits(const uint4 v, uint32_t t)
{
    if (DT == 0) {
        const float tf = __uint_as_float(t);
        return (uint32_t)!(__uint_as_float(v.x) < tf) | ((uint32_t)!(__uint_as_float(v.y) < tf) << 1) |
               ((uint32_t)!(__uint_as_float(v.z) < tf) << 2) |
               ((uint32_t)!(__uint_as_float(v.w) < tf) << 3);
    } else {
        const uint32_t m0 = geu2_mask<DT>(v.x, t);
        const uint32_t m1 = geu2_mask<DT>(v.y, t);
        const uint32_t m2 = geu2_mask<DT>(v.z, t);
        const uint32_t m3 = geu2_mask<DT>(v.w, t);
        const uint32_t lo4 = __byte_perm(m0, m1, 0x7531) & 0x01010101u;
        const uint32_t hi4 = __byte_perm(m2, m3, 0x7531) & 0x01010101u;
        return (uint32_t)__dp4a(lo4, 0x08040201u, 0u) | ((uint32_t)__dp4a(hi4, 0x08040201u, 0u) << 4);
    }
}

template <int DT>
__device__ __forceinline__ uint32_t element_bits(const uint4 v, int e)
{
    if (DT == 0) {
        return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    } else {
        const uint32_t w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
        return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
    }
}

// Exact survivor mask of chunk c of a block that is not plain: elements past
// hi are dropped, and with `refine` every candidate is compared as a
// composite against T.
template <int DT>
__device__ __forceinline__ uint32_t chunk_fixup(uint32_t mask, const uint4 v, int c, const BlockView &bv,
                                                const Threshold &thr)
{
    using E = Elem<DT>;
    const int first = bv.lo + c * E::kPerChunk;
    const int valid = bv.hi - first;
    if (valid < E::kPerChunk)
        mask &= (1u << valid) - 1u;
    if (bv.refine && mask) {
        uint32_t m = mask;
        while (m) {
            const int e = __ffs(m) - 1;
            m &= m - 1u;
            const unsigned long long comp =
                ((unsigned long long)E::key(element_bits<DT>(v, e)) << 32) |
                (unsigned long long)(~(uint32_t)(first + e));
            if (!(comp > thr.comp))
                mask &= ~(1u << e);
        }
    }
    return mask;
}

// Exact survivor masks of one lane's chunks, kept in registers: round r
// (chunk c0 + lane + 32r) occupies kPerChunk bits of the mask words.
template <int DT, int MAXR>
struct MaskRegs {
    static constexpr int kBits = Elem<DT>::kPerChunk;
    static constexpr int kPerWord = 32 / kBits;
    static constexpr int kWords = (MAXR + kPerWord - 1) / kPerWord;
    uint32_t w[kWords];
    __device__ __forceinline__ uint32_t get(int r) const
    {
        return (w[r / kPerWord] >> ((r % kPerWord) * kBits)) & ((1u << kBits) - 1u);
    }
};

// NaN-propagating maxima: if any operand is NaN the result is NaN, so
// !(max < t) holds exactly when !(x < t) holds for some element x.
__device__ __forceinline__ uint32_t max_nan_f32(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.f32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t max_nan_f16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// NaN-propagating maximum of two packed (DT = 1, 2) or single (DT = 0) values.
template <int DT>
__device__ __forceinline__ uint32_t max_nan(uint32_t a, uint32_t b)
{
    return DT == 0 ? max_nan_f32(a, b) : DT == 1 ? max_nan_bf16x2(a, b) : max_nan_f16x2(a, b);
}

template <int DT>
__device__ __forceinline__ uint32_t chunk_max(const uint4 v)
{
    return max_nan<DT>(max_nan<DT>(v.x, v.y), max_nan<DT>(v.z, v.w));
}

// true if some element summarised by the running maximum m passes !(x < t)
template <int DT>
__device__ __forceinline__ bool max_passes(uint32_t m, uint32_t t)
{
    if (DT == 0)
        return !(__uint_as_float(m) < __uint_as_float(t));
    return geu2_mask<DT>(m, t) != 0u;
}

// Survivors of this warp's chunks.  Fast path: every lane folds its chunks
// into one NaN-propagating maximum and compares it once (about half an
// instruction per element); only when some lane passes do the passing lanes
// build exact per-chunk masks, kept in registers (round r = chunk c0 + lane +
// 32r, kPerChunk bits each).  Returns the warp's survivor count; lane_cnt is
// this lane's.
template <int DT, int MAXR>
__device__ __forceinline__ int warp_filter(const BlockView &bv, const Threshold &thr, int lane,
                                           MaskRegs<DT, MAXR> &mk, uint32_t &lane_cnt)
{
    using M = MaskRegs<DT, MAXR>;
    lane_cnt = 0u;
#pragma unroll
    for (int i = 0; i < M::kWords; ++i)
        mk.w[i] = 0u;
    // the identity of the maximum: -inf (any real element or NaN replaces it)
    uint32_t mx = Elem<DT>::splat(Elem<DT>::kNegInfBits);
#pragma unroll
    for (int r = 0; r < MAXR; ++r) {
        const int c = bv.c0 + lane + 32 * r;
        if (c < bv.c1)
            mx = max_nan<DT>(mx, chunk_max<DT>(lds128(bv.slot + c * 16)));
    }
    const bool pass = bv.c0 + lane < bv.c1 && max_passes<DT>(mx, bv.t);
    if (!__any_sync(kFull, pass))
        return 0;
    if (pass) {
#pragma unroll
        for (int r = 0; r < MAXR; ++r) {
            const int c = bv.c0 + lane + 32 * r;
            if (c < bv.c1) {
                const uint4 v = lds128(bv.slot + c * 16);
                uint32_t m = prefilter_bits<DT>(v, bv.t);
                if (!bv.plain)
                    m = chunk_fixup<DT>(m, v, c, bv, thr);
                mk.w[r / M::kPerWord] |= m << ((r % M::kPerWord) * M::kBits);
                lane_cnt += __popc(m);
            }
        }
    }
    return (int)__reduce_add_sync(kFull, lane_cnt);
}

// Appends this warp's survivors at cand[base, base + count): one warp scan of
// the lane counts gives every lane its slot range (predicate / exclusive scan
// / scatter of "Compact"); each lane walks its masks with __ffs.
template <int DT, int MAXR>
__device__ __forceinline__ void warp_append(const BlockView &bv, int lane, const MaskRegs<DT, MAXR> &mk,
                                            uint32_t lane_cnt, unsigned long long *cand, int base)
{
    using E = Elem<DT>;
    const uint32_t incl = warp_inclusive_scan(lane_cnt, lane);
    int pos = base + (int)(incl - lane_cnt);
    if (lane_cnt == 0u)
        return;
#pragma unroll
    for (int r = 0; r < MAXR; ++r) {
        uint32_t m = mk.get(r);
        if (m) {
            const int c = bv.c0 + lane + 32 * r;
            const uint4 v = lds128(bv.slot + c * 16);
            const int first = bv.lo + c * E::kPerChunk;
            do {
                const int e = __ffs(m) - 1;
                m &= m - 1u;
                cand[pos++] = ((unsigned long long)E::key(element_bits<DT>(v, e)) << 32) |
                              (unsigned long long)(~(uint32_t)(first + e));
            } while (m);
        }
    }
}

// ---------------------------------------------------------------------------
// Final order and output: every selected composite goes straight to its rank
// in the output row: index = ~low word, value = the bits its key came from
// (the input is read again only for +-0 and NaN, whose keys do not determine
// the bits).  Positions past cnt get index -1 and -inf.  Caller synchronises.
// ---------------------------------------------------------------------------
// Output pointers of the call and k (what the epilogue needs of Params).
struct Out {
    int32_t *idx;
    void *val;
    int k;
};

template <int DT>
__device__ __forceinline__ void emit(const Out &p, long long obase, int pos,
                                     unsigned long long c, const unsigned char *xrow)
{
    using E = Elem<DT>;
    const int32_t idx = (int32_t)(~(uint32_t)c);
    const uint32_t key = (uint32_t)(c >> 32);
    uint32_t bits;
    if (key == E::kNanKey || key == E::kZeroKey)
        bits = DT == 0 ? reinterpret_cast<const uint32_t *>(xrow)[idx]
                       : reinterpret_cast<const uint16_t *>(xrow)[idx];
    else
        bits = E::bits_of_key(key);
    p.idx[obase + pos] = idx;
    if (DT == 0)
        reinterpret_cast<uint32_t *>(p.val)[obase + pos] = bits;
    else
        reinterpret_cast<uint16_t *>(p.val)[obase + pos] = (uint16_t)bits;
}

template <int DT, int E>
__device__ __forceinline__ void emit_runs(unsigned long long *arr, int cnt, const Out &p,
                                          long long obase, const unsigned char *xrow)
{
    const int P = 256 * E;
    for (int i = cnt + threadIdx.x; i < P; i += kThreads)
        arr[i] = 0ull;
    __syncthreads();
    unsigned long long vals[E];
    int ranks[E];
    rank_desc_runs<E>(arr, vals, ranks);
#pragma unroll
    for (int j = 0; j < E; ++j)
        if (vals[j] != 0ull && ranks[j] < p.k)
            emit<DT>(p, obase, ranks[j], vals[j], xrow);
}

// Outputs a thread holds in registers in one round of a merge-path sort.
constexpr int kMergeOut = 16;
// Split rows whose union of slice results (splits * k) exceeds
// kClusterSelectMinUnion take the select across the cluster when k is at
// most kClusterSelectMaxK (a slice's entries fit the register select after
// its own select at most); smaller unions go to CTA 0 whole, and unions of
// larger k go there pruned.
constexpr int kClusterSelectMaxK = 24 * kThreads;
constexpr int kClusterSelectMinUnion = 24 * kThreads;

// Outputs [t0, t1) (at most kMergeOut) of the descending merge of runs A[0, la)
// and B[0, lb): a merge-path search finds how many of the first t0 come from
// A, then the two runs are walked.  Distinct nonzero entries; 0 pads.
__device__ __forceinline__ void merge_chunk(const unsigned long long *A, int la,
                                            const unsigned long long *B, int lb, int t0, int t1,
                                            unsigned long long (&out)[kMergeOut])
{
    int lo = t0 - lb > 0 ? t0 - lb : 0, hi = t0 < la ? t0 : la;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (A[mid] > B[t0 - mid - 1])
            lo = mid + 1;
        else
            hi = mid;
    }
    int i = lo, j = t0 - lo;
#pragma unroll
    for (int q = 0; q < kMergeOut; ++q) {
        if (q < t1 - t0) {
            const unsigned long long a = i < la ? A[i] : 0ull;
            const unsigned long long b = j < lb ? B[j] : 0ull;
            const bool ta = a > b;
            out[q] = ta ? a : b;
            i += ta ? 1 : 0;
            j += ta ? 0 : 1;
        }
    }
}


// Sorts the cnt distinct nonzero entries arr[0, cnt) descending, 256 < cnt
// <= 2048 (used above 1024, where it beats ranking across runs of 256 per
// warp); arr holds pow2_ceil(cnt) entries (the pads are 0 and sort last).
// Each warp sorts runs of 64 in registers (bitonic), then runs are merged
// pairwise in rounds of doubling width: every thread produces its own
// consecutive outputs of a merge (merge-path search, then a walk), holds
// them in registers across a barrier and stores them in place.  With TO_OUT
// the last round writes the first kout outputs to the row instead.
template <int DT, bool TO_OUT>
__device__ __forceinline__ void merge_sort_desc(unsigned long long *arr, int cnt, int kout,
                                                const Out &p, long long obase,
                                                const unsigned char *xrow)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = pow2_ceil(cnt);  // 512, 1024 or 2048
    for (int i = cnt + tid; i < P; i += kThreads)
        arr[i] = 0ull;
    __syncthreads();
    for (int r = warp; r < P / 64; r += kWarps) {
        unsigned long long v[2] = {arr[64 * r + lane], arr[64 * r + 32 + lane]};
        warp_bitonic_regs<2>(v, lane, true);
        arr[64 * r + lane] = v[0];
        arr[64 * r + 32 + lane] = v[1];
    }
    __syncthreads();
    const int per = P / kThreads;  // outputs per thread: 2, 4 or 8
    const int t0 = tid * per;
    const int lim = cnt < kout ? cnt : kout;
    for (int w = 64; w < P; w *= 2) {
        const int pair = t0 / (2 * w), local = t0 % (2 * w);
        const unsigned long long *A = arr + (size_t)pair * 2 * w;
        unsigned long long out[kMergeOut];
        merge_chunk(A, w, A + w, w, local, local + per, out);
        if (TO_OUT && 2 * w == P) {
#pragma unroll
            for (int q = 0; q < kMergeOut; ++q)
                if (q < per && t0 + q < lim)
                    emit<DT>(p, obase, t0 + q, out[q], xrow);
            return;
        }
        __syncthreads();  // every read of this round's runs is done
#pragma unroll
        for (int q = 0; q < kMergeOut; ++q)
            if (q < per)
                arr[t0 + q] = out[q];
        __syncthreads();
    }
}

// Orders 256 < cnt <= 1024 distinct entries and writes them: entries are
// bucketed by their top eight varying bits (histogram, a scan from the top
// bucket down, scatter into bucket order) and each entry is then ranked only
// against the members of its own bucket.  Returns false, having written
// nothing, when a bucket holds more than kBucketMax entries (the caller then
// ranks across warp runs).  `scratch` is 768 free words of shared memory.
constexpr int kBucketMax = 128;

template <int DT>
__device__ __forceinline__ bool bucket_sort_write(unsigned long long *arr, int cnt, const Out &p,
                                                  long long obase, const unsigned char *xrow,
                                                  uint32_t *scratch, Misc *ms)
{
    constexpr int R = 4;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t hi[R], lo[R], dg[R], valid = 0u;
    uint32_t oh = 0u, ol = 0u, ah = ~0u, al = ~0u;
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const int i = tid + kThreads * j;
        hi[j] = 0u;
        lo[j] = 0u;
        if (i < cnt) {
            const unsigned long long c = arr[i];
            hi[j] = (uint32_t)(c >> 32);
            lo[j] = (uint32_t)c;
            valid |= 1u << j;
            oh |= hi[j];
            ol |= lo[j];
            ah &= hi[j];
            al &= lo[j];
        }
    }
    oh = __reduce_or_sync(kFull, oh);
    ol = __reduce_or_sync(kFull, ol);
    ah = __reduce_and_sync(kFull, ah);
    al = __reduce_and_sync(kFull, al);
    if (lane == 0) {
        ms->wor[warp] = ((unsigned long long)oh << 32) | ol;
        ms->wand[warp] = ((unsigned long long)ah << 32) | al;
    }
    uint32_t *cntb = scratch, *offb = scratch + 256, *fillb = scratch + 512;
    cntb[tid] = 0u;
    fillb[tid] = 0u;
    __syncthreads();  // also: every load of arr is done
    unsigned long long vo = 0ull, va = ~0ull;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        vo |= ms->wor[w];
        va &= ms->wand[w];
    }
    const unsigned long long vary = vo ^ va;
    const int h = 63 - __clzll((long long)vary);  // cnt > 1 distinct entries: vary != 0
    const int sh = h >= 7 ? h - 7 : 0;
#pragma unroll
    for (int j = 0; j < R; ++j) {
        dg[j] = (sh >= 32 ? hi[j] >> (sh - 32) : __funnelshift_r(lo[j], hi[j], sh)) & 255u;
        if ((valid >> j) & 1u)
            atomicAdd(&cntb[dg[j]], 1u);
    }
    __syncthreads();
    if (warp == 0) {
        // offb[d] = entries in higher buckets; lane l owns buckets 8l .. 8l+7
        const uint4 q0 = *reinterpret_cast<const uint4 *>(cntb + lane * 8);
        const uint4 q1 = *reinterpret_cast<const uint4 *>(cntb + lane * 8 + 4);
        const uint32_t c[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const uint32_t tot = ((c[0] + c[1]) + (c[2] + c[3])) + ((c[4] + c[5]) + (c[6] + c[7]));
        uint32_t suf = tot;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_down_sync(kFull, suf, d);
            if (lane + d < 32)
                suf += o;
        }
        uint32_t run = suf - tot;  // entries in the buckets of higher lanes
        uint32_t mx = 0u;
#pragma unroll
        for (int t = 7; t >= 0; --t) {
            offb[lane * 8 + t] = run;
            run += c[t];
            mx = c[t] > mx ? c[t] : mx;
        }
        mx = __reduce_max_sync(kFull, mx);
        if (lane == 0)
            ms->sel_eq = mx;
    }
    __syncthreads();
    if (ms->sel_eq > (uint32_t)kBucketMax)
        return false;  // uniform: every thread read the same word
    int slot[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
        slot[j] = 0;
        if ((valid >> j) & 1u) {
            slot[j] = (int)offb[dg[j]] + (int)atomicAdd(&fillb[dg[j]], 1u);
            arr[slot[j]] = ((unsigned long long)hi[j] << 32) | lo[j];
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < R; ++j) {
        if ((valid >> j) & 1u) {
            const unsigned long long e = ((unsigned long long)hi[j] << 32) | lo[j];
            const int b0 = (int)offb[dg[j]], bn = (int)cntb[dg[j]];
            int r = 0;
            for (int i = b0; i < b0 + bn; ++i)
                r += arr[i] > e ? 1 : 0;
            if (b0 + r < p.k)
                emit<DT>(p, obase, b0 + r, e, xrow);
        }
    }
    return true;
}

template <int DT>
__device__ __forceinline__ void sort_and_write(unsigned long long *arr, int cnt, const Out &p, int row,
                                               const unsigned char *xrow, uint32_t *scratch, Misc *ms,
                                               int room)
{
    using E = Elem<DT>;
    const long long obase = (long long)row * p.k;
    for (int i = cnt + threadIdx.x; i < p.k; i += kThreads) {
        p.idx[obase + i] = -1;
        if (DT == 0)
            reinterpret_cast<uint32_t *>(p.val)[obase + i] = E::kNegInfBits;
        else
            reinterpret_cast<uint16_t *>(p.val)[obase + i] = (uint16_t)E::kNegInfBits;
    }
    if (cnt <= kThreads && cnt > 64 && room >= kThreads) {
        // ranks from warp-sorted runs and binary searches; with cnt > k only
        // ranks below k are written, so this also selects
        for (int i = cnt + threadIdx.x; i < kThreads; i += kThreads)
            arr[i] = 0ull;
        __syncthreads();
        unsigned long long vals[1];
        int ranks[1];
        rank_desc_runs<1>(arr, vals, ranks);
        if (vals[0] != 0ull && ranks[0] < p.k)
            emit<DT>(p, obase, ranks[0], vals[0], xrow);
    } else if (cnt <= kThreads) {
        // every thread ranks one entry; with cnt > k only ranks below k are
        // written, so this also selects
        const int t = threadIdx.x;
        if (t < cnt) {
            const unsigned long long e = arr[t];
            int rank = 0;
#pragma unroll 8
            for (int j = 0; j < cnt; ++j)
                rank += arr[j] > e ? 1 : 0;
            if (rank < p.k)
                emit<DT>(p, obase, rank, e, xrow);
        }
    } else if (cnt <= 1024) {
        if (!bucket_sort_write<DT>(arr, cnt, p, obase, xrow, scratch, ms)) {
            if (cnt <= 512)
                emit_runs<DT, 2>(arr, cnt, p, obase, xrow);
            else
                emit_runs<DT, 4>(arr, cnt, p, obase, xrow);
        }
    } else if (cnt <= 2048) {
        merge_sort_desc<DT, true>(arr, cnt, p.k, p, obase, xrow);
    } else {
        const int P = pow2_ceil(cnt);
        for (int i = cnt + threadIdx.x; i < P; i += kThreads)
            arr[i] = 0ull;
        __syncthreads();
        bitonic_sort_smem(arr, P, true);
        for (int i = threadIdx.x; i < cnt; i += kThreads)
            emit<DT>(p, obase, i, arr[i], xrow);
    }
}

// Sorts the cnt distinct entries arr[0, cnt) descending, in place (the same
// rank computations as sort_and_write; every entry moves to its rank).  arr
// holds pow2_ceil(cnt) entries.  Caller synchronises before; ends
// synchronised.
// ---------------------------------------------------------------------------
// The top k of a split row by one RadixSelectTopK ("算法", step 3) over the
// union of the slices' candidates, taken across the cluster: no slice
// selects, sorts or ships its own top k first.  Each pass every CTA counts
// its live entries into its own 256-bin histogram; after a cluster barrier
// every CTA sums the S histograms through distributed shared memory, so all
// of them see the same counts and take the same digit decisions (warp 0's
// digit search, as in radix_select_regs).  The passes go on until every
// entry of the chosen digit is needed; the composites are distinct, so the
// selected entries (higher digits, plus that digit) are exactly the k
// largest of the union.  Each CTA then copies its selected entries into
// CTA 0's buffer `dst0` after those of the lower slices.  Histograms rotate
// over three buffers (cleared on entry), and a buffer is cleared again one
// cluster barrier after the pass whose sums read it; the sums go to a fourth
// 256-word buffer, and all four are left zero.  All
// threads of all CTAs of the cluster call it (every CTA passes the same
// cluster barriers); it returns the number of entries in dst0, which is
// min(k, size of the union), and ends with CTA 0's copy complete.
// ---------------------------------------------------------------------------
static_assert(4 * kHistBins <= kHistWords, "the cluster select uses four histogram buffers");

template <int R>
static __device__ __noinline__ int cluster_select(const unsigned long long *cand, int n, int k, int S,
                                                  unsigned long long *dst0, int dst_room,
                                                  uint32_t *whist, Misc *ms)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slice = (int)cluster.block_rank();
    uint32_t hi[R], lo[R], dg[R];
    uint32_t valid = 0u;
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const int i = tid + kThreads * j;
        hi[j] = 0u;
        lo[j] = 0u;
        dg[j] = 0u;
        if (i < n) {
            const unsigned long long c = cand[i];
            hi[j] = (uint32_t)(c >> 32);
            lo[j] = (uint32_t)c;
            valid |= 1u << j;
        }
    }
    // bits that vary over the union, and its size
    uint32_t oh = 0u, ol = 0u, ah = ~0u, al = ~0u;
#pragma unroll
    for (int j = 0; j < R; ++j) {
        if (valid & (1u << j)) {
            oh |= hi[j];
            ol |= lo[j];
            ah &= hi[j];
            al &= lo[j];
        }
    }
    oh = __reduce_or_sync(kFull, oh);
    ol = __reduce_or_sync(kFull, ol);
    ah = __reduce_and_sync(kFull, ah);
    al = __reduce_and_sync(kFull, al);
    if (lane == 0) {
        ms->wor[warp] = ((unsigned long long)oh << 32) | ol;
        ms->wand[warp] = ((unsigned long long)ah << 32) | al;
    }
    // the selects of the scan leave two of their three rotating buffers
    // dirty: clear all four here (nothing reads them remotely yet)
#pragma unroll
    for (int b = 0; b < 4; ++b)
        whist[b * kHistBins + tid] = 0u;
    __syncthreads();
    if (tid == 0) {
        unsigned long long vo = 0ull, va = ~0ull;
        for (int w = 0; w < kWarps; ++w) {
            vo |= ms->wor[w];
            va &= ms->wand[w];
        }
        ms->cl_or = vo;
        ms->cl_and = va;
        ms->cl_n = n;
    }
    cluster.sync();  // every slice's summary is published; the buffers are clear
    unsigned long long go = 0ull, ga = ~0ull;
    long long tot = 0;
    for (int s = 0; s < S; ++s) {
        const Misc *pm = cluster.map_shared_rank(ms, s);
        go |= pm->cl_or;  // an empty slice has OR 0 and AND all ones
        ga &= pm->cl_and;
        tot += pm->cl_n;
    }
    uint32_t sel = valid;
    int last = -1;  // histogram buffer of the last pass
    uint32_t *sums = whist + 3 * kHistBins;
    if (tot > k) {
        const unsigned long long vary = go ^ ga;  // nonzero: at least two distinct entries
        uint32_t need = (uint32_t)k, live = valid, above = 0u;
        int h = 63 - __clzll((long long)vary);
        int pass = 0;
        while (true) {
            const int sh = h >= 7 ? h - 7 : 0;
            uint32_t *cur = whist + (pass % 3) * kHistBins;
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const uint32_t d = (sh >= 32 ? hi[j] >> (sh - 32) : __funnelshift_r(lo[j], hi[j], sh)) & 255u;
                dg[j] = d;
                if (live & (1u << j))
                    atomicAdd(&cur[d], 1u);
            }
            cluster.sync();  // every slice's counts of this pass are in
            if (pass >= 1)
                whist[((pass - 1) % 3) * kHistBins + tid] = 0u;  // every slice summed it before the barrier
            uint32_t g = 0u;
            for (int s = 0; s < S; ++s)
                g += cluster.map_shared_rank(cur, s)[tid];
            sums[tid] = g;
            __syncthreads();
            if (warp == 0)
                digit_search(sums, need, lane, ms);
            __syncthreads();
            const uint32_t dsel = ms->sel_digit, eq = ms->sel_eq;
            need -= ms->sel_above;
            last = pass % 3;
            ++pass;
#pragma unroll
            for (int j = 0; j < R; ++j) {
                if (live & (1u << j)) {
                    if (dg[j] > dsel)
                        above |= 1u << j;
                    if (dg[j] != dsel)
                        live &= ~(1u << j);
                }
            }
            if (eq == need)
                break;
            const unsigned long long below = sh > 0 ? (vary & ((1ull << sh) - 1ull)) : 0ull;
            if (below == 0ull)
                break;  // unreachable for distinct composites; keeps the loop finite
            h = 63 - __clzll((long long)below);
        }
        sel = above | live;
    }
    // this slice's selected entries go to CTA 0 after the lower slices' ones
    const int mine = warp_count<R>(sel);
    if (lane == 0)
        ms->wsum[warp] = (uint32_t)mine;
    __syncthreads();
    int wbase = 0, cnt = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        wbase += w < warp ? (int)ms->wsum[w] : 0;
        cnt += (int)ms->wsum[w];
    }
    if (tid == 0)
        ms->cl_cnt = cnt;
    cluster.sync();  // counts published; every slice has summed the last histograms
    if (last >= 0)
        whist[last * kHistBins + tid] = 0u;
    sums[tid] = 0u;
    int base = 0, total = 0;
    for (int s = 0; s < S; ++s) {
        const int c = cluster.map_shared_rank(ms, s)->cl_cnt;
        base += s < slice ? c : 0;
        total += c;
    }
    if (DS_GUARD(ms, base + cnt <= dst_room, 64u))
        warp_scatter<R>(sel, hi, lo, cluster.map_shared_rank(dst0, 0) + base + wbase, lane);
    cluster.sync();  // CTA 0 holds the selected entries
    return total;
}

// A split row with a large union: the row's top k by one select across
// the cluster into CTA 0's ring (free once every CTA has finished
// streaming, which the select's first cluster barrier ensures), then CTA 0
// orders it.  cnt = this slice's entries in cand.  A function of its own:
// inside finish_slice it grew the stream kernel's stack frame (ptxas).
template <int DT>
static __device__ __noinline__ void finish_by_cluster(const Out o, unsigned char *ring, unsigned long long *cand,
                                                      uint32_t *whist, Misc *ms, int cnt, int S, int row,
                                                      int slice, const unsigned char *xrow)
{
    unsigned long long *dst = reinterpret_cast<unsigned long long *>(ring);
    const int droom = (int)(cand - dst);
    int total;
    if (cnt <= 4 * kThreads)
        total = cluster_select<4>(cand, cnt, o.k, S, dst, droom, whist, ms);
    else if (cnt <= 8 * kThreads)
        total = cluster_select<8>(cand, cnt, o.k, S, dst, droom, whist, ms);
    else if (cnt <= 12 * kThreads)
        total = cluster_select<12>(cand, cnt, o.k, S, dst, droom, whist, ms);
    else
        total = cluster_select<24>(cand, cnt, o.k, S, dst, droom, whist, ms);
    if (slice == 0)
        sort_and_write<DT>(dst, total < o.k ? total : o.k, o, row, xrow, whist, ms, droom);
}

// ---------------------------------------------------------------------------
// Epilogue of one slice: final TopK, counters, then the ordered output (one
// CTA per row) or the cluster merge (split rows).  A separate function so
// that the streaming loop is compiled on its own.  Called by all threads
// after the scan; the candidate buffer holds n entries.  WIDE = false
// leaves out the select across the cluster, for callers whose splits * k
// never exceeds kClusterSelectMinUnion.
// ---------------------------------------------------------------------------
template <int DT, bool WIDE = true>
static __device__ __noinline__ void finish_slice(const Out o, long long *stats, unsigned char *ring,
                                                 unsigned long long *cand, int room, uint32_t *whist,
                                                 uint16_t *holes, Misc *ms, int n, int S, int row,
                                                 int slice, const unsigned char *xrow, int A, int R,
                                                 int W, int peak)
{
    const int tid = threadIdx.x;
    W += n;
    // one CTA per row with at most 1024 entries: ordering them all and
    // writing the first k selects them too (sort_and_write), cheaper than a
    // select followed by the order of k (DSA index scores: 552 entries, k = 512)
    const bool rank_all = S == 1 && (n <= kThreads || (n <= 4 * kThreads && room >= 4 * kThreads));
    // a split row with a large union: one select over the whole cluster,
    // which takes a slice's candidates as they are when they fit registers
    const bool by_cluster =
        WIDE && S > 1 && o.k <= kClusterSelectMaxK && (long long)S * o.k > kClusterSelectMinUnion;
    const bool whole = by_cluster && n <= 24 * kThreads;
    unsigned long long tk = 0ull;  // this slice's k-th composite (0: fewer than k entries)
    if (n > o.k && !rank_all && !whole)
        tk = select_topk(cand, n, o.k, room, whist, holes, ms);
    const int cnt = rank_all || whole ? n : (n < o.k ? n : o.k);
    if (stats != nullptr && tid == 0) {
        long long *s = stats + ((long long)row * S + slice) * 4;
        s[0] = A;
        s[1] = R;
        s[2] = W;
        s[3] = peak;
    }

    if (S == 1) {
        sort_and_write<DT>(cand, cnt, o, row, xrow, whist, ms, room);
        return;
    }

    // -- split rows: partial top-k of every slice into CTA 0 -------------------
    cg::cluster_group cluster = cg::this_cluster();
    if (by_cluster) {
        finish_by_cluster<DT>(o, ring, cand, whist, ms, cnt, S, row, slice, xrow);
        return;
    }
    // otherwise CTA 0 selects the top k of the union and orders it.  For a
    // large union: the row's k-th composite is at least every slice's k-th
    // (that slice alone holds k entries at or above it), so a slice sends
    // CTA 0 only its entries at or above the largest slice threshold --
    // exact, and often only k entries in all (sorted or heavily tied rows).
    // Used when the union would not fit the register select (S*k > 6144).
    const bool prune = (long long)S * o.k > 24LL * kThreads;
    if (prune && tid < S)
        *cluster.map_shared_rank(&ms->tslice[slice], tid) = tk;
    cluster.sync();  // thresholds published; every CTA has finished streaming; CTA 0's ring is free
    unsigned long long tmax = 0ull;
    if (prune)
        for (int s2 = 0; s2 < S; ++s2)
            tmax = ms->tslice[s2] > tmax ? ms->tslice[s2] : tmax;
    if (!prune) {
        if (tid == 0)
            ms->merge_off = atomicAdd(cluster.map_shared_rank(&ms->merge_count, 0), cnt);
        __syncthreads();
        unsigned long long *dst =
            cluster.map_shared_rank(reinterpret_cast<unsigned long long *>(ring), 0) + ms->merge_off;
        if (DS_GUARD(ms, ms->merge_off + cnt <= cand - reinterpret_cast<unsigned long long *>(ring), 16u))
            for (int i = tid; i < cnt; i += kThreads)
                dst[i] = cand[i];
    } else {
        // the kept entries of each warp's stripes, then one remote atomic per
        // CTA for the slots in CTA 0, then the stores
        const int lane = tid & 31, warp = tid >> 5;
        uint32_t mine = 0u;
        for (int i0 = warp * 32; i0 < cnt; i0 += kThreads) {
            const int i = i0 + lane;
            mine += (uint32_t)__popc(__ballot_sync(kFull, i < cnt && cand[i] >= tmax));
        }
        if (lane == 0)
            ms->wsum[warp] = mine;
        __syncthreads();
        if (tid == 0) {
            int tot = 0;
            for (int w = 0; w < kWarps; ++w)
                tot += (int)ms->wsum[w];
            ms->merge_off = tot ? atomicAdd(cluster.map_shared_rank(&ms->merge_count, 0), tot) : 0;
        }
        __syncthreads();
        int base = ms->merge_off;
        for (int w = 0; w < warp; ++w)
            base += (int)ms->wsum[w];
        unsigned long long *dst = cluster.map_shared_rank(reinterpret_cast<unsigned long long *>(ring), 0);
        if (DS_GUARD(ms, base + (int)mine <= cand - reinterpret_cast<unsigned long long *>(ring), 32u))
        for (int i0 = warp * 32; i0 < cnt; i0 += kThreads) {
            const int i = i0 + lane;
            const unsigned long long c = i < cnt ? cand[i] : 0ull;
            const bool keep = i < cnt && c >= tmax;
            const uint32_t b = __ballot_sync(kFull, keep);
            if (keep)
                dst[base + __popc(b & lanemask_lt(lane))] = c;
            base += __popc(b);
        }
    }
    cluster.sync();
    if (slice != 0)
        return;
    const int total = ms->merge_count;
    const int kk = total < o.k ? total : o.k;
    unsigned long long *merged = reinterpret_cast<unsigned long long *>(ring);
    if (total > kk)
        select_topk(merged, total, kk, (int)(cand - merged), whist, holes, ms);
    sort_and_write<DT>(merged, kk, o, row, xrow, whist, ms, (int)(cand - merged));
}

// ---------------------------------------------------------------------------
// The kernel.  grid = rows * splits, cluster = (splits, 1, 1) when splits > 1.
// ---------------------------------------------------------------------------
template <int DT, bool ASYNC, int MAXR>
__global__ void __launch_bounds__(kThreads, 2) deepselect_topk_kernel(const Params p)
{
    allow_dependent_grid();
    dependent_grid_wait();  // before the first read of x, row_len or the outputs
    using E = Elem<DT>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = p.splits;
    const int row = blockIdx.x / S, slice = blockIdx.x % S;

    unsigned char *ring = smem;
    unsigned long long *cand = reinterpret_cast<unsigned long long *>(smem + p.off_cand);
    unsigned long long *perm = reinterpret_cast<unsigned long long *>(smem + p.off_perm);
    uint32_t *whist = reinterpret_cast<uint32_t *>(smem + p.off_hist);
    uint16_t *holes = reinterpret_cast<uint16_t *>(smem + p.off_holes);
    Misc *ms = reinterpret_cast<Misc *>(smem + p.off_misc);

    long long len_ll = p.row_len ? (long long)p.row_len[row] : p.total - (long long)row * p.N;
    len_ll = len_ll < 0 ? 0 : (len_ll > p.N ? p.N : len_ll);
    const int len = (int)len_ll;
    const int B = p.B;
    const int m = (int)((len_ll + B - 1) / B);
    const int per = (m + S - 1) / S;
    const int first_block = slice * per;
    const int msl = max(0, min(per, m - first_block));  // blocks of this slice
    const unsigned char *xrow =
        reinterpret_cast<const unsigned char *>(p.x) + (size_t)row * (size_t)p.N * E::kSize;

    // -- random block order: ascending (Philox word 0, block id) -------------
    const int P = pow2_ceil(msl > 32 ? msl : 32);
    for (int i = tid; i < P; i += kThreads) {
        unsigned long long v = ~0ull;
        if (i < msl) {
            const uint32_t b = (uint32_t)(first_block + i);
            const uint32_t w =
                p.identity ? 0u : philox_word0(b, (uint32_t)row, (uint32_t)slice, 0u, p.seed_lo, p.seed_hi);
            v = ((unsigned long long)w << 32) | b;
        }
        perm[i] = v;
    }
    if (tid == 0) {
        ms->merge_count = 0;
        ms->pass = 0;
        ms->check = p.check;
    }
    __syncthreads();
    sort_asc_small(perm, msl, P, reinterpret_cast<unsigned long long *>(whist));  // histogram space as scratch
    for (int i = tid; i < p.hist_words; i += kThreads)
        whist[i] = 0u;  // ordered before the first select by its barriers

    const int bps = p.bps;
    const int nst = (msl + bps - 1) / bps;
    const int esz = E::kSize;
    const int g = warp >> p.wpb_shift, sub = warp & (p.wpb - 1);
    const int NS = ASYNC ? p.stages : 1;  // ring slots

    // Every lane copies its own 16-byte chunks of this warp's part of the
    // block at stage st into ring slot `slot` with cp.async and commits one
    // group per stage (possibly empty).  A lane later reads only chunks it
    // copied itself, so waiting on its own groups is all the synchronisation
    // the ring needs.  The partial last chunk of a row is loaded at use.
    auto prefetch = [&](int st, int slot) {
        const int q = st * bps + g;
        if (st < nst && q < msl) {
            const int lo = (int)(uint32_t)perm[q] * B;
            const int nbytes = (min(lo + B, len) - lo) * esz;
            const int nch = (nbytes + 15) >> 4;
            const int c0 = min(sub * p.cpw, nch), c1 = min(c0 + p.cpw, nch);
            unsigned char *dst = ring + (size_t)(slot * bps + g) * p.slot_bytes;
            const unsigned char *src = xrow + (size_t)lo * esz;
            for (int c = c0 + lane; c < c1; c += 32)
                if ((c + 1) * 16 <= nbytes)
                    cp_async16(smem_addr(dst + c * 16), src + c * 16);
        }
        cp_async_commit();
    };
    if (ASYNC)
        for (int s = 0; s < NS - 1; ++s)
            prefetch(s, s);

    Threshold thr = threshold_initial<DT>();
    int n = 0;                          // candidates in the buffer
    int A = 0, R = 0, W = 0, peak = 0;  // counters of the slice (all below 2^31)
    int ip = 0;                         // parity of the survivor-count buffer
    int slot = 0;                       // ring slot of the current stage
    const int kB2 = p.k + p.B2;

    for (int st = 0; st < nst; ++st) {
        if (ASYNC) {
            // refill the slot this lane finished with (stage st-1)
            prefetch(st + NS - 1, slot == 0 ? NS - 1 : slot - 1);
            cp_async_wait_pending(NS - 1);  // this lane's copies of stage st landed
        }

        BlockView bv;
        const int q = st * bps + g;
        const bool has = q < msl;
        bv.slot = ring + (size_t)(slot * bps + g) * p.slot_bytes;
        bv.lo = has ? (int)(uint32_t)perm[q] * B : 0;
        bv.hi = has ? min(bv.lo + B, len) : 0;
        const int nbytes = (bv.hi - bv.lo) * esz;
        const int nch = (nbytes + 15) >> 4;
        bv.c0 = min(sub * p.cpw, nch);
        bv.c1 = min(bv.c0 + p.cpw, nch);
        slot = slot + 1 == NS ? 0 : slot + 1;

        // chunks not copied ahead (plain-load path, or the ragged tail of a
        // row) are loaded by the lane that will filter them
        if (has && (!ASYNC || (nbytes & 15))) {
            const int async_end = ASYNC ? (nbytes & ~15) : 0;
            for (int c = bv.c0 + lane; c < bv.c1; c += 32) {
                if (c * 16 >= async_end) {
                    unsigned char *dst = const_cast<unsigned char *>(bv.slot) + c * 16;
                    for (int e = 0; e < E::kPerChunk; ++e) {
                        const int j = bv.lo + c * E::kPerChunk + e;
                        if (j < bv.hi) {
                            if (DT == 0)
                                reinterpret_cast<uint32_t *>(dst)[e] =
                                    reinterpret_cast<const uint32_t *>(xrow)[j];
                            else
                                reinterpret_cast<uint16_t *>(dst)[e] =
                                    reinterpret_cast<const uint16_t *>(xrow)[j];
                        }
                    }
                }
            }
        }

        int gstart = 0;
        while (true) {
            const bool mine = has && g >= gstart;
            MaskRegs<DT, MAXR> mk;
            uint32_t lane_cnt = 0u;
            int cnt = 0;
            if (mine) {
                const bool ge = (uint32_t)bv.lo < thr.ti;
                bv.t = ge ? thr.t_ge : thr.t_gt;
                bv.refine = ge ? (thr.nan_ge || (uint32_t)bv.hi > thr.ti) : thr.nan_gt;
                bv.plain = !bv.refine && ((bv.hi - bv.lo) & (E::kPerChunk - 1)) == 0;
                cnt = warp_filter<DT, MAXR>(bv, thr, lane, mk, lane_cnt);
            }
            int *cw = ms->cntw[ip];
            ip ^= 1;
            if (lane == 0)
                cw[warp] = cnt;
            if (!__syncthreads_or(cnt != 0))
                break;
            // blocks in stage order; find the first one after which the
            // buffer reaches k + B2
            int run = n, trig = -1, before_me = 0;
            {
                const int4 ca = reinterpret_cast<const int4 *>(cw)[0];
                const int4 cb = reinterpret_cast<const int4 *>(cw)[1];
                const int cv[kWarps] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
                const int wmask = p.wpb - 1;
#pragma unroll
                for (int w2 = 0; w2 < kWarps; ++w2) {
                    if (trig < 0 && w2 >= (gstart << p.wpb_shift)) {
                        if (w2 < warp)
                            before_me += cv[w2];
                        run += cv[w2];
                        if ((w2 & wmask) == wmask && run >= kB2)
                            trig = w2 >> p.wpb_shift;
                    }
                }
            }
            const int gend = trig >= 0 ? trig : bps - 1;
            if (mine && g <= gend && cnt &&
                DS_GUARD(ms, n + before_me + cnt <= ((p.off_perm - p.off_cand) >> 3), 1u))
                warp_append<DT, MAXR>(bv, lane, mk, lane_cnt, cand, n + before_me);
            A += run - n;
            peak = run > peak ? run : peak;
            n = run;
            if (trig < 0)
                break;  // the next barrier orders these appends before any reader
            W += n;
            R += 1;
            __syncthreads();  // every warp's appends are in the buffer
            const unsigned long long tcomp =
                select_topk(cand, n, p.k, (p.off_perm - p.off_cand) >> 3, whist, holes, ms);
            n = p.k;
            thr = threshold_from<DT>(tcomp);
            gstart = trig + 1;
            if (gstart >= bps)
                break;
        }
    }
    if (ASYNC)
        cp_async_wait_pending(0);
    __syncthreads();  // appends of the last stage are visible

    finish_slice<DT>(Out{p.out_idx, p.out_val, p.k}, p.stats, ring, cand, (p.off_perm - p.off_cand) >> 3,
                     whist, holes, ms, n, S, row, slice, xrow, A, R, W, peak);
}

typedef void (*KernelFn)(Params);

// Kernel entry points of one dtype, defined in ds_kernels_<dtype>.cu.
KernelFn kernel_fp32(bool async, bool wide);
KernelFn kernel_bf16(bool async, bool wide);
KernelFn kernel_fp16(bool async, bool wide);

}  // namespace ds
