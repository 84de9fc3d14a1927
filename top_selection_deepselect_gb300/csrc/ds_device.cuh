// ds_device.cuh -- device-side building blocks of the DeepSelect top-k kernel
// for sm_103a: order keys, Philox4x32-10, asynchronous-copy wrappers, warp
// scans, the shared-memory radix select and the ordering of the final k.
//
// Sources (page title, section):
//   PFCCLab/DeepSelect "DeepSelect-deep-dive", "算法" (scan / filter /
//     compact loop, RadixSelectTopK) and "实现" (one-pass bit-mask filter
//     walked with __ffs, warp prefix sums, histograms, cluster split rows);
//   milkfeng.top "CUDA 算子笔记 4", "Top K Selection" / "改造 Radix Sort"
//     (order-preserving float -> unsigned key, 8-bit digit select, bitonic
//     order of the final k);
//   elainafan.one "并行算法（一）", "Scan" and "Compact" (Hillis-Steele scan,
//     predicate / scan / scatter compaction);
//   Salmon et al., SC'11 (Philox4x32-10).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ds {

constexpr int kThreads = 256;             // threads per CTA
constexpr int kWarps = kThreads / 32;     // warps per CTA
constexpr int kMaxStages = 4;             // deepest shared-memory ring

// Bounds-checked builds (-DDS_CHECKED, built by the tests): DS_GUARD(ms,
// cond, bit) records `bit` in the word ms->check and yields false when a
// computed shared-memory range is out of bounds, so the write is skipped
// instead of corrupting memory (nothing traps).  In the product build it is
// the constant true and its condition is not compiled.
#ifdef DS_CHECKED
#define DS_GUARD(ms, cond, bit) ::ds::ds_guard((cond), (bit), (ms)->check)
#else
#define DS_GUARD(ms, cond, bit) true
#endif
constexpr int kMaxSplits = 16;            // largest thread-block cluster used
constexpr unsigned kFull = 0xFFFFFFFFu;

// ---------------------------------------------------------------------------
// Element traits.  A candidate is one 64-bit composite
//     (order key << 32) | ~index
// so that unsigned comparison of composites is the total order of the
// result: larger key first, and among equal keys the lower index first.
// The order key is the sign-flip map of "改造 Radix Sort" applied after
// sending every NaN to the largest key and -0.0 to the key of +0.0.
// ---------------------------------------------------------------------------
template <int DT>
struct Elem;

template <>
struct Elem<0> {  // fp32
    static constexpr int kSize = 4;
    static constexpr int kPerChunk = 4;                  // elements per 16-byte chunk
    static constexpr int kKeyTopShift = 56;              // shift of the highest key digit
    static constexpr int kKeyDigits = 4;
    static constexpr uint32_t kNanKey = 0xFFFFFFFFu;
    static constexpr uint32_t kInfKey = 0xFF800000u;     // key of +inf
    static constexpr uint32_t kZeroKey = 0x80000000u;    // key of +-0
    static constexpr uint32_t kNegInfBits = 0xFF800000u;
    static constexpr uint32_t kNanBits = 0x7FC00000u;
    static constexpr uint32_t kThresholdInit = 0xFF800000u;  // -inf: admits every element

    __device__ static __forceinline__ uint32_t key(uint32_t u)
    {
        uint32_t flipped = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
        uint32_t mag = u & 0x7FFFFFFFu;
        flipped = (mag == 0u) ? kZeroKey : flipped;
        return (mag > 0x7F800000u) ? kNanKey : flipped;
    }
    // value bits of a non-NaN key (zero comes back as +0.0)
    __device__ static __forceinline__ uint32_t bits_of_key(uint32_t kk)
    {
        return (kk & 0x80000000u) ? (kk ^ 0x80000000u) : ~kk;
    }
    // threshold operand for the packed prefilter
    __device__ static __forceinline__ uint32_t splat(uint32_t bits) { return bits; }
};

template <>
struct Elem<1> {  // bf16
    static constexpr int kSize = 2;
    static constexpr int kPerChunk = 8;
    static constexpr int kKeyTopShift = 40;
    static constexpr int kKeyDigits = 2;
    static constexpr uint32_t kNanKey = 0xFFFFu;
    static constexpr uint32_t kInfKey = 0xFF80u;
    static constexpr uint32_t kZeroKey = 0x8000u;
    static constexpr uint32_t kNegInfBits = 0xFF80u;
    static constexpr uint32_t kNanBits = 0x7FC0u;
    static constexpr uint32_t kThresholdInit = 0xFF80u;

    __device__ static __forceinline__ uint32_t key(uint32_t u)
    {
        u &= 0xFFFFu;
        uint32_t flipped = (u & 0x8000u) ? (~u & 0xFFFFu) : (u | 0x8000u);
        uint32_t mag = u & 0x7FFFu;
        flipped = (mag == 0u) ? kZeroKey : flipped;
        return (mag > 0x7F80u) ? kNanKey : flipped;
    }
    __device__ static __forceinline__ uint32_t bits_of_key(uint32_t kk)
    {
        return (kk & 0x8000u) ? (kk ^ 0x8000u) : (~kk & 0xFFFFu);
    }
    __device__ static __forceinline__ uint32_t splat(uint32_t bits) { return bits | (bits << 16); }
};

template <>
struct Elem<2> {  // IEEE binary16: +inf is 0x7C00, larger magnitudes are NaN
    static constexpr int kSize = 2;
    static constexpr int kPerChunk = 8;
    static constexpr int kKeyTopShift = 40;
    static constexpr int kKeyDigits = 2;
    static constexpr uint32_t kNanKey = 0xFFFFu;
    static constexpr uint32_t kInfKey = 0xFC00u;
    static constexpr uint32_t kZeroKey = 0x8000u;
    static constexpr uint32_t kNegInfBits = 0xFC00u;
    static constexpr uint32_t kNanBits = 0x7E00u;
    static constexpr uint32_t kThresholdInit = 0xFC00u;

    __device__ static __forceinline__ uint32_t key(uint32_t u)
    {
        u &= 0xFFFFu;
        uint32_t flipped = (u & 0x8000u) ? (~u & 0xFFFFu) : (u | 0x8000u);
        uint32_t mag = u & 0x7FFFu;
        flipped = (mag == 0u) ? kZeroKey : flipped;
        return (mag > 0x7C00u) ? kNanKey : flipped;
    }
    __device__ static __forceinline__ uint32_t bits_of_key(uint32_t kk)
    {
        return (kk & 0x8000u) ? (kk ^ 0x8000u) : (~kk & 0xFFFFu);
    }
    __device__ static __forceinline__ uint32_t splat(uint32_t bits) { return bits | (bits << 16); }
};

// ---------------------------------------------------------------------------
// Running threshold T of the scan ("算法": starts at -inf, raised to the
// smallest kept element after every compaction), held as the composite of
// that element plus the two prefilter operands derived from it.
//
// The prefilter of a block is a single unordered compare per element,
// pass = !(v < t), which admits NaN and treats -0 == +0 exactly like the key
// order.  Elements equal to T pass only when their index is below T's, so a
// block whose indices all lie below T's index uses t = value(T) ("key >= T")
// and a block whose indices all lie at or above it uses t = the next value
// up ("key > T").  A block that straddles T's index, or a NaN operand, is
// resolved exactly per element by comparing composites ("refine").
// ---------------------------------------------------------------------------
struct Threshold {
    unsigned long long comp;  // composite of T; 0 admits every element
    uint32_t ti;              // index of T (elements with T's key pass iff index < ti)
    uint32_t t_ge, t_gt;      // prefilter operands (fp32 bits or packed bf16x2 / f16x2)
    bool nan_ge, nan_gt;      // operand is NaN: the prefilter admits all, refine
};

template <int DT>
__device__ __forceinline__ Threshold threshold_initial()
{
    using E = Elem<DT>;
    Threshold t;
    t.comp = 0ull;
    t.ti = 0xFFFFFFFFu;
    t.t_ge = E::splat(E::kThresholdInit);
    t.t_gt = t.t_ge;
    t.nan_ge = false;
    t.nan_gt = false;
    return t;
}

template <int DT>
__device__ __forceinline__ Threshold threshold_from(unsigned long long comp)
{
    using E = Elem<DT>;
    Threshold t;
    const uint32_t tk = (uint32_t)(comp >> 32);
    t.comp = comp;
    t.ti = ~(uint32_t)comp;
    t.nan_ge = (tk == E::kNanKey);
    t.t_ge = E::splat(t.nan_ge ? E::kNanBits : E::bits_of_key(tk));
    t.nan_gt = (tk >= E::kInfKey);
    t.t_gt = E::splat(t.nan_gt ? E::kNanBits : E::bits_of_key(tk + 1u));
    return t;
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC'11), first output word only.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2,
                                                 uint32_t c3, uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0;
        const uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c0;
}

// ---------------------------------------------------------------------------
// A keyed pseudorandom permutation of [0, n), evaluated per position without
// a table (the free-running kernel needs the block at a position without
// sorting the whole order first).  A balanced Feistel network of 4 rounds on
// 2h bits, 2^(2h) >= n: (L, R) -> (R, L ^ F(R ^ key_r)), F multiplying by
// odd constants with xor-shifts, is a permutation of [0, 2^(2h)); positions
// that map past n are walked on along their cycle ("cycle walking"), which
// returns below n at the latest when it comes back to the start, so the
// result is a bijection of [0, n).  Keys come from one Philox word per row
// slice, so the order is random and independent of the data.
// ---------------------------------------------------------------------------
struct BlockOrder {
    uint32_t n, h, mask;
    uint32_t key[4];

    __device__ __forceinline__ static uint32_t mix(uint32_t x)
    {
        x *= 0xD2511F53u;
        x ^= x >> 15;
        x *= 0xCD9E8D57u;
        x ^= x >> 13;
        return x;
    }

    __device__ __forceinline__ void init(uint32_t count, uint32_t word)
    {
        n = count;
        h = 0;
        while (h < 16 && (1u << (2 * h)) < count)
            ++h;
        mask = (1u << h) - 1u;
#pragma unroll
        for (int r = 0; r < 4; ++r)
            key[r] = mix(word + (uint32_t)r * 0x9E3779B9u);
    }

    __device__ __forceinline__ uint32_t operator()(uint32_t q) const
    {
        if (n <= 1u)
            return 0u;
        uint32_t x = q;
        const unsigned long long domain = 1ull << (2 * h);
        for (unsigned long long walk = 0; walk < domain; ++walk) {
            uint32_t L = x >> h, R = x & mask;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t f = mix(R ^ key[r]) & mask;
                const uint32_t t = R;
                R = L ^ f;
                L = t;
            }
            x = (L << h) | R;
            if (x < n)
                break;
        }
        return x;
    }
};

// ---------------------------------------------------------------------------
// PTX wrappers: shared-memory address, asynchronous copies, 128-bit loads.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte asynchronous copy global -> shared (L1 bypassed); both addresses
// 16-byte aligned.  Completion is tracked per thread by commit groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Waits until at most `pending` (0..5; larger values wait as for 5) of this
// thread's newest commit groups are still in flight.
__device__ __forceinline__ void cp_async_wait_pending(int pending)
{
    switch (pending) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    }
}

// Programmatic dependent launch: let the next grid on the stream be
// scheduled now (its CTAs start once this grid's CTAs have all started and
// wait in dependent_grid_wait), and wait until the previous grid on the
// stream has completed and its memory is visible.  Both are no-ops for a
// launch without the programmatic attribute.
__device__ __forceinline__ void allow_dependent_grid()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void dependent_grid_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(const unsigned char *p)
{
    return *reinterpret_cast<const uint4 *>(p);
}

// ---------------------------------------------------------------------------
// Warp primitives.
// ---------------------------------------------------------------------------
// Hillis-Steele inclusive scan over the 32 lanes ("Scan").
__device__ __forceinline__ uint32_t warp_inclusive_scan(uint32_t v, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(kFull, v, d);
        if (lane >= d)
            v += o;
    }
    return v;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v)
{
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        v += __shfl_xor_sync(kFull, v, d);
    return v;
}

__device__ __forceinline__ unsigned long long warp_min_reduce(unsigned long long v)
{
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const unsigned long long o = __shfl_xor_sync(kFull, v, d);
        v = o < v ? o : v;
    }
    return v;
}

__device__ __forceinline__ uint32_t lanemask_lt(int lane) { return (1u << lane) - 1u; }

// ---------------------------------------------------------------------------
// 64-bit warp helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long shfl_idx_u64(unsigned long long v, int src)
{
    const uint32_t lo = __shfl_sync(kFull, (uint32_t)v, src);
    const uint32_t hi = __shfl_sync(kFull, (uint32_t)(v >> 32), src);
    return ((unsigned long long)hi << 32) | lo;
}

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m)
{
    const uint32_t lo = __shfl_xor_sync(kFull, (uint32_t)v, m);
    const uint32_t hi = __shfl_xor_sync(kFull, (uint32_t)(v >> 32), m);
    return ((unsigned long long)hi << 32) | lo;
}

__device__ __forceinline__ unsigned long long warp_or_u64(unsigned long long v)
{
    const uint32_t lo = __reduce_or_sync(kFull, (uint32_t)v);
    const uint32_t hi = __reduce_or_sync(kFull, (uint32_t)(v >> 32));
    return ((unsigned long long)hi << 32) | lo;
}

__device__ __forceinline__ unsigned long long warp_and_u64(unsigned long long v)
{
    const uint32_t lo = __reduce_and_sync(kFull, (uint32_t)v);
    const uint32_t hi = __reduce_and_sync(kFull, (uint32_t)(v >> 32));
    return ((unsigned long long)hi << 32) | lo;
}

__device__ __forceinline__ unsigned long long min_u64(unsigned long long a, unsigned long long b)
{
    return a < b ? a : b;
}

__device__ __forceinline__ unsigned long long max_u64(unsigned long long a, unsigned long long b)
{
    return a > b ? a : b;
}

__host__ __device__ __forceinline__ int pow2_ceil(int v)
{
    int p = 1;
    while (p < v)
        p <<= 1;
    return p;
}

// ---------------------------------------------------------------------------
// Ordering the selected entries.  A sort network of k entries needs
// O(log^2 k) dependent steps; here the final position of every entry is its
// rank -- the number of entries that come before it -- computed with few
// dependent steps:
//   * up to 256 entries: every thread counts the entries above its own one;
//   * up to 2048: each warp sorts a run of 32E entries held in registers
//     (bitonic, shuffles for strides below 32, register swaps above), then
//     every entry's rank is its place in its own run plus, for each other
//     run, the number of entries above it found by binary search.
// Entries must be distinct; padding entries (0 when descending) never count.
// ---------------------------------------------------------------------------

// Sorts the 32E entries of one warp's run in registers (all lanes call).
template <int E>
__device__ __forceinline__ void warp_bitonic_regs(unsigned long long (&r)[E], int lane, bool desc)
{
    constexpr int span = 32 * E;
#pragma unroll
    for (int size = 2; size <= span; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride >= 32) {
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const int q = stride / 32;
                    if ((j & q) == 0) {
                        const int i = 32 * j + lane;
                        const bool up = ((i & size) == 0) != desc;
                        const unsigned long long x = r[j], y = r[j + q];
                        if (up ? (x > y) : (x < y)) {
                            r[j] = y;
                            r[j + q] = x;
                        }
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const int i = 32 * j + lane;
                    const unsigned long long o = shfl_xor_u64(r[j], stride);
                    const bool up = ((i & size) == 0) != desc;
                    const bool lower = (lane & stride) == 0;
                    r[j] = (lower == up) ? min_u64(r[j], o) : max_u64(r[j], o);
                }
            }
        }
    }
}

// Ranks (descending order: number of entries greater) of the cnt distinct
// entries a[0, cnt), 256 < cnt <= 32*E*8.  a is padded with zeros to 256E
// entries by the caller and synchronised.  Each thread gets the entries
// a[base + 32j + lane] of its warp's run after the call (returned through
// `vals`) together with their ranks; entries at positions >= cnt are pads.
// On return a[] holds the warp-sorted runs and the CTA is synchronised.
template <int E>
__device__ __forceinline__ void rank_desc_runs(unsigned long long *a, unsigned long long (&vals)[E],
                                               int (&ranks)[E])
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int span = 32 * E;
    const int base = warp * span;
#pragma unroll
    for (int j = 0; j < E; ++j)
        vals[j] = a[base + 32 * j + lane];
    warp_bitonic_regs<E>(vals, lane, true);
#pragma unroll
    for (int j = 0; j < E; ++j)
        a[base + 32 * j + lane] = vals[j];
    __syncthreads();
    // branch-free binary searches, the eight runs in lockstep so that the
    // loads of one step are independent: pos[w] = entries of run w above e
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const unsigned long long e = vals[j];
        int pos[kWarps];
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            pos[w] = 0;
#pragma unroll
        for (int step = span / 2; step >= 1; step >>= 1) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w)
                pos[w] += a[w * span + pos[w] + step - 1] > e ? step : 0;
        }
        int rank = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const int q = pos[w] + (a[w * span + pos[w]] > e ? 1 : 0);
            rank += (w == warp) ? (32 * j + lane) : q;
        }
        ranks[j] = rank;
    }
    __syncthreads();
}

// Plain shared-memory bitonic sort (any power of two); ends synchronised.
__device__ __forceinline__ void bitonic_sort_smem(unsigned long long *a, int P, bool desc)
{
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = threadIdx.x; t < (P >> 1); t += kThreads) {
                const int lo = 2 * t - (t & (stride - 1));
                const int hi = lo + stride;
                const bool pair_desc = (((lo & size) == 0) == desc);
                const unsigned long long x = a[lo], y = a[hi];
                if (pair_desc ? (x < y) : (x > y)) {
                    a[lo] = y;
                    a[hi] = x;
                }
            }
            __syncthreads();
        }
    }
}

// Sorts the cnt distinct entries a[0, cnt) ascending, in place (block
// order); positions past cnt are left as they are.  Up to 64 entries every
// thread counts; up to 256 the complements are ranked in descending order
// in `scratch` (256 entries;
// the complement of a real entry is never 0, and 0 pads rank last) by
// warp-sorted runs and binary searches; larger sets use the shared-memory
// bitonic network in a itself (cap_pow2 entries).  Caller synchronises
// before; ends synchronised.
__device__ __forceinline__ void sort_asc_small(unsigned long long *a, int cnt, int cap_pow2,
                                               unsigned long long *scratch)
{
    if (cnt <= 64) {
        // few entries: every thread counts the entries below its own
        const int t = threadIdx.x;
        unsigned long long e = 0ull;
        int rank = 0;
        if (t < cnt) {
            e = a[t];
            for (int j = 0; j < cnt; ++j)
                rank += a[j] < e ? 1 : 0;
        }
        __syncthreads();
        if (t < cnt)
            a[rank] = e;
        __syncthreads();
    } else if (cnt <= kThreads) {
        const int t = threadIdx.x;
        scratch[t] = t < cnt ? ~a[t] : 0ull;
        __syncthreads();
        unsigned long long vals[1];
        int ranks[1];
        rank_desc_runs<1>(scratch, vals, ranks);
        if (vals[0] != 0ull)
            a[ranks[0]] = ~vals[0];
        __syncthreads();
    } else {
        for (int i = cnt + threadIdx.x; i < cap_pow2; i += kThreads)
            a[i] = ~0ull;
        __syncthreads();
        bitonic_sort_smem(a, cap_pow2, false);
    }
}

// Shared scratch words of one CTA.
struct Misc {
    unsigned long long wor[kWarps];      // per-warp OR / AND / min of composites
    unsigned long long wand[kWarps];
    unsigned long long wmin[kWarps];
    unsigned long long group[32];        // small tie group of the select
    unsigned long long texact;           // exact k-th composite, when resolved
    __align__(16) int cntw[2][kWarps];   // survivors per warp, double-buffered
    uint32_t wsum[kWarps];               // per-warp totals of block scans
    uint32_t sel_digit, sel_above, sel_eq;
    int merge_count;                     // CTA 0 of a cluster: entries received
    int merge_off;                       // this CTA's offset in CTA 0's merge buffer
    unsigned int *check;                 // bounds-checked builds: violation bits (null otherwise)
    unsigned long long tslice[16];       // split rows: every slice's k-th composite (0: fewer than k)
    int pass;                            // select: digit passes so far (histogram rotation)
    int ctr[2];                          // free-running scan: buffer length, one word per epoch
    __align__(16) int rem[kWarps];       // free-running scan: warp still has stages (at a sync point)
    unsigned long long cl_or, cl_and;    // split rows: OR / AND of this slice's candidates
    int cl_n, cl_cnt;                    // split rows: this slice's candidates / entries selected
};

// Digit histograms: the register select uses one 256-bin histogram of 32-bit
// counters per CTA, three rotating buffers; each pass clears the buffer of
// the next, so the buffer a call starts with (ms->pass mod 3) is clear, while
// up to two others may be left dirty.  The shared-memory select uses one
// histogram per warp over the whole region and clears it on entry.
constexpr int kHistBins = 256;
constexpr int kHistWords = kWarps * kHistBins;  // 8 KiB
static_assert(3 * kHistBins <= kHistWords, "rotating buffers fit the region");

// Exclusive scan of one value per thread over the CTA (thread order).
// Uses ms->wsum; ends synchronised.  Returns the exclusive prefix.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, Misc *ms)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t incl = warp_inclusive_scan(v, lane);
    if (lane == 31)
        ms->wsum[warp] = incl;
    __syncthreads();
    uint32_t before = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
        before += (w < warp) ? ms->wsum[w] : 0u;
    return before + incl - v;
}

// ---------------------------------------------------------------------------
// RadixSelectTopK ("算法", step 3) on n > k distinct composites in shared
// memory.  After the call cand[0, k) holds the k largest (in no particular
// order); returns the smallest of them, the new threshold.  Called by all
// threads; ends synchronised.
//
// Every thread loads its entries cand[tid + 256j] into registers once (up to
// R of them), as two 32-bit halves; all passes then work on registers.  The
// select is bound by issued instructions (every warp of the SM runs it), so
// each step is kept to few instructions per entry:
//  1. OR and AND of all composites (warp reductions): only bits where they
//     differ can separate entries, so digits start at the highest such bit
//     and skip bits that never vary.
//  2. Digit passes of 8 bits from the top: every entry still matching the
//     chosen prefix adds one to its bin of the CTA's 256-bin histogram (one
//     shared atomic per entry); warp 0 then scans the histogram from the top
//     bin down, finds the digit that holds the need-th entry and publishes it.
//     Entries of higher digits are selected for good, those of other digits
//     drop out.  Histogram buffers rotate over three, so clearing the next
//     one needs no extra barrier.
//  3. The loop stops when every entry of the chosen digit is needed, or when
//     at most 32 remain tied; the tied entries are gathered and every warp
//     ranks them (shuffles) to find the exact k-th composite.
//  4. Compaction: the selected entries of each register slot are counted by
//     a warp ballot; after one barrier every warp's slots in cand[0, k)
//     start after those of the warps below it, and the buffer is overwritten
//     in place (all entries are in registers).  Counts and minima travel
//     through per-warp words rather than shared atomics, which serialise
//     when eight warps hit one word.
// ---------------------------------------------------------------------------
// Warp 0's decision for one digit pass over histogram `hb`: lane l owns bins
// 8l .. 8l+7; bins are ranked from the top.  Publishes the digit that holds
// the need-th entry, the number of entries in higher bins and its own count.
__device__ __forceinline__ void digit_search(const uint32_t *hb, uint32_t need, int lane, Misc *ms)
{
    const uint4 q0 = *reinterpret_cast<const uint4 *>(hb + lane * 8);
    const uint4 q1 = *reinterpret_cast<const uint4 *>(hb + lane * 8 + 4);
    // cu_t: entries in this lane's bins 8l+7 down to 8l+t (a sum tree, three
    // dependent adds deep)
    const uint32_t s76 = q1.w + q1.z, s54 = q1.y + q1.x, s32 = q0.w + q0.z, s10 = q0.y + q0.x;
    const uint32_t s74 = s76 + s54, s30 = s32 + s10;
    const uint32_t cu7 = q1.w, cu6 = s76, cu5 = s76 + q1.y, cu4 = s74;
    const uint32_t cu3 = s74 + q0.w, cu2 = s74 + s32, cu1 = (s74 + s32) + q0.y, cu0 = s74 + s30;
    uint32_t suf = cu0;  // entries in the bins of this lane and all lanes above
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_down_sync(kFull, suf, d);
        if (lane + d < 32)
            suf += o;
    }
    const uint32_t excl = suf - cu0;
    const bool found = excl < need && need <= suf;
    const uint32_t r = need - excl;
    // bins of this lane lying wholly above the need-th entry
    const uint32_t nb = (((uint32_t)(cu7 < r) + (uint32_t)(cu6 < r)) +
                         ((uint32_t)(cu5 < r) + (uint32_t)(cu4 < r))) +
                        (((uint32_t)(cu3 < r) + (uint32_t)(cu2 < r)) + (uint32_t)(cu1 < r));
    // before = cu_{8-nb} (0 for nb = 0), through = cu_{7-nb}: three levels of selects
    const bool b0 = nb & 1u, b1 = nb & 2u, b2 = nb & 4u;
    const uint32_t bA = b0 ? cu7 : 0u, bB = b0 ? cu5 : cu6, bC = b0 ? cu3 : cu4, bD = b0 ? cu1 : cu2;
    const uint32_t before = b2 ? (b1 ? bD : bC) : (b1 ? bB : bA);
    const uint32_t tA = b0 ? cu6 : cu7, tB = b0 ? cu4 : cu5, tC = b0 ? cu2 : cu3, tD = b0 ? cu0 : cu1;
    const uint32_t through = b2 ? (b1 ? tD : tC) : (b1 ? tB : tA);
    if (found) {
        ms->sel_digit = 8u * (uint32_t)lane + 7u - nb;
        ms->sel_above = excl + before;
        ms->sel_eq = through - before;
    }
}

#ifdef DS_CHECKED
__device__ __forceinline__ bool ds_guard(bool ok, unsigned int bit, unsigned int *word)
{
    if (!ok && word != nullptr)
        atomicOr(word, bit);
    return ok;
}
#endif

// Entries flagged in `bits` (bit j = register slot j) over the whole warp.
template <int R>
__device__ __forceinline__ int warp_count(uint32_t bits)
{
    int tot = 0;
#pragma unroll
    for (int j = 0; j < R; ++j)
        tot += __popc(__ballot_sync(kFull, (bits >> j) & 1u));
    return tot;
}

// Writes the flagged entries to dst[0, count): slot by slot, each lane's
// position is the flagged lanes below it plus the earlier slots' totals.
template <int R>
__device__ __forceinline__ void warp_scatter(uint32_t bits, const uint32_t (&hi)[R],
                                             const uint32_t (&lo)[R], unsigned long long *dst,
                                             int lane)
{
    int run = 0;
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const uint32_t b = __ballot_sync(kFull, (bits >> j) & 1u);
        if ((bits >> j) & 1u)
            dst[run + __popc(b & lanemask_lt(lane))] = ((unsigned long long)hi[j] << 32) | lo[j];
        run += __popc(b);
    }
}

template <int R>
static __device__ __noinline__ unsigned long long radix_select_regs(unsigned long long *cand, int n,
                                                                    int k, uint32_t *hist,
                                                                    Misc *ms)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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
    int pass = ms->pass;  // published before the previous barrier

    // 1. varying bits
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
    __syncthreads();  // also: all loads of cand are done, every warp read ms->pass
    unsigned long long vo = 0ull, va = ~0ull;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        vo |= ms->wor[w];
        va &= ms->wand[w];
    }
    const unsigned long long vary = vo ^ va;

    // 2./3. digit passes
    uint32_t need = (uint32_t)k;
    uint32_t live = valid;  // entries still matching the chosen prefix
    uint32_t above = 0u;    // entries selected by a higher digit
    bool exact = false;
    unsigned long long texact = 0ull;
    int h = 63 - __clzll((long long)vary);
    while (true) {
        const int sh = h >= 7 ? h - 7 : 0;
        uint32_t *cur = hist + (pass % 3) * kHistBins;
        hist[((pass + 1) % 3) * kHistBins + tid] = 0u;
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const uint32_t d = (sh >= 32 ? hi[j] >> (sh - 32) : __funnelshift_r(lo[j], hi[j], sh)) & 255u;
            dg[j] = d;
            if (live & (1u << j))
                atomicAdd(&cur[d], 1u);
        }
        __syncthreads();
        if (warp == 0)
            digit_search(cur, need, lane, ms);
        __syncthreads();
        const uint32_t dsel = ms->sel_digit, eq = ms->sel_eq;
        need -= ms->sel_above;
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
        if (eq <= 32u) {
            // gather the tied entries (each warp's at the offset of the
            // warps below it) and let every warp rank them
            const int mine = warp_count<R>(live);
            if (lane == 0)
                ms->wsum[warp] = (uint32_t)mine;
            __syncthreads();
            int base = 0;
#pragma unroll
            for (int w = 0; w < kWarps; ++w)
                base += w < warp ? (int)ms->wsum[w] : 0;
            if (DS_GUARD(ms, base + mine <= 32, 4u))
                warp_scatter<R>(live, hi, lo, ms->group + base, lane);
            __syncthreads();
            const unsigned long long g = lane < (int)eq ? ms->group[lane] : 0ull;
            uint32_t rank = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const unsigned long long o = shfl_idx_u64(g, j);
                rank += (j < (int)eq && o > g) ? 1u : 0u;
            }
            const int src = __ffs(__ballot_sync(kFull, lane < (int)eq && rank == need - 1u)) - 1;
            texact = shfl_idx_u64(g, src);
            exact = true;
            break;
        }
        // eq > need >= 1 and composites are distinct: lower bits still vary
        const unsigned long long below = sh > 0 ? (vary & ((1ull << sh) - 1ull)) : 0ull;
        if (below == 0ull)
            break;  // unreachable for distinct composites; keeps the loop finite
        h = 63 - __clzll((long long)below);
    }

    // 4. compaction
    uint32_t sel = above;
    if (exact) {
#pragma unroll
        for (int j = 0; j < R; ++j)
            if (((live >> j) & 1u) && (((unsigned long long)hi[j] << 32) | lo[j]) >= texact)
                sel |= 1u << j;
    } else {
        sel |= live;
    }
    // every warp's count (and smallest taken entry) goes to shared memory; the
    // warp's slots start after those of the warps below it
    const int mine = warp_count<R>(sel);
    unsigned long long wmin = ~0ull;
    if (!exact) {
        // the chosen digit's entries are taken whole: the smallest of them
        // is the k-th composite.  A warp with no such entry reports the
        // all-ones composite, which is below no entry (at most equal to a
        // NaN at index 0), so it never changes the minimum.
        uint32_t mh = ~0u, ml = ~0u;
#pragma unroll
        for (int j = 0; j < R; ++j)
            if ((live >> j) & 1u)
                mh = min(mh, hi[j]);
        mh = __reduce_min_sync(kFull, mh);
#pragma unroll
        for (int j = 0; j < R; ++j)
            if (((live >> j) & 1u) && hi[j] == mh)
                ml = min(ml, lo[j]);
        ml = __reduce_min_sync(kFull, ml);
        wmin = ((unsigned long long)mh << 32) | ml;
    }
    if (lane == 0) {
        ms->wsum[warp] = (uint32_t)mine;
        ms->wmin[warp] = wmin;
    }
    if (tid == 0)
        ms->pass = pass;
    __syncthreads();
    int cbase = 0;
    unsigned long long tmin = ~0ull;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        cbase += w < warp ? (int)ms->wsum[w] : 0;
        tmin = min_u64(tmin, ms->wmin[w]);
    }
    if (DS_GUARD(ms, cbase + mine <= n, 2u))
        warp_scatter<R>(sel, hi, lo, cand + cbase, lane);
    __syncthreads();
    return exact ? texact : tmin;
}

// The same for sets too large for registers: every pass reads shared memory.
static __device__ __noinline__ unsigned long long radix_select_smem(unsigned long long *cand, int n,
                                                                    int k, uint32_t *whist,
                                                                    uint16_t *holes, Misc *ms)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // this variant counts in 32-bit words over the histogram region; start
    // from zero (it leaves the region zero for the rotating buffers)
    for (int i = tid; i < kHistWords; i += kThreads)
        whist[i] = 0u;
    unsigned long long vo = 0ull, va = ~0ull;
    for (int i = tid; i < n; i += kThreads) {
        const unsigned long long c = cand[i];
        vo |= c;
        va &= c;
    }
    vo = warp_or_u64(vo);
    va = warp_and_u64(va);
    if (lane == 0) {
        ms->wor[warp] = vo;
        ms->wand[warp] = va;
    }
    __syncthreads();
    vo = 0ull;
    va = ~0ull;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        vo |= ms->wor[w];
        va &= ms->wand[w];
    }
    const unsigned long long vary = vo ^ va;
    unsigned long long prefix = 0ull, pmask = 0ull;
    uint32_t need = (uint32_t)k;
    int h = 63 - __clzll((long long)vary);
    uint32_t *wh = whist + warp * 256;
    while (true) {
        const int lo = h >= 7 ? h - 7 : 0;
        for (int i = tid; i < n; i += kThreads) {
            const unsigned long long c = cand[i];
            if ((c & pmask) == prefix)
                atomicAdd(&wh[(uint32_t)(c >> lo) & 255u], 1u);
        }
        __syncthreads();
        const int bin = 255 - tid;
        uint32_t cnt = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            cnt += whist[w * 256 + bin];
            whist[w * 256 + bin] = 0u;
        }
        const uint32_t excl = block_exclusive_scan(cnt, ms);
        if (excl < need && need <= excl + cnt) {
            ms->sel_digit = (uint32_t)bin;
            ms->sel_above = excl;
            ms->sel_eq = cnt;
        }
        __syncthreads();
        const uint32_t dsel = ms->sel_digit, eq = ms->sel_eq;
        need -= ms->sel_above;
        prefix |= (unsigned long long)dsel << lo;
        pmask |= 255ull << lo;
        if (eq == need)
            break;
        const unsigned long long below = lo > 0 ? (vary & ((1ull << lo) - 1ull)) : 0ull;
        if (below == 0ull)
            break;  // unreachable for distinct composites; keeps the loop finite
        h = 63 - __clzll((long long)below);
    }
    // in-place compaction: unselected slots below k are listed, selected
    // entries at or above k move into them
    uint32_t nh = 0, nm = 0;
    unsigned long long mn = ~0ull;
    for (int i = tid; i < n; i += kThreads) {
        const unsigned long long c = cand[i];
        const bool sel = (c & pmask) >= prefix;
        if (sel)
            mn = min_u64(mn, c);
        if (i < k)
            nh += sel ? 0u : 1u;
        else
            nm += sel ? 1u : 0u;
    }
    mn = warp_min_reduce(mn);
    if (lane == 0)
        ms->wmin[warp] = mn;
    const uint32_t off = block_exclusive_scan(nh | (nm << 16), ms);
    uint32_t oh = off & 0xFFFFu, om = off >> 16;
    for (int i = tid; i < k; i += kThreads)
        if (!((cand[i] & pmask) >= prefix))
            holes[oh++] = (uint16_t)i;
    __syncthreads();
    for (int i = tid + kThreads * (k / kThreads); i < n; i += kThreads) {
        if (i < k)
            continue;
        const unsigned long long c = cand[i];
        if ((c & pmask) >= prefix)
            cand[holes[om++]] = c;
    }
    __syncthreads();
    unsigned long long t = ~0ull;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
        t = min_u64(t, ms->wmin[w]);
    return t;
}

__device__ __forceinline__ unsigned long long radix_select_topk(unsigned long long *cand, int n, int k,
                                                                uint32_t *hist, uint16_t *holes,
                                                                Misc *ms)
{
    if (n <= 4 * kThreads)
        return radix_select_regs<4>(cand, n, k, hist, ms);
    if (n <= 8 * kThreads)
        return radix_select_regs<8>(cand, n, k, hist, ms);
    if (n <= 12 * kThreads)
        return radix_select_regs<12>(cand, n, k, hist, ms);
    if (n <= 24 * kThreads)
        return radix_select_regs<24>(cand, n, k, hist, ms);
    return radix_select_smem(cand, n, k, hist, holes, ms);
}

// The select between streaming phases and at the end.  `room` = entries the
// buffer at cand can hold (kept for selects that need scratch beyond n).
__device__ __forceinline__ unsigned long long select_topk(unsigned long long *cand, int n, int k,
                                                          int room, uint32_t *hist, uint16_t *holes,
                                                          Misc *ms)
{
    (void)room;
    return radix_select_topk(cand, n, k, hist, holes, ms);
}

}  // namespace ds
