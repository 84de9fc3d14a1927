// ds_device.cuh -- device-side building blocks of the DeepSelect top-k kernel
// for sm_103a: order keys, Philox4x32-10, mbarrier / bulk-copy wrappers, warp
// scans, the shared-memory radix select and the bitonic sort.
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
#include <cuda_runtime.h>
#include <stdint.h>

namespace ds {

constexpr int kThreads = 256;             // threads per CTA
constexpr int kWarps = kThreads / 32;     // warps per CTA
constexpr int kMaxStages = 4;             // deepest shared-memory ring
constexpr int kMaxSplits = 16;            // largest thread-block cluster used
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // bound on any mbarrier wait

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
    uint32_t t_ge, t_gt;      // prefilter operands (fp32 bits or packed bf16x2)
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
// PTX wrappers: shared-memory address, global timer, mbarrier, bulk copy.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_timer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0u;
}

// Waits for phase `parity` of the barrier; gives up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs)
            return false;
    }
    return true;
}

// Bulk (TMA, non-tensor) copy global -> own shared memory, completion
// counted in bytes on `bar`.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Orders earlier generic-proxy shared-memory accesses before later bulk copies.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v)
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
// Bitonic sort of P (a power of two) 64-bit entries in shared memory by the
// whole CTA.  The caller synchronises before; the sort ends synchronised.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bitonic_sort_u64(unsigned long long *a, int P, bool descending)
{
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = threadIdx.x; t < (P >> 1); t += kThreads) {
                const int lo = 2 * t - (t & (stride - 1));
                const int hi = lo + stride;
                const bool pair_desc = (((lo & size) == 0) == descending);
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

__host__ __device__ __forceinline__ int pow2_ceil(int v)
{
    int p = 1;
    while (p < v)
        p <<= 1;
    return p;
}

// Scratch words of one CTA's radix select and stage decisions.
struct Misc {
    unsigned long long bar[kMaxStages];  // one mbarrier per ring stage
    unsigned long long tmin;             // smallest selected composite
    int cntw[kWarps];                    // survivors per warp in the current stage
    uint32_t sel_digit, sel_above, sel_eq;
    int hole_count, mover_count;
    int flag;                            // a wait timed out
    int merge_count[kMaxSplits];         // partial-result sizes (CTA 0 of a cluster)
};

// ---------------------------------------------------------------------------
// RadixSelectTopK ("算法", step 3) on n > k composites in shared memory.
//
// Digits of 8 bits are taken from the most significant end: first the order
// key (4 digits for fp32, 2 for bf16), then the complemented index (only its
// low idx_bits bits vary).  Each pass builds a 256-bin histogram of the
// entries that still match the selected prefix, with warp-aggregated shared
// atomics (one atomic per distinct digit per warp), and one warp scans the
// bins from the top to find the digit holding the k-th entry.  The loop stops
// as soon as every entry matching the prefix is needed, so distinct keys
// rarely reach the index digits.
//
// Afterwards the k selected entries -- (c & pmask) >= prefix -- are moved to
// cand[0, k) in place: unselected slots below k are listed, selected entries
// at or above k are moved into them.  Returns the smallest selected
// composite, the new threshold.  Called by all threads; ends synchronised.
// ---------------------------------------------------------------------------
template <int DT>
__device__ unsigned long long radix_select_topk(unsigned long long *cand, int n, int k,
                                                uint32_t *hist /* 2 x 256 */,
                                                uint16_t *holes, Misc *ms, int idx_bits)
{
    using E = Elem<DT>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned long long prefix = 0ull, pmask = 0ull;
    uint32_t need = (uint32_t)k;

    hist[tid] = 0u;  // kThreads == 256 bins
    if (tid == 0) {
        ms->hole_count = 0;
        ms->mover_count = 0;
        ms->tmin = ~0ull;
    }
    __syncthreads();

    const int ndigits = E::kKeyDigits + idx_bits / 8;
    for (int d = 0; d < ndigits; ++d) {
        const int sh = d < E::kKeyDigits ? E::kKeyTopShift - 8 * d
                                         : idx_bits - 8 - 8 * (d - E::kKeyDigits);
        uint32_t *h = hist + (d & 1) * 256;
        for (int base = 0; base < n; base += kThreads) {
            const int i = base + tid;
            uint32_t dig = 256u;  // not counted
            if (i < n) {
                const unsigned long long c = cand[i];
                if ((c & pmask) == prefix)
                    dig = (uint32_t)(c >> sh) & 255u;
            }
            const uint32_t peers = __match_any_sync(kFull, dig);
            if (dig < 256u && lane == __ffs(peers) - 1)
                atomicAdd(&h[dig], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns bins 255-8l down to 248-8l; scan in descending bin order
            uint32_t c8[8], s = 0;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                c8[t] = h[255 - 8 * lane - t];
                s += c8[t];
            }
            const uint32_t incl = warp_inclusive_scan(s, lane);
            uint32_t cum = incl - s;
            if (cum < need && need <= incl) {
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    if (cum + c8[t] >= need) {
                        ms->sel_digit = (uint32_t)(255 - 8 * lane - t);
                        ms->sel_above = cum;
                        ms->sel_eq = c8[t];
                        break;
                    }
                    cum += c8[t];
                }
            }
        } else {
            uint32_t *next = hist + ((d + 1) & 1) * 256;
            for (int b = tid - 32; b < 256; b += kThreads - 32)
                next[b] = 0u;
        }
        __syncthreads();
        const uint32_t dsel = ms->sel_digit;
        need -= ms->sel_above;
        prefix |= (unsigned long long)dsel << sh;
        pmask |= 255ull << sh;
        if (ms->sel_eq == need)
            break;
    }

    // in-place compaction of the selected entries into cand[0, k)
    unsigned long long my_min = ~0ull;
    for (int base = 0; base < k; base += kThreads) {
        const int i = base + tid;
        bool hole = false;
        if (i < k) {
            const unsigned long long c = cand[i];
            if ((c & pmask) >= prefix)
                my_min = c < my_min ? c : my_min;
            else
                hole = true;
        }
        const uint32_t b = __ballot_sync(kFull, hole);
        if (b) {
            int off = 0;
            if (lane == 0)
                off = atomicAdd(&ms->hole_count, __popc(b));
            off = __shfl_sync(kFull, off, 0);
            if (hole)
                holes[off + __popc(b & lanemask_lt(lane))] = (uint16_t)i;
        }
    }
    __syncthreads();
    for (int base = k; base < n; base += kThreads) {
        const int i = base + tid;
        bool mover = false;
        unsigned long long c = 0ull;
        if (i < n) {
            c = cand[i];
            mover = (c & pmask) >= prefix;
            if (mover)
                my_min = c < my_min ? c : my_min;
        }
        const uint32_t b = __ballot_sync(kFull, mover);
        if (b) {
            int off = 0;
            if (lane == 0)
                off = atomicAdd(&ms->mover_count, __popc(b));
            off = __shfl_sync(kFull, off, 0);
            if (mover)
                cand[holes[off + __popc(b & lanemask_lt(lane))]] = c;
        }
    }
    my_min = warp_min_u64(my_min);
    if (lane == 0)
        atomicMin(&ms->tmin, my_min);
    __syncthreads();
    return ms->tmin;
}

}  // namespace ds
