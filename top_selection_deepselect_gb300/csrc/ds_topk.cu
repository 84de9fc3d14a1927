// ds_topk.cu -- DeepSelect top-k for GB300 (sm_103a): the streaming kernel
// and the C-ABI launcher declared in include/ds_topk.h.
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
//   * blocks are staged into a ring of shared-memory stages by bulk (TMA)
//     copies issued by one thread, completion tracked by mbarriers, several
//     stages ahead of the filter;
//   * a stage holds one B-block per `warps_per_block` warps; each warp filters
//     its part with one unordered compare per element (fp32 FSETP, bf16 packed
//     set.geu) and only when a warp sees a survivor does it build exact bit
//     masks, which are placed with __ffs after a warp prefix sum (section
//     "实现": one-pass mask + __ffs placement);
//   * the blocks of a stage are filtered in parallel against the same T; a
//     stage is cut at the first block after which the buffer would reach
//     k + B2, the buffer is compacted, and the rest of the stage is filtered
//     again with the new T -- exactly the block-by-block semantics, so the
//     counters A, R, W and the peak length equal the step-by-step model's;
//   * split rows (section "实现", last paragraph): each CTA of the cluster
//     selects the top k of its contiguous slice and stores it into CTA 0's
//     shared memory (distributed shared memory), CTA 0 selects and sorts.

#include "ds_topk.h"

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "ds_device.cuh"

namespace cg = cooperative_groups;

namespace ds {

// Device status word: bit 0 = a kernel gave up waiting for a bulk copy.
__device__ unsigned int g_status;

struct Params {
    const void *x;
    const int32_t *row_len;
    int32_t *out_idx;
    void *out_val;
    long long *stats;
    long long N;
    int k, B, B2;
    uint32_t seed_lo, seed_hi;
    int splits;          // CTAs per row
    int wpb;             // warps per B-block
    int bps;             // B-blocks per stage (kWarps / wpb)
    int stages;          // ring depth (1 for the plain-load path)
    int slot_bytes;      // bytes of one staged block (B * size rounded up to 16)
    int cpw;             // 16-byte chunks per warp of a block
    int idx_bits;        // index bits that vary (multiple of 8)
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
};

template <int DT>
__device__ __forceinline__ uint32_t prefilter_any(const uint4 v, uint32_t t)
{
    if (DT == 0) {
        const float tf = __uint_as_float(t);
        const bool p = !(__uint_as_float(v.x) < tf) | !(__uint_as_float(v.y) < tf) |
                       !(__uint_as_float(v.z) < tf) | !(__uint_as_float(v.w) < tf);
        return p ? 1u : 0u;
    } else {
        const __nv_bfloat162 t2 = *reinterpret_cast<const __nv_bfloat162 *>(&t);
        return __hgeu2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&v.x), t2) |
               __hgeu2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&v.y), t2) |
               __hgeu2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&v.z), t2) |
               __hgeu2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&v.w), t2);
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

// Exact survivor mask of chunk c (bit e = element lo + c*kPerChunk + e).
template <int DT>
__device__ __forceinline__ uint32_t chunk_mask(const uint4 v, int c, const BlockView &bv,
                                               const Threshold &thr)
{
    using E = Elem<DT>;
    uint32_t mask;
    if (DT == 0) {
        const float tf = __uint_as_float(bv.t);
        mask = (uint32_t)!(__uint_as_float(v.x) < tf) | ((uint32_t)!(__uint_as_float(v.y) < tf) << 1) |
               ((uint32_t)!(__uint_as_float(v.z) < tf) << 2) |
               ((uint32_t)!(__uint_as_float(v.w) < tf) << 3);
    } else {
        const __nv_bfloat162 t2 = *reinterpret_cast<const __nv_bfloat162 *>(&bv.t);
        const uint32_t m0 = __hgeu2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&v.x), t2);
        const uint32_t m1 = __hgeu2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&v.y), t2);
        const uint32_t m2 = __hgeu2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&v.z), t2);
        const uint32_t m3 = __hgeu2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&v.w), t2);
        mask = (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) |
               ((m2 & 1u) << 4) | ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 128u);
    }
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

// Survivors of this warp's chunks (warp total, in every lane).
template <int DT>
__device__ __forceinline__ int warp_count(const BlockView &bv, const Threshold &thr, int lane)
{
    uint32_t any = 0u;
    for (int c = bv.c0 + lane; c < bv.c1; c += 32)
        any |= prefilter_any<DT>(lds128(bv.slot + c * 16), bv.t);
    if (!__any_sync(kFull, any != 0u))
        return 0;
    uint32_t cnt = 0u;
    for (int c = bv.c0 + lane; c < bv.c1; c += 32)
        cnt += __popc(chunk_mask<DT>(lds128(bv.slot + c * 16), c, bv, thr));
    return (int)warp_sum(cnt);
}

// Appends this warp's survivors at cand[base ...] in chunk order
// (predicate / exclusive scan / scatter of "Compact", mask walked with __ffs).
template <int DT>
__device__ __forceinline__ void warp_append(const BlockView &bv, const Threshold &thr, int lane,
                                            unsigned long long *cand, int base)
{
    using E = Elem<DT>;
    const int rounds = (bv.c1 - bv.c0 + 31) >> 5;
    for (int r = 0; r < rounds; ++r) {
        const int c = bv.c0 + lane + 32 * r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        uint32_t mask = 0u;
        if (c < bv.c1) {
            v = lds128(bv.slot + c * 16);
            mask = chunk_mask<DT>(v, c, bv, thr);
        }
        const uint32_t cnt = __popc(mask);
        const uint32_t incl = warp_inclusive_scan(cnt, lane);
        int pos = base + (int)(incl - cnt);
        const int first = bv.lo + c * E::kPerChunk;
        while (mask) {
            const int e = __ffs(mask) - 1;
            mask &= mask - 1u;
            cand[pos++] = ((unsigned long long)E::key(element_bits<DT>(v, e)) << 32) |
                          (unsigned long long)(~(uint32_t)(first + e));
        }
        base += (int)__shfl_sync(kFull, incl, 31);
    }
}

// ---------------------------------------------------------------------------
// Final order and output: bitonic sort of the cnt selected composites, then
// index = ~low word and value = the bits the key came from (the input is read
// again only for +-0 and NaN, whose keys do not determine the bits).
// ---------------------------------------------------------------------------
template <int DT>
__device__ void sort_and_write(unsigned long long *arr, int cnt, const Params &p, int row,
                               const unsigned char *xrow)
{
    using E = Elem<DT>;
    const int P = pow2_ceil(cnt > 0 ? cnt : 1);
    for (int i = cnt + threadIdx.x; i < P; i += kThreads)
        arr[i] = 0ull;
    __syncthreads();
    bitonic_sort_u64(arr, P, true);
    const long long obase = (long long)row * p.k;
    for (int i = threadIdx.x; i < p.k; i += kThreads) {
        int32_t idx = -1;
        uint32_t bits = E::kNegInfBits;
        if (i < cnt) {
            const unsigned long long c = arr[i];
            idx = (int32_t)(~(uint32_t)c);
            const uint32_t key = (uint32_t)(c >> 32);
            if (key == E::kNanKey || key == E::kZeroKey)
                bits = DT == 0 ? reinterpret_cast<const uint32_t *>(xrow)[idx]
                               : reinterpret_cast<const uint16_t *>(xrow)[idx];
            else
                bits = E::bits_of_key(key);
        }
        p.out_idx[obase + i] = idx;
        if (DT == 0)
            reinterpret_cast<uint32_t *>(p.out_val)[obase + i] = bits;
        else
            reinterpret_cast<uint16_t *>(p.out_val)[obase + i] = (uint16_t)bits;
    }
}

// ---------------------------------------------------------------------------
// The kernel.  grid = rows * splits, cluster = (splits, 1, 1) when splits > 1.
// ---------------------------------------------------------------------------
template <int DT, bool BULK, bool STATS>
__global__ void __launch_bounds__(kThreads, 1) deepselect_topk_kernel(const Params p)
{
    using E = Elem<DT>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = p.splits;
    const int row = blockIdx.x / S, slice = blockIdx.x % S;

    unsigned char *ring = smem;
    unsigned long long *cand = reinterpret_cast<unsigned long long *>(smem + p.off_cand);
    unsigned long long *perm = reinterpret_cast<unsigned long long *>(smem + p.off_perm);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + p.off_hist);
    uint16_t *holes = reinterpret_cast<uint16_t *>(smem + p.off_holes);
    Misc *ms = reinterpret_cast<Misc *>(smem + p.off_misc);

    long long len_ll = p.row_len ? (long long)p.row_len[row] : p.N;
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
    const int P = pow2_ceil(msl > 0 ? msl : 1);
    for (int i = tid; i < P; i += kThreads) {
        unsigned long long v = ~0ull;
        if (i < msl) {
            const uint32_t b = (uint32_t)(first_block + i);
            const uint32_t w = philox_word0(b, (uint32_t)row, (uint32_t)slice, 0u, p.seed_lo, p.seed_hi);
            v = ((unsigned long long)w << 32) | b;
        }
        perm[i] = v;
    }
    if (tid == 0) {
        ms->flag = 0;
        if (BULK) {
            for (int s = 0; s < p.stages; ++s)
                mbar_init(smem_addr(&ms->bar[s]), 1u);
            mbar_fence_init();
        }
    }
    __syncthreads();
    bitonic_sort_u64(perm, P, false);

    const int bps = p.bps;
    const int nst = (msl + bps - 1) / bps;
    const int esz = E::kSize;

    // thread 0 issues the bulk copies of stage st into ring slot st % stages
    int issued = 0;  // stages issued so far (thread 0)
    auto issue_stage = [&](int st) {
        issued = st + 1;
        const int buf = st % p.stages;
        const uint32_t bar = smem_addr(&ms->bar[buf]);
        uint32_t total = 0u;
        for (int g = 0; g < bps; ++g) {
            const int q = st * bps + g;
            if (q < msl) {
                const int lo = (int)(uint32_t)perm[q] * B;
                const int hi = min(lo + B, len);
                total += (uint32_t)((hi - lo) * esz) & ~15u;
            }
        }
        mbar_arrive_expect_tx(bar, total);
        for (int g = 0; g < bps; ++g) {
            const int q = st * bps + g;
            if (q < msl) {
                const int lo = (int)(uint32_t)perm[q] * B;
                const int hi = min(lo + B, len);
                const uint32_t nb = (uint32_t)((hi - lo) * esz) & ~15u;
                if (nb)
                    bulk_copy_g2s(smem_addr(ring + (size_t)(buf * bps + g) * p.slot_bytes),
                                  xrow + (size_t)lo * esz, nb, bar);
            }
        }
    };
    if (BULK && tid == 0) {
        const int pre = min(p.stages, nst);
        for (int st = 0; st < pre; ++st)
            issue_stage(st);
    }

    Threshold thr = threshold_initial<DT>();
    int n = 0;                              // candidates in the buffer
    long long A = 0, R = 0, W = 0, peak = 0;
    bool failed = false;
    int failed_stage = 0;
    const int kB2 = p.k + p.B2;
    const int g = warp / p.wpb, sub = warp % p.wpb;

    for (int st = 0; st < nst; ++st) {
        const int buf = BULK ? st % p.stages : 0;
        if (BULK && !mbar_wait_bounded(smem_addr(&ms->bar[buf]), (uint32_t)((st / p.stages) & 1)))
            ms->flag = 1;

        BlockView bv;
        const int q = st * bps + g;
        const bool has = q < msl;
        bv.slot = ring + (size_t)(buf * bps + g) * p.slot_bytes;
        bv.lo = has ? (int)(uint32_t)perm[q] * B : 0;
        bv.hi = has ? min(bv.lo + B, len) : 0;
        const int nbytes = (bv.hi - bv.lo) * esz;
        const int nch = (nbytes + 15) >> 4;
        bv.c0 = min(sub * p.cpw, nch);
        bv.c1 = min(bv.c0 + p.cpw, nch);

        // chunks not delivered by a bulk copy (plain-load path, or the ragged
        // tail of a row) are loaded by the lane that will filter them
        if (has) {
            const int bulk_end = BULK ? (nbytes & ~15) : 0;
            for (int c = bv.c0 + lane; c < bv.c1; c += 32) {
                if (c * 16 >= bulk_end) {
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
            if (mine) {
                const bool ge = (uint32_t)bv.lo < thr.ti;
                bv.t = ge ? thr.t_ge : thr.t_gt;
                bv.refine = ge ? (thr.nan_ge || (uint32_t)bv.hi > thr.ti) : thr.nan_gt;
            }
            const int cnt = mine ? warp_count<DT>(bv, thr, lane) : 0;
            if (lane == 0)
                ms->cntw[warp] = cnt;
            const int any = __syncthreads_or(cnt != 0);
            if (ms->flag) {
                failed = true;
                break;
            }
            // every thread is past stage st-1: its ring slot can be refilled
            if (BULK && gstart == 0 && tid == 0 && st > 0 && st - 1 + p.stages < nst) {
                fence_proxy_async_smem();
                issue_stage(st - 1 + p.stages);
            }
            if (!any)
                break;
            // blocks in stage order; find the first one after which the
            // buffer reaches k + B2
            int run = n, trig = -1, before_me = 0;
            for (int w2 = gstart * p.wpb; w2 < bps * p.wpb; ++w2) {
                const int c = ms->cntw[w2];
                if (w2 < warp)
                    before_me += c;
                run += c;
                if ((w2 % p.wpb) == p.wpb - 1 && run >= kB2) {
                    trig = w2 / p.wpb;
                    break;
                }
            }
            const int gend = trig >= 0 ? trig : bps - 1;
            if (mine && g <= gend && cnt)
                warp_append<DT>(bv, thr, lane, cand, n + before_me);
            A += run - n;
            peak = run > peak ? run : peak;
            n = run;
            __syncthreads();
            if (trig < 0)
                break;
            W += n;
            R += 1;
            const unsigned long long tcomp =
                radix_select_topk<DT>(cand, n, p.k, hist, holes, ms, p.idx_bits);
            n = p.k;
            thr = threshold_from<DT>(tcomp);
            gstart = trig + 1;
            if (gstart >= bps)
                break;
        }
        if (failed) {
            failed_stage = st;
            break;
        }
    }

    if (failed) {
        // wait (bounded) for every copy still in flight, record the failure
        // and give up the slice
        if (tid == 0) {
            if (BULK)
                for (int s = failed_stage; s < issued; ++s)
                    (void)mbar_wait_bounded(smem_addr(&ms->bar[s % p.stages]),
                                            (uint32_t)((s / p.stages) & 1));
            atomicOr(&g_status, 1u);
        }
        n = 0;
        __syncthreads();
    }

    // -- final TopK of the slice ---------------------------------------------
    W += n;
    if (n > p.k)
        radix_select_topk<DT>(cand, n, p.k, hist, holes, ms, p.idx_bits);
    const int cnt = n < p.k ? n : p.k;
    if (STATS && tid == 0) {
        long long *s = p.stats + ((long long)row * S + slice) * 4;
        s[0] = A;
        s[1] = R;
        s[2] = W;
        s[3] = peak;
    }

    if (S == 1) {
        sort_and_write<DT>(cand, cnt, p, row, xrow);
        return;
    }

    // -- split rows: partial top-k of every slice into CTA 0 -------------------
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();  // every CTA has finished streaming; CTA 0's ring is free
    unsigned long long *dst =
        cluster.map_shared_rank(reinterpret_cast<unsigned long long *>(ring), 0) +
        (size_t)slice * p.k;
    for (int i = tid; i < p.k; i += kThreads)
        dst[i] = i < cnt ? cand[i] : 0ull;  // 0 sorts below every real composite
    if (tid == 0)
        *cluster.map_shared_rank(&ms->merge_count[slice], 0) = cnt;
    cluster.sync();
    if (slice != 0)
        return;
    int total = 0;
    for (int s = 0; s < S; ++s)
        total += ms->merge_count[s];
    const int kk = total < p.k ? total : p.k;
    unsigned long long *merged = reinterpret_cast<unsigned long long *>(ring);
    const int nm = S * p.k;
    if (kk > 0 && nm > kk)
        radix_select_topk<DT>(merged, nm, kk, hist, holes, ms, p.idx_bits);
    sort_and_write<DT>(merged, kk, p, row, xrow);
}

}  // namespace ds

// ===========================================================================
// Host side: argument checks, launch planning, C ABI.
// ===========================================================================
namespace {

using ds::Params;

thread_local char g_detail[512];

int fail(int status, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
    va_end(ap);
    return status;
}

int fail_cuda(cudaError_t e, const char *what)
{
    return fail(DS_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct ClusterFit {
    const void *fn;
    int splits, smem, nclusters;
};

struct DevInfo {
    bool ready = false;
    ClusterFit fits[32];   // cached cluster-capacity answers (no query during graph capture)
    int nfits = 0;
    int sms = 0;
    int smem_optin = 0;    // max dynamic shared memory per CTA
    int smem_per_sm = 0;   // shared memory per SM
    int smem_reserved = 0; // reserved shared memory per CTA
    unsigned attr_set = 0; // kernels whose smem attribute was raised
};

constexpr int kMaxDevices = 64;
DevInfo g_devs[kMaxDevices];
std::mutex g_mu;

int device_info(DevInfo **out, int *dev_out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(DS_EUNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    DevInfo &d = g_devs[dev];
    if (!d.ready) {
        int v = 0;
        if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail_cuda(e, "cudaDeviceGetAttribute(SM count)");
        d.sms = v;
        if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return fail_cuda(e, "cudaDeviceGetAttribute(smem opt-in)");
        d.smem_optin = v;
        if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
            return fail_cuda(e, "cudaDeviceGetAttribute(smem per SM)");
        d.smem_per_sm = v;
        if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess)
            return fail_cuda(e, "cudaDeviceGetAttribute(reserved smem)");
        d.smem_reserved = v;
        d.ready = true;
    }
    *out = &d;
    if (dev_out)
        *dev_out = dev;
    return DS_OK;
}

typedef void (*KernelFn)(Params);

KernelFn kernel_for(int dtype, bool bulk, bool stats, int *slot)
{
    static const KernelFn table[8] = {
        ds::deepselect_topk_kernel<0, false, false>, ds::deepselect_topk_kernel<0, false, true>,
        ds::deepselect_topk_kernel<0, true, false>,  ds::deepselect_topk_kernel<0, true, true>,
        ds::deepselect_topk_kernel<1, false, false>, ds::deepselect_topk_kernel<1, false, true>,
        ds::deepselect_topk_kernel<1, true, false>,  ds::deepselect_topk_kernel<1, true, true>,
    };
    const int i = dtype * 4 + (bulk ? 2 : 0) + (stats ? 1 : 0);
    *slot = i;
    return table[i];
}

int ensure_attributes(DevInfo &d, int dtype, bool bulk, bool stats, KernelFn *fn)
{
    int slot = 0;
    *fn = kernel_for(dtype, bulk, stats, &slot);
    std::lock_guard<std::mutex> lock(g_mu);
    if (d.attr_set & (1u << slot))
        return DS_OK;
    cudaError_t e = cudaFuncSetAttribute((const void *)*fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         d.smem_optin);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaFuncSetAttribute(max dynamic smem)");
    e = cudaFuncSetAttribute((const void *)*fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaFuncSetAttribute(non-portable cluster size)");
    d.attr_set |= 1u << slot;
    return DS_OK;
}

int check_args(const void *x, int dtype, int rows, int64_t N, int k, int B, int B2, int splits,
               const void *out_idx, const void *out_val)
{
    if (dtype != DS_FP32 && dtype != DS_BF16)
        return fail(DS_EUNSUPPORTED, "dtype %d is not DS_FP32 (0) or DS_BF16 (1)", dtype);
    if (rows < 0)
        return fail(DS_EINVAL, "rows = %d is negative", rows);
    if (N < 1 || N >= (int64_t)1 << 31)
        return fail(DS_EINVAL, "N = %lld is outside [1, 2^31)", (long long)N);
    if (k < 1 || (int64_t)k > N)
        return fail(DS_EINVAL, "k = %d is outside [1, N = %lld]", k, (long long)N);
    if (B < 1 || B2 < 1)
        return fail(DS_EINVAL, "B = %d and B2 = %d must both be >= 1", B, B2);
    if (splits < 0 || splits > ds::kMaxSplits)
        return fail(DS_EINVAL, "splits = %d is outside [0, %d]", splits, ds::kMaxSplits);
    if (rows > 0 && (!x || !out_idx || !out_val))
        return fail(DS_EINVAL, "x, out_idx and out_val must be non-NULL when rows > 0");
    return DS_OK;
}

struct Plan {
    Params p;
    int grid;
    int smem;
    int ctas_per_sm;
    bool bulk;
};

int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Shared-memory layout for a given split factor and ring depth.
long long layout(Plan &pl, int stages, int splits)
{
    Params &p = pl.p;
    const long long ring_stream = (long long)stages * p.bps * p.slot_bytes;
    const long long ring_merge = splits > 1 ? (long long)splits * p.k * 8 : 0;
    long long off = align_up((int)(ring_stream > ring_merge ? ring_stream : ring_merge), 128);
    const long long cap = (long long)(p.k + (long long)p.B + p.B2) > ds::pow2_ceil(p.k)
                              ? (long long)p.k + p.B + p.B2
                              : ds::pow2_ceil(p.k);
    p.off_cand = (int)off;
    off += cap * 8;
    const long long m = (p.N + p.B - 1) / p.B;
    const long long per = (m + splits - 1) / splits;
    p.off_perm = (int)off;
    off += (long long)ds::pow2_ceil((int)(per > 0 ? per : 1)) * 8;
    p.off_hist = (int)off;
    off += 2 * 256 * 4;
    p.off_holes = (int)off;
    off += align_up(p.k * 2, 16);
    p.off_misc = (int)off;
    off += align_up((int)sizeof(ds::Misc), 16);
    return off;
}

constexpr long long kMaxPermBlocks = 4096;  // blocks per slice the in-CTA order holds

int make_plan(const void *x, int dtype, int rows, int64_t N, int k, int B, int B2, int splits_req,
              bool stats, DevInfo &d, Plan &pl)
{
    memset(&pl, 0, sizeof(pl));
    Params &p = pl.p;
    const int esz = dtype == DS_FP32 ? 4 : 2;
    p.N = N;
    p.k = k;
    p.B = B;
    p.B2 = B2;
    const long long cap = (long long)k + B + B2;
    if (cap > 65535)
        return fail(DS_EUNSUPPORTED,
                    "k + B + B2 = %lld exceeds the 65535-entry candidate buffer; query ds_topk_max_k",
                    cap);
    const long long slot = ((long long)B * esz + 15) / 16 * 16;
    if (slot > 64 * 1024)
        return fail(DS_EUNSUPPORTED, "B * sizeof(elem) = %lld bytes exceeds 64 KiB", (long long)B * esz);
    pl.bulk = ((uintptr_t)x % 16 == 0) && ((N * esz) % 16 == 0) && (((long long)B * esz) % 16 == 0);
    p.slot_bytes = (int)slot;
    int wpb = 1;
    while (wpb < ds::kWarps && p.slot_bytes / (wpb * 2) >= 2048)
        wpb *= 2;
    p.wpb = wpb;
    p.bps = ds::kWarps / wpb;
    p.cpw = (p.slot_bytes / 16 + wpb - 1) / wpb;
    int bits = 1;
    while (bits < 31 && ((long long)1 << bits) < N)
        ++bits;
    p.idx_bits = (bits + 7) / 8 * 8;
    if (p.idx_bits > 32)
        p.idx_bits = 32;

    const long long m = (N + B - 1) / B;
    const long long budget_one = d.smem_optin;
    const long long half_sm = d.smem_per_sm / 2 - d.smem_reserved;

    auto fits = [&](int stages, int splits, long long limit) -> long long {
        Plan tmp = pl;
        const long long per = (m + splits - 1) / splits;
        if (per > kMaxPermBlocks)
            return -1;
        const long long bytes = layout(tmp, stages, splits);
        return bytes <= limit ? bytes : -1;
    };

    // split factor
    int splits = splits_req;
    if (splits == 0) {
        // aim for at least one CTA per SM when rows are few
        const int stages_guess = pl.bulk ? 4 : 1;
        long long bytes1 = fits(stages_guess, 1, half_sm);
        int per_sm = bytes1 > 0 ? 2 : 1;
        const long long slots = (long long)d.sms * per_sm;
        splits = 1;
        if ((long long)rows * 2 < slots) {
            long long want = slots / (rows > 0 ? rows : 1);
            if (want > 8)
                want = 8;
            if (want > m)
                want = m;
            splits = (int)(want < 1 ? 1 : want);
        }
        while (splits > 1 && fits(pl.bulk ? 2 : 1, splits, budget_one) < 0)
            --splits;
    }
    if (splits > 1 && (long long)splits * k * 8 > budget_one)
        return fail(DS_EUNSUPPORTED, "splits * k * 8 = %lld bytes does not fit shared memory",
                    (long long)splits * k * 8);
    p.splits = splits;
    if ((m + splits - 1) / splits > kMaxPermBlocks)
        return fail(DS_EUNSUPPORTED,
                    "ceil(N/B) / splits = %lld blocks per slice exceeds %lld; raise B or splits",
                    (m + splits - 1) / splits, kMaxPermBlocks);

    // ring depth: deepest that keeps two CTAs per SM, else deepest that fits
    int stages = 0;
    long long bytes = -1;
    if (pl.bulk) {
        for (int s = ds::kMaxStages; s >= 2 && bytes < 0; --s) {
            bytes = fits(s, splits, half_sm);
            if (bytes >= 0)
                stages = s;
        }
        for (int s = ds::kMaxStages; s >= 2 && bytes < 0; --s) {
            bytes = fits(s, splits, budget_one);
            if (bytes >= 0)
                stages = s;
        }
    }
    if (bytes < 0) {
        // two bulk stages do not fit (or the layout forbids bulk copies):
        // one stage filled by plain loads
        pl.bulk = false;
        bytes = fits(1, splits, budget_one);
        stages = 1;
    }
    if (bytes < 0)
        return fail(DS_EUNSUPPORTED,
                    "working set for k=%d, B=%d, B2=%d, splits=%d exceeds %d bytes of shared "
                    "memory; query ds_topk_max_k",
                    k, B, B2, splits, d.smem_optin);
    p.stages = stages;
    pl.smem = (int)layout(pl, stages, splits);
    pl.grid = rows * splits;
    pl.ctas_per_sm = (int)((d.smem_per_sm) / (pl.smem + d.smem_reserved));
    if (pl.ctas_per_sm > 2048 / ds::kThreads)
        pl.ctas_per_sm = 2048 / ds::kThreads;
    (void)stats;
    return DS_OK;
}

// Clusters of this plan's size that can be resident at once (0: none).
// Answers are cached per device so that steady-state calls make no query.
int cluster_capacity(DevInfo &d, KernelFn fn, const Plan &pl, int *nclusters)
{
    {
        std::lock_guard<std::mutex> lock(g_mu);
        for (int i = 0; i < d.nfits; ++i)
            if (d.fits[i].fn == (const void *)fn && d.fits[i].splits == pl.p.splits &&
                d.fits[i].smem == pl.smem) {
                *nclusters = d.fits[i].nclusters;
                return DS_OK;
            }
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)pl.p.splits, 1, 1);
    cfg.blockDim = dim3(ds::kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)pl.smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)pl.p.splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaOccupancyMaxActiveClusters(nclusters, (const void *)fn, &cfg);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        *nclusters = 0;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (d.nfits < 32)
        d.fits[d.nfits++] = ClusterFit{(const void *)fn, pl.p.splits, pl.smem, *nclusters};
    return DS_OK;
}

int launch(const void *x, int dtype, int rows, const int32_t *row_len, int64_t N, int k, int B,
           int B2, uint64_t seed, int splits_req, int32_t *out_idx, void *out_val, int64_t *stats,
           cudaStream_t stream)
{
    int rc = check_args(x, dtype, rows, N, k, B, B2, splits_req, out_idx, out_val);
    if (rc != DS_OK)
        return rc;
    if (stats && splits_req < 1)
        return fail(DS_EINVAL, "stats need an explicit splits >= 1");
    if (rows == 0)
        return DS_OK;
    DevInfo *d = nullptr;
    if ((rc = device_info(&d, nullptr)) != DS_OK)
        return rc;
    Plan pl;
    if ((rc = make_plan(x, dtype, rows, N, k, B, B2, splits_req, stats != nullptr, *d, pl)) != DS_OK)
        return rc;
    KernelFn fn = nullptr;
    if ((rc = ensure_attributes(*d, dtype, pl.bulk, stats != nullptr, &fn)) != DS_OK)
        return rc;
    // a cluster must fit on one GPC: shrink an automatic split factor until
    // the hardware can hold at least one cluster
    while (pl.p.splits > 1) {
        int nclusters = 0;
        if ((rc = cluster_capacity(*d, fn, pl, &nclusters)) != DS_OK)
            return rc;
        if (nclusters >= 1)
            break;
        if (splits_req != 0)
            return fail(DS_EUNSUPPORTED,
                        "a cluster of %d CTAs with %d bytes of shared memory each cannot be "
                        "scheduled on this device",
                        pl.p.splits, pl.smem);
        if ((rc = make_plan(x, dtype, rows, N, k, B, B2, pl.p.splits - 1, stats != nullptr, *d,
                            pl)) != DS_OK)
            return rc;
    }
    if ((long long)rows * pl.p.splits > 0x7FFFFFFFLL)
        return fail(DS_EINVAL, "rows * splits exceeds the grid limit");
    Params &p = pl.p;
    p.x = x;
    p.row_len = row_len;
    p.out_idx = out_idx;
    p.out_val = out_val;
    p.stats = reinterpret_cast<long long *>(stats);
    p.seed_lo = (uint32_t)seed;
    p.seed_hi = (uint32_t)(seed >> 32);

    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
    cfg.blockDim = dim3(ds::kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.splits > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)p.splits;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, p);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaLaunchKernelEx");
    return DS_OK;
}

size_t elem_size(int dtype) { return dtype == DS_FP32 ? 4 : 2; }

}  // namespace

extern "C" {

int ds_topk(const void *x, int dtype, int rows, const int32_t *row_len, int64_t N, int k, int B,
            int B2, uint64_t seed, int32_t *out_idx, void *out_val, void *stream)
{
    g_detail[0] = '\0';
    return launch(x, dtype, rows, row_len, N, k, B, B2, seed, 0, out_idx, out_val, nullptr,
                  (cudaStream_t)stream);
}

int ds_topk_ex(const void *x, int dtype, int rows, const int32_t *row_len, int64_t N, int k,
               int B, int B2, uint64_t seed, int splits, int32_t *out_idx, void *out_val,
               int64_t *stats, void *stream)
{
    g_detail[0] = '\0';
    return launch(x, dtype, rows, row_len, N, k, B, B2, seed, splits, out_idx, out_val, stats,
                  (cudaStream_t)stream);
}

int ds_topk_host(const void *x_host, int dtype, int rows, const int32_t *row_len_host, int64_t N,
                 int k, int B, int B2, uint64_t seed, int32_t *out_idx_host, void *out_val_host,
                 void *x_dev, int32_t *row_len_dev, int32_t *out_idx_dev, void *out_val_dev,
                 void *stream)
{
    g_detail[0] = '\0';
    int rc = check_args(x_host, dtype, rows, N, k, B, B2, 0, out_idx_host, out_val_host);
    if (rc != DS_OK)
        return rc;
    if (rows > 0 && (!x_dev || !out_idx_dev || !out_val_dev))
        return fail(DS_EINVAL, "device staging buffers must be non-NULL when rows > 0");
    if ((row_len_host == nullptr) != (row_len_dev == nullptr))
        return fail(DS_EINVAL, "row_len_host and row_len_dev must both be given or both be NULL");
    if (rows == 0)
        return DS_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t es = elem_size(dtype);
    cudaError_t e = cudaMemcpyAsync(x_dev, x_host, (size_t)rows * (size_t)N * es,
                                    cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaMemcpyAsync(x)");
    if (row_len_host) {
        e = cudaMemcpyAsync(row_len_dev, row_len_host, (size_t)rows * 4, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess)
            return fail_cuda(e, "cudaMemcpyAsync(row_len)");
    }
    rc = launch(x_dev, dtype, rows, row_len_dev, N, k, B, B2, seed, 0, out_idx_dev, out_val_dev,
                nullptr, s);
    if (rc != DS_OK)
        return rc;
    e = cudaMemcpyAsync(out_idx_host, out_idx_dev, (size_t)rows * k * 4, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaMemcpyAsync(out_idx)");
    e = cudaMemcpyAsync(out_val_host, out_val_dev, (size_t)rows * k * es, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaMemcpyAsync(out_val)");
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaStreamSynchronize");
    return DS_OK;
}

int ds_topk_plan(const void *x, int dtype, int rows, int64_t N, int k, int B, int B2, int splits,
                 ds_plan_t *plan)
{
    g_detail[0] = '\0';
    if (!plan)
        return fail(DS_EINVAL, "plan must be non-NULL");
    int rc = check_args(x ? x : (const void *)16, dtype, rows, N, k, B, B2, splits,
                        (const void *)16, (const void *)16);
    if (rc != DS_OK)
        return rc;
    DevInfo *d = nullptr;
    if ((rc = device_info(&d, nullptr)) != DS_OK)
        return rc;
    Plan pl;
    if ((rc = make_plan(x, dtype, rows, N, k, B, B2, splits, false, *d, pl)) != DS_OK)
        return rc;
    plan->splits = pl.p.splits;
    plan->threads = ds::kThreads;
    plan->stages = pl.p.stages;
    plan->blocks_per_stage = pl.p.bps;
    plan->warps_per_block = pl.p.wpb;
    plan->bulk = pl.bulk ? 1 : 0;
    plan->smem_bytes = pl.smem;
    plan->capacity = (pl.p.off_perm - pl.p.off_cand) / 8;
    plan->grid = pl.grid;
    plan->ctas_per_sm = pl.ctas_per_sm;
    return DS_OK;
}

int ds_topk_max_k(int dtype, int B, int B2)
{
    g_detail[0] = '\0';
    if (dtype != DS_FP32 && dtype != DS_BF16)
        return fail(DS_EUNSUPPORTED, "dtype %d is not DS_FP32 or DS_BF16", dtype);
    if (B < 1 || B2 < 1)
        return fail(DS_EINVAL, "B and B2 must be >= 1");
    DevInfo *d = nullptr;
    int rc = device_info(&d, nullptr);
    if (rc != DS_OK)
        return rc;
    const long long N = (long long)B * kMaxPermBlocks < ((long long)1 << 31) - 1
                            ? (long long)B * kMaxPermBlocks
                            : ((long long)1 << 31) - 1;
    int lo = 0, hi = 65535;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        Plan pl;
        if (mid <= N && make_plan((const void *)16, dtype, 1, N, mid, B, B2, 1, false, *d, pl) == DS_OK)
            lo = mid;
        else
            hi = mid - 1;
    }
    g_detail[0] = '\0';
    if (lo == 0)
        return fail(DS_EUNSUPPORTED, "no k fits shared memory for B=%d, B2=%d", B, B2);
    return lo;
}

int ds_topk_device_status(void)
{
    g_detail[0] = '\0';
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaDeviceSynchronize");
    unsigned int v = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&v, ds::g_status, sizeof(v));
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaMemcpyFromSymbol(status)");
    e = cudaMemcpyToSymbol(ds::g_status, &zero, sizeof(zero));
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaMemcpyToSymbol(status)");
    if (v)
        return fail(DS_EDEVICE, "a kernel gave up waiting for a bulk copy (status 0x%x)", v);
    return DS_OK;
}

const char *ds_strerror(int status)
{
    switch (status) {
    case DS_OK: return "success";
    case DS_EINVAL: return "invalid argument";
    case DS_EUNSUPPORTED: return "unsupported dtype or working set too large for shared memory";
    case DS_ECUDA: return "CUDA runtime error";
    case DS_EDEVICE: return "a kernel timed out waiting for a bulk copy";
    default: return "unknown status";
    }
}

const char *ds_last_error_detail(void) { return g_detail; }

}  // extern "C"
