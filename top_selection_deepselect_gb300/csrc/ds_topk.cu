// ds_topk.cu -- host side of the DeepSelect top-k library: argument checks,
// launch planning (kernel, split factor, ring depth, shared-memory layout)
// and the C ABI declared in include/ds_topk.h.  The kernels are in
// ds_kernel.cuh (block by block, with counters) and ds_stream.cuh (free-running
// warps), instantiated per dtype in ds_kernels_fp32.cu, ds_kernels_bf16.cu and
// ds_kernels_fp16.cu.

#include "ds_topk.h"

#include <cuda_runtime.h>

#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "ds_stream.cuh"

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
    unsigned char *noalloc_ws = nullptr;  // device address of g_noalloc_ws on this device
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

using ds::KernelFn;

// 18 instantiations: the block-by-block kernel per dtype x asynchronous
// copies x mask rounds (4 rounds cover blocks of up to 2 KiB per warp, 16 up
// to 8 KiB per warp), and the free-running kernel per dtype x pairs.
KernelFn kernel_for(int dtype, bool stream, bool pairs, bool async, bool wide, int *slot)
{
    if (stream) {
        *slot = 12 + dtype * 2 + (pairs ? 1 : 0);
        return dtype == DS_FP32 ? ds::stream_kernel_fp32(pairs)
             : dtype == DS_BF16 ? ds::stream_kernel_bf16(pairs) : ds::stream_kernel_fp16(pairs);
    }
    *slot = dtype * 4 + (async ? 2 : 0) + (wide ? 1 : 0);
    return dtype == DS_FP32 ? ds::kernel_fp32(async, wide)
         : dtype == DS_BF16 ? ds::kernel_bf16(async, wide) : ds::kernel_fp16(async, wide);
}

int ensure_attributes(DevInfo &d, int dtype, bool stream, bool pairs, bool async, bool wide,
                      KernelFn *fn)
{
    int slot = 0;
    *fn = kernel_for(dtype, stream, pairs, async, wide, &slot);
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
    if (dtype != DS_FP32 && dtype != DS_BF16 && dtype != DS_FP16)
        return fail(DS_EUNSUPPORTED, "dtype %d is not DS_FP32 (0), DS_BF16 (1) or DS_FP16 (2)", dtype);
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
    bool async;
    bool stream;    // free-running kernel (no counters)
    int per_chunk;  // elements per 16-byte chunk
};


// Shared-memory layout for a given split factor and ring depth.  Every region
// starts on a 128-byte boundary (asynchronous-copy destinations need 16 bytes, the
// scratch words are read with 128-bit loads).
long long align128(long long v) { return (v + 127) / 128 * 128; }

long long layout(Plan &pl, int stages, int splits)
{
    Params &p = pl.p;
    const long long ring_stream = pl.stream ? (long long)ds::kWarps * stages * ds::kStageBytes
                                            : (long long)stages * p.bps * p.slot_bytes;
    const long long ring_merge = splits > 1 ? (long long)splits * p.k * 8 : 0;
    long long off = align128(ring_stream > ring_merge ? ring_stream : ring_merge);
    // block by block: k + B + B2 (the largest length the loop reaches);
    // free-running: k + B2 + the largest reservation, a pair of pieces
    // (reservations beyond that are filled with the composite 0 and retried
    // after a compaction; the first reservation after a compaction starts
    // at k and always fits, so every retry makes progress)
    // pairs only where the first threshold is seeded (small k): from -inf a
    // pair reserves two whole pieces, and the larger buffer makes the first
    // select larger (DSA index scores, k = 512: 27.7 -> 38.9 us with pairs)
    p.pairs = pl.stream && p.k <= ds::kSeedMaxK ? 1 : 0;
    long long cap = pl.stream ? (long long)p.k + p.B2 +
                                    (long long)(p.pairs ? ds::kPairChunks : ds::kStageChunks) * pl.per_chunk
                              : (long long)p.k + p.B + p.B2;
    if (cap < ds::pow2_ceil(p.k))
        cap = ds::pow2_ceil(p.k);
    if (cap < 32)
        cap = 32;
    p.cap = (int)cap;
    p.off_cand = (int)off;
    off = align128(off + cap * 8);
    const long long m = (p.N + p.B - 1) / p.B;
    const long long per = (m + splits - 1) / splits;
    // block order: (Philox word, id) pairs sorted in place (block by block), or
    // the block id at each position (free-running)
    p.off_perm = (int)off;
    off = align128(off + (pl.stream ? per * 4 : (long long)ds::pow2_ceil((int)(per > 32 ? per : 32)) * 8));
    // digit histograms: three rotating 256-bin buffers for the register
    // select; the per-warp histograms of the shared-memory select only when
    // a select can exceed the register select's 6144 entries (the buffer, or
    // the union of a split row in CTA 0).  The cluster select of a split row
    // (splits * k above 8192) uses four 256-bin buffers of that region.
    const long long reg_max = 24LL * ds::kThreads;
    const bool big_select = cap > reg_max || (splits > 1 && (long long)splits * p.k > reg_max);
    p.hist_words = big_select ? ds::kHistWords : 3 * ds::kHistBins;
    p.off_hist = (int)off;
    off = align128(off + (long long)p.hist_words * 4);
    p.off_holes = (int)off;
    off = align128(off + (long long)p.k * 2);
    p.off_misc = (int)off;
    off = align128(off + (long long)sizeof(ds::Misc));
    return off;
}

constexpr long long kMaxPermBlocks = 4096;  // blocks per slice the in-CTA order holds
constexpr long long kMaxAutoSplits = 16;     // largest automatic split factor
constexpr long long kStreamSliceBytes = 128 * 1024;  // slices that keep a second CTA per SM busy
constexpr long long kMinSliceBytes = 64 * 1024;      // free-running kernel: smallest automatic slice

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
    pl.async = ((uintptr_t)x % 16 == 0) && ((N * esz) % 16 == 0) && (((long long)B * esz) % 16 == 0);
    pl.per_chunk = 16 / esz;
    // the free-running kernel serves every call without counters whose rows
    // take 16-byte copies; counters follow the block-by-block loop exactly
    pl.stream = !stats && pl.async;
    p.slot_bytes = (int)slot;
    int wpb = 1;
    while (wpb < ds::kWarps && p.slot_bytes / (wpb * 2) >= 2048)
        wpb *= 2;
    p.wpb = wpb;
    p.wpb_shift = wpb == 1 ? 0 : wpb == 2 ? 1 : wpb == 4 ? 2 : 3;
    p.bps = ds::kWarps / wpb;
    p.cpw = (p.slot_bytes / 16 + wpb - 1) / wpb;

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

    // split factor (automatic): a power of two, at most kMaxAutoSplits and
    // one block per slice.  Rows that are short for the GPU run latency
    // bound, and two CTAs on one SM slow each other down, so the default
    // fills the SMs with one CTA each; a second CTA per SM is taken only
    // when its slices still stream at least kStreamSliceBytes each.
    int splits = splits_req;
    if (splits == 0) {
        const long long r = rows > 0 ? rows : 1;
        auto pow2_floor = [](long long v) {
            long long q = 1;
            while (2 * q <= v)
                q *= 2;
            return q;
        };
        auto cap = [&](long long v) {
            v = v < kMaxAutoSplits ? v : kMaxAutoSplits;
            v = v < m ? v : m;
            return pow2_floor(v < 1 ? 1 : v);
        };
        long long one = cap((long long)d.sms / r);
        while (one > 1 && fits(pl.async ? 2 : 1, (int)one, budget_one) < 0)
            one /= 2;
        long long two = cap(2LL * d.sms / r);
        while (two > one && fits(pl.async ? 2 : 1, (int)two, half_sm) < 0)
            two /= 2;
        const long long slice_bytes = (m + two - 1) / two * (long long)B * esz;
        splits = (int)(two > one && slice_bytes >= kStreamSliceBytes ? two : one);
        // the free-running kernel's first threshold leaves short slices with
        // few or no compactions, and then the cluster merge costs more than
        // the parallel scan saves: its slices keep kMinSliceBytes at least
        while (pl.stream && splits > 1 && (m + splits - 1) / splits * (long long)B * esz < kMinSliceBytes)
            splits /= 2;
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
    if (pl.stream) {
        for (int s = ds::kMaxStreamStages; s >= 2 && bytes < 0; --s) {
            bytes = fits(s, splits, half_sm);
            if (bytes >= 0)
                stages = s;
        }
        for (int s = ds::kMaxStreamStages; s >= 2 && bytes < 0; --s) {
            bytes = fits(s, splits, budget_one);
            if (bytes >= 0)
                stages = s;
        }
        if (bytes < 0)
            pl.stream = false;  // the block-by-block kernel's smaller ring may fit
    }
    if (!pl.stream && pl.async) {
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
        // two ring slots do not fit (or the layout forbids 16-byte copies):
        // one stage filled by plain loads
        pl.async = false;
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

#ifdef DS_CHECKED
// Bounds-checked builds only (the tests build one): a device word that the
// kernels' DS_GUARD checks OR their violation bits into.
unsigned int *g_check = nullptr;

int check_word(unsigned int **out)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_check == nullptr) {
        cudaError_t e = cudaMalloc(&g_check, sizeof(unsigned int));
        if (e == cudaSuccess)
            e = cudaMemset(g_check, 0, sizeof(unsigned int));
        if (e != cudaSuccess)
            return fail_cuda(e, "bounds-check word");
    }
    *out = g_check;
    return DS_OK;
}
#endif

// `total` = elements in x when row_len is NULL (rows * N for a matrix; less
// when the rows are consecutive pieces of one long row with a short last piece).
// With enqueue = false every check and planning step runs and nothing is launched.
int launch(const void *x, int dtype, int rows, const int32_t *row_len, int64_t N, int64_t total,
           int k, int B, int B2, uint64_t seed, int splits_req, int32_t *out_idx, void *out_val,
           int64_t *stats, cudaStream_t stream, bool enqueue = true, int order = DS_ORDER_RANDOM)
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
    if ((rc = ensure_attributes(*d, dtype, pl.stream, pl.p.pairs != 0, pl.async, pl.p.cpw > 128, &fn)) !=
        DS_OK)
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
        if ((rc = make_plan(x, dtype, rows, N, k, B, B2, pl.p.splits / 2, stats != nullptr, *d,
                            pl)) != DS_OK)
            return rc;
    }
    if ((long long)rows * pl.p.splits > 0x7FFFFFFFLL)
        return fail(DS_EINVAL, "rows * splits exceeds the grid limit");
    if (!enqueue)
        return DS_OK;
    Params &p = pl.p;
    p.x = x;
    p.row_len = row_len;
    p.total = total;
    p.out_idx = out_idx;
    p.out_val = out_val;
    p.stats = reinterpret_cast<long long *>(stats);
    p.seed_lo = (uint32_t)seed;
#ifdef DS_CHECKED
    if ((rc = check_word(&p.check)) != DS_OK)
        return rc;
#else
    p.check = nullptr;
#endif
    p.seed_hi = (uint32_t)(seed >> 32);
    p.identity = order == DS_ORDER_IDENTITY ? 1 : 0;

    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
    cfg.blockDim = dim3(ds::kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)pl.smem;
    cfg.stream = stream;
    // Programmatic dependent launch: the grid may be scheduled while the
    // previous kernel on the stream drains; the kernels wait for that kernel
    // to complete (griddepcontrol.wait) before they read or write memory.
    // Taken when the grid overfills the SMs anyway, or is small: a grid of
    // one CTA per SM scheduled early lands two CTAs on the SMs that happen
    // to be free, and its latency-bound rows then run slower (DSA index
    // scores: 27.2 -> 31.3 us).
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (pl.grid > d->sms || 2 * pl.grid <= d->sms) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (p.splits > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.splits;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, p);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaLaunchKernelEx");
    return DS_OK;
}

size_t elem_size(int dtype) { return dtype == DS_FP32 ? 4 : 2; }

// ---------------------------------------------------------------------------
// One long row over the whole GPU.  The row is cut into G pieces of P
// elements (the last one shorter), viewed as a [G x P] matrix: the first
// launch takes the exact top k of every piece, the second the top k of the
// G*k piece results laid end to end, and a gather maps each chosen position
// q back to the row index (q / k) * P + (index within piece q / k).
//
// Why the second launch's order is the row's order: a piece's results are
// sorted by (value desc, index asc), pieces are laid out in row order, so
// among equal values a smaller position means a smaller row index.  A last
// piece shorter than k is padded with -inf at its end; with k <= N there are
// at least k real entries, all ranked ahead of every pad (a pad ties only
// with real -inf values and sits after all of them), so no pad is chosen.
// ---------------------------------------------------------------------------
constexpr long long kRowPieceMin = 64;  // pieces hold at least this many k
constexpr size_t kWsAlign = 256;

size_t align_ws(size_t v) { return (v + kWsAlign - 1) / kWsAlign * kWsAlign; }

struct RowPlan {
    long long P;        // piece length (a multiple of B and of 8 elements)
    int G;              // pieces (1: the row is selected directly)
    long long N2;       // row pitch of the second launch (G*k rounded up to 8)
    size_t off_val1, off_q2, bytes;  // workspace layout; idx1 at offset 0
};

long long gcd_ll(long long a, long long b)
{
    while (b) {
        const long long t = a % b;
        a = b;
        b = t;
    }
    return a;
}

int row_plan(int dtype, int64_t N, int k, int B, int sms, RowPlan &rp)
{
    memset(&rp, 0, sizeof(rp));
    const long long unit = (long long)B / gcd_ll(B, 8) * 8;  // lcm(B, 8)
    long long g = (long long)N / (kRowPieceMin * k);
    if (g > 2LL * sms)
        g = 2LL * sms;
    if (g >= 8)
        g = g / 8 * 8;
    if (g < 2 && N > kMaxAutoSplits * kMaxPermBlocks * B)
        g = 2;  // longer than one cluster's block orders hold: cut it anyway
    if (g < 2) {
        rp.G = 1;
        rp.P = N;
        return DS_OK;
    }
    long long P = ((N + g - 1) / g + unit - 1) / unit * unit;
    const long long Pmax = kMaxPermBlocks * B / unit * unit;  // the block order of one CTA
    P = P < Pmax ? P : Pmax;
    const long long Pk = ((long long)k + unit - 1) / unit * unit;
    P = P > Pk ? P : Pk;
    const long long G = (N + P - 1) / P;
    if (G < 2) {
        rp.G = 1;
        rp.P = N;
        return DS_OK;
    }
    rp.P = P;
    rp.G = (int)G;
    rp.N2 = (G * k + 7) / 8 * 8;
    if (rp.N2 >= (long long)1 << 31)
        return fail(DS_EUNSUPPORTED, "pieces * k = %lld exceeds 2^31", G * k);
    const size_t es = elem_size(dtype);
    rp.off_val1 = align_ws((size_t)G * k * 4);
    rp.off_q2 = rp.off_val1 + align_ws((size_t)rp.N2 * es);
    rp.bytes = rp.off_q2 + align_ws((size_t)k * 4);
    return DS_OK;
}

__global__ void long_row_gather(const int32_t *__restrict__ q2, const int32_t *__restrict__ idx1,
                                int k, long long P, int32_t *__restrict__ out_idx)
{
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j < k) {
        const int q = q2[j];
        const int li = q >= 0 ? idx1[q] : -1;
        out_idx[j] = li >= 0 ? (int32_t)((long long)(q / k) * P + li) : -1;
    }
}

int long_row_check(const void *x, int dtype, int64_t N, int k, int B, int B2, const void *out_idx,
                   const void *out_val)
{
    return check_args(x, dtype, 1, N, k, B, B2, 0, out_idx, out_val);
}

int long_row_plan(int dtype, int64_t N, int k, int B, RowPlan &rp)
{
    DevInfo *d = nullptr;
    int rc = device_info(&d, nullptr);
    if (rc != DS_OK)
        return rc;
    return row_plan(dtype, N, k, B, d->sms, rp);
}

// Workspace of ds_topk_long_row_noalloc: one fixed array per device that
// loads the library, held until the process exits.  Every call shares it.
constexpr size_t kNoAllocBytes = 8u << 20;
static __device__ __align__(256) unsigned char g_noalloc_ws[kNoAllocBytes];

// The array's device address on the current device, looked up once per
// device (host code cannot use the symbol itself as a device pointer).
int noalloc_workspace(unsigned char **out)
{
    DevInfo *d = nullptr;
    int dev = 0;
    int rc = device_info(&d, &dev);
    if (rc != DS_OK)
        return rc;
    std::lock_guard<std::mutex> lock(g_mu);
    if (d->noalloc_ws == nullptr) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_ws);
        if (e != cudaSuccess)
            return fail_cuda(e, "cudaGetSymbolAddress(g_noalloc_ws)");
        d->noalloc_ws = static_cast<unsigned char *>(ptr);
    }
    *out = d->noalloc_ws;
    return DS_OK;
}

int long_row_run(const void *x, int dtype, int64_t N, int k, int B, int B2, uint64_t seed,
                 const RowPlan &rp, unsigned char *ws, int32_t *out_idx, void *out_val,
                 cudaStream_t stream)
{
    if (rp.G == 1)
        return launch(x, dtype, 1, nullptr, N, N, k, B, B2, seed, 0, out_idx, out_val, nullptr,
                      stream);
    int32_t *idx1 = reinterpret_cast<int32_t *>(ws);
    void *val1 = ws + rp.off_val1;
    int32_t *q2 = reinterpret_cast<int32_t *>(ws + rp.off_q2);
    // both launches are planned before either is enqueued, so that a size
    // the second one cannot take is reported with nothing enqueued
    for (int pass = 0; pass < 2; ++pass) {
        const bool enqueue = pass == 1;
        int rc = launch(x, dtype, rp.G, nullptr, rp.P, N, k, B, B2, seed, 0, idx1, val1, nullptr,
                        stream, enqueue);
        if (rc != DS_OK)
            return rc;
        rc = launch(val1, dtype, 1, nullptr, rp.N2, (int64_t)rp.G * k, k, B, B2, seed, 0, q2,
                    out_val, nullptr, stream, enqueue);
        if (rc != DS_OK)
            return rc;
    }
    long_row_gather<<<(k + 255) / 256, 256, 0, stream>>>(q2, idx1, k, rp.P, out_idx);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DS_OK : fail_cuda(e, "long_row_gather launch");
}

}  // namespace

extern "C" {

int ds_topk(const void *x, int dtype, int rows, const int32_t *row_len, int64_t N, int k, int B,
            int B2, uint64_t seed, int32_t *out_idx, void *out_val, void *stream)
{
    g_detail[0] = '\0';
    return launch(x, dtype, rows, row_len, N, (int64_t)rows * N, k, B, B2, seed, 0, out_idx, out_val,
                  nullptr, (cudaStream_t)stream);
}

int ds_topk_ex(const void *x, int dtype, int rows, const int32_t *row_len, int64_t N, int k,
               int B, int B2, uint64_t seed, int splits, int32_t *out_idx, void *out_val,
               int64_t *stats, void *stream)
{
    g_detail[0] = '\0';
    return launch(x, dtype, rows, row_len, N, (int64_t)rows * N, k, B, B2, seed, splits, out_idx,
                  out_val, stats, (cudaStream_t)stream);
}

int ds_topk_stats_order(const void *x, int dtype, int rows, const int32_t *row_len, int64_t N,
                        int k, int B, int B2, uint64_t seed, int splits, int order,
                        int32_t *out_idx, void *out_val, int64_t *stats, void *stream)
{
    g_detail[0] = '\0';
    if (order != DS_ORDER_RANDOM && order != DS_ORDER_IDENTITY)
        return fail(DS_EINVAL, "order = %d is not DS_ORDER_RANDOM (0) or DS_ORDER_IDENTITY (1)", order);
    if (!stats && rows > 0)
        return fail(DS_EINVAL, "stats must be non-NULL: the block order only changes the counters");
    return launch(x, dtype, rows, row_len, N, (int64_t)rows * N, k, B, B2, seed, splits, out_idx,
                  out_val, stats, (cudaStream_t)stream, true, order);
}

static int host_call(const void *x_host, int dtype, int rows, const int32_t *row_len_host, int64_t N,
                     int k, int B, int B2, uint64_t seed, int32_t *out_idx_host, void *out_val_host,
                     void *x_dev, int32_t *row_len_dev, int32_t *out_idx_dev, void *out_val_dev,
                     void *stream, bool sync)
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
    rc = launch(x_dev, dtype, rows, row_len_dev, N, (int64_t)rows * N, k, B, B2, seed, 0,
                out_idx_dev, out_val_dev, nullptr, s);
    if (rc != DS_OK)
        return rc;
    e = cudaMemcpyAsync(out_idx_host, out_idx_dev, (size_t)rows * k * 4, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaMemcpyAsync(out_idx)");
    e = cudaMemcpyAsync(out_val_host, out_val_dev, (size_t)rows * k * es, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaMemcpyAsync(out_val)");
    if (!sync)
        return DS_OK;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaStreamSynchronize");
    return DS_OK;
}

int ds_topk_host(const void *x_host, int dtype, int rows, const int32_t *row_len_host, int64_t N,
                 int k, int B, int B2, uint64_t seed, int32_t *out_idx_host, void *out_val_host,
                 void *x_dev, int32_t *row_len_dev, int32_t *out_idx_dev, void *out_val_dev,
                 void *stream)
{
    return host_call(x_host, dtype, rows, row_len_host, N, k, B, B2, seed, out_idx_host,
                     out_val_host, x_dev, row_len_dev, out_idx_dev, out_val_dev, stream, true);
}

int ds_topk_host_async(const void *x_host, int dtype, int rows, const int32_t *row_len_host,
                       int64_t N, int k, int B, int B2, uint64_t seed, int32_t *out_idx_host,
                       void *out_val_host, void *x_dev, int32_t *row_len_dev, int32_t *out_idx_dev,
                       void *out_val_dev, void *stream)
{
    return host_call(x_host, dtype, rows, row_len_host, N, k, B, B2, seed, out_idx_host,
                     out_val_host, x_dev, row_len_dev, out_idx_dev, out_val_dev, stream, false);
}

int ds_topk_long_row_workspace(int dtype, int64_t N, int k, int B, int B2, size_t *bytes,
                               int64_t *piece_len, int *pieces)
{
    g_detail[0] = '\0';
    if (!bytes)
        return fail(DS_EINVAL, "bytes must be non-NULL");
    int rc = long_row_check((const void *)16, dtype, N, k, B, B2, (const void *)16,
                            (const void *)16);
    if (rc != DS_OK)
        return rc;
    RowPlan rp;
    if ((rc = long_row_plan(dtype, N, k, B, rp)) != DS_OK)
        return rc;
    *bytes = rp.bytes;
    if (piece_len)
        *piece_len = rp.P;
    if (pieces)
        *pieces = rp.G;
    return DS_OK;
}

int ds_topk_long_row(const void *x, int dtype, int64_t N, int k, int B, int B2, uint64_t seed,
                     void *workspace, size_t workspace_bytes, int32_t *out_idx, void *out_val,
                     void *stream)
{
    g_detail[0] = '\0';
    int rc = long_row_check(x, dtype, N, k, B, B2, out_idx, out_val);
    if (rc != DS_OK)
        return rc;
    RowPlan rp;
    if ((rc = long_row_plan(dtype, N, k, B, rp)) != DS_OK)
        return rc;
    if (rp.bytes > 0 && (!workspace || workspace_bytes < rp.bytes))
        return fail(DS_EINVAL, "workspace of %zu bytes at %p is smaller than the %zu bytes needed; "
                    "query ds_topk_long_row_workspace", workspace_bytes, workspace, rp.bytes);
    if (rp.bytes > 0 && (uintptr_t)workspace % kWsAlign != 0)
        return fail(DS_EINVAL, "workspace must be %zu-byte aligned", kWsAlign);
    return long_row_run(x, dtype, N, k, B, B2, seed, rp, static_cast<unsigned char *>(workspace),
                        out_idx, out_val, (cudaStream_t)stream);
}

int ds_topk_long_row_noalloc(const void *x, int dtype, int64_t N, int k, int B, int B2,
                             uint64_t seed, int32_t *out_idx, void *out_val, void *stream)
{
    g_detail[0] = '\0';
    int rc = long_row_check(x, dtype, N, k, B, B2, out_idx, out_val);
    if (rc != DS_OK)
        return rc;
    RowPlan rp;
    if ((rc = long_row_plan(dtype, N, k, B, rp)) != DS_OK)
        return rc;
    if (rp.bytes > kNoAllocBytes)
        return fail(DS_EUNSUPPORTED,
                    "the piece results need %zu bytes, more than the %zu-byte built-in workspace; "
                    "use ds_topk_long_row with a workspace of your own",
                    rp.bytes, kNoAllocBytes);
    unsigned char *ws = nullptr;
    if (rp.bytes > 0 && (rc = noalloc_workspace(&ws)) != DS_OK)
        return rc;
    return long_row_run(x, dtype, N, k, B, B2, seed, rp, ws, out_idx, out_val,
                        (cudaStream_t)stream);
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
    plan->async_copy = pl.async ? 1 : 0;
    plan->smem_bytes = pl.smem;
    plan->capacity = pl.p.cap;
    plan->grid = pl.grid;
    plan->ctas_per_sm = pl.ctas_per_sm;
    plan->kernel = pl.stream ? 1 : 0;
    return DS_OK;
}

int ds_topk_max_k(int dtype, int B, int B2)
{
    g_detail[0] = '\0';
    if (dtype != DS_FP32 && dtype != DS_BF16 && dtype != DS_FP16)
        return fail(DS_EUNSUPPORTED, "dtype %d is not DS_FP32, DS_BF16 or DS_FP16", dtype);
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

#ifdef DS_CHECKED
// Bounds-checked builds only: the violation bits so far (0: none); `reset`
// clears them.  Synchronises the device.
int ds_check_word(uint32_t *out, int reset)
{
    unsigned int *w = nullptr;
    int rc = check_word(&w);
    if (rc != DS_OK)
        return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(out, w, sizeof(unsigned int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && reset)
        e = cudaMemset(w, 0, sizeof(unsigned int));
    return e == cudaSuccess ? DS_OK : fail_cuda(e, "bounds-check word");
}
#endif

const char *ds_strerror(int status)
{
    switch (status) {
    case DS_OK: return "success";
    case DS_EINVAL: return "invalid argument";
    case DS_EUNSUPPORTED: return "unsupported dtype or working set too large for shared memory";
    case DS_ECUDA: return "CUDA runtime error";
    default: return "unknown status";
    }
}

const char *ds_last_error_detail(void) { return g_detail; }

}  // extern "C"
