// ds_stream.cuh -- the free-running variant of the DeepSelect top-k kernel
// (sm_103a, device code), used whenever the caller asks for no counters.
//
// The method is the one of PFCCLab/DeepSelect "DeepSelect-deep-dive",
// section "算法": the row's B-blocks are visited in a random order drawn
// from Philox, elements above the running threshold T are appended to a
// candidate buffer, and when the buffer reaches k + B2 a radix select
// shrinks it to k and raises T.  Any T that is at most the row's k-th
// element gives the same answer (the result is unique under the total
// order), so this kernel lets the eight warps of a CTA run independently:
//   * warp w scans the blocks at positions w, w + 8, w + 16, ... of the
//     CTA's block order, in stages of 2 KiB (128 chunks of 16 bytes, four
//     per lane), through its own ring of asynchronous copies: every lane
//     copies and later reads only its own chunks, so a warp never waits for
//     another warp while it streams;
//   * every warp filters against the T of the last compaction it took part
//     in and reserves its survivors' slots with one shared atomic on the
//     buffer length; survivors are written in rounds across the lanes, so
//     the 8-byte stores of a round land on consecutive slots;
//   * a warp that finds the buffer at k + B2 or more at a stage boundary, or
//     whose reservation would run past the buffer's capacity, or that has no
//     stages left, waits at the CTA barrier; when all eight are there the
//     CTA compacts (radix select) if the buffer reached k + B2, and the
//     warps go on with the new T.  A reservation that runs past the capacity
//     fills its slots below the capacity with the composite 0, which is
//     below every element (no key is 0), and its stage is filtered again
//     after the compaction.  The capacity is k + B2 + one stage, so at least
//     k + B2 real entries precede any such filler.
// The epilogue (final select, order, or the split-row merge through the
// cluster) is the block-by-block kernel's.
#pragma once

#include "ds_kernel.cuh"

namespace ds {

constexpr int kStageChunks = 128;                 // 16-byte chunks of one warp stage
constexpr int kStageBytes = kStageChunks * 16;    // 2 KiB
constexpr int kLaneChunks = kStageChunks / 32;    // chunks per lane and stage
constexpr int kMaxStreamStages = 6;               // deepest per-warp ring

__device__ __forceinline__ int ld_volatile_shared(const int *p)
{
    return *reinterpret_cast<const volatile int *>(p);
}

// Survivor bits of this lane's chunks of one stage (bit i*kPerChunk + e =
// element e of chunk c0 + lane + 32i).  `sp` is the stage's slot: chunk c is
// at sp + (c - c0)*16.  Fast path as in warp_filter: one NaN-propagating
// maximum per lane, one unordered compare; exact masks only for lanes whose
// maximum passes.  Warp-uniform return value of zero: no survivor.
template <int DT>
__device__ __forceinline__ uint32_t stage_filter(const unsigned char *sp, const BlockView &bv,
                                                 const Threshold &thr, int lane)
{
    using E = Elem<DT>;
    constexpr int kB = E::kPerChunk;
    uint4 v[kLaneChunks];
    uint32_t mx = E::splat(E::kNegInfBits);
#pragma unroll
    for (int i = 0; i < kLaneChunks; ++i) {
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (bv.c0 + lane + 32 * i < bv.c1) {
            v[i] = lds128(sp + (lane + 32 * i) * 16);
            mx = max_nan<DT>(mx, chunk_max<DT>(v[i]));
        }
    }
    const bool pass = bv.c0 + lane < bv.c1 && max_passes<DT>(mx, bv.t);
    if (!__any_sync(kFull, pass))
        return 0u;
    uint32_t mword = 0u;
    if (pass) {
#pragma unroll
        for (int i = 0; i < kLaneChunks; ++i) {
            const int c = bv.c0 + lane + 32 * i;
            if (c < bv.c1) {
                uint32_t m = prefilter_bits<DT>(v[i], bv.t);
                if (!bv.plain)
                    m = chunk_fixup<DT>(m, v[i], c, bv, thr);
                mword |= m << (i * kB);
            }
        }
    }
    return mword;
}

// Writes the survivors flagged in `mword` to dst[0, count) in rounds: in
// every round each lane with survivors left writes its next one, at the
// slot after those of the lower lanes, so consecutive lanes store to
// consecutive 8-byte slots.
template <int DT>
__device__ __forceinline__ void stage_append(const unsigned char *sp, const BlockView &bv, int lane,
                                             uint32_t mword, unsigned long long *dst)
{
    using E = Elem<DT>;
    constexpr int kB = E::kPerChunk;
    int run = 0;
    while (true) {
        const uint32_t b = __ballot_sync(kFull, mword != 0u);
        if (b == 0u)
            break;
        if (mword) {
            const int bit = __ffs(mword) - 1;
            mword &= mword - 1u;
            const int i = bit / kB, e = bit % kB;
            const unsigned char *ep = sp + (lane + 32 * i) * 16 + e * E::kSize;
            const uint32_t bits = DT == 0 ? *reinterpret_cast<const uint32_t *>(ep)
                                          : (uint32_t)*reinterpret_cast<const uint16_t *>(ep);
            const uint32_t idx = (uint32_t)(bv.lo + (bv.c0 + lane + 32 * i) * kB + e);
            dst[run + __popc(b & lanemask_lt(lane))] =
                ((unsigned long long)E::key(bits) << 32) | (unsigned long long)(~idx);
        }
        run += __popc(b);
    }
}

// grid = rows * splits, cluster = (splits, 1, 1) when splits > 1.  Needs
// 16-byte aligned rows and blocks (the planner checks).
template <int DT>
__global__ void __launch_bounds__(kThreads, 2) deepselect_stream_kernel(const Params p)
{
    using E = Elem<DT>;
    constexpr int kB = E::kPerChunk;
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
            const uint32_t w = philox_word0(b, (uint32_t)row, (uint32_t)slice, 0u, p.seed_lo, p.seed_hi);
            v = ((unsigned long long)w << 32) | b;
        }
        perm[i] = v;
    }
    for (int i = tid; i < kHistWords; i += kThreads)
        whist[i] = 0u;
    if (tid == 0) {
        ms->merge_count = 0;
        ms->pass = 0;
        ms->check = p.check;
        ms->ctr[0] = 0;
        ms->ctr[1] = 0;
    }
    __syncthreads();
    sort_asc_small(perm, msl, P);

    const int NS = p.stages;
    unsigned char *wring = ring + (size_t)warp * NS * kStageBytes;
    const int esz = E::kSize;
    const int trigger = p.k + p.B2;
    const int cap = p.cap;

    // producer cursor: block order position and stage within the block
    int pq = warp, pp = 0;
    auto prefetch = [&](int slot) {
        if (pq < msl) {
            const int lo = (int)(uint32_t)perm[pq] * B;
            const int nbytes = (min(lo + B, len) - lo) * esz;
            const int nch = (nbytes + 15) >> 4;
            const int c0 = pp * kStageChunks;
            unsigned char *dst = wring + slot * kStageBytes;
            const unsigned char *src = xrow + (size_t)lo * esz;
#pragma unroll
            for (int i = 0; i < kLaneChunks; ++i) {
                const int c = c0 + lane + 32 * i;
                if ((c + 1) * 16 <= nbytes)
                    cp_async16(smem_addr(dst + (lane + 32 * i) * 16), src + (size_t)c * 16);
            }
            if (c0 + kStageChunks >= nch) {
                pq += kWarps;
                pp = 0;
            } else {
                ++pp;
            }
        }
        cp_async_commit();
    };
    for (int s = 0; s < NS - 1; ++s)
        prefetch(s);

    int ps = NS - 1;          // slot the next prefetch fills
    int cq = warp, cpc = 0;   // consumer cursor
    int cs = 0;               // slot of the consumer's stage
    int epoch = 0;            // compactions so far (selects the length word)
    bool pending = false;     // the current stage waits for a compaction
    Threshold thr = threshold_initial<DT>();

    while (true) {
        while (cq < msl) {
            if (!pending) {
                if (ld_volatile_shared(&ms->ctr[epoch & 1]) >= trigger)
                    break;  // a compaction is due
                prefetch(ps);
                ps = ps + 1 == NS ? 0 : ps + 1;
                cp_async_wait_pending(NS - 1);  // this lane's copies of the stage landed
            }
            BlockView bv;
            bv.lo = (int)(uint32_t)perm[cq] * B;
            bv.hi = min(bv.lo + B, len);
            const int nbytes = (bv.hi - bv.lo) * esz;
            const int nch = (nbytes + 15) >> 4;
            bv.c0 = cpc * kStageChunks;
            bv.c1 = min(bv.c0 + kStageChunks, nch);
            bv.slot = nullptr;
            unsigned char *sp = wring + cs * kStageBytes;
            // the partial last chunk of a row is loaded by the lane that filters it
            if (!pending && (nbytes & 15) && nch - 1 < bv.c1 && ((nch - 1 - bv.c0) & 31) == lane) {
                const int c = nch - 1;
                unsigned char *dst = sp + (c - bv.c0) * 16;
                for (int e = 0; e < kB; ++e) {
                    const int j = bv.lo + c * kB + e;
                    if (j < bv.hi) {
                        if (DT == 0)
                            reinterpret_cast<uint32_t *>(dst)[e] = reinterpret_cast<const uint32_t *>(xrow)[j];
                        else
                            reinterpret_cast<uint16_t *>(dst)[e] = reinterpret_cast<const uint16_t *>(xrow)[j];
                    }
                }
            }
            // prefilter operand for the stage's element range (see Threshold)
            const int slo = bv.lo + bv.c0 * kB;
            const int shi = min(bv.lo + bv.c1 * kB, bv.hi);
            const bool ge = (uint32_t)slo < thr.ti;
            bv.t = ge ? thr.t_ge : thr.t_gt;
            bv.refine = ge ? (thr.nan_ge || (uint32_t)shi > thr.ti) : thr.nan_gt;
            bv.plain = !bv.refine && shi - slo == (bv.c1 - bv.c0) * kB;
            const uint32_t mword = stage_filter<DT>(sp, bv, thr, lane);
            const int cnt = (int)__reduce_add_sync(kFull, (uint32_t)__popc(mword));
            if (cnt) {
                int base = 0;
                if (lane == 0)
                    base = atomicAdd(&ms->ctr[epoch & 1], cnt);
                base = __shfl_sync(kFull, base, 0);
                if (base + cnt > cap) {
                    // no room: fill what lies below the capacity with the
                    // composite 0 and filter this stage again after the
                    // compaction
                    for (int i = base + lane; i < cap; i += 32)
                        cand[i] = 0ull;
                    pending = true;
                    break;
                }
                stage_append<DT>(sp, bv, lane, mword, cand + base);
            }
            pending = false;
            if (bv.c1 >= nch) {
                cq += kWarps;
                cpc = 0;
            } else {
                ++cpc;
            }
            cs = cs + 1 == NS ? 0 : cs + 1;
        }

        // -- sync point: all eight warps ------------------------------------
        if (lane == 0)
            ms->rem[warp] = cq < msl ? 1 : 0;
        __syncthreads();
        const int n_now = ms->ctr[epoch & 1];
        const int4 ra = reinterpret_cast<const int4 *>(ms->rem)[0];
        const int4 rb = reinterpret_cast<const int4 *>(ms->rem)[1];
        const bool more = (ra.x | ra.y | ra.z | ra.w | rb.x | rb.y | rb.z | rb.w) != 0;
        if (n_now >= trigger) {
            if (tid == 0)
                ms->ctr[(epoch + 1) & 1] = p.k;  // ordered by the select's first barrier
            const unsigned long long tcomp =
                radix_select_topk(cand, n_now < cap ? n_now : cap, p.k, whist, holes, ms);
            ++epoch;
            thr = threshold_from<DT>(tcomp);
            continue;
        }
        if (!more)
            break;
    }
    cp_async_wait_pending(0);
    const int n = ms->ctr[epoch & 1];
    __syncthreads();  // every thread read the length; this thread's copies have landed

    finish_slice<DT>(Out{p.out_idx, p.out_val, p.k}, nullptr, ring, cand, whist, holes, ms, n, S, row,
                     slice, xrow, 0, 0, 0, 0);
}

// Free-running kernel entry points of one dtype, defined in ds_kernels_<dtype>.cu.
KernelFn stream_kernel_fp32();
KernelFn stream_kernel_bf16();
KernelFn stream_kernel_fp16();

}  // namespace ds
