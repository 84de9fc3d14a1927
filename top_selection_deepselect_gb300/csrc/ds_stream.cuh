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
//   * the block order is a keyed pseudorandom permutation (BlockOrder);
//     every warp evaluates its own positions in parallel across its lanes,
//     so it issues its first copies at once, with no CTA-wide sort first;
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
//     below every element (no key is 0), and its pieces are filtered again
//     after the compaction.  The capacity is k + B2 + the largest
//     reservation (one piece, or a pair of pieces when pairs are on), so at
//     least k + B2 real entries precede any such filler, and the first
//     reservation after a compaction (at k) always fits.
// The epilogue (final select, order, or the split-row merge through the
// cluster) is the block-by-block kernel's.
#pragma once

#include "ds_kernel.cuh"

namespace ds {

constexpr int kStageChunks = 128;                 // 16-byte chunks of one warp stage
constexpr int kStageBytes = kStageChunks * 16;    // 2 KiB
constexpr int kLaneChunks = kStageChunks / 32;    // chunks per lane and stage
constexpr int kMaxStreamStages = 6;               // deepest per-warp ring
constexpr int kPairChunks = 2 * kStageChunks;      // chunks one reservation covers (two pieces)

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

// The first threshold for small k.  The pages start from -inf, so the first
// k + B2 elements all enter the buffer and the first compaction selects
// from them.  Any T with k elements of the row above it gives the same
// answer, so here every lane takes the largest element of its chunks of
// its warp's first kSeedStages stages (256 distinct elements of the row;
// chunks not yet copied are left out), and T is placed just below the k-th
// largest of these maxima: every element with that key passes, and the k maxima at or
// above it guarantee k elements above T.  The k-th is found by ranking the 256
// maxima (keys made distinct by the thread index; warp-sorted runs and
// binary searches) in the candidate buffer, which is still empty.  Lanes without elements count as
// key 0, below every element.  Called by all threads before the first
// stage is consumed (its copies are waited for here).
constexpr int kSeedMaxK = 128;
#ifndef DS_SEED_STAGES
#define DS_SEED_STAGES 4
#endif
constexpr int kSeedStages = DS_SEED_STAGES;  // stages per warp the maxima are taken over

template <int DT>
__device__ __forceinline__ uint32_t max_key_of(uint32_t mx)
{
    using E = Elem<DT>;
    if (DT == 0)
        return E::key(mx);
    const uint32_t a = E::key(mx & 0xFFFFu), b = E::key(mx >> 16);
    return a > b ? a : b;
}

template <int DT>
__device__ __noinline__ Threshold seed_threshold(const unsigned char *wring, const int *btab, int msl,
                                                 int len, int B, int k, int NS,
                                                 unsigned long long *cand, Misc *ms)
{
    using E = Elem<DT>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nseed = kSeedStages < NS - 1 ? kSeedStages : NS - 1;
    cp_async_wait_pending(NS - 1 - nseed);  // this lane's copies of its first nseed stages landed
    uint32_t mx = E::splat(E::kNegInfBits);
    bool any = false;
    int q = warp, pc = 0;  // the producer cursor's first steps
    for (int st = 0; st < nseed && q < msl; ++st) {
        const int lo = btab[q] * B;
        const int nbytes = (min(lo + B, len) - lo) * E::kSize;
        const int nch = (nbytes + 15) >> 4;
        const int c0 = pc * kStageChunks;
#pragma unroll
        for (int i = 0; i < kLaneChunks; ++i) {
            const int c = c0 + lane + 32 * i;
            if ((c + 1) * 16 <= nbytes) {
                mx = max_nan<DT>(mx, chunk_max<DT>(lds128(wring + st * kStageBytes + (lane + 32 * i) * 16)));
                any = true;
            }
        }
        if (c0 + kStageChunks >= nch) {
            q += kWarps;
            pc = 0;
        } else {
            ++pc;
        }
    }
    const uint32_t key = any ? max_key_of<DT>(mx) : 0u;
    cand[tid] = ((unsigned long long)key << 32) | (uint32_t)tid;
    if (tid == 0)
        ms->texact = 0ull;
    __syncthreads();
    unsigned long long vals[1];
    int ranks[1];
    rank_desc_runs<1>(cand, vals, ranks);  // the one 0 composite (thread 0 without elements) ranks last
    if (ranks[0] == k - 1)
        ms->texact = vals[0];
    __syncthreads();  // texact is published
    const uint32_t tkey = (uint32_t)(ms->texact >> 32);
    return tkey == 0u ? threshold_initial<DT>() : threshold_from<DT>((unsigned long long)tkey << 32);
}

// The first threshold for larger k (kSeedMaxK < k <= kSeedMaxWideK).  256
// lane maxima are too few, so the maxima of single 16-byte chunks are used
// (four per lane and stage, each a different element of the row), and T is
// not their exact k-th but the lower edge of the histogram bin that holds
// it: any key with k chunk maxima at or above it has k elements at or above
// it.  One pass of 256 bins spans [kmin, kmax] of the maxima, where kmin is
// already a lower bound on their k-th largest: each lane's chunk slots are
// cut into G >= k/256 groups (by chunk position; for G = 8 also by stage
// parity; G = 16: every slot), and the smallest of a lane's G group maxima
// has G maxima of that lane at or above it, so the minimum of these over
// the lanes has 256G >= k maxima above it.  Lanes with an empty group drop
// out of that minimum; when fewer than k/G lanes remain, kmin is the
// smallest maximum.  With fewer than k maxima in all, T stays -inf.
constexpr int kSeedMaxWideK = 16 * kThreads;
static_assert((long long)kMaxSplits * kSeedMaxK <= kClusterSelectMinUnion,
              "the pairs instance (k <= kSeedMaxK) never needs the select across the cluster");
static_assert(kHistBins == kThreads, "one histogram bin per thread");

template <int DT>
__device__ __noinline__ Threshold seed_threshold_wide(const unsigned char *wring, const int *btab, int msl,
                                                      int len, int B, int k, int NS, uint32_t *hist,
                                                      Misc *ms)
{
    using E = Elem<DT>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nseed = kSeedStages < NS - 1 ? kSeedStages : NS - 1;
    cp_async_wait_pending(NS - 1 - nseed);  // this lane's copies of its first nseed stages landed
    uint32_t ck[4][kLaneChunks];  // chunk maximum keys by stage and slot; 0: no chunk
    int q = warp, pc = 0;
#pragma unroll
    for (int st = 0; st < 4; ++st) {
        const bool have = st < nseed && q < msl;
        int nbytes = 0, c0 = 0;
        if (have) {
            const int lo = btab[q] * B;
            nbytes = (min(lo + B, len) - lo) * E::kSize;
            c0 = pc * kStageChunks;
        }
#pragma unroll
        for (int i = 0; i < kLaneChunks; ++i) {
            const int c = c0 + lane + 32 * i;
            ck[st][i] = (have && (c + 1) * 16 <= nbytes)
                            ? max_key_of<DT>(chunk_max<DT>(lds128(wring + st * kStageBytes + (lane + 32 * i) * 16)))
                            : 0u;
        }
        if (have) {
            if (c0 + kStageChunks >= ((nbytes + 15) >> 4)) {
                q += kWarps;
                pc = 0;
            } else {
                ++pc;
            }
        }
    }
    const int G = k <= kThreads ? 1 : k <= 2 * kThreads ? 2 : k <= 4 * kThreads ? 4
                                    : k <= 8 * kThreads ? 8 : 16;
    uint32_t gp[2][kLaneChunks], gi[kLaneChunks];
    uint32_t vmin = 0xFFFFFFFFu, nvalid = 0u, all_min = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < kLaneChunks; ++i) {
        gp[0][i] = max(ck[0][i], ck[2][i]);
        gp[1][i] = max(ck[1][i], ck[3][i]);
        gi[i] = max(gp[0][i], gp[1][i]);
#pragma unroll
        for (int st = 0; st < 4; ++st) {
            vmin = ck[st][i] ? min(vmin, ck[st][i]) : vmin;
            nvalid += ck[st][i] ? 1u : 0u;
            all_min = min(all_min, ck[st][i]);
        }
    }
    const uint32_t vmax = max(max(gi[0], gi[1]), max(gi[2], gi[3]));
    uint32_t bound;  // the smallest of this lane's G group maxima (0: a group is empty)
    if (G == 1)
        bound = vmax;
    else if (G == 2)
        bound = min(max(gi[0], gi[2]), max(gi[1], gi[3]));
    else if (G == 4)
        bound = min(min(gi[0], gi[1]), min(gi[2], gi[3]));
    else if (G == 8)
        bound = min(min(min(gp[0][0], gp[0][1]), min(gp[0][2], gp[0][3])),
                    min(min(gp[1][0], gp[1][1]), min(gp[1][2], gp[1][3])));
    else
        bound = all_min;
    const uint32_t wmax = __reduce_max_sync(kFull, vmax);
    const uint32_t wbound = __reduce_min_sync(kFull, bound ? bound : 0xFFFFFFFFu);
    const uint32_t wlanes = (uint32_t)__popc(__ballot_sync(kFull, bound != 0u));
    const uint32_t wvmin = __reduce_min_sync(kFull, vmin);
    const uint32_t wvalid = __reduce_add_sync(kFull, nvalid);
    if (lane == 0) {
        ms->wor[warp] = ((unsigned long long)wmax << 32) | wbound;
        ms->wand[warp] = ((unsigned long long)wvmin << 32) | wlanes;
        ms->wsum[warp] = wvalid;
    }
    __syncthreads();
    uint32_t kmax = 0u, kbound = 0xFFFFFFFFu, kvmin = 0xFFFFFFFFu, lanes = 0u, valid = 0u;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const unsigned long long a = ms->wor[w], b = ms->wand[w];
        kmax = max(kmax, (uint32_t)(a >> 32));
        kbound = min(kbound, (uint32_t)a);
        kvmin = min(kvmin, (uint32_t)(b >> 32));
        lanes += (uint32_t)b;
        valid += ms->wsum[w];
    }
    uint32_t kmin;
    if (lanes * (uint32_t)G >= (uint32_t)k)
        kmin = kbound;
    else if (valid >= (uint32_t)k)
        kmin = kvmin;
    else
        return threshold_initial<DT>();  // the same decision in every thread
    const uint32_t span = kmax - kmin;
    const int sh = span >= 256u ? (32 - __clz(span)) - 8 : 0;  // (span >> sh) < 256
#pragma unroll
    for (int st = 0; st < 4; ++st)
#pragma unroll
        for (int i = 0; i < kLaneChunks; ++i)
            if (ck[st][i] >= kmin)
                atomicAdd(&hist[(ck[st][i] - kmin) >> sh], 1u);
    __syncthreads();
    if (warp == 0)
        digit_search(hist, (uint32_t)k, lane, ms);  // at least k maxima are counted
    __syncthreads();
    const uint32_t tkey = kmin + (ms->sel_digit << sh);
    hist[tid] = 0u;  // the histogram is left zero (one bin per thread)
    return threshold_from<DT>((unsigned long long)tkey << 32);
}

// The survivors of a pair of pieces in one loop: bits 0..31 of `m` are
// piece A's (as stage_filter numbers them), bits 32..63 piece B's.  Every
// round each lane with survivors left writes its next one at the slot after
// those of the lower lanes; the number of rounds is the largest count of a
// lane, known before the loop.
template <int DT>
__device__ __forceinline__ void pair_append(const unsigned char *spA, const BlockView &bvA,
                                            const unsigned char *spB, const BlockView &bvB, int lane,
                                            unsigned long long m, unsigned long long *dst)
{
    using E = Elem<DT>;
    constexpr int kB = E::kPerChunk;
    const int rounds = (int)__reduce_max_sync(kFull, (uint32_t)__popcll(m));
    int run = 0;
    for (int r = 0; r < rounds; ++r) {
        const bool has = m != 0ull;
        const uint32_t b = __ballot_sync(kFull, has);
        if (has) {
            const int bit = __ffsll((long long)m) - 1;
            m &= m - 1ull;
            const bool inB = bit >= 32;
            const int i = (bit & 31) / kB, e = (bit & 31) % kB;
            const unsigned char *ep = (inB ? spB : spA) + (lane + 32 * i) * 16 + e * E::kSize;
            const uint32_t bits = DT == 0 ? *reinterpret_cast<const uint32_t *>(ep)
                                          : (uint32_t)*reinterpret_cast<const uint16_t *>(ep);
            const int lo = inB ? bvB.lo : bvA.lo, c0 = inB ? bvB.c0 : bvA.c0;
            const uint32_t idx = (uint32_t)(lo + (c0 + lane + 32 * i) * kB + e);
            dst[run + __popc(b & lanemask_lt(lane))] =
                ((unsigned long long)E::key(bits) << 32) | (unsigned long long)(~idx);
        }
        run += __popc(b);
    }
}

// Exact survivor bits of one whole piece held in registers (4 chunks per
// lane): bits only for the chunks whose own maximum passes (small k, where
// survivors are sparse).
template <int DT>
__device__ __forceinline__ uint32_t whole_piece_bits(const uint4 (&v)[kLaneChunks], const uint32_t (&cm)[kLaneChunks],
                                                     uint32_t t)
{
    constexpr int kB = Elem<DT>::kPerChunk;
    uint32_t m = 0u;
#pragma unroll
    for (int i = 0; i < kLaneChunks; ++i)
        if (max_passes<DT>(cm[i], t))
            m |= prefilter_bits<DT>(v[i], t) << (i * kB);
    return m;
}

// grid = rows * splits, cluster = (splits, 1, 1) when splits > 1.  Needs
// 16-byte aligned rows and blocks (the planner checks).
template <int DT, bool PAIRS>
__global__ void __launch_bounds__(kThreads, 2) deepselect_stream_kernel(const Params p)
{
    allow_dependent_grid();
    // Rows of full length: everything up to the first copies (block order,
    // shared-memory set-up) reads no input, so it runs before waiting for
    // the previous grid on the stream; with row_len the wait comes first.
    const bool wait_late = p.row_len == nullptr;
    if (!wait_late)
        dependent_grid_wait();
    using E = Elem<DT>;
    constexpr int kB = E::kPerChunk;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = p.splits;
    const int row = blockIdx.x / S, slice = blockIdx.x % S;

    unsigned char *ring = smem;
    unsigned long long *cand = reinterpret_cast<unsigned long long *>(smem + p.off_cand);
    int *btab = reinterpret_cast<int *>(smem + p.off_perm);  // block at each position
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

    // -- random block order: a keyed permutation of the slice's blocks (keyed
    // by Philox from seed, row and slice).  Every warp evaluates the
    // positions it will scan (w, w+8, ...), one per lane, into a table it
    // alone reads: no sort and no CTA barrier before the first copies.
    {
        BlockOrder order;
        order.init((uint32_t)msl, philox_word0((uint32_t)row, (uint32_t)slice, 0u, 1u, p.seed_lo, p.seed_hi));
        for (int q = warp + kWarps * lane; q < msl; q += kWarps * 32)
            btab[q] = first_block + (int)order((uint32_t)q);
        __syncwarp();
    }

    const int NS = p.stages;
    unsigned char *wring = ring + (size_t)warp * NS * kStageBytes;
    const int esz = E::kSize;
    const int trigger = p.k + p.B2;
    const int cap = p.cap;

    // Producer: block order position pq and stage pp within the block; the
    // block's byte count and this lane's source address are set once per
    // block.  Lane l copies the 16-byte chunks l, l+32, l+64, l+96 of a
    // stage, at the same offsets of the slot.
    int pq = warp, pp = 0, p_nbytes = 0;
    const unsigned char *p_src = nullptr;
    auto p_enter = [&]() {
        if (pq < msl) {
            const int lo = btab[pq] * B;
            p_nbytes = (min(lo + B, len) - lo) * esz;
            p_src = xrow + (size_t)lo * esz + lane * 16;
        }
    };
    p_enter();
    const uint32_t ring_lane = smem_addr(wring) + lane * 16;
    auto prefetch = [&](int slot) {
        if (pq < msl) {
            const int b0 = pp * kStageBytes;  // the stage's first byte in the block
            const uint32_t dst = ring_lane + slot * kStageBytes;
            const unsigned char *src = p_src + b0;
            if (b0 + kStageBytes <= p_nbytes) {
#pragma unroll
                for (int i = 0; i < kLaneChunks; ++i)
                    cp_async16(dst + i * 512, src + i * 512);
            } else {
#pragma unroll
                for (int i = 0; i < kLaneChunks; ++i)
                    if (b0 + (lane + 32 * i + 1) * 16 <= p_nbytes)
                        cp_async16(dst + i * 512, src + i * 512);
            }
            if (b0 + kStageBytes >= p_nbytes) {
                pq += kWarps;
                pp = 0;
                p_enter();
            } else {
                ++pp;
            }
        }
        cp_async_commit();
    };
    if (tid == 0) {
        ms->merge_count = 0;
        ms->pass = 0;
        ms->check = p.check;
        ms->ctr[0] = 0;
        ms->ctr[1] = 0;
    }
    for (int i = tid; i < p.hist_words; i += kThreads)
        whist[i] = 0u;
    if (wait_late)
        dependent_grid_wait();  // before the first read of x or the outputs
    for (int s = 0; s < NS - 1; ++s)
        prefetch(s);  // each warp's first copies go out before the CTA barrier
    __syncthreads();  // the buffer length words and the histograms are set

    int ps = NS - 1;          // slot the next prefetch fills
    int cs = 0;               // slot of the consumer's stage
    int epoch = 0;            // compactions so far (selects the length word)
    bool pending = false;     // the current stage waits for a compaction
    // consumer: the same walk, with the block's bounds set once per block
    int cq = warp, cpc = 0, c_lo = 0, c_hi = 0, c_nbytes = 0;
    auto c_enter = [&]() {
        if (cq < msl) {
            c_lo = btab[cq] * B;
            c_hi = min(c_lo + B, len);
            c_nbytes = (c_hi - c_lo) * esz;
        }
    };
    c_enter();
    Threshold thr = threshold_initial<DT>();
    if (p.k <= kSeedMaxK && msl >= kWarps)
        thr = seed_threshold<DT>(wring, btab, msl, len, B, p.k, NS, cand, ms);
    else if (p.k <= kSeedMaxWideK && msl >= kWarps && (long long)msl * B >= (long long)trigger)
        thr = seed_threshold_wide<DT>(wring, btab, msl, len, B, p.k, NS, whist, ms);

    // The partial last chunk of a row is loaded by the lane that filters it.
    auto load_tail = [&](unsigned char *sp, const BlockView &bv, int nbytes) {
        const int nch = (nbytes + 15) >> 4;
        if ((nbytes & 15) && nch - 1 < bv.c1 && ((nch - 1 - bv.c0) & 31) == lane) {
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
    };

    while (true) {
        // For small k (seeded threshold, few survivors) pieces are consumed in
        // pairs (A = the cursor's piece, B = the next one of the walk): both
        // are folded in one trip, one vote covers them, and their survivors
        // share one reservation.  With a ring of NS >= 3 pieces, one refill
        // goes out before the pair is waited for and one after it is
        // consumed, so NS - 2 pieces stay in flight.  Otherwise B is empty
        // and a trip consumes one piece.
        while (cq < msl) {
            const int b0A = cpc * kStageBytes;
            int qB = cq, pcB = cpc + 1, loB = c_lo, hiB = c_hi, nbB = c_nbytes;
            if (b0A + kStageBytes >= c_nbytes) {
                qB = cq + kWarps;
                pcB = 0;
                if (qB < msl) {
                    loB = btab[qB] * B;
                    hiB = min(loB + B, len);
                    nbB = (hiB - loB) * esz;
                }
            }
            const bool hasB = PAIRS && NS >= 3 && qB < msl;
            const int csB = cs + 1 == NS ? 0 : cs + 1;
            if (!pending) {
                if (ld_volatile_shared(&ms->ctr[epoch & 1]) >= trigger)
                    break;  // a compaction is due
                prefetch(ps);
                ps = ps + 1 == NS ? 0 : ps + 1;
                if (hasB)
                    cp_async_wait_pending(NS - 2);  // this lane's copies of A and B landed
                else
                    cp_async_wait_pending(NS - 1);  // this lane's copies of A landed
            }
            // prefilter operands per piece, for the block's index range (see Threshold)
            const bool geA = (uint32_t)c_lo < thr.ti, geB = (uint32_t)loB < thr.ti;
            BlockView bvA, bvB;
            bvA.lo = c_lo;
            bvA.hi = c_hi;
            bvA.c0 = cpc * kStageChunks;
            bvA.t = geA ? thr.t_ge : thr.t_gt;
            bvA.refine = geA ? (thr.nan_ge || (uint32_t)c_hi > thr.ti) : thr.nan_gt;
            bvA.slot = nullptr;
            bvB.lo = loB;
            bvB.hi = hiB;
            bvB.c0 = pcB * kStageChunks;
            bvB.t = geB ? thr.t_ge : thr.t_gt;
            bvB.refine = geB ? (thr.nan_ge || (uint32_t)hiB > thr.ti) : thr.nan_gt;
            bvB.slot = nullptr;
            const bool fastA = !bvA.refine && b0A + kStageBytes <= c_nbytes;
            const bool fastB = hasB && !bvB.refine && (pcB + 1) * kStageBytes <= nbB;
            unsigned char *spA = wring + cs * kStageBytes;
            unsigned char *spB = wring + csB * kStageBytes;
            uint32_t mA = 0u, mB = 0u;
            // whole pieces clear of T's index: four 16-byte loads at fixed
            // offsets, one maximum per lane, exact bits for passing lanes
            if (fastA) {
                const unsigned char *lp = spA + lane * 16;
                const uint4 v[kLaneChunks] = {lds128(lp), lds128(lp + 512), lds128(lp + 1024), lds128(lp + 1536)};
                const uint32_t cm[kLaneChunks] = {chunk_max<DT>(v[0]), chunk_max<DT>(v[1]), chunk_max<DT>(v[2]),
                                                  chunk_max<DT>(v[3])};
                const uint32_t mx = max_nan<DT>(max_nan<DT>(cm[0], cm[1]), max_nan<DT>(cm[2], cm[3]));
                if (max_passes<DT>(mx, bvA.t))
                    mA = PAIRS ? whole_piece_bits<DT>(v, cm, bvA.t)
                               : prefilter_bits<DT>(v[0], bvA.t) | (prefilter_bits<DT>(v[1], bvA.t) << kB) |
                                     (prefilter_bits<DT>(v[2], bvA.t) << (2 * kB)) |
                                     (prefilter_bits<DT>(v[3], bvA.t) << (3 * kB));
            }
            if (fastB) {
                const unsigned char *lp = spB + lane * 16;
                const uint4 v[kLaneChunks] = {lds128(lp), lds128(lp + 512), lds128(lp + 1024), lds128(lp + 1536)};
                const uint32_t cm[kLaneChunks] = {chunk_max<DT>(v[0]), chunk_max<DT>(v[1]), chunk_max<DT>(v[2]),
                                                  chunk_max<DT>(v[3])};
                const uint32_t mx = max_nan<DT>(max_nan<DT>(cm[0], cm[1]), max_nan<DT>(cm[2], cm[3]));
                if (max_passes<DT>(mx, bvB.t))
                    mB = whole_piece_bits<DT>(v, cm, bvB.t);
            }
            // other pieces (a row's partial last piece, a block that
            // straddles T's index, a NaN operand): chunk bounds and
            // per-element checks
            if (!fastA) {
                bvA.c1 = min(bvA.c0 + kStageChunks, (c_nbytes + 15) >> 4);
                if (!pending)
                    load_tail(spA, bvA, c_nbytes);
                const int slo = bvA.lo + bvA.c0 * kB, shi = min(bvA.lo + bvA.c1 * kB, bvA.hi);
                bvA.plain = !bvA.refine && shi - slo == (bvA.c1 - bvA.c0) * kB;
                mA = stage_filter<DT>(spA, bvA, thr, lane);
            }
            if (hasB && !fastB) {
                bvB.c1 = min(bvB.c0 + kStageChunks, (nbB + 15) >> 4);
                if (!pending)
                    load_tail(spB, bvB, nbB);
                const int slo = bvB.lo + bvB.c0 * kB, shi = min(bvB.lo + bvB.c1 * kB, bvB.hi);
                bvB.plain = !bvB.refine && shi - slo == (bvB.c1 - bvB.c0) * kB;
                mB = stage_filter<DT>(spB, bvB, thr, lane);
            }
            if (__any_sync(kFull, (mA | mB) != 0u)) {
                // one reservation for both pieces
                const int cnt = (int)__reduce_add_sync(kFull, (uint32_t)(__popc(mA) + __popc(mB)));
                int base = 0;
                if (lane == 0)
                    base = atomicAdd(&ms->ctr[epoch & 1], cnt);
                base = __shfl_sync(kFull, base, 0);
                if (base + cnt > cap) {
                    // no room: fill what lies below the capacity with the
                    // composite 0 and filter both pieces again after the
                    // compaction
                    for (int i = base + lane; i < cap; i += 32)
                        cand[i] = 0ull;
                    pending = true;
                    break;
                }
                if (PAIRS)  // few survivors: one loop over both pieces
                    pair_append<DT>(spA, bvA, spB, bvB, lane,
                                    (unsigned long long)mA | ((unsigned long long)mB << 32), cand + base);
                else        // dense pieces at the start of a large-k scan
                    stage_append<DT>(spA, bvA, lane, mA, cand + base);
            }
            pending = false;
            if (hasB) {
                // past B; then refill A's slot (its loads are done)
                cq = qB;
                cpc = pcB;
                c_lo = loB;
                c_hi = hiB;
                c_nbytes = nbB;
                cs = csB;
            }
            if ((cpc + 1) * kStageBytes >= c_nbytes) {
                cq += kWarps;
                cpc = 0;
                c_enter();
            } else {
                ++cpc;
            }
            cs = cs + 1 == NS ? 0 : cs + 1;
            if (hasB) {
                prefetch(ps);
                ps = ps + 1 == NS ? 0 : ps + 1;
            }
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
                select_topk(cand, n_now < cap ? n_now : cap, p.k, cap, whist, holes, ms);
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

    // with pairs (k <= 128) a union of slices holds at most 16 * 128 entries,
    // so that instance leaves out the select across the cluster
    finish_slice<DT, !PAIRS>(Out{p.out_idx, p.out_val, p.k}, nullptr, ring, cand, cap, whist, holes, ms,
                             n, S, row, slice, xrow, 0, 0, 0, 0);
}

// Free-running kernel entry points of one dtype (pairs of pieces or single
// pieces), defined in ds_kernels_<dtype>.cu.
KernelFn stream_kernel_fp32(bool pairs);
KernelFn stream_kernel_bf16(bool pairs);
KernelFn stream_kernel_fp16(bool pairs);

}  // namespace ds
