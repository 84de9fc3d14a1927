/*
 * ds_topk.h -- C ABI of the GB300 DeepSelect top-k library (libds_topk.so).
 *
 * Operation (PFCCLab/DeepSelect "DeepSelect-deep-dive", section "算法", and
 * milkfeng.top "CUDA 算子笔记 4", section "Top K Selection"): for every row r
 * of a [rows x N] score matrix (fp32, bf16 or IEEE fp16), return the k largest of its first row_len[r]
 * elements and their indices.  The result is exact and unique:
 *   - order: value descending; NaN (any payload) above +inf; -0.0 == +0.0;
 *     equal values by lower index first;
 *   - out_idx[r*k + i] = row-local index (int32) of the i-th element,
 *     out_val[r*k + i] = its value, bit for bit as it was read (same dtype
 *     as x);
 *   - a row with fewer than k valid elements fills the rest with index -1
 *     and value -inf.
 * The result does not depend on `seed`, on the split factor or on any other
 * launch choice; `seed` only fixes the random block order the scan uses
 * (section "算法": the block order must be random and independent of x), and
 * with it the amount of selection work and the counters of ds_topk_ex.
 *
 * Memory: every pointer passed to ds_topk / ds_topk_ex / ds_topk_long_row is
 * device memory owned by the caller.  The library allocates nothing on the
 * device and keeps no per-call state; it caches a few attributes per device.
 * The one device buffer it holds is the fixed 8 MiB workspace of
 * ds_topk_long_row_noalloc, part of the library's image on every device that
 * loads it.
 *
 * Layout: x is row-major with a row pitch of N elements; row r starts at
 * element r*N.  Outputs are row-major [rows][k].  Any alignment of x works;
 * when x is 16-byte aligned and N*sizeof(elem) and B*sizeof(elem) are
 * multiples of 16 the rows are staged into shared memory by 16-byte
 * asynchronous copies several stages ahead, otherwise by plain loads.
 *
 * Asynchrony: ds_topk and ds_topk_ex only enqueue work on `stream` (a
 * cudaStream_t, NULL for the legacy default stream) and return; they never
 * synchronise the host.  ds_topk_host synchronises before it returns.
 *
 * Errors: functions return DS_OK (0) or a negative status; argument errors
 * are reported before anything is enqueued.  ds_strerror gives a fixed text
 * per status and ds_last_error_detail a message for the calling thread's
 * most recent failure.  Device-side conditions that cannot be reported
 * synchronously: row_len[r] > N is read as N, row_len[r] < 0 as 0.
 */
#ifndef DS_TOPK_H
#define DS_TOPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DS_OK 0
#define DS_EINVAL (-1)       /* an argument is out of range or a pointer is NULL */
#define DS_EUNSUPPORTED (-2) /* dtype unknown, or the working set does not fit in shared memory */
#define DS_ECUDA (-3)        /* a CUDA runtime call failed (see ds_last_error_detail) */

#define DS_FP32 0
#define DS_BF16 1
#define DS_FP16 2 /* IEEE binary16; the same key order (NaN above +inf, -0 == +0) */

/* Launch plan chosen for a call (filled by ds_topk_plan). */
typedef struct {
    int splits;           /* CTAs cooperating on one row (thread-block cluster size) */
    int threads;          /* threads per CTA */
    int stages;           /* shared-memory ring slots, in stages */
    int blocks_per_stage; /* B-blocks staged per ring stage */
    int warps_per_block;  /* warps filtering one B-block */
    int async_copy;       /* 1: 16-byte asynchronous copies into shared memory; 0: plain loads */
    int smem_bytes;       /* dynamic shared memory per CTA */
    int capacity;         /* candidate-buffer capacity in entries: >= k + B + B2 (kernel 0),
                             >= k + B2 + one warp stage of 2 KiB (kernel 1) */
    int grid;             /* CTAs launched (rows * splits) */
    int ctas_per_sm;      /* resident CTAs per SM for this plan */
    int kernel;           /* 0: block by block, the pages' loop step for step (counters);
                             1: free-running warps (calls without counters whose rows take
                             16-byte copies) */
} ds_plan_t;

/*
 * ds_topk -- top-k of every row, sorted by (value desc, index asc).
 *   x        device, [rows][N] elements of `dtype` (DS_FP32, DS_BF16 or DS_FP16)
 *   rows     >= 0 (0 is a no-op)
 *   row_len  device int32[rows] valid lengths, or NULL for N in every row
 *   N        row pitch and maximum length, 1 <= N < 2^31
 *   k        1 <= k <= N
 *   B, B2    block size and compaction slack of the scan, both >= 1
 *            (section "算法": compaction runs when the buffer reaches k + B2)
 *   seed     key of the random block order
 *   out_idx  device int32[rows][k]
 *   out_val  device [rows][k] elements of `dtype`
 *   stream   cudaStream_t or NULL
 * The split factor is chosen automatically.
 */
int ds_topk(const void *x, int dtype, int rows, const int32_t *row_len, int64_t N, int k, int B,
            int B2, uint64_t seed, int32_t *out_idx, void *out_val, void *stream);

/*
 * ds_topk_ex -- ds_topk with an explicit split factor and optional counters.
 *   splits   0: automatic; 1: one CTA per row; 2..16: the m = ceil(len/B)
 *            blocks of a row are cut into `splits` contiguous slices of
 *            ceil(m/splits) blocks, one CTA of a thread-block cluster scans
 *            each slice, and the top k of the slices' union is selected by
 *            one radix select across the cluster (splits * k > 6144 and
 *            k <= 6144) or in CTA 0 (otherwise; for k > 6144 only entries at
 *            or above the largest slice k-th are sent) (section "实现", last
 *            paragraph).  The automatic factor
 *            is a power of two that fills the SMs with one CTA each (two when
 *            slices still hold 128 KiB); calls without counters keep slices of
 *            at least 64 KiB.
 *   stats    device int64[rows][splits][4] or NULL; when given, every slice
 *            writes {A, R, W, peak}: elements appended to the candidate
 *            buffer, compactions inside the loop, total input length of all
 *            selection calls including the final one, and the largest buffer
 *            length reached (section "RadixSelectTopK 总处理元素数的期望上界").
 *            Requires an explicit splits >= 1.
 */
int ds_topk_ex(const void *x, int dtype, int rows, const int32_t *row_len, int64_t N, int k,
               int B, int B2, uint64_t seed, int splits, int32_t *out_idx, void *out_val,
               int64_t *stats, void *stream);

/*
 * ds_topk_stats_order -- ds_topk_ex with counters and a chosen block order,
 * for studying the scan's work (a diagnostic; the result is the same).
 *   order   DS_ORDER_RANDOM: the random order of ds_topk_ex (the method);
 *           DS_ORDER_IDENTITY: blocks in index order.  DeepSelect-deep-dive,
 *           section "算法", requires an order that is random and independent
 *           of x: on a row sorted ascending, index order makes every block
 *           beat the threshold, so every element is appended and the work W
 *           grows with the row instead of staying within the bound of
 *           section "RadixSelectTopK 总处理元素数的期望上界".
 *   stats   required (non-NULL when rows > 0), as in ds_topk_ex; splits >= 1.
 * Other arguments and errors as ds_topk_ex; DS_EINVAL for another order.
 */
#define DS_ORDER_RANDOM 0
#define DS_ORDER_IDENTITY 1
int ds_topk_stats_order(const void *x, int dtype, int rows, const int32_t *row_len, int64_t N,
                        int k, int B, int B2, uint64_t seed, int splits, int order,
                        int32_t *out_idx, void *out_val, int64_t *stats, void *stream);

/*
 * ds_topk_host -- the same operation on HOST buffers.
 *   x_host, row_len_host (nullable), out_idx_host, out_val_host: host memory
 *   (page-locked memory gives asynchronous copies; pageable memory works).
 *   x_dev, row_len_dev (NULL iff row_len_host is NULL), out_idx_dev,
 *   out_val_dev: caller-owned device staging buffers of the same sizes.
 * Enqueues the host->device copies, the selection and the device->host
 * copies on `stream`, then synchronises the stream and returns.
 */
int ds_topk_host(const void *x_host, int dtype, int rows, const int32_t *row_len_host, int64_t N,
                 int k, int B, int B2, uint64_t seed, int32_t *out_idx_host, void *out_val_host,
                 void *x_dev, int32_t *row_len_dev, int32_t *out_idx_dev, void *out_val_dev,
                 void *stream);

/*
 * ds_topk_host_async -- ds_topk_host without the final synchronisation: the
 * copies and the selection are only enqueued on `stream`; the host buffers
 * must stay valid and unmodified (inputs) or unread (outputs) until the
 * stream reaches this point (cudaStreamSynchronize or an event).  With two
 * streams and two sets of staging buffers, consecutive calls overlap one
 * call's copies with the other's selection.  Page-locked host memory is
 * needed for the copies to be asynchronous.
 */
int ds_topk_host_async(const void *x_host, int dtype, int rows, const int32_t *row_len_host,
                       int64_t N, int k, int B, int B2, uint64_t seed, int32_t *out_idx_host,
                       void *out_val_host, void *x_dev, int32_t *row_len_dev, int32_t *out_idx_dev,
                       void *out_val_dev, void *stream);

/*
 * ds_topk_long_row -- top-k of ONE row of N elements spread over the whole
 * GPU, sorted by (value desc, index asc), the same result as ds_topk with
 * rows = 1.  The row is cut into G pieces of P elements (P a multiple of B;
 * the last piece shorter), every piece is selected by its own CTA(s)
 * (DeepSelect-deep-dive, section "实现", last paragraph: a sequence is cut
 * into parts that are selected separately), the top k of the G*k piece
 * results is selected by a second launch, and a gather maps the chosen
 * positions back to row indices (the multi-pass selection of one long row in
 * "CUDA 算子笔记 4", section "Top K Selection", takes the same place).  G
 * grows with N / k up to two pieces per SM, and beyond that only when a
 * piece would exceed the 4096 blocks one CTA orders; when it would be 1 the
 * row is selected directly and no workspace is used.
 *   x          device, N elements of `dtype`
 *   N, k, B, B2, seed  as in ds_topk (rows = 1)
 *   workspace  caller-owned device memory, 256-byte aligned, of at least the
 *              size ds_topk_long_row_workspace returns (may be NULL when that
 *              size is 0); it holds the piece results between the launches
 *              and must not be used by another call until this one is done
 *              on `stream`
 *   out_idx    device int32[k], row indices
 *   out_val    device [k] elements of `dtype`
 *   stream     cudaStream_t or NULL; three kernels are enqueued, nothing is
 *              synchronised
 * Errors: the argument checks of ds_topk, and DS_EINVAL when the workspace is
 * NULL, misaligned or smaller than needed.
 */
int ds_topk_long_row(const void *x, int dtype, int64_t N, int k, int B, int B2, uint64_t seed,
                     void *workspace, size_t workspace_bytes, int32_t *out_idx, void *out_val,
                     void *stream);

/* Plan of ds_topk_long_row for these arguments on the current device:
 * *bytes = workspace bytes it needs (0: none); when non-NULL, *piece_len = P
 * and *pieces = G (G = 1: the row is selected directly, P = N). */
int ds_topk_long_row_workspace(int dtype, int64_t N, int k, int B, int B2, size_t *bytes,
                               int64_t *piece_len, int *pieces);

/*
 * ds_topk_long_row_noalloc -- ds_topk_long_row for callers that cannot
 * allocate device memory: the same operation, arguments and result, with the
 * piece results kept in a workspace built into the library instead of one
 * the caller passes.  The pages have no counterpart; this is an interface
 * convenience.
 *   Workspace: one 8 MiB array per device, held from the library's load
 *   until the process exits.  Calls whose pieces need more than that (G*k
 *   entries of 4 + sizeof(elem) bytes each, plus 4*k bytes; see
 *   ds_topk_long_row_workspace) return DS_EUNSUPPORTED before anything is
 *   enqueued.  The call itself allocates nothing.
 *   Sharing: every call on a device uses the same array and leaves its
 *   contents behind; nothing in it needs to start at zero (each launch writes
 *   what the next one reads).  Calls that overlap on the GPU (on different
 *   streams, or from different host threads without ordering) race on the
 *   array and give wrong results: order them on one stream.
 *   Set-up: the first call on a device looks up the array's device address
 *   (once per device, with that device current).  Make that first call
 *   before capturing a CUDA graph that contains later calls.
 */
int ds_topk_long_row_noalloc(const void *x, int dtype, int64_t N, int k, int B, int B2,
                             uint64_t seed, int32_t *out_idx, void *out_val, void *stream);

/*
 * ds_topk_plan -- the launch plan ds_topk_ex would use on the current device
 * (x is only inspected for its alignment).  splits as in ds_topk_ex.
 */
int ds_topk_plan(const void *x, int dtype, int rows, int64_t N, int k, int B, int B2, int splits,
                 ds_plan_t *plan);

/* Largest k that fits one CTA's shared memory for this dtype, B and B2 on
 * the current device (N taken as large as the block order allows), or a
 * negative status. */
int ds_topk_max_k(int dtype, int B, int B2);

/* Fixed description of a status code. */
const char *ds_strerror(int status);

/* Message describing the calling thread's most recent failure ("" if none). */
const char *ds_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* DS_TOPK_H */
