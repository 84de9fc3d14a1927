// Test kernels for the device primitives of the DeepSelect library (test
// infrastructure only: the library's C ABI does not expose these).  Each
// kernel runs one warp on the inputs of a worked example and writes what the
// primitive produced.
#include <stdint.h>

#include "ds_device.cuh"

using namespace ds;

// warp_inclusive_scan over lanes 0..n-1 (other lanes hold 0)
__global__ void k_scan(const uint32_t *in, int n, uint32_t *incl, uint32_t *excl)
{
    const int lane = threadIdx.x;
    const uint32_t v = lane < n ? in[lane] : 0u;
    const uint32_t s = warp_inclusive_scan(v, lane);
    if (lane < n) {
        incl[lane] = s;
        excl[lane] = s - v;
    }
}

// compaction as the select does it: keep flags per register slot, a warp
// ballot count (the warp's slots start after the lower warps' counts; one
// warp here), ballot ranks for the positions
__global__ void k_compact(const uint32_t *x, const uint32_t *p, int n, unsigned long long *out,
                          int *count)
{
    const int lane = threadIdx.x;
    uint32_t hi[1] = {0u}, lo[1] = {lane < n ? x[lane] : 0u};
    const uint32_t keep = (lane < n && p[lane]) ? 1u : 0u;
    const int total = warp_count<1>(keep);
    warp_scatter<1>(keep, hi, lo, out, lane);
    if (lane == 0)
        *count = total;
}

// the mask walk of the append: lane 0 holds a bit mask of kept positions
// and writes x at them in order with __ffs / mask &= mask - 1
__global__ void k_mask_walk(const uint32_t *x, uint32_t mask, uint32_t *out, int *count)
{
    if (threadIdx.x != 0)
        return;
    int pos = 0;
    uint32_t m = mask;
    while (m) {
        const int e = __ffs(m) - 1;
        m &= m - 1u;
        out[pos++] = x[e];
    }
    *count = pos;
}

// the free-running kernel's block order: position q -> block id, for q < n
__global__ void k_block_order(uint32_t n, uint32_t word, uint32_t *out)
{
    BlockOrder order;
    order.init(n, word);
    for (uint32_t q = blockIdx.x * blockDim.x + threadIdx.x; q < n; q += gridDim.x * blockDim.x)
        out[q] = order(q);
}

extern "C" int prim_block_order(uint32_t n, uint32_t word, uint32_t *out)
{
    k_block_order<<<64, 256>>>(n, word, out);
    return (int)cudaDeviceSynchronize();
}

extern "C" int prim_scan(const uint32_t *in, int n, uint32_t *incl, uint32_t *excl)
{
    k_scan<<<1, 32>>>(in, n, incl, excl);
    return (int)cudaDeviceSynchronize();
}

extern "C" int prim_compact(const uint32_t *x, const uint32_t *p, int n, unsigned long long *out,
                            int *count)
{
    k_compact<<<1, 32>>>(x, p, n, out, count);
    return (int)cudaDeviceSynchronize();
}

extern "C" int prim_mask_walk(const uint32_t *x, uint32_t mask, uint32_t *out, int *count)
{
    k_mask_walk<<<1, 32>>>(x, mask, out, count);
    return (int)cudaDeviceSynchronize();
}
