// ds_kernels_bf16.cu -- bf16 instantiations of the DeepSelect top-k kernels.
#include "ds_stream.cuh"

namespace ds {

KernelFn kernel_bf16(bool async, bool wide)
{
    if (async)
        return wide ? deepselect_topk_kernel<1, true, 16> : deepselect_topk_kernel<1, true, 4>;
    return wide ? deepselect_topk_kernel<1, false, 16> : deepselect_topk_kernel<1, false, 4>;
}

KernelFn stream_kernel_bf16(bool pairs)
{
    return pairs ? deepselect_stream_kernel<1, true> : deepselect_stream_kernel<1, false>;
}

}  // namespace ds
