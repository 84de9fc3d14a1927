// ds_kernels_fp16.cu -- IEEE fp16 instantiations of the DeepSelect top-k kernels.
#include "ds_stream.cuh"

namespace ds {

KernelFn kernel_fp16(bool async, bool wide)
{
    if (async)
        return wide ? deepselect_topk_kernel<2, true, 16> : deepselect_topk_kernel<2, true, 4>;
    return wide ? deepselect_topk_kernel<2, false, 16> : deepselect_topk_kernel<2, false, 4>;
}

KernelFn stream_kernel_fp16(bool pairs)
{
    return pairs ? deepselect_stream_kernel<2, true> : deepselect_stream_kernel<2, false>;
}

}  // namespace ds
