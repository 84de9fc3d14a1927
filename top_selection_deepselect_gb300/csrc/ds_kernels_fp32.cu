// ds_kernels_fp32.cu -- fp32 instantiations of the DeepSelect top-k kernels.
#include "ds_stream.cuh"

namespace ds {

KernelFn kernel_fp32(bool async, bool wide)
{
    if (async)
        return wide ? deepselect_topk_kernel<0, true, 16> : deepselect_topk_kernel<0, true, 4>;
    return wide ? deepselect_topk_kernel<0, false, 16> : deepselect_topk_kernel<0, false, 4>;
}

KernelFn stream_kernel_fp32(bool pairs)
{
    return pairs ? deepselect_stream_kernel<0, true> : deepselect_stream_kernel<0, false>;
}

}  // namespace ds
