// ds_kernels_bf16.cu -- bf16 instantiations of the DeepSelect top-k kernel.
#include "ds_kernel.cuh"

namespace ds {

KernelFn kernel_bf16(bool async, bool wide)
{
    if (async)
        return wide ? deepselect_topk_kernel<1, true, 16> : deepselect_topk_kernel<1, true, 4>;
    return wide ? deepselect_topk_kernel<1, false, 16> : deepselect_topk_kernel<1, false, 4>;
}

}  // namespace ds
