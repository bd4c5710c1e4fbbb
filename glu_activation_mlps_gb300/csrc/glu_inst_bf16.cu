// Kernel instantiations for storage dtype bf16 (all activations, both directions).
#include "glu_kernels.cuh"

namespace glu {

KernelFn kernel_bf16(int act, int dir, int vb_sel, int unroll_sel)
{
    return select_kernel<__nv_bfloat16>(act, dir, vb_sel, unroll_sel);
}

}  // namespace glu
