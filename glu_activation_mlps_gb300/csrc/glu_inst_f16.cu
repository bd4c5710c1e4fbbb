// Kernel instantiations for storage dtype f16 (all activations, both directions).
#include "glu_kernels.cuh"

namespace glu {

KernelFn kernel_f16(int act, int dir, int vb_sel, int unroll_sel)
{
    return select_kernel<__half>(act, dir, vb_sel, unroll_sel);
}

}  // namespace glu
