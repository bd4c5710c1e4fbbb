// Instantiations and host side of the bulk-copy staging kernels (all
// activations, dtypes and directions), and the counter of waits that ran out.
#include "glu_bulk.cuh"

namespace glu {

namespace {

template <class T, class Act>
BulkFn bulk_pick(int dir, bool narrow)
{
    if (narrow) return dir == kBwd ? glu_bulk_kernel<Act, T, kBwd, true> : glu_bulk_kernel<Act, T, kFwd, true>;
    return dir == kBwd ? glu_bulk_kernel<Act, T, kBwd, false> : glu_bulk_kernel<Act, T, kFwd, false>;
}

template <class T>
BulkFn bulk_for_dtype(int act, int dir, bool narrow)
{
    switch (act) {
    case 0: return bulk_pick<T, Silu>(dir, narrow);
    case 1: return bulk_pick<T, GeluErf>(dir, narrow);
    case 2: return bulk_pick<T, GeluTanh>(dir, narrow);
    case 3: return bulk_pick<T, Relu>(dir, narrow);
    default: return nullptr;
    }
}

}  // namespace

BulkFn bulk_kernel(int dtype, int act, int dir, bool narrow)
{
    switch (dtype) {
    case 0: return bulk_for_dtype<float>(act, dir, narrow);
    case 1: return bulk_for_dtype<__half>(act, dir, narrow);
    case 2: return bulk_for_dtype<__nv_bfloat16>(act, dir, narrow);
    default: return nullptr;
    }
}

int bulk_smem_bytes(int dir, bool narrow)
{
    if (narrow) return dir == kBwd ? BulkShape<kBwd, true>::kSmemBytes : BulkShape<kFwd, true>::kSmemBytes;
    return dir == kBwd ? BulkShape<kBwd, false>::kSmemBytes : BulkShape<kFwd, false>::kSmemBytes;
}

int bulk_threads(bool narrow)
{
    return narrow ? BulkShape<kFwd, true>::kThreads : BulkShape<kFwd, false>::kThreads;
}

cudaError_t bulk_timeouts(unsigned int *count, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(count, g_bulk_timeouts, sizeof(unsigned int));
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_bulk_timeouts, &zero, sizeof(unsigned int));
    }
    return e;
}

}  // namespace glu
