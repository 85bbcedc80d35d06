// Instantiations of the paged prefill kernel (tcgen05), head_dim 128, G = 1, 2, 4, 8.
#include "pkv_prefill_tc.cuh"

namespace pkv {

cudaError_t launch_prefill_d128(int G, const CUtensorMap *tmq, const CUtensorMap *tmk,
                               const CUtensorMap *tmv, const PrefillParams &p, dim3 grid,
                               size_t smem, cudaStream_t stream)
{
    return launch_prefill_tc_d<128>(G, tmq, tmk, tmv, p, grid, smem, stream);
}

const void *prefill_kernel_d128(int G) { return prefill_tc_kernel_d<128>(G); }

} // namespace pkv
