// Instantiations of the paged decode kernel: head_dim 128, 8 workers per CTA,
// FP8 (E4M3) caches, G = 1, 2, 4, 8, boxes of 16 or 32 tokens.
#include "pkv_decode.cuh"

namespace pkv {

cudaError_t launch_decode8_d128_w8(int G, int bt, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                   const DecodeParams &p, int grid, size_t smem, cudaStream_t stream)
{
    return bt == 2 * kBox ? launch_decode_shape<128, 8, true, 2 * kBox>(G, tmk, tmv, p, grid, smem, stream)
                          : launch_decode_shape<128, 8, true, kBox>(G, tmk, tmv, p, grid, smem, stream);
}

const void *decode_kernel8_d128_w8(int G, int bt)
{
    return bt == 2 * kBox ? decode_kernel_shape<128, 8, true, 2 * kBox>(G)
                          : decode_kernel_shape<128, 8, true, kBox>(G);
}

} // namespace pkv
