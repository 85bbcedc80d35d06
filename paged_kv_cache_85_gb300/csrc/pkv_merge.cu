// Log-sum-exp merge of split-K partial results.
//
// A sequence whose context was cut into k > 1 partitions has, per query
// head, k partial states (acc_c, m_c, l_c): acc_c = sum over the partition
// of 2^(s_t - m_c) v_t, l_c = sum of 2^(s_t - m_c), with scores s in log2
// units.  The full softmax result is
//     M = max_c m_c,  out = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c.
// Sequences with one partition were written by the decode kernel directly;
// sequences with context length 0 get zeros here.
//
// One warp per (sequence, query head); each lane owns D/32 output columns.
#include <cuda_bf16.h>

#include "pkv_kernels.h"
#include "pkv_ptx.cuh"

namespace pkv {

constexpr int kMergeWarps = 4;

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_partitions_kernel(const DecodeParams p)
{
    constexpr int DPL = D / 32;
    grid_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kMergeWarps + warp;
    if (row >= (long long)p.B * p.Hq)
        return;
    const int b = (int)(row / p.Hq);
    int n = __ldg(p.context_lens + b);
    const int maxctx = p.MBS * p.bs;
    n = n < 0 ? 0 : (n > maxctx ? maxctx : n);
    const int nc = (n + p.chunk - 1) / p.chunk;
    if (nc == 1)
        return;
    // Partials come from the decode kernel just before this one.
    grid_dependency_wait();
    uint16_t *o = p.out + row * D + lane * DPL;
    if (nc == 0) {
#pragma unroll
        for (int i = 0; i < DPL; i++)
            o[i] = 0;
        return;
    }
    const float *ml = p.ws_ml + (size_t)row * p.S * 2;
    float M = -INFINITY;
    for (int c = lane; c < nc; c += 32)
        M = fmaxf(M, ml[2 * c]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float Ls = 0.f;
    for (int c = lane; c < nc; c += 32)
        Ls += ml[2 * c + 1] * fast_exp2(ml[2 * c] - M);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        Ls += __shfl_xor_sync(0xffffffffu, Ls, off);

    const float *a = p.ws_acc + (size_t)row * p.S * D + lane * DPL;
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; i++)
        acc[i] = 0.f;
    for (int c = 0; c < nc; c++) {
        const float w = fast_exp2(ml[2 * c] - M);
        if constexpr (DPL == 4) {
            const float4 x = *reinterpret_cast<const float4 *>(a + (size_t)c * D);
            acc[0] += w * x.x;
            acc[1] += w * x.y;
            acc[2] += w * x.z;
            acc[3] += w * x.w;
        } else {
            const float2 x = *reinterpret_cast<const float2 *>(a + (size_t)c * D);
            acc[0] += w * x.x;
            acc[1] += w * x.y;
        }
    }
#pragma unroll
    for (int i = 0; i < DPL; i++)
        o[i] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[i] / Ls));
}

cudaError_t launch_merge(int D, const DecodeParams &p, cudaStream_t stream)
{
    const long long rows = (long long)p.B * p.Hq;
    if (rows == 0)
        return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)((rows + kMergeWarps - 1) / kMergeWarps));
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (D == 128)
        return cudaLaunchKernelEx(&cfg, merge_partitions_kernel<128>, p);
    if (D == 64)
        return cudaLaunchKernelEx(&cfg, merge_partitions_kernel<64>, p);
    return cudaErrorInvalidValue;
}

} // namespace pkv
