// Log-sum-exp merge of the pieces of streams that straddle workers.
//
// The decode kernel concatenated the box streams KV-head-major and cut each
// region (one per KV head, or one for all heads on tiny grids) into equal
// slices of P boxes, Wr workers per region.  A stream [s, e) of region r
// that lies in one slice was finished by its worker and written to `out`
// directly.  A stream spanning workers r*Wr + s/P .. r*Wr + (e-1)/P left one
// partial per worker, each (acc_i, m_i, l_i) per query head with
// acc_i = sum over the piece of 2^(s_t - m_i) v_t and l_i = sum of
// 2^(s_t - m_i) (scores in log2 units).  Worker w0's piece sits in its first
// slot if the stream starts its slice, else in its second slot (the last
// piece of that slice); every later worker's piece is its first.  The result
// is
//     M = max_i m_i,  out = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i.
// Sequences with context length 0 get zeros here.
//
// One warp per (sequence, query head); each lane owns D/32 output columns.
#include <cuda_bf16.h>

#include <type_traits>

#include "pkv_kernels.h"
#include "pkv_ptx.cuh"

namespace pkv {

constexpr int kMergeWarps = 4;
constexpr int kFastPieces = 8;  // rows with at most this many pieces load everything at once

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_pieces_kernel(const DecodeParams p)
{
    constexpr int DPL = D / 32;
    grid_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kMergeWarps + warp;
    if (row >= (long long)p.B * p.Hq)
        return;
    const int b = (int)(row / p.Hq);
    const int hq = (int)(row - (long long)b * p.Hq);
    const int G = p.Hq / p.Hkv;
    const int kvh = hq / G, g = hq - kvh * G;
    // The box layout and the partials come from the decode kernel just before.
    grid_dependency_wait();
    const int P = p.ws_hdr[1];
    const int Wr = p.ws_hdr[2];
    const int R = p.ws_hdr[4];
    const int *pb = p.ws_hdr + kWsHeaderInts;
    const int nb = pb[b + 1] - pb[b];
    uint16_t *o = p.out + row * D + lane * DPL;
    if (nb == 0) {
#pragma unroll
        for (int i = 0; i < DPL; i++)
            o[i] = 0;
        return;
    }
    // Position of the stream inside its region (one region per KV head, or
    // a single region holding all heads head-major).
    const int r = R == p.Hkv ? kvh : 0;
    const int s = (R == p.Hkv ? 0 : kvh * pb[p.B]) + pb[b];
    const int e = s + nb;
    const int w0 = r * Wr + s / P, w1 = r * Wr + (e - 1) / P;
    if (w0 == w1)
        return;  // finished inside one worker
    const int n = w1 - w0 + 1;
    const int slot0 = (s % P == 0) ? 0 : 1;
    auto piece = [&](int i) -> const float * {
        const int w = w0 + i;
        const int slot = i == 0 ? slot0 : 0;
        return p.ws_part + (((size_t)w * 2 + slot) * G + g) * (D + 4);
    };

    using Vec = typename std::conditional<DPL == 4, float4, float2>::type;
    if (n <= kFastPieces) {
        // Few pieces (the common case): every load of the row in flight at once.
        Vec x[kFastPieces];
        float mi[kFastPieces], li[kFastPieces];
#pragma unroll
        for (int i = 0; i < kFastPieces; i++) {
            if (i < n) {
                const float *pc = piece(i);
                x[i] = *reinterpret_cast<const Vec *>(pc + lane * DPL);
                mi[i] = pc[D];
                li[i] = pc[D + 1];
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < kFastPieces; i++)
            if (i < n)
                M = fmaxf(M, mi[i]);
        float acc[DPL], Ls = 0.f;
#pragma unroll
        for (int c = 0; c < DPL; c++)
            acc[c] = 0.f;
        if (M != -INFINITY) {  // else no token of the stream could be read: zeros
#pragma unroll
            for (int i = 0; i < kFastPieces; i++) {
                if (i < n) {
                    const float w = fast_exp2(mi[i] - M);
                    Ls += li[i] * w;
                    const float *xv = reinterpret_cast<const float *>(&x[i]);
#pragma unroll
                    for (int c = 0; c < DPL; c++)
                        acc[c] += w * xv[c];
                }
            }
        }
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
        for (int c = 0; c < DPL; c++)
            o[c] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[c] * inv));
        return;
    }

    float M = -INFINITY;
    for (int i = lane; i < n; i += 32)
        M = fmaxf(M, piece(i)[D]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (M == -INFINITY) {  // no token of the stream could be read
#pragma unroll
        for (int i = 0; i < DPL; i++)
            o[i] = 0;
        return;
    }
    float Ls = 0.f;
    for (int i = lane; i < n; i += 32)
        Ls += piece(i)[D + 1] * fast_exp2(piece(i)[D] - M);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        Ls += __shfl_xor_sync(0xffffffffu, Ls, off);

    // Weighted sum of the partial outputs; 8 pieces' loads in flight at once.
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; i++)
        acc[i] = 0.f;
    for (int c0 = 0; c0 < n; c0 += 32) {
        const int m = min(32, n - c0);
        const float wl = lane < m ? fast_exp2(piece(c0 + lane)[D] - M) : 0.f;
        for (int j0 = 0; j0 < m; j0 += 8) {
            Vec x[8];
#pragma unroll
            for (int j = 0; j < 8; j++)
                if (j0 + j < m)
                    x[j] = *reinterpret_cast<const Vec *>(piece(c0 + j0 + j) + lane * DPL);
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const float w = __shfl_sync(0xffffffffu, wl, (j0 + j) & 31);
                if (j0 + j < m) {
                    const float *xv = reinterpret_cast<const float *>(&x[j]);
#pragma unroll
                    for (int i = 0; i < DPL; i++)
                        acc[i] += w * xv[i];
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < DPL; i++)
        o[i] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[i] / Ls));
}

cudaError_t launch_merge(int D, int G, const DecodeParams &p, cudaStream_t stream)
{
    (void)G;
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
        return cudaLaunchKernelEx(&cfg, merge_pieces_kernel<128>, p);
    if (D == 64)
        return cudaLaunchKernelEx(&cfg, merge_pieces_kernel<64>, p);
    return cudaErrorInvalidValue;
}

} // namespace pkv
