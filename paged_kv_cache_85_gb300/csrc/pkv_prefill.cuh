// Paged prefill attention (causal, variable-length, GQA) on sm_103a.
//
// What it computes (MinivLLM guide "HowToApproachvLLM" §4.5 prepare_prefill:
// the new tokens of all sequences are flattened into one list with
// cu_seqlens_q / cu_seqlens_k boundaries and KV is read through block_tables;
// "Nano-vLLM 源码学习(2)" §2: the prefix-hit prefill path reads paged KV):
// sequence b has q_len = cu_q[b+1] - cu_q[b] new tokens and k_len =
// cu_k[b+1] - cu_k[b] keys (cached prefix + the new tokens, already stored);
// new token i sits at position k_len - q_len + i and attends to positions
// 0 .. that one:  out = softmax(scale q.K^T) V over those keys.
//
// Design.  One CTA per (query tile, KV head, sequence).  A tile is 112 rows
// of (token, head-in-group) pairs, token-major, so every K/V byte a CTA
// loads serves all G query heads of its KV head.  Seven consumer warps own
// 16 rows each; one producer warp streams 64-key K/V tiles (four 16-token
// boxes, each resolved through the block table and fetched by TMA with the
// 128-byte swizzle) through a 4-stage mbarrier ring.  Each consumer warp
// keeps its Q fragments and O accumulators in registers (mma.sync m16n8k16,
// bf16 in, fp32 accumulate), runs the online softmax in the log2 domain on
// the score fragments, and splits P into bf16 hi + lo parts for P.V so that
// P keeps ~16 significant bits.  The running max moves only when a row's
// tile max exceeds it by more than 2^8 (P <= 256, exact in bf16's range).
// Warps skip the MMAs of tiles that lie entirely above their rows' causal
// limit; tiles entirely below it skip the masking.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_kernels.h"
#include "pkv_prefill.h"
#include "pkv_ptx.cuh"

namespace pkv {

constexpr int kPfWarps = 7;                // consumer warps, 16 rows each
constexpr int kPfRows = kPfWarps * 16;     // (token, head) rows per CTA: 112 = 16 * 7, a
                                           // multiple of every G; 8 warps in all keep two
                                           // warps per SM sub-partition (255 registers)
constexpr int kPfKeys = 64;                // keys per K/V tile
constexpr int kPfBoxes = kPfKeys / kBox;   // 16-token boxes per tile
constexpr int kPfStages = 4;

struct PrefillSmem {
    size_t kv, full, empty, meta, total;
};

__host__ __device__ inline PrefillSmem prefill_smem_layout(int D)
{
    PrefillSmem L;
    size_t o = 0;
    L.kv = o;  // per stage: K tile [4 boxes][D/64 halves][16][64], then V tile alike
    o += (size_t)kPfStages * 2 * kPfBoxes * kBox * D * 2;
    L.full = o;
    o += kPfStages * 8;
    L.empty = o;
    o += kPfStages * 8;
    L.meta = o;  // per stage: bit i set when box i was loaded
    o += kPfStages * 4;
    L.total = align_up(o, 16) + 1024;  // slack to align the base to 1024 B
    return L;
}

// Byte offset of 16-byte chunk `c` (0 .. D/8-1) of token row `t` in a
// 16-token box stored as D/64 halves of [16 rows][128 B], 128-byte swizzle.
__device__ __forceinline__ uint32_t pf_chunk(int t, int c)
{
    return (uint32_t)((c >> 3) * kHalfBytes + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

template <int D>
__device__ __forceinline__ void prefill_producer(const CUtensorMap *tmk, const CUtensorMap *tmv,
                                                 const PrefillParams &p, uint8_t *smem,
                                                 const PrefillSmem &L, int lane, int b, int kvh,
                                                 int k_len, int nkt)
{
    constexpr unsigned FULL = 0xffffffffu;
    constexpr int kBoxBytes = kBox * D * 2;
    constexpr int kTileBytes = kPfBoxes * kBoxBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    uint32_t *meta = reinterpret_cast<uint32_t *>(smem + L.meta);
    if (lane == 0) {
        prefetch_tensormap(tmk);
        prefetch_tensormap(tmv);
    }
    const int32_t *table = p.block_tables + (size_t)b * p.MBS;
    // The K/V may have just been written by store_kvcache on this stream.
    grid_dependency_wait();
    int stage = 0;
    uint32_t phase = 0;
    for (int j = 0; j < nkt; j++) {
        if (!__all_sync(FULL, mbar_wait(&empty[stage], phase ^ 1))) {
            if (lane == 0)
                flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
            return;
        }
        // lanes 0..3: one 16-token box each
        const int key0 = j * kPfKeys + lane * kBox;
        bool loaded = false;
        int row = 0;
        if (lane < kPfBoxes && key0 < k_len) {
            const int blk = __ldg(table + key0 / p.bs);
            loaded = blk >= 0 && blk < p.NB;
            if (!loaded)
                flag_error(p.err_flag, 0x2 /* PKV_FLAG_BAD_BLOCK */);
            row = blk * p.bs + key0 % p.bs;
        }
        const uint32_t mask = __ballot_sync(FULL, loaded);
        const uint32_t bytes = (uint32_t)__popc(mask) * 2u * kBoxBytes;
        if (lane == 0) {
            meta[stage] = mask;
            mbar_arrive_expect_tx(&full[stage], bytes);
        }
        __syncwarp();
        if (loaded) {
            uint8_t *kd = smem + L.kv + (size_t)stage * 2 * kTileBytes + lane * kBoxBytes;
#pragma unroll
            for (int half = 0; half < D / 64; half++) {
                tma_load_4d(kd + half * kHalfBytes, tmk, 0, half, kvh, row, &full[stage]);
                tma_load_4d(kd + kTileBytes + half * kHalfBytes, tmv, 0, half, kvh, row,
                            &full[stage]);
            }
        }
        if (++stage == kPfStages) {
            stage = 0;
            phase ^= 1;
        }
    }
}

template <int D, int G>
__device__ __forceinline__ void prefill_consumer(const PrefillParams &p, uint8_t *smem,
                                                 const PrefillSmem &L, int warp, int lane, int b,
                                                 int kvh, int cq0, int q_len, int k_len, int tok0,
                                                 int nkt)
{
    constexpr unsigned FULL = 0xffffffffu;
    constexpr int KS = D / 16;                 // k-steps of q.K^T
    constexpr int NT = D / 8;                  // n-tiles of O
    constexpr int kBoxBytes = kBox * D * 2;
    constexpr int kTileBytes = kPfBoxes * kBoxBytes;
    constexpr float kLazy = 8.f;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    const uint32_t *meta = reinterpret_cast<const uint32_t *>(smem + L.meta);

    const int quad = lane & 3;
    const int mat = lane >> 3, mrow = lane & 7;
    // this lane's two rows (CTA rows r0, r0 + 8), their tokens and heads
    const int r0 = warp * 16 + (lane >> 2), r1 = r0 + 8;
    const int t0 = tok0 + r0 / G, t1 = tok0 + r1 / G;
    const int g0 = r0 % G, g1 = r1 % G;
    const bool ok0 = t0 < q_len, ok1 = t1 < q_len;
    const int base = k_len - q_len;            // position of new token 0
    const int pos0 = base + t0, pos1 = base + t1;
    // the warp's causal range: its first row's position .. its last valid row's
    const int wt_first = tok0 + (warp * 16) / G;
    const int wt_last = min(tok0 + (warp * 16 + 15) / G, q_len - 1);
    const int w_nkt = wt_first < q_len ? (base + wt_last) / kPfKeys + 1 : 0;
    const int wpos_first = base + wt_first;

    // Q fragments straight from global memory (rows past q_len are zero)
    grid_dependency_wait();
    const uint16_t *q0 = p.q + ((size_t)(cq0 + t0) * p.Hq + kvh * G + g0) * D + 2 * quad;
    const uint16_t *q1 = p.q + ((size_t)(cq0 + t1) * p.Hq + kvh * G + g1) * D + 2 * quad;
    uint32_t qa[KS][4];
#pragma unroll
    for (int k = 0; k < KS; k++) {
        qa[k][0] = ok0 ? __ldg(reinterpret_cast<const uint32_t *>(q0 + 16 * k)) : 0u;
        qa[k][1] = ok1 ? __ldg(reinterpret_cast<const uint32_t *>(q1 + 16 * k)) : 0u;
        qa[k][2] = ok0 ? __ldg(reinterpret_cast<const uint32_t *>(q0 + 16 * k + 8)) : 0u;
        qa[k][3] = ok1 ? __ldg(reinterpret_cast<const uint32_t *>(q1 + 16 * k + 8)) : 0u;
    }
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; n++)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    const int ktok = mrow + ((mat >> 1) << 3);  // K rows this lane addresses for ldmatrix
    const int vtok = mrow + ((mat & 1) << 3);   // V rows (transposed loads)
    int stage = 0;
    uint32_t phase = 0;
    for (int j = 0; j < nkt; j++) {
        if (!__all_sync(FULL, mbar_wait(&full[stage], phase))) {
            if (lane == 0)
                flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
            return;
        }
        if (j < w_nkt) {
            const uint32_t mask = meta[stage];
            const uint32_t kb = smem_u32(smem + L.kv + (size_t)stage * 2 * kTileBytes);
            const uint32_t vb = kb + kTileBytes;
            // ---- S = Q K^T: 16 rows x 64 keys (n-tile n = keys 8n .. 8n+7) ----
            float s[8][4];
#pragma unroll
            for (int n = 0; n < 8; n++)
                s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
            for (int k = 0; k < KS; k++) {
#pragma unroll
                for (int bx = 0; bx < kPfBoxes; bx++) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(kb + bx * kBoxBytes + pf_chunk(ktok, 2 * k + (mat & 1)), b0, b1,
                                b2, b3);
                    mma_bf16_16816(s[2 * bx], qa[k][0], qa[k][1], qa[k][2], qa[k][3], b0, b1);
                    mma_bf16_16816(s[2 * bx + 1], qa[k][0], qa[k][1], qa[k][2], qa[k][3], b2, b3);
                }
            }
            // ---- scale (log2 domain) and mask ----
            const int key_base = j * kPfKeys;
            const bool all_loaded = mask == (1u << kPfBoxes) - 1u;
#pragma unroll
            for (int n = 0; n < 8; n++) {
                s[n][0] *= p.scale_log2;
                s[n][1] *= p.scale_log2;
                s[n][2] *= p.scale_log2;
                s[n][3] *= p.scale_log2;
            }
            if (!all_loaded || key_base + kPfKeys - 1 > wpos_first) {
#pragma unroll
                for (int n = 0; n < 8; n++) {
                    const bool bl = (mask >> (n >> 1)) & 1u;
                    const int key = key_base + 8 * n + 2 * quad;
                    if (!bl || key > pos0) s[n][0] = -INFINITY;
                    if (!bl || key + 1 > pos0) s[n][1] = -INFINITY;
                    if (!bl || key > pos1) s[n][2] = -INFINITY;
                    if (!bl || key + 1 > pos1) s[n][3] = -INFINITY;
                }
            }
            // ---- online softmax per row ----
            float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
            for (int n = 0; n < 8; n++) {
                x0 = fmaxf(x0, fmaxf(s[n][0], s[n][1]));
                x1 = fmaxf(x1, fmaxf(s[n][2], s[n][3]));
            }
            x0 = fmaxf(x0, __shfl_xor_sync(FULL, x0, 1));
            x0 = fmaxf(x0, __shfl_xor_sync(FULL, x0, 2));
            x1 = fmaxf(x1, __shfl_xor_sync(FULL, x1, 1));
            x1 = fmaxf(x1, __shfl_xor_sync(FULL, x1, 2));
            if (__any_sync(FULL, x0 > m0 + kLazy || x1 > m1 + kLazy)) {
                const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
                const float a0 = n0 == -INFINITY ? 1.f : fast_exp2(m0 - n0);
                const float a1 = n1 == -INFINITY ? 1.f : fast_exp2(m1 - n1);
                m0 = n0;
                m1 = n1;
                l0 *= a0;
                l1 *= a1;
#pragma unroll
                for (int n = 0; n < NT; n++) {
                    o[n][0] *= a0;
                    o[n][1] *= a0;
                    o[n][2] *= a1;
                    o[n][3] *= a1;
                }
            }
            const float mu0 = m0 == -INFINITY ? 0.f : m0, mu1 = m1 == -INFINITY ? 0.f : m1;
#pragma unroll
            for (int n = 0; n < 8; n++) {
                s[n][0] = fast_exp2(s[n][0] - mu0);
                s[n][1] = fast_exp2(s[n][1] - mu0);
                s[n][2] = fast_exp2(s[n][2] - mu1);
                s[n][3] = fast_exp2(s[n][3] - mu1);
                l0 += s[n][0] + s[n][1];
                l1 += s[n][2] + s[n][3];
            }
            // ---- O += P V, one 16-key box per k-step, P split hi + lo ----
            const bool vmask = !all_loaded || key_base + kPfKeys > k_len;
#pragma unroll
            for (int bx = 0; bx < kPfBoxes; bx++) {
                uint32_t ah[4], al[4];
                {
                    const float pv[4][2] = {{s[2 * bx][0], s[2 * bx][1]},
                                            {s[2 * bx][2], s[2 * bx][3]},
                                            {s[2 * bx + 1][0], s[2 * bx + 1][1]},
                                            {s[2 * bx + 1][2], s[2 * bx + 1][3]}};
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        ah[i] = pack_bf16x2(pv[i][0], pv[i][1]);
                        const float2 h = bf16x2_to_float2(ah[i]);
                        al[i] = pack_bf16x2(pv[i][0] - h.x, pv[i][1] - h.y);
                    }
                }
                // keys of this box past k_len, or in a box not loaded, must not
                // reach the MMA (0 * NaN is NaN): clear their V halves
                uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
                if (vmask) {
                    const int kb0 = key_base + bx * kBox + 2 * quad;  // keys of b0 halves
                    const bool bl = (mask >> bx) & 1u;
                    keep_lo = (bl && kb0 < k_len ? 0x0000ffffu : 0u) |
                              (bl && kb0 + 1 < k_len ? 0xffff0000u : 0u);
                    keep_hi = (bl && kb0 + 8 < k_len ? 0x0000ffffu : 0u) |
                              (bl && kb0 + 9 < k_len ? 0xffff0000u : 0u);
                }
#pragma unroll
                for (int n2 = 0; n2 < NT / 2; n2++) {
                    uint32_t v0, v1, v2, v3;
                    ldmatrix_x4_trans(vb + bx * kBoxBytes + pf_chunk(vtok, 2 * n2 + (mat >> 1)),
                                      v0, v1, v2, v3);
                    v0 &= keep_lo;
                    v1 &= keep_hi;
                    v2 &= keep_lo;
                    v3 &= keep_hi;
                    mma_bf16_16816(o[2 * n2], ah[0], ah[1], ah[2], ah[3], v0, v1);
                    mma_bf16_16816(o[2 * n2], al[0], al[1], al[2], al[3], v0, v1);
                    mma_bf16_16816(o[2 * n2 + 1], ah[0], ah[1], ah[2], ah[3], v2, v3);
                    mma_bf16_16816(o[2 * n2 + 1], al[0], al[1], al[2], al[3], v2, v3);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[stage]);
        if (++stage == kPfStages) {
            stage = 0;
            phase ^= 1;
        }
    }
    // ---- normalise and store ----
    l0 += __shfl_xor_sync(FULL, l0, 1);
    l0 += __shfl_xor_sync(FULL, l0, 2);
    l1 += __shfl_xor_sync(FULL, l1, 1);
    l1 += __shfl_xor_sync(FULL, l1, 2);
    const float f0 = l0 > 0.f ? 1.f / l0 : 0.f, f1 = l1 > 0.f ? 1.f / l1 : 0.f;
    if (ok0) {
        uint16_t *dst = p.out + ((size_t)(cq0 + t0) * p.Hq + kvh * G + g0) * D + 2 * quad;
#pragma unroll
        for (int n = 0; n < NT; n++)
            *reinterpret_cast<uint32_t *>(dst + 8 * n) = pack_bf16x2(o[n][0] * f0, o[n][1] * f0);
    }
    if (ok1) {
        uint16_t *dst = p.out + ((size_t)(cq0 + t1) * p.Hq + kvh * G + g1) * D + 2 * quad;
#pragma unroll
        for (int n = 0; n < NT; n++)
            *reinterpret_cast<uint32_t *>(dst + 8 * n) = pack_bf16x2(o[n][2] * f1, o[n][3] * f1);
    }
    (void)b;
}

template <int D, int G>
__global__ void __launch_bounds__((kPfWarps + 1) * 32, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const PrefillParams p)
{
    constexpr int TPC = kPfRows / G;  // query tokens per CTA
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const PrefillSmem L = prefill_smem_layout(D);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, kvh = blockIdx.y;
    const int tile = (int)gridDim.x - 1 - (int)blockIdx.x;  // the longest tiles start first

    grid_launch_dependents();
    const int cq0 = __ldg(p.cu_q + b), cq1 = __ldg(p.cu_q + b + 1);
    const int ck0 = __ldg(p.cu_k + b), ck1 = __ldg(p.cu_k + b + 1);
    const int q_len = cq1 - cq0, k_len = ck1 - ck0;
    const bool sane = cq0 >= 0 && q_len >= 0 && (long long)cq1 <= p.Tq && k_len >= q_len &&
                      k_len <= p.MBS * p.bs && q_len <= p.max_q;
    if (!sane) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0)
            flag_error(p.err_flag, 0x4 /* PKV_FLAG_BAD_CONTEXT_LEN */);
        return;
    }
    const int tok0 = tile * TPC;
    if (tok0 >= q_len)
        return;
    const int last_pos = (k_len - q_len) + min(q_len, tok0 + TPC) - 1;
    const int nkt = last_pos / kPfKeys + 1;

    if (threadIdx.x == 0) {
        uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
        uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
        for (int s = 0; s < kPfStages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPfWarps);
        }
        fence_mbarrier_init();
    }
    __syncthreads();
    if (warp == kPfWarps)
        prefill_producer<D>(&tmk, &tmv, p, smem, L, lane, b, kvh, k_len, nkt);
    else
        prefill_consumer<D, G>(p, smem, L, warp, lane, b, kvh, cq0, q_len, k_len, tok0, nkt);
}

template <int D>
inline cudaError_t launch_prefill_d(int G, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                    const PrefillParams &p, dim3 grid, size_t smem,
                                    cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = dim3((kPfWarps + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (G) {
    case 1: return cudaLaunchKernelEx(&cfg, paged_prefill_kernel<D, 1>, *tmk, *tmv, p);
    case 2: return cudaLaunchKernelEx(&cfg, paged_prefill_kernel<D, 2>, *tmk, *tmv, p);
    case 4: return cudaLaunchKernelEx(&cfg, paged_prefill_kernel<D, 4>, *tmk, *tmv, p);
    case 8: return cudaLaunchKernelEx(&cfg, paged_prefill_kernel<D, 8>, *tmk, *tmv, p);
    default: return cudaErrorInvalidValue;
    }
}

template <int D> inline const void *prefill_kernel_d(int G)
{
    switch (G) {
    case 1: return reinterpret_cast<const void *>(&paged_prefill_kernel<D, 1>);
    case 2: return reinterpret_cast<const void *>(&paged_prefill_kernel<D, 2>);
    case 4: return reinterpret_cast<const void *>(&paged_prefill_kernel<D, 4>);
    case 8: return reinterpret_cast<const void *>(&paged_prefill_kernel<D, 8>);
    default: return nullptr;
    }
}

} // namespace pkv
