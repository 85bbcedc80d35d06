// Paged prefill: kernel parameters and host-side launch entry points
// (internal; the public ABI is pkv.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

struct PrefillParams {
    const uint16_t *q;            // bf16 [Tq, Hq, D]: the sequences' new tokens, concatenated
    uint16_t *out;                // bf16 [Tq, Hq, D]
    const int32_t *block_tables;  // [B, MBS]
    const int32_t *cu_q;          // [B + 1] boundaries of the new tokens
    const int32_t *cu_k;          // [B + 1] boundaries of the contexts (cached + new)
    int32_t *err_flag;            // nullable
    long long Tq;
    int B, Hq, Hkv, MBS, bs, NB;
    int max_q;                    // the caller's bound on q_len (sizes the work space)
    int X;                        // query tile pairs per sequence at max_q
    int n_items;                  // work items: X tile pairs x Hkv heads x B sequences
    float scale_log2;             // |scale| * log2(e)
    int neg_scale;                // scale < 0: the score MMA negates Q
    int tile_copies;              // bs % 64 == 0: K/V maps copy whole 64-token tiles
};

cudaError_t launch_prefill(int D, int G, const CUtensorMap *tmq, const CUtensorMap *tmk,
                           const CUtensorMap *tmv, const PrefillParams &p, dim3 grid, size_t smem,
                           cudaStream_t stream);
const void *prefill_kernel(int D, int G);
size_t prefill_smem_bytes(int D);
constexpr int kPrefillRows = 128;  // (token, head) rows per query tile (two tiles per work item)
constexpr int kPrefillKeys = 64;   // keys per K/V tile
constexpr int kPrefillThreads = 11 * 32;

} // namespace pkv
