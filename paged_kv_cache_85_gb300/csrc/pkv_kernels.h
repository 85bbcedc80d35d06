// Kernel parameters and host-side launch entry points shared by the
// translation units of the CUDA library (internal; the public ABI is pkv.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

// Decode pipeline geometry.
constexpr int kTile = 64;          // context tokens per pipeline stage
constexpr int kBox = 16;           // tokens per TMA box; divides every block size
constexpr int kConsumerWarps = 4;  // each owns one 16-token box of a stage
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kSegTokens = 32 * kBox;  // tokens whose block ids one producer load covers
constexpr int kAutoChunk = 256;    // default partition length (split-K)
constexpr int kMaxSplits = 1024;   // most partitions one sequence may have
constexpr int kMaxBatch = 8192;    // sequences per call (unit map lives in shared memory)

struct DecodeParams {
    const uint16_t *q;            // bf16 [B, Hq, D]
    const int32_t *block_tables;  // [B, MBS]
    const int32_t *context_lens;  // [B]
    uint16_t *out;                // bf16 [B, Hq, D]
    float *ws_acc;                // [B, Hq, S, D]   unnormalised partial outputs
    float *ws_ml;                 // [B, Hq, S, 2]   (running max in log2 units, sum)
    int32_t *err_flag;            // nullable
    int B, Hq, Hkv, MBS, bs;
    int chunk;                    // partition length in tokens, multiple of kTile
    int S;                        // ceil(MBS*bs / chunk)
    int NB;
    float scale_log2;             // scale * log2(e)
};

// Partition choice shared by the workspace query and the launch.
inline void choose_partition(int MBS, int bs, int num_splits, int *chunk, int *S)
{
    long long maxctx = (long long)MBS * bs;
    if (maxctx < 1)
        maxctx = 1;
    long long c = num_splits > 0 ? (maxctx + num_splits - 1) / num_splits : kAutoChunk;
    c = (c + kTile - 1) / kTile * kTile;
    long long cap = (maxctx + kTile - 1) / kTile * kTile;
    if (c > cap)
        c = cap;
    long long s = (maxctx + c - 1) / c;
    if (s > kMaxSplits) {
        c = ((maxctx + kMaxSplits - 1) / kMaxSplits + kTile - 1) / kTile * kTile;
        s = (maxctx + c - 1) / c;
    }
    *chunk = (int)c;
    *S = (int)s;
}

// Host launchers (defined next to their kernels).
cudaError_t launch_store(const void *k, const void *v, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int64_t N, int row_bytes,
                         long long n_slots, int32_t *err_flag, cudaStream_t stream);

// Dynamic shared memory the decode kernel needs for (D, G, B, S).
size_t decode_smem_bytes(int D, int G, int B, int S);
// Resident CTAs per SM for that configuration (0 if it cannot launch).
int decode_occupancy(int D, int G, size_t smem);
cudaError_t launch_decode(int D, int G, const CUtensorMap *tmk, const CUtensorMap *tmv,
                          const DecodeParams &p, int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_merge(int D, const DecodeParams &p, cudaStream_t stream);

} // namespace pkv
