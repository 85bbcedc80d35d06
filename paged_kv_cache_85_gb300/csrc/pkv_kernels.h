// Kernel parameters and host-side launch entry points shared by the
// translation units of the CUDA library (internal; the public ABI is pkv.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

// Decode geometry.  Every (sequence, KV head) context is a stream of
// 16-token boxes; the concatenated streams are cut into equal contiguous
// slices, one per worker (a consumer warp).
constexpr int kBox = 16;         // tokens per box = per TMA copy; divides every block size
// Two CTA shapes: four workers (consumer warps) + one producer warp with a
// 3-stage ring, two CTAs per SM (preferred: less lock-step per stage, two
// producers per SM); or eight workers + one producer, one CTA per SM, for
// sizes whose shared memory does not fit twice on an SM.
constexpr int kPairWorkers = 4;
constexpr int kPairStages = 3;
constexpr int kWideWorkers = 8;
constexpr int kMaxStages = 4;    // pipeline depth cap (stage = one box per worker)
constexpr int kMinStages = 2;
constexpr size_t kSmemPerSm = 228 * 1024;   // shared memory per SM
constexpr size_t kSmemReserve = 1024;       // reserved per resident CTA
constexpr size_t kMaxDynSmem = 227 * 1024;  // opt-in maximum per CTA
constexpr int kMaxBatch = 8192;  // sequences per call (their prefix sums live in shared memory)
constexpr int kWsHeaderInts = 8; // workspace header: Tr, P, Wr, B, R (+ padding)
constexpr int kHalfBytes = kBox * 128;  // one 64-column half of a box: 16 rows of 128 B
__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct DecodeParams {
    const uint16_t *q;            // bf16 [B, Hq, D]
    const int32_t *block_tables;  // [B, MBS]
    const int32_t *context_lens;  // [B]
    uint16_t *out;                // bf16 [B, Hq, D]
    int32_t *ws_hdr;              // [kWsHeaderInts + B + 1] header + boxes-per-head prefix
    float *ws_part;               // [W][2][G][D + 2] partial (acc[D], max, sum) per worker slot
    int32_t *err_flag;            // nullable
    int B, Hq, Hkv, MBS, bs;
    int NB;
    int stages;                   // pipeline depth chosen on the host to fit shared memory
    float scale_log2;             // scale * log2(e) (FP8 caches: times k_scale)
    float v_scale;                // FP8 caches: dequant scale of V (1 for bf16)
};

struct PrefillParams {
    const uint16_t *q;            // bf16 [Tq, Hq, D]: the sequences' new tokens, concatenated
    uint16_t *out;                // bf16 [Tq, Hq, D]
    const int32_t *block_tables;  // [B, MBS]
    const int32_t *cu_q;          // [B + 1] boundaries of the new tokens
    const int32_t *cu_k;          // [B + 1] boundaries of the contexts (cached + new)
    int32_t *err_flag;            // nullable
    long long Tq;
    int B, Hq, Hkv, MBS, bs, NB;
    int max_q;                    // the caller's bound on q_len (sizes the grid)
    float scale_log2;             // scale * log2(e)
};

// Host launchers (defined next to their kernels).
cudaError_t launch_store(const void *k, const void *v, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int64_t N, int row_bytes,
                         long long n_slots, int32_t *err_flag, cudaStream_t stream);
cudaError_t launch_store_fp8(const void *k, const void *v, void *k_cache, void *v_cache,
                             const int64_t *slot_mapping, int64_t N, int row_elems,
                             long long n_slots, float kinv, float vinv, int32_t *err_flag,
                             cudaStream_t stream);
cudaError_t launch_merge(int D, int G, const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_prefill(int D, int G, const CUtensorMap *tmk, const CUtensorMap *tmv,
                           const PrefillParams &p, dim3 grid, size_t smem, cudaStream_t stream);
const void *prefill_kernel(int D, int G);
size_t prefill_smem_bytes(int D);
constexpr int kPrefillThreads = 8 * 32;  // 7 consumer warps + 1 producer warp
constexpr int kPrefillRows = 112;        // (token, head) rows per CTA

} // namespace pkv
