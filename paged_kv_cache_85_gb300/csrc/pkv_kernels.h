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

// Host launchers (defined next to their kernels).
cudaError_t launch_store(const void *k, const void *v, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int64_t N, int row_bytes,
                         long long n_slots, int32_t *err_flag, cudaStream_t stream);
cudaError_t launch_store_fp8(const void *k, const void *v, void *k_cache, void *v_cache,
                             const int64_t *slot_mapping, int64_t N, int row_elems,
                             long long n_slots, float kinv, float vinv, int32_t *err_flag,
                             cudaStream_t stream);
cudaError_t launch_merge(int D, int G, const DecodeParams &p, cudaStream_t stream);

} // namespace pkv
