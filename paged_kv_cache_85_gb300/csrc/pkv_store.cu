// store_kvcache: scatter the step's new K/V rows into the block-paged cache.
//
// MinivLLM guide "HowToApproachvLLM", section 4.5: slot_mapping names, for
// each new token only, the flat cache slot its K/V go to; the decode slot is
// block_table[-1]*block_size + last_block_num_tokens - 1.  Section 4.6: the
// padded entries of a CUDA-graph batch carry a sentinel (-1 here) and are
// skipped.  With the cache laid out as [NB, bs, Hkv, D], a slot's Hkv*D
// values are one contiguous row, so the scatter is a row copy.
//
// One CTA per new token copies its K row and V row with 16-byte vector
// loads/stores; the row is Hkv*D*2 bytes (2 KB for 8 KV heads x 128).
#include "pkv_kernels.h"
#include "pkv_ptx.cuh"

namespace pkv {

constexpr int kStoreThreads = 128;

__global__ void __launch_bounds__(kStoreThreads)
    store_kvcache_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                         uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                         const int64_t *__restrict__ slot_mapping, int row16, long long n_slots,
                         int32_t *err_flag)
{
    grid_launch_dependents();
    const int64_t i = blockIdx.x;
    const int64_t slot = __ldg(slot_mapping + i);
    if (slot == -1)
        return;
    if (slot < 0 || slot >= n_slots) {
        if (threadIdx.x == 0)
            flag_error(err_flag, 0x1 /* PKV_FLAG_BAD_SLOT */);
        return;
    }
    const uint4 *ks = k + i * row16;
    const uint4 *vs = v + i * row16;
    uint4 *kd = k_cache + slot * row16;
    uint4 *vd = v_cache + slot * row16;
    // The new rows are inputs no earlier kernel writes: fetch the first chunk
    // before waiting on the previous kernels, which may still read the cache.
    uint4 a0 = make_uint4(0, 0, 0, 0), b0 = a0;
    if ((int)threadIdx.x < row16) {
        a0 = __ldg(ks + threadIdx.x);
        b0 = __ldg(vs + threadIdx.x);
    }
    grid_dependency_wait();
    if ((int)threadIdx.x < row16) {
        kd[threadIdx.x] = a0;
        vd[threadIdx.x] = b0;
    }
    for (int c = threadIdx.x + kStoreThreads; c < row16; c += kStoreThreads) {
        const uint4 a = __ldg(ks + c);
        const uint4 b = __ldg(vs + c);
        kd[c] = a;
        vd[c] = b;
    }
}

// FP8 variant ("VLLM-0.7.3 源码" section 5.3: the KV cache stored in FP8 via
// kv_cache_dtype): every bf16 value is widened, multiplied by the reciprocal
// of its tensor's scale in fp32, and encoded as OCP E4M3 (nearest even,
// finite saturation).  One thread turns 8 values (16 B) into 8 codes (8 B).
__device__ __forceinline__ uint2 quantize8(uint4 a, float inv)
{
    const float2 f0 = bf16x2_to_float2(a.x), f1 = bf16x2_to_float2(a.y);
    const float2 f2 = bf16x2_to_float2(a.z), f3 = bf16x2_to_float2(a.w);
    const uint32_t c0 = f32x2_to_e4m3x2(__fmul_rn(f0.x, inv), __fmul_rn(f0.y, inv));
    const uint32_t c1 = f32x2_to_e4m3x2(__fmul_rn(f1.x, inv), __fmul_rn(f1.y, inv));
    const uint32_t c2 = f32x2_to_e4m3x2(__fmul_rn(f2.x, inv), __fmul_rn(f2.y, inv));
    const uint32_t c3 = f32x2_to_e4m3x2(__fmul_rn(f3.x, inv), __fmul_rn(f3.y, inv));
    return make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
}

__global__ void __launch_bounds__(kStoreThreads)
    store_kvcache_fp8_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                             uint2 *__restrict__ k_cache, uint2 *__restrict__ v_cache,
                             const int64_t *__restrict__ slot_mapping, int row8, long long n_slots,
                             float kinv, float vinv, int32_t *err_flag)
{
    grid_launch_dependents();
    const int64_t i = blockIdx.x;
    const int64_t slot = __ldg(slot_mapping + i);
    if (slot == -1)
        return;
    if (slot < 0 || slot >= n_slots) {
        if (threadIdx.x == 0)
            flag_error(err_flag, 0x1 /* PKV_FLAG_BAD_SLOT */);
        return;
    }
    const uint4 *ks = k + i * row8;
    const uint4 *vs = v + i * row8;
    uint2 *kd = k_cache + slot * row8;
    uint2 *vd = v_cache + slot * row8;
    uint4 a0 = make_uint4(0, 0, 0, 0), b0 = a0;
    if ((int)threadIdx.x < row8) {
        a0 = __ldg(ks + threadIdx.x);
        b0 = __ldg(vs + threadIdx.x);
    }
    grid_dependency_wait();  // the cache may still be read by earlier kernels
    if ((int)threadIdx.x < row8) {
        kd[threadIdx.x] = quantize8(a0, kinv);
        vd[threadIdx.x] = quantize8(b0, vinv);
    }
    for (int c = threadIdx.x + kStoreThreads; c < row8; c += kStoreThreads) {
        kd[c] = quantize8(__ldg(ks + c), kinv);
        vd[c] = quantize8(__ldg(vs + c), vinv);
    }
}

cudaError_t launch_store_fp8(const void *k, const void *v, void *k_cache, void *v_cache,
                             const int64_t *slot_mapping, int64_t N, int row_elems,
                             long long n_slots, float kinv, float vinv, int32_t *err_flag,
                             cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)N);
    cfg.blockDim = dim3(kStoreThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, store_kvcache_fp8_kernel, static_cast<const uint4 *>(k),
                              static_cast<const uint4 *>(v), static_cast<uint2 *>(k_cache),
                              static_cast<uint2 *>(v_cache), slot_mapping, row_elems / 8, n_slots,
                              kinv, vinv, err_flag);
}

cudaError_t launch_store(const void *k, const void *v, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int64_t N, int row_bytes,
                         long long n_slots, int32_t *err_flag, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)N);
    cfg.blockDim = dim3(kStoreThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, store_kvcache_kernel, static_cast<const uint4 *>(k),
                              static_cast<const uint4 *>(v), static_cast<uint4 *>(k_cache),
                              static_cast<uint4 *>(v_cache), slot_mapping, row_bytes / 16,
                              n_slots, err_flag);
}

} // namespace pkv
