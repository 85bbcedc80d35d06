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
