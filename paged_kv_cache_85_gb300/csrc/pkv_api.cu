// C ABI of the paged KV-cache decode library: argument checks, partition
// choice, TMA descriptors, grid sizing and kernel launches.  Nothing here
// allocates device memory or synchronises the host.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pkv.h"
#include "pkv_decode.cuh"
#include "pkv_kernels.h"

namespace pkv {
cudaError_t launch_decode_d64(int G, const CUtensorMap *tmk, const CUtensorMap *tmv,
                              const DecodeParams &p, int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_decode_d128(int G, const CUtensorMap *tmk, const CUtensorMap *tmv,
                               const DecodeParams &p, int grid, size_t smem, cudaStream_t stream);
const void *decode_kernel_d64(int G);
const void *decode_kernel_d128(int G);
} // namespace pkv

namespace {

thread_local char g_last_error[512] = "";

pkv_status fail(pkv_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool group_supported(int G) { return G == 1 || G == 2 || G == 4 || G == 8; }

constexpr int kMaxDevices = 64;
constexpr size_t kMaxDynSmem = 227 * 1024;

struct DeviceState {
    bool ready = false;
    int sms = 0;
    bool smem_set[2][9] = {};  // [D == 128][G]
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

pkv_status device_state(DeviceState **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &st = g_dev[dev];
    if (!st.ready) {
        e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return fail(PKV_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        st.ready = true;
    }
    *out = &st;
    return PKV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D view of a cache [NB*bs tokens, Hkv, D] with a box of 16 tokens x 1 head x D.
pkv_status make_cache_map(CUtensorMap *map, const void *cache, long long tokens, int Hkv, int D)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc)
        return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)pkv::kBox};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(cache), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PKV_OK;
}

size_t workspace_bytes_for(int B, int Hq, int D, int S)
{
    if (S <= 1)
        return 0;
    return pkv::align_up((size_t)B * Hq * S * (size_t)(D + 2) * 4, 256);
}

} // namespace

extern "C" {

const char *pkv_last_error(void) { return g_last_error; }

const char *pkv_status_string(pkv_status s)
{
    switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    }
    return "PKV_UNKNOWN_STATUS";
}

int pkv_version(void) { return 100; }

pkv_status pkv_store_kvcache(const void *k, const void *v, void *k_cache, void *v_cache,
                             const int64_t *slot_mapping, int64_t N, int Hkv, int D,
                             int64_t NB, int bs, int32_t *err_flag, void *stream)
{
    if (N < 0 || Hkv < 1 || D < 1 || NB < 1 || bs < 1)
        return fail(PKV_ERR_INVALID_ARG, "store_kvcache: bad sizes N=%lld Hkv=%d D=%d NB=%lld bs=%d",
                    (long long)N, Hkv, D, (long long)NB, bs);
    if (N > 0x7fffffffLL)
        return fail(PKV_ERR_INVALID_ARG, "store_kvcache: N=%lld exceeds 2^31-1", (long long)N);
    if (((long long)Hkv * D) % 8 != 0)
        return fail(PKV_ERR_UNSUPPORTED, "store_kvcache: Hkv*D must be a multiple of 8");
    if (N == 0)
        return PKV_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping)
        return fail(PKV_ERR_INVALID_ARG, "store_kvcache: null pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return fail(PKV_ERR_INVALID_ARG, "store_kvcache: pointers must be 16-byte aligned");
    const long long row_bytes = (long long)Hkv * D * 2;
    if (row_bytes > 0x7fffffffLL)
        return fail(PKV_ERR_INVALID_ARG, "store_kvcache: row too large");
    cudaError_t e = pkv::launch_store(k, v, k_cache, v_cache, slot_mapping, N, (int)row_bytes,
                                      (long long)NB * bs, err_flag,
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "store_kvcache launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

size_t pkv_decode_workspace_bytes(int B, int Hq, int D, int MBS, int bs, int num_splits)
{
    if (B < 0 || Hq < 1 || D < 1 || MBS < 1 || bs < 1 || num_splits < 0)
        return 0;
    int chunk = 0, S = 0;
    pkv::choose_partition(MBS, bs, num_splits, &chunk, &S);
    return workspace_bytes_for(B, Hq, D, S);
}

pkv_status pkv_paged_attn_decode(const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, int MBS,
                                 const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                                 int64_t NB, int bs, float scale, void *out, void *workspace,
                                 size_t workspace_bytes, int num_splits, int32_t *err_flag,
                                 void *stream)
{
    if (B < 0 || Hq < 1 || Hkv < 1 || MBS < 1 || NB < 1 || bs < 1 || num_splits < 0)
        return fail(PKV_ERR_INVALID_ARG,
                    "paged_attn_decode: bad sizes B=%d Hq=%d Hkv=%d MBS=%d NB=%lld bs=%d splits=%d",
                    B, Hq, Hkv, MBS, (long long)NB, bs, num_splits);
    if (Hq % Hkv != 0)
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
    const int G = Hq / Hkv;
    if (!group_supported(G))
        return fail(PKV_ERR_UNSUPPORTED, "paged_attn_decode: Hq/Hkv=%d not in {1,2,4,8}", G);
    if (D != 64 && D != 128)
        return fail(PKV_ERR_UNSUPPORTED, "paged_attn_decode: head_dim %d not in {64,128}", D);
    if (bs % pkv::kBox != 0)
        return fail(PKV_ERR_UNSUPPORTED, "paged_attn_decode: block_size %d not a multiple of 16", bs);
    if ((long long)NB * bs >= 0x7fffffffLL || (long long)MBS * bs >= 0x7fffffffLL)
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: NB*bs and MBS*bs must be < 2^31");
    if (B > pkv::kMaxBatch)
        return fail(PKV_ERR_UNSUPPORTED, "paged_attn_decode: B=%d above %d", B, pkv::kMaxBatch);
    if (!std::isfinite(scale))
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: scale is not finite");
    if (B == 0)
        return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: null pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        !aligned16(workspace) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: misaligned pointer");

    int chunk = 0, S = 0;
    pkv::choose_partition(MBS, bs, num_splits, &chunk, &S);
    const size_t need = workspace_bytes_for(B, Hq, D, S);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(PKV_ERR_WORKSPACE, "paged_attn_decode: workspace needs %zu bytes, got %zu", need,
                    workspace ? workspace_bytes : (size_t)0);

    const size_t smem = pkv::decode_smem_layout(D, G, D == 128 ? pkv::DecodeShape<128>::kStages
                                                               : pkv::DecodeShape<64>::kStages,
                                                B, S)
                            .total;
    if (smem > kMaxDynSmem)
        return fail(PKV_ERR_UNSUPPORTED,
                    "paged_attn_decode: B=%d with %d partitions needs %zu B of shared memory", B, S,
                    smem);

    DeviceState *st = nullptr;
    pkv_status ps = device_state(&st);
    if (ps != PKV_OK)
        return ps;
    const void *kfn = D == 128 ? pkv::decode_kernel_d128(G) : pkv::decode_kernel_d64(G);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        bool &set = st->smem_set[D == 128][G];
        if (!set) {
            cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kMaxDynSmem);
            if (e != cudaSuccess)
                return fail(PKV_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            set = true;
        }
    }
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kfn, pkv::kDecodeThreads, smem);
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "occupancy query: %s", cudaGetErrorString(e));
    if (occ < 1)
        return fail(PKV_ERR_UNSUPPORTED, "paged_attn_decode: kernel does not fit on an SM");

    const long long units_max = (long long)B * Hkv * S;
    long long grid = (long long)st->sms * occ;
    if (grid > units_max)
        grid = units_max;

    CUtensorMap tmk, tmv;
    const long long tokens = (long long)NB * bs;
    if ((ps = make_cache_map(&tmk, k_cache, tokens, Hkv, D)) != PKV_OK)
        return ps;
    if ((ps = make_cache_map(&tmv, v_cache, tokens, Hkv, D)) != PKV_OK)
        return ps;

    pkv::DecodeParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = static_cast<uint16_t *>(out);
    p.ws_acc = S > 1 ? static_cast<float *>(workspace) : nullptr;
    p.ws_ml = S > 1 ? static_cast<float *>(workspace) + (size_t)B * Hq * S * D : nullptr;
    p.err_flag = err_flag;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.MBS = MBS;
    p.bs = bs;
    p.chunk = chunk;
    p.S = S;
    p.NB = (int)NB;
    p.scale_log2 = scale * 1.4426950408889634f;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = D == 128 ? pkv::launch_decode_d128(G, &tmk, &tmv, p, (int)grid, smem, s)
                 : pkv::launch_decode_d64(G, &tmk, &tmv, p, (int)grid, smem, s);
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "paged_attn_decode launch: %s", cudaGetErrorString(e));
    e = pkv::launch_merge(D, p, s);
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

} // extern "C"
