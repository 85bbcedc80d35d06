// C ABI of the paged KV-cache decode library: argument checks, launch
// planning, TMA descriptors, grid sizing and kernel launches.  Nothing here
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
#include "pkv_prefill.h"
#include "pkv_prefill_tc.cuh"

namespace pkv {
#define PKV_DECLARE_SHAPE(D, NW)                                                                  \
    cudaError_t launch_decode_d##D##_w##NW(int G, const CUtensorMap *tmk, const CUtensorMap *tmv, \
                                           const DecodeParams &p, int grid, size_t smem,          \
                                           cudaStream_t stream);                                  \
    const void *decode_kernel_d##D##_w##NW(int G);
PKV_DECLARE_SHAPE(64, 4)
PKV_DECLARE_SHAPE(64, 8)
PKV_DECLARE_SHAPE(128, 4)
PKV_DECLARE_SHAPE(128, 8)
#undef PKV_DECLARE_SHAPE
#define PKV_DECLARE_SHAPE8(D, NW)                                                                 \
    cudaError_t launch_decode8_d##D##_w##NW(int G, int bt, const CUtensorMap *tmk,                \
                                            const CUtensorMap *tmv, const DecodeParams &p,        \
                                            int grid, size_t smem, cudaStream_t stream);          \
    const void *decode_kernel8_d##D##_w##NW(int G, int bt);
PKV_DECLARE_SHAPE8(64, 4)
PKV_DECLARE_SHAPE8(64, 8)
PKV_DECLARE_SHAPE8(128, 4)
PKV_DECLARE_SHAPE8(128, 8)
#undef PKV_DECLARE_SHAPE8
cudaError_t launch_prefill_d64(int G, const CUtensorMap *tmq, const CUtensorMap *tmk,
                               const CUtensorMap *tmv, const PrefillParams &p, dim3 grid,
                               size_t smem, cudaStream_t stream);
cudaError_t launch_prefill_d128(int G, const CUtensorMap *tmq, const CUtensorMap *tmk,
                                const CUtensorMap *tmv, const PrefillParams &p, dim3 grid,
                                size_t smem, cudaStream_t stream);
const void *prefill_kernel_d64(int G);
const void *prefill_kernel_d128(int G);

cudaError_t launch_prefill(int D, int G, const CUtensorMap *tmq, const CUtensorMap *tmk,
                           const CUtensorMap *tmv, const PrefillParams &p, dim3 grid, size_t smem,
                           cudaStream_t stream)
{
    return D == 128 ? launch_prefill_d128(G, tmq, tmk, tmv, p, grid, smem, stream)
                    : launch_prefill_d64(G, tmq, tmk, tmv, p, grid, smem, stream);
}

const void *prefill_kernel(int D, int G)
{
    return D == 128 ? prefill_kernel_d128(G) : prefill_kernel_d64(G);
}

size_t prefill_smem_bytes(int D) { return tc_smem_layout(D).total; }

// bt: tokens per box (16, or 32 for FP8 caches with block sizes divisible by 32)
const void *decode_kernel(int D, int NW, int G, bool f8, int bt)
{
    const bool pair = NW == kPairWorkers;
    if (f8) {
        if (D == 128)
            return pair ? decode_kernel8_d128_w4(G, bt) : decode_kernel8_d128_w8(G, bt);
        return pair ? decode_kernel8_d64_w4(G, bt) : decode_kernel8_d64_w8(G, bt);
    }
    if (D == 128)
        return pair ? decode_kernel_d128_w4(G) : decode_kernel_d128_w8(G);
    return pair ? decode_kernel_d64_w4(G) : decode_kernel_d64_w8(G);
}

cudaError_t launch_decode(int D, int NW, int G, bool f8, int bt, const CUtensorMap *tmk,
                          const CUtensorMap *tmv, const DecodeParams &p, int grid, size_t smem,
                          cudaStream_t stream)
{
    const bool pair = NW == kPairWorkers;
    if (f8) {
        if (D == 128)
            return pair ? launch_decode8_d128_w4(G, bt, tmk, tmv, p, grid, smem, stream)
                        : launch_decode8_d128_w8(G, bt, tmk, tmv, p, grid, smem, stream);
        return pair ? launch_decode8_d64_w4(G, bt, tmk, tmv, p, grid, smem, stream)
                    : launch_decode8_d64_w8(G, bt, tmk, tmv, p, grid, smem, stream);
    }
    if (D == 128)
        return pair ? launch_decode_d128_w4(G, tmk, tmv, p, grid, smem, stream)
                    : launch_decode_d128_w8(G, tmk, tmv, p, grid, smem, stream);
    return pair ? launch_decode_d64_w4(G, tmk, tmv, p, grid, smem, stream)
                : launch_decode_d64_w8(G, tmk, tmv, p, grid, smem, stream);
}
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
constexpr long long kMaxWorkersTotal = 2048;  // workers of one decode launch (256 SMs x 8)
using pkv::kMaxDynSmem;

struct DeviceState {
    bool ready = false;
    int dev = 0;
    int sms = 0;
    bool smem_set[2][2][2][2][9] = {};  // [fp8][32-token boxes][D == 128][NW == 8][G]
    bool pf_smem_set[2][9] = {};     // prefill: [D == 128][G]
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
        st.dev = dev;
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

// Occupancy per (kernel, dynamic shared memory), cached: the query is pure
// host arithmetic but not free, and decode calls repeat the same shapes.
struct OccEntry {
    const void *fn = nullptr;
    size_t smem = 0;
    int occ = 0;
};
constexpr int kOccCache = 32;
OccEntry g_occ[kMaxDevices][kOccCache];

pkv_status occupancy(int dev, const void *fn, int threads, size_t smem, int *occ)
{
    std::lock_guard<std::mutex> lk(g_mu);
    OccEntry *slot = nullptr;
    for (auto &e : g_occ[dev]) {
        if (e.fn == fn && e.smem == smem) {
            *occ = e.occ;
            return PKV_OK;
        }
        if (!e.fn && !slot)
            slot = &e;
    }
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "occupancy query: %s", cudaGetErrorString(e));
    if (slot) {
        slot->fn = fn;
        slot->smem = smem;
        slot->occ = n;
    }
    *occ = n;
    return PKV_OK;
}

// 4-D view of a cache [NB*bs tokens, Hkv, D] as (64 columns, D/64 halves,
// Hkv, tokens); a box is 64 columns x 1 half x 1 head x 16 tokens, landing as
// 16 rows of 128 B with the 128-byte swizzle (conflict-free ldmatrix reads).
pkv_status make_cache_map(CUtensorMap *map, const void *cache, long long tokens, int Hkv, int D)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc)
        return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[4] = {64, (cuuint64_t)(D / 64), (cuuint64_t)Hkv, (cuuint64_t)tokens};
    cuuint64_t strides[3] = {128, (cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
    cuuint32_t box[4] = {64, 1, 1, (cuuint32_t)pkv::kBox};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(cache), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PKV_OK;
}

// The same cache for the prefill kernel's copies of both halves at once: 4-D
// (64 columns, tokens, Hkv, D/64 halves), box 64 x rows x 1 x D/64, landing as
// the halves one after the other, each `rows` rows of 128 B with the 128-byte
// swizzle.  rows = 64: a whole K or V tile where a block holds whole 64-token
// tiles (bs % 64 == 0); rows = 16: one 16-token box of a V tile.
pkv_status make_cache_tile_map(CUtensorMap *map, const void *cache, long long tokens, int Hkv, int D,
                               int rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc)
        return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[4] = {64, (cuuint64_t)tokens, (cuuint64_t)Hkv, (cuuint64_t)(D / 64)};
    cuuint64_t strides[3] = {(cuuint64_t)Hkv * D * 2, (cuuint64_t)D * 2, 128};
    cuuint32_t box[4] = {64, (cuuint32_t)rows, 1, (cuuint32_t)(D / 64)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(cache), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (tile) failed (%d)", (int)r);
    return PKV_OK;
}

// Prefill queries q [Tq, Hq, D] bf16 as 4-D (64, D/64, Hq, Tq) like the cache;
// box 64 x 1 x G x 128/G: one 128-row (token, head) tile half per copy.
pkv_status make_q_map(CUtensorMap *map, const void *q, long long Tq, int Hq, int D, int G)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc)
        return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[4] = {64, (cuuint64_t)(D / 64), (cuuint64_t)Hq, (cuuint64_t)Tq};
    cuuint64_t strides[3] = {128, (cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)G, (cuuint32_t)(pkv::kPrefillRows / G)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(q), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (q) failed (%d)", (int)r);
    return PKV_OK;
}

// FP8 cache [NB*bs tokens, Hkv, D] as bytes: 3-D (D, Hkv, tokens), box
// D x 1 x rows (16 or 32 tokens), swizzled at the row width (128-byte rows
// for D = 128, 64-byte rows for D = 64).
pkv_status make_cache_map8(CUtensorMap *map, const void *cache, long long tokens, int Hkv, int D,
                           int rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc)
        return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)D, (cuuint64_t)Hkv * D};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(cache), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (fp8) failed (%d)", (int)r);
    return PKV_OK;
}

// Tensor maps of recently used caches, per host thread (a map is plain data:
// the same cache pointer and shape always encode the same map).
// Map kinds: 16-token boxes of a bf16 cache (one half per copy), 16- or
// 32-token boxes of an FP8 cache, or, for the prefill kernel, whole 64-token
// tiles or 16-token boxes of a bf16 cache with both halves per copy.
enum MapKind { kMapBox = 0, kMapBox8 = 1, kMapTile = 2, kMapBoxHalves = 3, kMapBox8Wide = 4 };
struct MapEntry {
    const void *ptr = nullptr;
    long long tokens = 0;
    int Hkv = 0, D = 0;
    int kind = kMapBox;
    CUtensorMap map;
};
constexpr int kMapCache = 8;
thread_local MapEntry t_maps[kMapCache];
thread_local int t_map_next = 0;

pkv_status cached_cache_map(CUtensorMap *map, const void *cache, long long tokens, int Hkv, int D,
                            int kind = kMapBox)
{
    for (const auto &e : t_maps)
        if (e.ptr == cache && e.tokens == tokens && e.Hkv == Hkv && e.D == D && e.kind == kind) {
            *map = e.map;
            return PKV_OK;
        }
    const pkv_status ps = kind == kMapBox8   ? make_cache_map8(map, cache, tokens, Hkv, D, pkv::kBox)
                          : kind == kMapBox8Wide ? make_cache_map8(map, cache, tokens, Hkv, D, 2 * pkv::kBox)
                          : kind == kMapTile ? make_cache_tile_map(map, cache, tokens, Hkv, D, pkv::kPrefillKeys)
                          : kind == kMapBoxHalves ? make_cache_tile_map(map, cache, tokens, Hkv, D, pkv::kBox)
                                                  : make_cache_map(map, cache, tokens, Hkv, D);
    if (ps != PKV_OK)
        return ps;
    MapEntry &e = t_maps[t_map_next];
    t_map_next = (t_map_next + 1) % kMapCache;
    e.ptr = cache;
    e.tokens = tokens;
    e.Hkv = Hkv;
    e.D = D;
    e.kind = kind;
    e.map = *map;
    return PKV_OK;
}

// Launch plan of one decode call: pipeline depth, shared memory, grid and
// workspace layout.  The workspace query and the launch share it, so they
// always agree.
struct DecodePlan {
    int G = 0, NW = 0, stages = 0, grid = 0;
    int bt = pkv::kBox;  // tokens per box
    size_t smem = 0, hdr_bytes = 0, ws_bytes = 0;
    const void *kernel = nullptr;
};

pkv_status plan_decode(int B, int Hq, int Hkv, int D, int MBS, int bs, int max_ctas,
                       bool with_device, DecodePlan *plan, bool f8 = false)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || MBS < 1 || bs < 1 || max_ctas < 0)
        return fail(PKV_ERR_INVALID_ARG,
                    "paged_attn_decode: bad sizes B=%d Hq=%d Hkv=%d MBS=%d bs=%d max_ctas=%d", B, Hq,
                    Hkv, MBS, bs, max_ctas);
    if (Hq % Hkv != 0)
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
    const int G = Hq / Hkv;
    if (!group_supported(G))
        return fail(PKV_ERR_UNSUPPORTED, "paged_attn_decode: Hq/Hkv=%d not in {1,2,4,8}", G);
    if (D != 64 && D != 128)
        return fail(PKV_ERR_UNSUPPORTED, "paged_attn_decode: head_dim %d not in {64,128}", D);
    if (bs % pkv::kBox != 0)
        return fail(PKV_ERR_UNSUPPORTED, "paged_attn_decode: block_size %d not a multiple of 16", bs);
    if (B > pkv::kMaxBatch)
        return fail(PKV_ERR_UNSUPPORTED, "paged_attn_decode: B=%d above %d", B, pkv::kMaxBatch);
    if ((long long)MBS * bs >= 0x7fffffffLL)
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: MBS*bs must be < 2^31");
    const long long box_max = (long long)B * Hkv * (((long long)MBS * bs + pkv::kBox - 1) / pkv::kBox);
    if (box_max >= 0x7fffffffLL)
        return fail(PKV_ERR_UNSUPPORTED, "paged_attn_decode: B*Hkv*MBS*bs/16 must be < 2^31");
    // Prefer 4-worker CTAs, three per SM for FP8 caches (their kernels are
    // built for three; up to four stages where they fit, since the FP8 path
    // is bound by the bytes its copies keep in flight) and two for bf16; fall
    // back to one 8-worker CTA per SM when they do not fit (large B, or G = 8
    // with D = 128).
    const size_t pair_smem = pkv::kSmemPerSm / 2 - pkv::kSmemReserve;
    const size_t trio_smem = pkv::kSmemPerSm / 3 - pkv::kSmemReserve;
    const int eb = f8 ? 1 : 2;  // bytes per cached element
    int NW = pkv::kPairWorkers;
    int stages = 0;
    int bt = pkv::kBox;
    if (f8) {
        stages = pkv::decode_stages_for(D, G, NW, B, pkv::kMaxStages, trio_smem, eb);
        // Where three CTAs per SM hold fewer than four stages of 16-token
        // boxes (large B or G), and the blocks hold whole 32-token boxes, two
        // stages of 32-token boxes keep as many bytes in flight while one is
        // consumed, with half the boxes (stage waits, descriptors, softmax
        // reductions) per byte.  With four 16-token stages the deeper ring
        // wins (measured).
        if (stages < pkv::kMaxStages && bs % (2 * pkv::kBox) == 0) {
            const int s32 = pkv::decode_stages_for(D, G, NW, B, pkv::kMaxStages, trio_smem, eb,
                                                   2 * pkv::kBox);
            if (s32 >= pkv::kMinStages) {
                bt = 2 * pkv::kBox;
                stages = s32;
            }
        }
    }
    if (bt == pkv::kBox && stages < pkv::kPairStages)
        stages = pkv::decode_stages_for(D, G, NW, B, pkv::kPairStages, pair_smem, eb);
    if (bt == pkv::kBox && stages < pkv::kPairStages) {
        NW = pkv::kWideWorkers;
        stages = pkv::decode_stages_for(D, G, NW, B, pkv::kMaxStages, kMaxDynSmem, eb);
    }
    if (stages == 0)
        return fail(PKV_ERR_UNSUPPORTED, "paged_attn_decode: B=%d does not fit shared memory", B);
    // The workspace is sized for the largest grid the launch may use, which
    // depends only on the arguments: no more CTAs than the boxes can keep
    // busy, at most kMaxWorkersTotal workers, and at most max_ctas.
    long long grid_cap = (box_max + NW - 1) / NW;
    if (grid_cap > kMaxWorkersTotal / NW)
        grid_cap = kMaxWorkersTotal / NW;
    if (max_ctas > 0 && grid_cap > max_ctas)
        grid_cap = max_ctas;
    if (grid_cap < 1)
        grid_cap = 1;
    // Partial slots: bounded for either CTA shape (and either cache type) by
    // boxes + 7, by kMaxWorkersTotal, and by max_ctas CTAs of 8 workers.
    long long workers_cap = box_max + pkv::kWideWorkers - 1;
    if (workers_cap > kMaxWorkersTotal)
        workers_cap = kMaxWorkersTotal;
    if (max_ctas > 0 && workers_cap > (long long)max_ctas * pkv::kWideWorkers)
        workers_cap = (long long)max_ctas * pkv::kWideWorkers;
    plan->G = G;
    plan->NW = NW;
    plan->stages = stages;
    plan->bt = bt;
    plan->smem = pkv::decode_smem_layout(D, G, NW, stages, B, eb, bt).total;
    plan->hdr_bytes = pkv::align_up((size_t)(pkv::kWsHeaderInts + B + 1) * 4, 256);
    plan->ws_bytes = plan->hdr_bytes +
                     (size_t)workers_cap * 2 * G * (size_t)(D + 4) * sizeof(float);
    plan->grid = (int)grid_cap;
    if (!with_device)
        return PKV_OK;
    DeviceState *st = nullptr;
    pkv_status ps = device_state(&st);
    if (ps != PKV_OK)
        return ps;
    const void *kfn = pkv::decode_kernel(D, NW, G, f8, bt);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        bool &set = st->smem_set[f8][bt != pkv::kBox][D == 128][NW == pkv::kWideWorkers][G];
        if (!set) {
            cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kMaxDynSmem);
            if (e != cudaSuccess)
                return fail(PKV_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            set = true;
        }
    }
    int occ = 0;
    if ((ps = occupancy(st->dev, kfn, (NW + 1) * 32, plan->smem, &occ)) != PKV_OK)
        return ps;
    if (occ < 1)
        return fail(PKV_ERR_UNSUPPORTED, "paged_attn_decode: kernel does not fit on an SM");
    const long long resident = (long long)st->sms * occ;
    if (resident < plan->grid)
        plan->grid = (int)resident;
    plan->kernel = kfn;
    return PKV_OK;
}

} // namespace

namespace pkv {
// Record a message for pkv_last_error() from another translation unit.
pkv_status report_error(pkv_status s, const char *msg)
{
    return fail(s, "%s", msg);
}
} // namespace pkv

static pkv_status decode_impl(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int MBS, const int32_t *context_lens,
                              int B, int Hq, int Hkv, int D, int64_t NB, int bs, float scale,
                              void *out, void *workspace, size_t workspace_bytes, int max_ctas,
                              int32_t *err_flag, void *stream, bool f8, float k_scale,
                              float v_scale)
{
    if (B < 0 || NB < 1)
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: bad sizes B=%d NB=%lld", B, (long long)NB);
    if (!std::isfinite(scale))
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: scale is not finite");
    if (B == 0) {
        // validate the remaining sizes even though there is nothing to do
        if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
            return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: bad head counts");
        return PKV_OK;
    }
    if ((long long)NB * bs >= 0x7fffffffLL)
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: NB*bs must be < 2^31");
    DecodePlan plan;
    if (f8 && (!std::isfinite(k_scale) || !std::isfinite(v_scale) || k_scale <= 0.f ||
               v_scale <= 0.f))
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode_fp8: scales must be finite and > 0");
    pkv_status ps = plan_decode(B, Hq, Hkv, D, MBS, bs, max_ctas, true, &plan, f8);
    if (ps != PKV_OK)
        return ps;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: null pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        !aligned16(workspace) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode: misaligned pointer");
    if (!workspace || workspace_bytes < plan.ws_bytes)
        return fail(PKV_ERR_WORKSPACE, "paged_attn_decode: workspace needs %zu bytes, got %zu",
                    plan.ws_bytes, workspace ? workspace_bytes : (size_t)0);

    CUtensorMap tmk, tmv;
    const long long tokens = (long long)NB * bs;
    const int kind = !f8 ? kMapBox : plan.bt == pkv::kBox ? kMapBox8 : kMapBox8Wide;
    if ((ps = cached_cache_map(&tmk, k_cache, tokens, Hkv, D, kind)) != PKV_OK)
        return ps;
    if ((ps = cached_cache_map(&tmv, v_cache, tokens, Hkv, D, kind)) != PKV_OK)
        return ps;

    pkv::DecodeParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = static_cast<uint16_t *>(out);
    p.ws_hdr = static_cast<int32_t *>(workspace);
    p.ws_part = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + plan.hdr_bytes);
    p.err_flag = err_flag;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.MBS = MBS;
    p.bs = bs;
    p.NB = (int)NB;
    p.stages = plan.stages;
    p.scale_log2 = scale * 1.4426950408889634f * (f8 ? k_scale : 1.f);
    p.v_scale = f8 ? v_scale : 1.f;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = pkv::launch_decode(D, plan.NW, plan.G, f8, plan.bt, &tmk, &tmv, p, plan.grid,
                                       plan.smem, s);
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "paged_attn_decode launch: %s", cudaGetErrorString(e));
    e = pkv::launch_merge(D, plan.G, p, s);
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}


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

size_t pkv_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int MBS, int bs, int max_ctas)
{
    DecodePlan plan;
    if (B == 0 || plan_decode(B, Hq, Hkv, D, MBS, bs, max_ctas, false, &plan) != PKV_OK)
        return 0;
    return plan.ws_bytes;
}

pkv_status pkv_paged_attn_decode(const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, int MBS,
                                 const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                                 int64_t NB, int bs, float scale, void *out, void *workspace,
                                 size_t workspace_bytes, int max_ctas, int32_t *err_flag,
                                 void *stream)
{
    return decode_impl(q, k_cache, v_cache, block_tables, MBS, context_lens, B, Hq, Hkv, D, NB, bs,
                       scale, out, workspace, workspace_bytes, max_ctas, err_flag, stream, false,
                       1.f, 1.f);
}

pkv_status pkv_paged_attn_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *block_tables, int MBS,
                                     const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                                     int64_t NB, int bs, float scale, float k_scale,
                                     float v_scale, void *out, void *workspace,
                                     size_t workspace_bytes, int max_ctas, int32_t *err_flag,
                                     void *stream)
{
    return decode_impl(q, k_cache, v_cache, block_tables, MBS, context_lens, B, Hq, Hkv, D, NB, bs,
                       scale, out, workspace, workspace_bytes, max_ctas, err_flag, stream, true,
                       k_scale, v_scale);
}

pkv_status pkv_paged_prefill(const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, int MBS, const int32_t *cu_seqlens_q,
                             const int32_t *cu_seqlens_k, int B, int64_t Tq, int max_seqlen_q,
                             int Hq, int Hkv, int D, int64_t NB, int bs, float scale, void *out,
                             int32_t *err_flag, void *stream)
{
    if (B < 0 || Tq < 0 || max_seqlen_q < 0 || NB < 1 || MBS < 1 || bs < 1 || Hq < 1 || Hkv < 1)
        return fail(PKV_ERR_INVALID_ARG, "paged_prefill: bad sizes B=%d Tq=%lld max_seqlen_q=%d "
                    "NB=%lld MBS=%d bs=%d Hq=%d Hkv=%d", B, (long long)Tq, max_seqlen_q,
                    (long long)NB, MBS, bs, Hq, Hkv);
    if (Hq % Hkv != 0)
        return fail(PKV_ERR_INVALID_ARG, "paged_prefill: Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
    const int G = Hq / Hkv;
    if (!group_supported(G))
        return fail(PKV_ERR_UNSUPPORTED, "paged_prefill: Hq/Hkv=%d not in {1,2,4,8}", G);
    if (D != 64 && D != 128)
        return fail(PKV_ERR_UNSUPPORTED, "paged_prefill: head_dim %d not in {64,128}", D);
    if (bs % pkv::kBox != 0)
        return fail(PKV_ERR_UNSUPPORTED, "paged_prefill: block_size %d not a multiple of 16", bs);
    if (!std::isfinite(scale))
        return fail(PKV_ERR_INVALID_ARG, "paged_prefill: scale is not finite");
    if ((long long)NB * bs >= 0x7fffffffLL || (long long)MBS * bs >= 0x7fffffffLL)
        return fail(PKV_ERR_INVALID_ARG, "paged_prefill: NB*bs and MBS*bs must be < 2^31");
    if (Tq >= 0x7fffffffLL || B > 65535)
        return fail(PKV_ERR_UNSUPPORTED, "paged_prefill: Tq must be < 2^31 and B <= 65535");
    if (B == 0 || Tq == 0 || max_seqlen_q == 0)
        return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !cu_seqlens_q || !cu_seqlens_k || !out)
        return fail(PKV_ERR_INVALID_ARG, "paged_prefill: null pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) ||
        (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
        return fail(PKV_ERR_INVALID_ARG, "paged_prefill: misaligned pointer");
    // work items: pairs of adjacent 128-row query tiles of one sequence and KV head
    const long long pairs =
        ((long long)max_seqlen_q * G + 2 * pkv::kPrefillRows - 1) / (2 * pkv::kPrefillRows);
    if (pairs * Hkv * B > 0x7fffffffLL)
        return fail(PKV_ERR_UNSUPPORTED, "paged_prefill: query tile pairs x Hkv x B must be < 2^31");

    DeviceState *st = nullptr;
    pkv_status ps = device_state(&st);
    if (ps != PKV_OK)
        return ps;
    const void *kfn = pkv::prefill_kernel(D, G);
    const size_t smem = pkv::prefill_smem_bytes(D);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        bool &set = st->pf_smem_set[D == 128][G];
        if (!set) {
            cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess)
                return fail(PKV_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            set = true;
        }
    }
    CUtensorMap tmq, tmk, tmv;
    const long long tokens = (long long)NB * bs;
    // blocks of whole 64-token tiles: one copy per K or V tile; else K one
    // copy per 16-token box and 64-column half, V one per box
    const bool tile_copies = bs % pkv::kPrefillKeys == 0;
    if ((ps = cached_cache_map(&tmk, k_cache, tokens, Hkv, D, tile_copies ? kMapTile : kMapBox)) != PKV_OK)
        return ps;
    if ((ps = cached_cache_map(&tmv, v_cache, tokens, Hkv, D, tile_copies ? kMapTile : kMapBoxHalves)) !=
        PKV_OK)
        return ps;
    if ((ps = make_q_map(&tmq, q, Tq, Hq, D, G)) != PKV_OK)
        return ps;
    pkv::PrefillParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.out = static_cast<uint16_t *>(out);
    p.block_tables = block_tables;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.err_flag = err_flag;
    p.Tq = Tq;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.MBS = MBS;
    p.bs = bs;
    p.NB = (int)NB;
    p.max_q = max_seqlen_q;
    p.X = (int)pairs;
    p.n_items = (int)(pairs * Hkv * B);
    p.scale_log2 = std::fabs(scale) * 1.4426950408889634f;
    p.neg_scale = scale < 0.f;
    p.tile_copies = tile_copies ? 1 : 0;
    // Persistent grid: one CTA per SM (each holds all of the SM's TMEM
    // columns, and asks for more than half of its shared memory so that no
    // second CTA lands beside it), each walking its share of the work items.
    static_assert(pkv::kPrefillThreads * 168 <= 65536, "prefill registers per thread");
    long long grid = (long long)st->sms;
    if (grid > p.n_items)
        grid = p.n_items;
    if (grid < 1)
        return PKV_OK;
    cudaError_t e = pkv::launch_prefill(D, G, &tmq, &tmk, &tmv, p, dim3((unsigned)grid),
                                        smem, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "paged_prefill launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

pkv_status pkv_store_kvcache_fp8(const void *k, const void *v, void *k_cache, void *v_cache,
                                 const int64_t *slot_mapping, int64_t N, int Hkv, int D,
                                 int64_t NB, int bs, float k_scale, float v_scale,
                                 int32_t *err_flag, void *stream)
{
    if (N < 0 || Hkv < 1 || D < 1 || NB < 1 || bs < 1)
        return fail(PKV_ERR_INVALID_ARG, "store_kvcache_fp8: bad sizes");
    if (N > 0x7fffffffLL)
        return fail(PKV_ERR_INVALID_ARG, "store_kvcache_fp8: N exceeds 2^31-1");
    if (((long long)Hkv * D) % 16 != 0)
        return fail(PKV_ERR_UNSUPPORTED, "store_kvcache_fp8: Hkv*D must be a multiple of 16");
    if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || k_scale <= 0.f || v_scale <= 0.f)
        return fail(PKV_ERR_INVALID_ARG, "store_kvcache_fp8: scales must be finite and > 0");
    if (N == 0)
        return PKV_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping)
        return fail(PKV_ERR_INVALID_ARG, "store_kvcache_fp8: null pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return fail(PKV_ERR_INVALID_ARG, "store_kvcache_fp8: pointers must be 16-byte aligned");
    const long long row = (long long)Hkv * D;
    if (row > 0x7fffffffLL)
        return fail(PKV_ERR_INVALID_ARG, "store_kvcache_fp8: row too large");
    // The reciprocal is formed once here in IEEE fp32, so the kernel's
    // products are exactly x * (1 / scale) rounded once.
    const float kinv = 1.0f / k_scale, vinv = 1.0f / v_scale;
    cudaError_t e = pkv::launch_store_fp8(k, v, k_cache, v_cache, slot_mapping, N, (int)row,
                                          (long long)NB * bs, kinv, vinv, err_flag,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "store_kvcache_fp8 launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

} // extern "C"
