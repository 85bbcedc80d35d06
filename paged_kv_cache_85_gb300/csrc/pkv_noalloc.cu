// pkv_paged_attn_decode_noalloc: paged decode attention for callers that
// cannot allocate device memory.
//
// Some callers may not call cudaMalloc (or any allocating routine) at the
// point where they run decode attention: code running inside a memory pool
// or allocator that forbids nested allocation, runtimes that must not touch
// the allocator mid-step, or hosts that only hand over input and output
// buffers.  pkv_paged_attn_decode needs a caller-provided scratch buffer;
// this entry point instead uses a fixed scratch array that lives in the
// library's own device memory, so the caller passes only inputs and outputs.
//
// The scratch is a file-scope __device__ array of PKV_NOALLOC_SCRATCH_BYTES
// (16 MiB).  Every GPU on which the library's device code is loaded holds it
// until the process exits.  Host code cannot use the array's name as a
// device address (it is a host-side stand-in), so the first call on each
// device looks the address up with cudaGetSymbolAddress while that device is
// current and caches it together with the id of the device's current
// context; a later call on a different context (after cudaDeviceReset, for
// instance, which reloads the module) looks it up again.  Make the first call
// on a device before any CUDA stream capture.
//
// All calls share the one array and it keeps whatever the last call left.
// Nothing in it has to start at zero: each call writes the box layout and
// every partial result before its merge kernel reads them.  Calls that
// overlap on the GPU (different streams, or different host threads, on the
// same device) race on the array and must be serialised by the caller.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "pkv.h"
#include "pkv_kernels.h"

namespace pkv {
pkv_status report_error(pkv_status s, const char *msg);
}

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

// The largest one-CTA need of any supported size: the header of kMaxBatch
// sequences plus the partial slots of one eight-worker CTA at G = 8, D = 128.
static_assert(((size_t)(pkv::kWsHeaderInts + pkv::kMaxBatch + 1) * 4 + 255) / 256 * 256 +
                      (size_t)pkv::kWideWorkers * 2 * 8 * (128 + 4) * sizeof(float) <=
                  (size_t)PKV_NOALLOC_SCRATCH_BYTES,
              "every supported size must fit at least one CTA in the built-in scratch");

namespace {

constexpr int kMaxDevices = 64;
struct ScratchAddr {
    bool valid = false;
    unsigned long long ctx_id = 0;
    void *addr = nullptr;
};
ScratchAddr g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Id of the calling thread's current context (0 when unknown): the driver's
// cuCtxGetCurrent / cuCtxGetId, reached through the runtime's entry-point
// query.  Neither call allocates.
unsigned long long current_context_id()
{
    static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_cur || !get_id)
        return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device, looked up once
// per device and context.
pkv_status scratch_address(void **addr, const char **why)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *why = "no usable current CUDA device";
        return PKV_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchAddr &e = g_scratch_addr[dev];
    const unsigned long long id = current_context_id();
    if (!e.valid || id == 0 || id != e.ctx_id) {
        void *p = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess || !p) {
            *why = cudaGetErrorString(err);
            e.valid = false;
            return PKV_ERR_CUDA;
        }
        e.addr = p;
        e.ctx_id = current_context_id();  // the lookup made the context current if it was not
        e.valid = true;
    }
    *addr = e.addr;
    return PKV_OK;
}

} // namespace

extern "C" pkv_status pkv_paged_attn_decode_noalloc(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables, int MBS,
    const int32_t *context_lens, int B, int Hq, int Hkv, int D, int64_t NB, int bs, float scale,
    void *out, int32_t *err_flag, void *stream)
{
    if (B == 0)
        return pkv_paged_attn_decode(q, k_cache, v_cache, block_tables, MBS, context_lens, B, Hq,
                                     Hkv, D, NB, bs, scale, out, nullptr, 0, 0, err_flag, stream);
    // The scratch holds a per-call header plus two partial results per
    // worker of the grid; use the largest grid whose scratch fits.
    const size_t one = pkv_decode_workspace_bytes(B, Hq, Hkv, D, MBS, bs, 1);
    if (one == 0)  // invalid or unsupported sizes: let the regular checks report them
        return pkv_paged_attn_decode(q, k_cache, v_cache, block_tables, MBS, context_lens, B, Hq,
                                     Hkv, D, NB, bs, scale, out, nullptr, 0, 1, err_flag, stream);
    if (one > (size_t)PKV_NOALLOC_SCRATCH_BYTES) {  // not reached: see the static_assert above
        char msg[200];
        snprintf(msg, sizeof msg,
                 "paged_attn_decode_noalloc: these sizes need %zu bytes of scratch even on one "
                 "CTA; the built-in scratch holds %zu (use pkv_paged_attn_decode)",
                 one, (size_t)PKV_NOALLOC_SCRATCH_BYTES);
        return pkv::report_error(PKV_ERR_WORKSPACE, msg);
    }
    const size_t two = pkv_decode_workspace_bytes(B, Hq, Hkv, D, MBS, bs, 2);
    const size_t per_cta = two - one;
    int max_ctas = 1;
    if (per_cta > 0)
        max_ctas = (int)(1 + ((size_t)PKV_NOALLOC_SCRATCH_BYTES - one) / per_cta);
    if (max_ctas > 1024)
        max_ctas = 1024;
    // Where the workspace of the uncapped grid fits, launch exactly what the
    // regular call launches (max_ctas = 0: as many CTAs as the device holds).
    const size_t full = pkv_decode_workspace_bytes(B, Hq, Hkv, D, MBS, bs, 0);
    if (full > 0 && full <= (size_t)PKV_NOALLOC_SCRATCH_BYTES)
        max_ctas = 0;
    void *scratch = nullptr;
    const char *why = "";
    const pkv_status st = scratch_address(&scratch, &why);
    if (st != PKV_OK) {
        char msg[200];
        snprintf(msg, sizeof msg, "paged_attn_decode_noalloc: scratch address lookup: %s", why);
        return pkv::report_error(st, msg);
    }
    return pkv_paged_attn_decode(q, k_cache, v_cache, block_tables, MBS, context_lens, B, Hq, Hkv,
                                 D, NB, bs, scale, out, scratch, (size_t)PKV_NOALLOC_SCRATCH_BYTES,
                                 max_ctas, err_flag, stream);
}
