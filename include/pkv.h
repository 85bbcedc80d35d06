/*
 * pkv.h - C ABI of a GB300 (sm_103a) paged-KV-cache decode library.
 *
 * Two operations make up one decode step of PagedAttention over a
 * block-paged KV cache:
 *
 *   pkv_store_kvcache    scatter the step's new K/V rows into the cache
 *                        through slot_mapping;
 *   pkv_paged_attn_decode for every running sequence and query head,
 *                        softmax(scale * q . K^T) . V over the sequence's
 *                        context_len cached tokens, gathered through its
 *                        block table, with grouped-query head sharing.
 *
 * Where these come from:
 *   - MinivLLM guide "HowToApproachvLLM", section 4.4 (allocate_kv_cache:
 *     the cache is preallocated and carved into blocks; slot_mapping tracks
 *     where each token is written) and section 4.5 (prepare_prefill /
 *     prepare_decode: a block's tokens are the slice
 *     [block_id*block_size, (block_id+1)*block_size) of the token axis;
 *     slot_mapping holds only the new tokens; the decode slot is
 *     block_table[-1]*block_size + last_block_num_tokens - 1; block_tables
 *     and context_lens tell the attention kernel where to read KV), and
 *     section 4.6 (sentinel padding of slot_mapping and context_lens).
 *   - "Nano-vLLM 源码学习(2)", section 2 Config (kvcache_block_size 256,
 *     max_num_seqs 512, max_model_len 4096; the decode path reads paged KV
 *     through block_table; heads and KV heads are separate counts).
 *   - "VLLM-0.7.3 源码", section 3.1 (block table: logical blocks mapped to
 *     physical blocks anywhere in memory; block_size 16 by default).
 *   The pages do not print the attention formula; the plain reading
 *   (softmax(scale q.K^T).V over the first context_len tokens, no other
 *   mask) is used.
 *
 * Conventions common to every call:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, except
 *     that the `out` of the decode, FP8 decode and prefill calls may instead
 *     be page-locked host memory the device can address (cudaHostAlloc /
 *     cudaHostRegister, the same pointer on host and device): the kernels
 *     then write the result over the host link while they run, in place of
 *     a separate device-to-host copy after them.  The library never
 *     allocates or frees device memory.  The one piece of
 *     device memory it keeps is the fixed scratch array of
 *     pkv_paged_attn_decode_noalloc (PKV_NOALLOC_SCRATCH_BYTES, a static
 *     __device__ array held by every GPU that loads the library).
 *   - Tensors are dense row-major; bf16 data is passed as `const void *`.
 *     Every pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *     pkv_store_kvcache, pkv_paged_attn_decode, pkv_paged_prefill and the FP8
 *     calls only enqueue work: they never synchronise the host and never
 *     allocate, so they can be captured into a CUDA graph.
 *   - Argument errors are reported by the return status before any launch;
 *     pkv_last_error() then gives a message.  Data errors found on the
 *     device (an out-of-range slot or block id, a context length above
 *     MBS*bs) never trap: the offending item is skipped (or clamped) and a
 *     PKV_FLAG_* bit is OR-ed into *err_flag when err_flag is non-NULL.
 *     err_flag is a device int32 the caller zeroes and reads back.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, Hq % Hkv != 0 ... */
    PKV_ERR_UNSUPPORTED = 2, /* valid but not built: head_dim or group size */
    PKV_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
    PKV_ERR_CUDA = 4         /* a CUDA runtime/driver call failed */
} pkv_status;

/* Device-side error bits OR-ed into *err_flag. */
#define PKV_FLAG_BAD_SLOT 0x1        /* slot_mapping[i] not -1 and outside [0, NB*bs) */
#define PKV_FLAG_BAD_BLOCK 0x2       /* a needed block_tables entry outside [0, NB) */
#define PKV_FLAG_BAD_CONTEXT_LEN 0x4 /* context_lens[b] < 0 or > MBS*bs (clamped) */
#define PKV_FLAG_TIMEOUT 0x8         /* an internal pipeline wait gave up (a bug) */
#define PKV_FLAG_V_RANGE 0x10        /* paged_prefill: a V value beyond f16's range was clamped */

/*
 * pkv_store_kvcache - write the step's new K/V rows into the paged cache.
 *
 * For every i in [0, N) with slot_mapping[i] != -1, copies the Hkv*D bf16
 * values of k[i] and v[i] (bit for bit) to flat slot s = slot_mapping[i],
 * i.e. block s / bs, offset s % bs of k_cache and v_cache.  slot -1 is the
 * padding sentinel and is skipped (MinivLLM guide 4.5/4.6).
 *
 *   k, v          bf16 [N, Hkv, D]            new rows (read)
 *   k_cache,
 *   v_cache       bf16 [NB, bs, Hkv, D]       caches (written in place)
 *   slot_mapping  int64 [N]                   flat slots, -1 = skip
 *   N >= 0, Hkv >= 1, D in {64, 128}, NB >= 1, bs >= 16 and bs % 16 == 0
 *   err_flag      int32 device word or NULL   PKV_FLAG_BAD_SLOT
 *
 * Valid slots are expected to be distinct (the block manager never hands
 * one slot to two tokens); with duplicates the surviving row is unspecified.
 * N == 0 enqueues nothing and returns PKV_OK.
 */
pkv_status pkv_store_kvcache(const void *k, const void *v, void *k_cache, void *v_cache,
                             const int64_t *slot_mapping, int64_t N, int Hkv, int D,
                             int64_t NB, int bs, int32_t *err_flag, void *stream);

/*
 * pkv_decode_workspace_bytes - device scratch pkv_paged_attn_decode needs.
 *
 * Depends only on its arguments (no device query); pass the same values,
 * including max_ctas, to the decode call.  The scratch holds the per-call
 * box layout (a few bytes per sequence) and, for every worker of the grid,
 * two fp32 partial results (G query rows of D outputs plus running max and
 * sum) for the pieces of contexts that straddle workers.  Returns 0 for
 * invalid or unsupported arguments or B == 0.
 */
size_t pkv_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int MBS, int bs, int max_ctas);

/*
 * pkv_paged_attn_decode - one decode step of paged attention.
 *
 * For each sequence b < B and query head h < Hq, with G = Hq / Hkv and
 * n = context_lens[b]:
 *   token t < n lives at block block_tables[b*MBS + t/bs], offset t % bs;
 *   s_t  = scale * sum_d q[b,h,d] * k_cache[block, offset, h/G, d]
 *   out[b,h,:] = sum_t exp(s_t - max s) v_cache[block, offset, h/G, :]
 *                / sum_t exp(s_t - max s)
 * computed with fp32 accumulation and an fp32 online softmax, rounded to
 * bf16 (nearest-even).  n == 0 gives zeros.  Only the first ceil(n/bs)
 * entries of a table row are read (the rest may be -1); slots of the last
 * block past n are never used, whatever they hold.
 *
 * Work split: every (sequence, KV head) context is a stream of 16-token
 * boxes; the concatenated streams are cut into equal slices, one per worker
 * warp of a persistent grid (two CTAs of four workers per SM, or one CTA of
 * eight workers per SM where the smaller CTAs do not fit twice in shared
 * memory: large B, or G = 8 at D = 128), and a second kernel merges, by
 * log-sum-exp, the pieces of contexts that straddle workers.  Both kernels
 * run on `stream`.
 *
 *   q             bf16 [B, Hq, D]
 *   k_cache,
 *   v_cache       bf16 [NB, bs, Hkv, D]
 *   block_tables  int32 [B, MBS]
 *   context_lens  int32 [B], 0 <= n <= MBS*bs
 *   scale         softmax scale (commonly 1/sqrt(D))
 *   out           bf16 [B, Hq, D]             written (device, or page-locked host)
 *   workspace     device scratch of at least
 *                 pkv_decode_workspace_bytes(B, Hq, Hkv, D, MBS, bs, max_ctas)
 *                 bytes; contents on entry do not matter; it is overwritten,
 *                 so calls that may overlap need separate workspaces
 *   max_ctas      0 = as many CTAs as the device holds at once (at most
 *                 2048 worker warps in all);
 *                 k >= 1 = at most k CTAs (moves where contexts are split;
 *                 results agree within rounding)
 *   B >= 0, Hq % Hkv == 0, Hq/Hkv in {1, 2, 4, 8}, D in {64, 128},
 *   bs >= 16 and bs % 16 == 0, B <= 8192, NB*bs < 2^31,
 *   B*Hkv*ceil(MBS*bs/16) < 2^31
 *   err_flag      int32 device word or NULL   PKV_FLAG_BAD_BLOCK |
 *                                             PKV_FLAG_BAD_CONTEXT_LEN
 *
 * Call pkv_store_kvcache for the step's new tokens first on the same
 * stream; context_lens then counts the new token.
 */
pkv_status pkv_paged_attn_decode(const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, int MBS,
                                 const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                                 int64_t NB, int bs, float scale, void *out, void *workspace,
                                 size_t workspace_bytes, int max_ctas, int32_t *err_flag,
                                 void *stream);

/*
 * pkv_paged_prefill - causal attention of a prefill step's new tokens over
 * their sequences' paged contexts.
 *
 * MinivLLM guide "HowToApproachvLLM", section 4.5 (prepare_prefill): the
 * new tokens of all B sequences are flattened into one list, cu_seqlens_q
 * and cu_seqlens_k mark the sequences' boundaries, slot_mapping writes the
 * uncached tokens' K/V (pkv_store_kvcache, called first) and block_tables
 * say where KV is read; "Nano-vLLM 源码学习(2)" section 2: the prefix-hit
 * prefill path reads paged KV through block_table.  The pages give no mask;
 * the plain causal reading is used: sequence b has q_len = cu_seqlens_q[b+1]
 * - cu_seqlens_q[b] new tokens and k_len = cu_seqlens_k[b+1] -
 * cu_seqlens_k[b] context tokens (cached prefix + the new tokens); new token
 * i sits at position k_len - q_len + i and attends to positions 0 .. that
 * one, read through block_tables[b]:
 *   out[cu_seqlens_q[b] + i, h, :] = softmax(scale * q . K^T) . V
 * with query head h reading KV head h / (Hq / Hkv).
 *
 *   q             device, bf16 [Tq, Hq, D] contiguous, 16-byte aligned
 *   k_cache/v_cache device, bf16 [NB, bs, Hkv, D] (as pkv_store_kvcache)
 *   block_tables  device, int32 [B, MBS]; entries past ceil(k_len / bs) unread
 *   cu_seqlens_q  device, int32 [B + 1], non-decreasing, cu_seqlens_q[B] <= Tq
 *   cu_seqlens_k  device, int32 [B + 1]; q_len <= k_len <= MBS * bs
 *   max_seqlen_q  host bound on every q_len (sizes the work space; a loose
 *                 bound only adds empty work positions)
 *   out           bf16 [Tq, Hq, D], device or page-locked host memory; rows
 *                 not covered by cu_seqlens_q are left untouched.  Each
 *                 thread writes one output row in 16-byte pieces, which
 *                 cross a host link one by one: for a large step, writing
 *                 device memory and copying it out afterwards is faster
 *                 (a 67 MB result: the kernel ran ~1.5 ms writing host
 *                 memory, against 0.22 ms plus a 0.35 ms copy)
 * D in {64, 128}; Hq / Hkv in {1, 2, 4, 8}; bs a multiple of 16.  No
 * workspace.  Device-side problems set err_flag bits and never trap: a
 * sequence whose lengths are inconsistent (or q_len > max_seqlen_q) is
 * skipped with PKV_FLAG_BAD_CONTEXT_LEN; a table entry outside [0, NB) sets
 * PKV_FLAG_BAD_BLOCK and its 16-token boxes are left out of the softmax.
 * Host-side errors return a status before any launch; B, Tq or
 * max_seqlen_q == 0 is a no-op.
 *
 * Precision: q . K^T runs on the tensor cores in bf16 with fp32
 * accumulation; P . V runs in f16 with fp32 accumulation: P (at most 2^8
 * after the online max) is rounded to f16, and V to f16, which holds every
 * bf16 value of magnitude in [2^-17, 65504] exactly (smaller magnitudes
 * round to f16 subnormals, absolute error <= 2^-25).  V values beyond
 * +-65504 (and infinities) are clamped to +-65504 and set PKV_FLAG_V_RANGE;
 * NaN stays NaN.  Output rounded to bf16.
 *
 * The kernel runs one CTA per SM that holds all of the SM's tensor memory
 * (512 columns); a concurrent kernel that allocates tensor memory on the
 * same SMs waits for it.
 */
pkv_status pkv_paged_prefill(const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, int MBS, const int32_t *cu_seqlens_q,
                             const int32_t *cu_seqlens_k, int B, int64_t Tq, int max_seqlen_q,
                             int Hq, int Hkv, int D, int64_t NB, int bs, float scale, void *out,
                             int32_t *err_flag, void *stream);

/*
 * FP8 KV cache ("VLLM-0.7.3 源码" section 5.3: kv_cache_dtype can store the
 * KV cache in FP8 while the output side keeps higher-precision compute).
 * The page gives no scale convention; these calls take the plain one: a
 * cache element is the OCP E4M3 code (1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, max 448) of x * (1 / scale), with one
 * positive fp32 dequant scale per tensor (k_scale for K, v_scale for V), and
 * stands for code_value * scale.  Caches are uint8 [NB, bs, Hkv, D].
 */

/*
 * pkv_store_kvcache_fp8 - quantize and scatter the step's new K/V rows.
 *
 * As pkv_store_kvcache, except that each bf16 value x is multiplied by the
 * fp32 reciprocal of its tensor's scale (1/k_scale, 1/v_scale, each formed
 * once in IEEE fp32) and stored as the nearest E4M3 code (ties to even;
 * finite values beyond 448, and infinities, saturate to +-448; NaN stays
 * NaN).  Hkv*D must be a multiple of 16; scales finite and > 0.
 */
pkv_status pkv_store_kvcache_fp8(const void *k, const void *v, void *k_cache, void *v_cache,
                                 const int64_t *slot_mapping, int64_t N, int Hkv, int D,
                                 int64_t NB, int bs, float k_scale, float v_scale,
                                 int32_t *err_flag, void *stream);

/*
 * pkv_paged_attn_decode_fp8 - pkv_paged_attn_decode over FP8 caches.
 *
 * Same arguments, workspace (pkv_decode_workspace_bytes with the same
 * sizes) and results, reading K = code_value * k_scale and V = code_value *
 * v_scale.  The contractions run on the tensor cores with fp32 accumulation:
 *   - scores on the E4M3 path, K as the raw cache codes and q split per head
 *     into two E4M3 parts under a power-of-two scale sq,
 *     q = sq * (hi + lo / 16), which is exact for every bf16 element of
 *     magnitude >= max|q| * 2^-14 (smaller elements are within
 *     max|q| * 2^-21);
 *   - P.V in f16: V codes converted to f16 (exact), P rounded to f16;
 *   - output rounded to bf16.
 * Three CTAs of four workers run per SM (one CTA of eight where they do not
 * fit).  Where those CTAs would hold fewer than four pipeline stages of
 * 16-token boxes (large B or G) and bs is a multiple of 32, the streams are
 * cut into 32-token boxes instead (two stages), which halves the per-box
 * work for the same bytes in flight; the results agree within the
 * tolerance above, not bit for bit, with a 16-token split.
 */
pkv_status pkv_paged_attn_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *block_tables, int MBS,
                                     const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                                     int64_t NB, int bs, float scale, float k_scale,
                                     float v_scale, void *out, void *workspace,
                                     size_t workspace_bytes, int max_ctas, int32_t *err_flag,
                                     void *stream);

/*
 * pkv_paged_attn_decode_noalloc - pkv_paged_attn_decode without a workspace
 * argument, for callers that cannot allocate device memory.
 *
 * (No counterpart in the pages: this is an interface convenience.)  Some
 * callers must not call cudaMalloc or any allocating routine when they run
 * decode attention, for instance code running inside a custom allocator or
 * memory pool, or a runtime that only owns the step's input and output
 * buffers.  This call computes exactly what pkv_paged_attn_decode computes
 * (same arguments and results, within rounding) but keeps its scratch in a
 * fixed device array of PKV_NOALLOC_SCRATCH_BYTES (16 MiB) inside the
 * library, which every GPU that loads the library's device code holds until
 * the process exits.  It allocates nothing.  The decode grid is the one
 * pkv_paged_attn_decode launches with max_ctas = 0 whenever that grid's
 * partial results fit the array, which holds for every supported size on a
 * 152-SM GB300; otherwise the grid is capped so they fit (results then agree
 * within rounding, as for any max_ctas).  Every supported size fits at least
 * one CTA, so the call never fails for lack of scratch.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it with the id
 * of the device's current context; a call on a new context (after
 * cudaDeviceReset, for instance) looks it up again.  Make the first call on a
 * device before any CUDA stream capture.  All calls share the one array and
 * it keeps the last call's contents (nothing in it needs to start at zero).
 * Calls that overlap on the GPU race on it: serialise them (one stream per
 * device, or events between streams).
 */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)

pkv_status pkv_paged_attn_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables, int MBS,
                                         const int32_t *context_lens, int B, int Hq, int Hkv,
                                         int D, int64_t NB, int bs, float scale, void *out,
                                         int32_t *err_flag, void *stream);

/* Message describing the last non-OK status returned on this host thread. */
const char *pkv_last_error(void);

/* Name of a status code. */
const char *pkv_status_string(pkv_status status);

/* ABI version of this library (major * 100 + minor). */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
