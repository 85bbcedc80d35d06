// paged_attn_decode: one decode step of PagedAttention on sm_103a.
//
// What it computes (MinivLLM guide "HowToApproachvLLM" section 4.5; the
// "Nano-vLLM 源码学习(2)" Config section; "VLLM-0.7.3 源码" section 3.1):
// for each running sequence b and query head h, softmax(scale q.K^T).V over
// the sequence's context_lens[b] cached tokens, where token t is read from
// physical block block_tables[b][t / bs], offset t % bs, of KV head
// h / (Hq / Hkv).
//
// How (GB300 design):
//  * Work decomposition (stream-K).  Each (sequence, KV head) context is a
//    stream of 16-token boxes; all G query heads of the group ride along, so
//    every K/V byte is read from HBM once.  The streams are concatenated
//    (KV-head-major); each head's region is cut into equal contiguous
//    slices, one per worker, so the workers of different heads read the
//    same token rows at the same time; a worker is one consumer warp, and a
//    persistent grid of CTAs with eight workers each fills the 152 SMs.
//    Every worker therefore moves the same number of bytes (+-1 box), and a
//    stream is split only where a slice boundary falls into it.  Each CTA
//    rebuilds the per-sequence box prefix sums from context_lens in shared
//    memory, so the host never reads context lengths and the call needs no
//    host synchronisation.
//  * Producer warp.  Lane w runs worker w: every pipeline stage carries one
//    box per worker, and each lane walks its worker's slice, loading block
//    ids four boxes ahead of use, so no copy waits on a block-table read.  Boxes ([16 tokens x D] bf16 of one KV head, from
//    the [NB*bs, Hkv, D] cache view) arrive by TMA into a ring of
//    shared-memory stages completed on mbarriers with their byte counts; the
//    G query rows of a worker's new piece come with it by a bulk copy.
//  * Consumer warps (workers).  Per box, Q.K^T and P.V run on the tensor
//    cores as warp-level bf16 MMAs with the G query heads as the rows (one
//    GQA group per MMA), fp32 accumulation, and the online softmax in fp32
//    registers (log2 domain); P enters P.V as a bf16 hi + lo pair.  K/V boxes
//    arrive 128-byte swizzled so the ldmatrix reads are conflict-free.  When a worker finishes
//    a piece of a stream it either writes the normalised bf16 output (the
//    piece is the whole stream) or a partial (acc, max, sum) into one of its
//    two workspace slots (first / last piece of its slice); a second kernel
//    merges the partials of streams that straddle workers by log-sum-exp.
//  * Masking selects out tokens at or past context_len (scores -> -inf and
//    the P.V loop stops at the last valid token), so whatever the unused
//    slots of the last block hold (even NaN) never reaches the output.
#pragma once

#include <cuda_bf16.h>

#include "pkv_kernels.h"
#include "pkv_ptx.cuh"

namespace pkv {

constexpr int kLookahead = 4;  // boxes per worker whose block ids are loaded ahead of use
constexpr int kHalfBytes = kBox * 128;  // one 64-column half of a box: 16 rows of 128 B

// Per-worker box descriptor of a stage, written by the producer.
struct __align__(16) BoxMeta {
    int b, h, tok0, nvalid;
    int flags, blk, pad0, pad1;
};
constexpr int kBoxValid = 1;     // the worker has a box in this stage
constexpr int kBoxLoaded = 2;    // its K/V were copied (the block id was valid)
constexpr int kPieceFirst = 4;   // first box of the worker's piece of this stream (q comes with it)
constexpr int kPieceLast = 8;    // last box of the piece: finish it after this box
constexpr int kStreamFirst = 16; // box 0 of the stream
constexpr int kStreamLast = 32;  // last box of the stream
constexpr int kSlot1 = 64;       // a partial of this piece goes to the worker's second slot
constexpr int kStageStop = 1 << 30;

struct DecodeSmem {
    size_t kv, q, full, empty, meta, pb, len, scan, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline DecodeSmem decode_smem_layout(int D, int G, int NW, int stages, int B,
                                                         int kv_elem_bytes = 2)
{
    DecodeSmem L;
    size_t o = 0;
    L.kv = o;  // per stage: K boxes [NW][D/64][16][64], then V boxes alike (128B-swizzled rows)
    o += (size_t)stages * 2 * NW * kBox * D * kv_elem_bytes;
    L.q = o;  // per stage and worker: G query rows
    o = align_up(o + (size_t)stages * NW * G * D * 2, 16);
    L.full = o;
    o += (size_t)stages * 8;
    L.empty = o;
    o += (size_t)stages * 8;
    L.meta = o = align_up(o, 16);
    o += (size_t)stages * NW * sizeof(BoxMeta);
    L.pb = o;  // boxes per KV head before sequence b, b = 0..B
    o = align_up(o + (size_t)(B + 1) * 4, 16);
    L.len = o;  // clamped context length per sequence
    o = align_up(o + (size_t)B * 4, 16);
    L.scan = o;  // per-warp partial sums of the prefix scan
    o = align_up(o + (size_t)(NW + 2) * 4, 16);
    L.total = o + 1024;  // slack to align the base to 1024 B (128-byte swizzle atoms)
    return L;
}

// Deepest pipeline (2..max_stages) whose shared memory fits max_smem.
inline int decode_stages_for(int D, int G, int NW, int B, int max_stages, size_t max_smem,
                             int kv_elem_bytes = 2)
{
    for (int s = max_stages; s >= kMinStages; s--)
        if (decode_smem_layout(D, G, NW, s, B, kv_elem_bytes).total <= max_smem)
            return s;
    return 0;
}

// Streams are concatenated head-major: all sequences' streams of KV head 0,
// then of head 1, ...  Workers in different head regions then sit at the
// same (sequence, box) positions at the same time, so the Hkv slices of one
// token range are fetched together (DRAM row locality), and sequences that
// share prefix blocks read them together (L2 reuse).
// Box x -> (sequence b, KV head h, box j of the stream); pb[b] = boxes per
// KV head before sequence b, so each head region holds pb[B] boxes.
__device__ __forceinline__ void locate_box(int x, const int *pb, int B, int &b, int &h, int &j)
{
    const int per_head = pb[B];
    h = x / per_head;
    const int r = x - h * per_head;
    int lo = 0, hi = B - 1;  // largest b with pb[b] <= r (skips empty sequences)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pb[mid] <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    b = lo;
    j = r - pb[b];
}

// Advance a (sequence, KV head, box) cursor to the next box of the
// concatenated streams, skipping sequences without boxes.
__device__ __forceinline__ void next_box(const int *pb, int B, int &b, int &h, int &j)
{
    if (++j == pb[b + 1] - pb[b]) {
        j = 0;
        do {
            if (++b == B) {
                b = 0;
                ++h;
            }
        } while (pb[b + 1] == pb[b]);  // ends: the sequence just left has boxes
    }
}

__device__ __forceinline__ int box_block(const DecodeParams &p, int b, int j)
{
    return __ldg(p.block_tables + (size_t)b * p.MBS + (j * kBox) / p.bs);
}

// Producer warp: lane w < NW runs worker w of this CTA.  Each lane
// walks its own slice with two cursors: the issue cursor, and a look-ahead
// cursor kLookahead boxes further on whose block ids are loaded into a small
// register queue, so a copy never waits on a block-table read.  Per stage
// every lane writes its worker's box descriptor and issues its own TMA
// copies; lane 0 arms the stage's mbarrier with the summed byte count.
template <int D, int G, int NW, bool F8>
__device__ __forceinline__ void decode_producer(const CUtensorMap *tmk, const CUtensorMap *tmv,
                                                const DecodeParams &p, uint8_t *smem,
                                                const DecodeSmem &L, int lane, int R, int Tr,
                                                int Wr, int P)
{
    constexpr unsigned FULL = 0xffffffffu;
    constexpr int kBoxBytes = kBox * D * (F8 ? 1 : 2);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    BoxMeta *meta = reinterpret_cast<BoxMeta *>(smem + L.meta);
    const int *pb = reinterpret_cast<const int *>(smem + L.pb);
    const int *len = reinterpret_cast<const int *>(smem + L.len);

    if (lane == 0) {
        prefetch_tensormap(tmk);
        prefetch_tensormap(tmv);
    }
    // Worker gw owns slice gw % Wr of region gw / Wr (regions past R idle).
    const bool worker = lane < NW;
    const int gw = blockIdx.x * NW + lane;
    const int r = gw / Wr;
    int start = 0, end = 0;
    if (worker && r < R) {
        const long long lo = (long long)(gw - r * Wr) * P;
        start = r * Tr + (int)(lo < Tr ? lo : Tr);
        end = r * Tr + (int)(lo + P < Tr ? lo + P : Tr);
    }
    int pos = start;
    int cb = 0, ch = 0, cj = 0;  // issue cursor
    if (start < end)
        locate_box(start, pb, p.B, cb, ch, cj);
    int lb = cb, lh = ch, lj = cj, lpos = start;  // look-ahead cursor
    int qb[kLookahead];                          // block ids of boxes pos .. pos + kLookahead - 1
#pragma unroll
    for (int i = 0; i < kLookahead; i++) {
        qb[i] = -1;
        if (lpos < end) {
            qb[i] = box_block(p, lb, lj);
            next_box(pb, p.B, lb, lh, lj);
        }
        ++lpos;
    }
    bool first_done = false;

    // K/V may have just been written by store_kvcache on this stream.
    grid_dependency_wait();

    int stage = 0;
    uint32_t phase = 0;
    for (;;) {
        const bool mine = pos < end;
        if (!__any_sync(FULL, mine))
            break;
        if (!__all_sync(FULL, mbar_wait(&empty[stage], phase ^ 1))) {
            if (lane == 0)
                flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
            return;
        }
        uint32_t bytes = 0;
        int flags = 0, row = 0, b = cb, h = ch;
        if (mine) {
            const int j = cj;
            const int blk = qb[0];
            const int nb = pb[b + 1] - pb[b];
            const int tok0 = j * kBox;
            const bool loaded = blk >= 0 && blk < p.NB;
            if (!loaded)
                flag_error(p.err_flag, 0x2 /* PKV_FLAG_BAD_BLOCK */);
            const bool pf = pos == start || j == 0;
            const bool pl = pos == end - 1 || j == nb - 1;
            flags = kBoxValid | (loaded ? kBoxLoaded : 0) | (pf ? kPieceFirst : 0) |
                    (pl ? kPieceLast : 0) | (j == 0 ? kStreamFirst : 0) |
                    (j == nb - 1 ? kStreamLast : 0) | (first_done ? kSlot1 : 0);
            if (pl)
                first_done = true;
            bytes = (loaded ? 2u * kBoxBytes : 0u) + (pf ? (uint32_t)(G * D * 2) : 0u);
            row = loaded ? blk * p.bs + tok0 % p.bs : 0;
            BoxMeta &m = meta[stage * NW + lane];
            m.b = b;
            m.h = h;
            m.tok0 = tok0;
            m.nvalid = min(kBox, len[b] - tok0);
            m.flags = flags;
            m.blk = blk;
            // advance both cursors
            next_box(pb, p.B, cb, ch, cj);
            ++pos;
#pragma unroll
            for (int i = 0; i + 1 < kLookahead; i++)
                qb[i] = qb[i + 1];
            qb[kLookahead - 1] = -1;
            if (lpos < end) {
                qb[kLookahead - 1] = box_block(p, lb, lj);
                next_box(pb, p.B, lb, lh, lj);
            }
            ++lpos;
        } else if (worker) {
            meta[stage * NW + lane].flags = 0;
        }
        bytes = __reduce_add_sync(FULL, bytes);
        __syncwarp();
        if (lane == 0)
            mbar_arrive_expect_tx(&full[stage], bytes);
        __syncwarp();
        if (flags & kPieceFirst)
            bulk_load(smem + L.q + ((size_t)stage * NW + lane) * G * D * 2,
                      p.q + ((size_t)b * p.Hq + (size_t)h * G) * D, G * D * 2, &full[stage]);
        if ((flags & kBoxLoaded) && F8) {
            uint8_t *kd = smem + L.kv + ((size_t)stage * 2 * NW + lane) * kBoxBytes;
            tma_load_3d(kd, tmk, 0, h, row, &full[stage]);
            tma_load_3d(kd + (size_t)NW * kBoxBytes, tmv, 0, h, row, &full[stage]);
        } else if (flags & kBoxLoaded) {
            uint8_t *kd = smem + L.kv + ((size_t)stage * 2 * NW + lane) * kBoxBytes;
#pragma unroll
            for (int half = 0; half < D / 64; half++) {
                tma_load_4d(kd + half * kHalfBytes, tmk, 0, half, h, row, &full[stage]);
                tma_load_4d(kd + (size_t)NW * kBoxBytes + half * kHalfBytes, tmv, 0, half, h, row,
                            &full[stage]);
            }
        }
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1;
        }
    }
    // Tell the consumers there is no more work.
    if (!__all_sync(FULL, mbar_wait(&empty[stage], phase ^ 1))) {
        if (lane == 0)
            flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
        return;
    }
    if (worker)
        meta[stage * NW + lane].flags = kStageStop;
    __syncwarp();
    if (lane == 0)
        mbar_arrive(&full[stage]);
}

// Byte offset of 16-byte chunk `c` (0 .. D/8-1) of token row `t` inside a box
// stored as D/64 halves of [16 rows][128 B] with the 128-byte TMA swizzle
// (chunk index XOR row % 8 within each row).
__device__ __forceinline__ uint32_t box_chunk(int t, int c)
{
    return (uint32_t)((c >> 3) * kHalfBytes + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// Consumer warp (worker).  Per 16-token box, on the tensor cores
// (mma.sync m16n8k16, bf16 in, fp32 accumulate), with the G query heads as
// the M rows (zero-padded to 16):
//   S[G x 16] = Q[G x D] . K^T    16 MMAs (D=128), K fragments by ldmatrix
//   online softmax in fp32 on the S fragments (each lane owns one head's row)
//   O[G x D] += P . V             P split into bf16 hi + lo parts (2 MMAs per
//                                 n-tile) so P keeps ~16 mantissa bits; V
//                                 fragments by ldmatrix.trans
template <int D, int G, int NW>
__device__ __forceinline__ void decode_consumer(const DecodeParams &p, uint8_t *smem,
                                                const DecodeSmem &L, int warp, int lane)
{
    constexpr int KSTEPS = D / 16;   // k-steps of the score MMA
    constexpr int NT = D / 8;        // 8-column n-tiles of the output
    constexpr int kBoxBytes = kBox * D * 2;
    constexpr unsigned FULL = 0xffffffffu;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    const BoxMeta *meta = reinterpret_cast<const BoxMeta *>(smem + L.meta);

    const int hrow = lane >> 2;    // head row of this lane's accumulator fragments
    const int quad = lane & 3;     // column pair within a fragment
    const bool real = hrow < G;    // rows G..15 are padding
    const int mat = lane >> 3;     // ldmatrix: matrix whose row address this lane supplies
    const int mrow = lane & 7;
    const int gw = blockIdx.x * NW + warp;

    uint32_t qa[KSTEPS][2];        // A fragments of q (a0, a2); a1 = a3 = 0 (padding rows)
    float o[NT][4];
    float m_run = -INFINITY, l_run = 0.f;
    bool whole = false;            // the current piece began at its stream's first box
#pragma unroll
    for (int k = 0; k < KSTEPS; k++)
        qa[k][0] = qa[k][1] = 0u;
#pragma unroll
    for (int n = 0; n < NT; n++)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    int stage = 0;
    uint32_t phase = 0;
    for (;;) {
        if (!__all_sync(FULL, mbar_wait(&full[stage], phase))) {
            if (lane == 0)
                flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
            return;
        }
        const BoxMeta bm = meta[stage * NW + warp];
        if (bm.flags & kStageStop)
            break;
        if (bm.flags & kPieceFirst) {
            const uint8_t *qs = smem + L.q + ((size_t)stage * NW + warp) * G * D * 2;
#pragma unroll
            for (int k = 0; k < KSTEPS; k++) {
                qa[k][0] = real ? *reinterpret_cast<const uint32_t *>(
                                      qs + (hrow * D + k * 16 + 2 * quad) * 2)
                                : 0u;
                qa[k][1] = real ? *reinterpret_cast<const uint32_t *>(
                                      qs + (hrow * D + k * 16 + 8 + 2 * quad) * 2)
                                : 0u;
            }
            m_run = -INFINITY;
            l_run = 0.f;
#pragma unroll
            for (int n = 0; n < NT; n++)
                o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            whole = (bm.flags & kStreamFirst) != 0;
        }
        const int nvw = (bm.flags & kBoxLoaded) ? bm.nvalid : 0;
        if (nvw > 0) {
            uint8_t *Ks = smem + L.kv + ((size_t)stage * 2 * NW + warp) * kBoxBytes;
            uint8_t *Vs = Ks + (size_t)NW * kBoxBytes;
            if (nvw < kBox) {
                // Rows past the context take weight 0, and 0 * NaN would still be
                // NaN on the tensor cores: clear them (whole rows, any swizzle).
                for (int i = lane; i < (kBox - nvw) * (D / 8); i += 32) {
                    const int t = nvw + i / (D / 8), c = i % (D / 8);
                    *reinterpret_cast<uint4 *>(Vs + (c >> 3) * kHalfBytes + t * 128 + (c & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();  // before TMA refills this buffer
                __syncwarp();
            }
            const uint32_t kb = smem_u32(Ks), vb = smem_u32(Vs);
            // ---- scores S = Q K^T (two 8-token n-tiles) ----
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            const int ktok = mrow + ((mat >> 1) << 3);
#pragma unroll
            for (int k = 0; k < KSTEPS; k++) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(kb + box_chunk(ktok, 2 * k + (mat & 1)), b0, b1, b2, b3);
                mma_bf16_16816(sc[0], qa[k][0], 0u, qa[k][1], 0u, b0, b1);
                mma_bf16_16816(sc[1], qa[k][0], 0u, qa[k][1], 0u, b2, b3);
            }
            // ---- online softmax (log2 domain); this lane: head hrow, tokens
            //      2q, 2q+1, 8+2q, 9+2q ----
            float sv[4] = {sc[0][0], sc[0][1], sc[1][0], sc[1][1]};
            const int tq = 2 * quad;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int t = tq + (i & 1) + ((i >> 1) << 3);
                sv[i] = t < nvw ? sv[i] * p.scale_log2 : -INFINITY;
            }
            float mt = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
            mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 1));
            mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 2));
            const float m_new = fmaxf(m_run, mt);
            const float alpha = fast_exp2(m_run - m_new);
            m_run = m_new;
            float pr[4];
#pragma unroll
            for (int i = 0; i < 4; i++)
                pr[i] = real ? fast_exp2(sv[i] - m_new) : 0.f;
            l_run = l_run * alpha + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
#pragma unroll
            for (int n = 0; n < NT; n++) {
                o[n][0] *= alpha;
                o[n][1] *= alpha;
            }
            // ---- P as A fragments, split hi + lo ----
            const uint32_t ph0 = pack_bf16x2(pr[0], pr[1]);
            const uint32_t ph2 = pack_bf16x2(pr[2], pr[3]);
            const float2 h0 = bf16x2_to_float2(ph0), h2 = bf16x2_to_float2(ph2);
            const uint32_t pl0 = pack_bf16x2(pr[0] - h0.x, pr[1] - h0.y);
            const uint32_t pl2 = pack_bf16x2(pr[2] - h2.x, pr[3] - h2.y);
            // ---- O += P V ----
            const int vtok = mrow + ((mat & 1) << 3);
#pragma unroll
            for (int n2 = 0; n2 < NT / 2; n2++) {
                uint32_t v0, v1, v2, v3;
                ldmatrix_x4_trans(vb + box_chunk(vtok, 2 * n2 + (mat >> 1)), v0, v1, v2, v3);
                mma_bf16_16816(o[2 * n2], ph0, 0u, ph2, 0u, v0, v1);
                mma_bf16_16816(o[2 * n2], pl0, 0u, pl2, 0u, v0, v1);
                mma_bf16_16816(o[2 * n2 + 1], ph0, 0u, ph2, 0u, v2, v3);
                mma_bf16_16816(o[2 * n2 + 1], pl0, 0u, pl2, 0u, v2, v3);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[stage]);

        if (bm.flags & kPieceLast) {
            // ---- finish this worker's piece of the stream ----
            float l_tot = l_run + __shfl_xor_sync(FULL, l_run, 1);
            l_tot += __shfl_xor_sync(FULL, l_tot, 2);
            const bool complete = whole && (bm.flags & kStreamLast);
            if (real) {
                const size_t hq = (size_t)bm.b * p.Hq + (size_t)bm.h * G + hrow;
                if (complete) {
                    uint16_t *orow = p.out + hq * D + 2 * quad;
#pragma unroll
                    for (int n = 0; n < NT; n++)
                        *reinterpret_cast<uint32_t *>(orow + 8 * n) =
                            pack_bf16x2(l_tot > 0.f ? o[n][0] / l_tot : 0.f,
                                        l_tot > 0.f ? o[n][1] / l_tot : 0.f);
                } else {
                    float *pg = p.ws_part +
                                (((size_t)gw * 2 + ((bm.flags & kSlot1) ? 1 : 0)) * G + hrow) * (D + 4);
#pragma unroll
                    for (int n = 0; n < NT; n++)
                        *reinterpret_cast<float2 *>(pg + 8 * n + 2 * quad) = make_float2(o[n][0], o[n][1]);
                    if (quad == 0) {
                        pg[D] = m_run;
                        pg[D + 1] = l_tot;
                    }
                }
            }
        }
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1;
        }
    }
}

// Byte offset of 16-byte chunk `c` of row `t` in an FP8 box of 16 rows of D
// bytes, as TMA writes it with the 128-byte (D = 128) or 64-byte (D = 64)
// swizzle.
template <int D> __device__ __forceinline__ uint32_t box8_chunk(int t, int c)
{
    if constexpr (D == 128)
        return (uint32_t)(t * 128 + ((c ^ (t & 7)) << 4));
    else
        return (uint32_t)(t * 64 + ((c ^ ((t >> 1) & 3)) << 4));
}

// Consumer warp for FP8 (E4M3) caches.  Same pipeline and softmax as the
// bf16 consumer; the MMAs run in f16 (E4M3 values are exact in f16; q is
// converted to f16; P needs no hi/lo split with f16's 10 mantissa bits).
// Fragments come from single 32-bit shared-memory loads by reindexing:
//   * scores: the contraction index d is permuted inside each 16-wide
//     k-step so that a lane's four B values (k = 2q, 2q+1, 8+2q, 9+2q) are
//     the four consecutive bytes d = 16k + 4q .. +3 of its token row; q's A
//     fragments use the same permutation, so S is unchanged;
//   * P.V: output columns are permuted so that column c of n-tile 4g + r
//     holds d = 32g + 4c + r; one 32-bit load of a V row then feeds four
//     n-tiles, and each lane ends up owning 8 consecutive outputs per group.
// K scales are folded into the score scale, V's scale into the output.
template <int D, int G, int NW>
__device__ __forceinline__ void decode_consumer_fp8(const DecodeParams &p, uint8_t *smem,
                                                    const DecodeSmem &L, int warp, int lane)
{
    constexpr int KSTEPS = D / 16;
    constexpr int NT = D / 8;
    constexpr int NG = D / 32;       // groups of 4 n-tiles fed by one load per row
    constexpr int kBoxBytes = kBox * D;
    constexpr unsigned FULL = 0xffffffffu;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    const BoxMeta *meta = reinterpret_cast<const BoxMeta *>(smem + L.meta);

    const int hrow = lane >> 2;      // head row of the accumulators / token of K fragments
    const int quad = lane & 3;
    const bool real = hrow < G;
    const int gw = blockIdx.x * NW + warp;

    uint32_t qa[KSTEPS][2];
    float o[NT][4];
    float m_run = -INFINITY, l_run = 0.f;
    bool whole = false;
#pragma unroll
    for (int k = 0; k < KSTEPS; k++)
        qa[k][0] = qa[k][1] = 0u;
#pragma unroll
    for (int n = 0; n < NT; n++)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    int stage = 0;
    uint32_t phase = 0;
    for (;;) {
        if (!__all_sync(FULL, mbar_wait(&full[stage], phase))) {
            if (lane == 0)
                flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
            return;
        }
        const BoxMeta bm = meta[stage * NW + warp];
        if (bm.flags & kStageStop)
            break;
        if (bm.flags & kPieceFirst) {
            const uint8_t *qs = smem + L.q + ((size_t)stage * NW + warp) * G * D * 2;
#pragma unroll
            for (int k = 0; k < KSTEPS; k++) {
                uint2 w = make_uint2(0u, 0u);
                if (real)
                    w = *reinterpret_cast<const uint2 *>(qs + (hrow * D + k * 16 + 4 * quad) * 2);
                const float2 f01 = bf16x2_to_float2(w.x), f23 = bf16x2_to_float2(w.y);
                qa[k][0] = pack_f16x2(f01.x, f01.y);
                qa[k][1] = pack_f16x2(f23.x, f23.y);
            }
            m_run = -INFINITY;
            l_run = 0.f;
#pragma unroll
            for (int n = 0; n < NT; n++)
                o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            whole = (bm.flags & kStreamFirst) != 0;
        }
        const int nvw = (bm.flags & kBoxLoaded) ? bm.nvalid : 0;
        if (nvw > 0) {
            uint8_t *Ks = smem + L.kv + ((size_t)stage * 2 * NW + warp) * kBoxBytes;
            uint8_t *Vs = Ks + (size_t)NW * kBoxBytes;
            if (nvw < kBox) {
                // Rows past the context take weight 0; 0 * NaN is still NaN on
                // the tensor cores, so clear them (whole rows, any swizzle).
                for (int i = lane; i < (kBox - nvw) * (D / 16); i += 32) {
                    const int t = nvw + i / (D / 16), c = i % (D / 16);
                    *reinterpret_cast<uint4 *>(Vs + t * D + c * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            // ---- scores ----
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int k = 0; k < KSTEPS; k++) {
                const uint32_t w0 = *reinterpret_cast<const uint32_t *>(Ks + box8_chunk<D>(hrow, k) + 4 * quad);
                const uint32_t w1 = *reinterpret_cast<const uint32_t *>(Ks + box8_chunk<D>(hrow + 8, k) + 4 * quad);
                mma_f16_16816(sc[0], qa[k][0], 0u, qa[k][1], 0u, e4m3x2_to_f16x2(w0),
                              e4m3x2_to_f16x2(w0 >> 16));
                mma_f16_16816(sc[1], qa[k][0], 0u, qa[k][1], 0u, e4m3x2_to_f16x2(w1),
                              e4m3x2_to_f16x2(w1 >> 16));
            }
            // ---- online softmax (log2 domain) ----
            float sv[4] = {sc[0][0], sc[0][1], sc[1][0], sc[1][1]};
            const int tq = 2 * quad;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int t = tq + (i & 1) + ((i >> 1) << 3);
                sv[i] = t < nvw ? sv[i] * p.scale_log2 : -INFINITY;
            }
            float mt = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
            mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 1));
            mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 2));
            const float m_new = fmaxf(m_run, mt);
            const float alpha = fast_exp2(m_run - m_new);
            m_run = m_new;
            float pr[4];
#pragma unroll
            for (int i = 0; i < 4; i++)
                pr[i] = real ? fast_exp2(sv[i] - m_new) : 0.f;
            l_run = l_run * alpha + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
#pragma unroll
            for (int n = 0; n < NT; n++) {
                o[n][0] *= alpha;
                o[n][1] *= alpha;
            }
            const uint32_t ph0 = pack_f16x2(pr[0], pr[1]);
            const uint32_t ph2 = pack_f16x2(pr[2], pr[3]);
            // ---- O += P V ----
            const int c = hrow;  // this lane's column within every n-tile
#pragma unroll
            for (int g4 = 0; g4 < NG; g4++) {
                const int chunk = 2 * g4 + (c >> 2);
                const int wofs = 4 * (c & 3);
                const uint32_t v0 = *reinterpret_cast<const uint32_t *>(Vs + box8_chunk<D>(tq, chunk) + wofs);
                const uint32_t v1 = *reinterpret_cast<const uint32_t *>(Vs + box8_chunk<D>(tq + 1, chunk) + wofs);
                const uint32_t v2 = *reinterpret_cast<const uint32_t *>(Vs + box8_chunk<D>(tq + 8, chunk) + wofs);
                const uint32_t v3 = *reinterpret_cast<const uint32_t *>(Vs + box8_chunk<D>(tq + 9, chunk) + wofs);
#pragma unroll
                for (int r = 0; r < 4; r++) {
                    const uint32_t sel = (uint32_t)(r | ((4 + r) << 4));
                    const uint32_t b0 = e4m3x2_to_f16x2(prmt(v0, v1, sel));
                    const uint32_t b1 = e4m3x2_to_f16x2(prmt(v2, v3, sel));
                    mma_f16_16816(o[4 * g4 + r], ph0, 0u, ph2, 0u, b0, b1);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[stage]);

        if (bm.flags & kPieceLast) {
            float l_tot = l_run + __shfl_xor_sync(FULL, l_run, 1);
            l_tot += __shfl_xor_sync(FULL, l_tot, 2);
            const bool complete = whole && (bm.flags & kStreamLast);
            if (real) {
                const size_t hq = (size_t)bm.b * p.Hq + (size_t)bm.h * G + hrow;
                if (complete) {
                    const float f = l_tot > 0.f ? p.v_scale / l_tot : 0.f;
#pragma unroll
                    for (int g4 = 0; g4 < NG; g4++) {
                        // outputs d = 32 g4 + 8 quad + 0..7
                        const uint4 pk = make_uint4(
                            pack_bf16x2(o[4 * g4 + 0][0] * f, o[4 * g4 + 1][0] * f),
                            pack_bf16x2(o[4 * g4 + 2][0] * f, o[4 * g4 + 3][0] * f),
                            pack_bf16x2(o[4 * g4 + 0][1] * f, o[4 * g4 + 1][1] * f),
                            pack_bf16x2(o[4 * g4 + 2][1] * f, o[4 * g4 + 3][1] * f));
                        *reinterpret_cast<uint4 *>(p.out + hq * D + 32 * g4 + 8 * quad) = pk;
                    }
                } else {
                    float *pg = p.ws_part +
                                (((size_t)gw * 2 + ((bm.flags & kSlot1) ? 1 : 0)) * G + hrow) * (D + 4);
                    const float vs = p.v_scale;
#pragma unroll
                    for (int g4 = 0; g4 < NG; g4++) {
                        float *dst = pg + 32 * g4 + 8 * quad;
                        *reinterpret_cast<float4 *>(dst) =
                            make_float4(o[4 * g4 + 0][0] * vs, o[4 * g4 + 1][0] * vs,
                                        o[4 * g4 + 2][0] * vs, o[4 * g4 + 3][0] * vs);
                        *reinterpret_cast<float4 *>(dst + 4) =
                            make_float4(o[4 * g4 + 0][1] * vs, o[4 * g4 + 1][1] * vs,
                                        o[4 * g4 + 2][1] * vs, o[4 * g4 + 3][1] * vs);
                    }
                    if (quad == 0) {
                        pg[D] = m_run;
                        pg[D + 1] = l_tot;
                    }
                }
            }
        }
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1;
        }
    }
}

// Per-sequence clamped lengths and the exclusive prefix sum of their box
// counts (boxes per KV head before sequence b), b = 0..B.
__device__ __forceinline__ void build_prefix(const DecodeParams &p, int *pb, int *len, int *wsum)
{
    const int tid = threadIdx.x, nt = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int maxctx = p.MBS * p.bs;
    const int per = (p.B + nt - 1) / nt;
    const int lo = min(p.B, tid * per), hi = min(p.B, lo + per);
    bool bad = false;
    int local = 0;
    for (int b = lo; b < hi; b++) {
        int n = __ldg(p.context_lens + b);
        if (n < 0 || n > maxctx) {
            bad = true;
            n = n < 0 ? 0 : maxctx;
        }
        len[b] = n;
        local += (n + kBox - 1) / kBox;
    }
    if (bad && blockIdx.x == 0)
        flag_error(p.err_flag, 0x4 /* PKV_FLAG_BAD_CONTEXT_LEN */);
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off)
            incl += t;
    }
    if (lane == 31)
        wsum[warp] = incl;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < nt / 32; w++) {
            const int t = wsum[w];
            wsum[w] = run;
            run += t;
        }
        wsum[nt / 32] = run;
    }
    __syncthreads();
    int run = wsum[warp] + incl - local;
    for (int b = lo; b < hi; b++) {
        pb[b] = run;
        run += (len[b] + kBox - 1) / kBox;
    }
    if (tid == 0)
        pb[p.B] = wsum[nt / 32];
    __syncthreads();
}

template <int D, int G, int NW, bool F8>
__global__ void __launch_bounds__((NW + 1) * 32, NW == kPairWorkers ? 2 : 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const DecodeParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const DecodeSmem L = decode_smem_layout(D, G, NW, p.stages, p.B, F8 ? 1 : 2);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    grid_launch_dependents();
    if (threadIdx.x == 0) {
        uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
        uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
        for (int s = 0; s < p.stages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        fence_mbarrier_init();
    }
    int *pb = reinterpret_cast<int *>(smem + L.pb);
    int *len = reinterpret_cast<int *>(smem + L.len);
    build_prefix(p, pb, len, reinterpret_cast<int *>(smem + L.scan));  // ends with __syncthreads()

    // Slicing: with at least one worker per KV head, each head's region of
    // the concatenated streams gets W / Hkv workers and is cut on its own, so
    // worker w and worker w + W / Hkv read the same (sequence, box) of two
    // heads at the same time; otherwise one region spans all heads.
    const int W = (int)gridDim.x * NW;       // workers
    const int R = W >= p.Hkv ? p.Hkv : 1;    // regions
    const int Tr = pb[p.B] * (p.Hkv / R);    // boxes per region
    const int Wr = W / R;                    // workers per region
    const int P = Tr > 0 ? (Tr + Wr - 1) / Wr : 1;

    if (warp == NW) {
        decode_producer<D, G, NW, F8>(&tmk, &tmv, p, smem, L, lane, R, Tr, Wr, P);
    } else {
        if (blockIdx.x == 0) {
            // Publish the box layout for the merge kernel (after the previous
            // step's kernels, which may still read the workspace).
            grid_dependency_wait();
            for (int i = threadIdx.x; i <= p.B; i += NW * 32)
                p.ws_hdr[kWsHeaderInts + i] = pb[i];
            if (threadIdx.x == 0) {
                p.ws_hdr[0] = Tr;
                p.ws_hdr[1] = P;
                p.ws_hdr[2] = Wr;
                p.ws_hdr[3] = p.B;
                p.ws_hdr[4] = R;
            }
        }
        if constexpr (F8)
            decode_consumer_fp8<D, G, NW>(p, smem, L, warp, lane);
        else
            decode_consumer<D, G, NW>(p, smem, L, warp, lane);
    }
}

template <int D, int NW, bool F8>
inline cudaError_t launch_decode_shape(int G, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                       const DecodeParams &p, int grid, size_t smem,
                                       cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((NW + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (G) {
    case 1: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 1, NW, F8>, *tmk, *tmv, p);
    case 2: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 2, NW, F8>, *tmk, *tmv, p);
    case 4: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 4, NW, F8>, *tmk, *tmv, p);
    case 8: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 8, NW, F8>, *tmk, *tmv, p);
    default: return cudaErrorInvalidValue;
    }
}

template <int D, int NW, bool F8> inline const void *decode_kernel_shape(int G)
{
    switch (G) {
    case 1: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 1, NW, F8>);
    case 2: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 2, NW, F8>);
    case 4: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 4, NW, F8>);
    case 8: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 8, NW, F8>);
    default: return nullptr;
    }
}

} // namespace pkv
