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
//    stream of 16-token boxes (32-token boxes for FP8 caches where three
//    CTAs per SM hold fewer than four 16-token stages and whole 32-token
//    boxes fit in a block); all G query heads of the group ride along, so
//    every K/V byte is read from HBM once.  The streams are concatenated
//    (KV-head-major); each head's region is cut into equal contiguous
//    slices, one per worker, so the workers of different heads read the
//    same token rows at the same time; a worker is one consumer warp.  A
//    persistent grid fills the SMs: two CTAs of four workers (plus a
//    producer warp) per SM for bf16 caches, three for FP8 caches, and one
//    CTA of eight workers per SM where two smaller CTAs do not fit in shared
//    memory (large B, or G = 8 at D = 128).
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


__host__ __device__ inline DecodeSmem decode_smem_layout(int D, int G, int NW, int stages, int B,
                                                         int kv_elem_bytes = 2, int box_tokens = kBox)
{
    DecodeSmem L;
    size_t o = 0;
    L.kv = o;  // per stage: K boxes [NW][D/64][16][64], then V boxes alike (128B-swizzled rows);
               // FP8 boxes [NW][box_tokens][D]
    o += (size_t)stages * 2 * NW * box_tokens * D * kv_elem_bytes;
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
                             int kv_elem_bytes = 2, int box_tokens = kBox)
{
    for (int s = max_stages; s >= kMinStages; s--)
        if (decode_smem_layout(D, G, NW, s, B, kv_elem_bytes, box_tokens).total <= max_smem)
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

template <int BT>
__device__ __forceinline__ int box_block(const DecodeParams &p, int b, int j)
{
    return __ldg(p.block_tables + (size_t)b * p.MBS + (j * BT) / p.bs);
}

// Producer warp: lane w < NW runs worker w of this CTA.  Each lane
// walks its own slice with two cursors: the issue cursor, and a look-ahead
// cursor kLookahead boxes further on whose block ids are loaded into a small
// register queue, so a copy never waits on a block-table read.  Per stage
// every lane writes its worker's box descriptor and issues its own TMA
// copies; lane 0 arms the stage's mbarrier with the summed byte count.
template <int D, int G, int NW, bool F8, int BT>
__device__ __forceinline__ void decode_producer(const CUtensorMap *tmk, const CUtensorMap *tmv,
                                                const DecodeParams &p, uint8_t *smem,
                                                const DecodeSmem &L, int lane, int R, int Tr,
                                                int Wr, int P)
{
    constexpr unsigned FULL = 0xffffffffu;
    constexpr int kBoxBytes = BT * D * (F8 ? 1 : 2);
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
    int qb[kLookahead];  // qb[(pos - start) % kLookahead]: block id of box pos, loaded ahead
#pragma unroll
    for (int i = 0; i < kLookahead; i++) {
        qb[i] = -1;
        if (lpos < end) {
            qb[i] = box_block<BT>(p, lb, lj);
            next_box(pb, p.B, lb, lh, lj);
        }
        ++lpos;
    }
    bool first_done = false;

    // K/V may have just been written by store_kvcache on this stream.
    grid_dependency_wait();

    int stage = 0;
    uint32_t phase = 0;
    bool more = true;
    while (more) {
    // Unrolled by the queue depth: round u uses and refills qb[u] in place,
    // so a block id is first read kLookahead rounds after its load was issued
    // (a shifting queue would wait on the newest load every round).
#pragma unroll
    for (int u = 0; u < kLookahead; u++) {
        const bool mine = pos < end;
        if (!__any_sync(FULL, mine)) {
            more = false;
            break;
        }
        if (!__all_sync(FULL, mbar_wait(&empty[stage], phase ^ 1))) {
            if (lane == 0)
                flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
            return;
        }
        uint32_t bytes = 0;
        int flags = 0, row = 0, b = cb, h = ch;
        if (mine) {
            const int j = cj;
            const int blk = qb[u];
            const int nb = pb[b + 1] - pb[b];
            const int tok0 = j * BT;
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
            m.nvalid = min(BT, len[b] - tok0);
            m.flags = flags;
            m.blk = blk;
            // advance both cursors
            next_box(pb, p.B, cb, ch, cj);
            ++pos;
            qb[u] = -1;
            if (lpos < end) {
                qb[u] = box_block<BT>(p, lb, lj);
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

// Consumer warp for FP8 (E4M3) caches.  Same pipeline, slices and outputs as
// the bf16 consumer; a box of BT = 16 or 32 tokens is taken as BT / 16
// sub-boxes of 16 tokens (one MMA tile each) under one online-softmax update.
// The arithmetic is arranged around the 8-bit data:
//   * scores S^T = K q^T run on the E4M3 tensor-core path (m16n8k32) with the
//     box's 16 tokens as M and the group's heads as N, so K fragments are
//     the raw codes read from shared memory, four per 32-bit word.  q enters
//     as two E4M3 parts under a power-of-two scale per head, q = sq (hi +
//     lo / 16): hi is q / sq rounded to E4M3 and lo the remainder times 16,
//     which represents every bf16 element of magnitude >= max|q| 2^-14
//     exactly (the rest to within max|q| 2^-21).  The contraction index is
//     permuted so that each lane's bytes are one contiguous run of its row;
//   * P.V runs as O^T = V^T P^T in f16 (m16n8k16) with head dimension d as
//     M: E4M3 values are exact in f16, P is rounded to f16, and P^T's
//     fragments come from the score accumulators by one movmatrix transpose.
//     d is permuted so that a lane reads D/8 contiguous bytes of a token row
//     and owns D/8 contiguous outputs per head;
//   * the running max is only moved (and O, l rescaled) when a head's box
//     max exceeds it by more than 2^8, which bounds P by 256 (exact range of
//     f16) and skips the rescale on most boxes.
// k_scale is folded into the score scale and v_scale into the output.
template <int D, int G, int NW, int BT>
__device__ __forceinline__ void decode_consumer_fp8(const DecodeParams &p, uint8_t *smem,
                                                    const DecodeSmem &L, int warp, int lane)
{
    constexpr int KS = D / 32;   // k-steps of the score MMA
    constexpr int KW = D / 16;   // K words per lane per token row (D/4 bytes)
    constexpr int MT = D / 16;   // m-tiles of O^T
    constexpr int VW = D / 32;   // V words per lane per token row (D/8 bytes)
    constexpr int NSUB = BT / 16; // 16-token sub-boxes per box (one MMA M tile each)
    constexpr int kBoxBytes = BT * D;
    constexpr unsigned FULL = 0xffffffffu;
    constexpr float kLazy = 8.f;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    const BoxMeta *meta = reinterpret_cast<const BoxMeta *>(smem + L.meta);

    const int g = lane >> 2;     // token row of S^T, head of q's B fragments, d-group of V
    const int quad = lane & 3;   // heads 2quad, 2quad+1 of S^T and O^T; token pair of V
    const int h0 = 2 * quad, h1 = 2 * quad + 1;
    const int gw = blockIdx.x * NW + warp;

    // shared-memory offsets of this lane's bytes within a box
    uint32_t koff[2][KW / 4];    // rows g, g+8: 16-byte chunks quad*(D/64) + c
#pragma unroll
    for (int c = 0; c < KW / 4; c++) {
        koff[0][c] = box8_chunk<D>(g, quad * (KW / 4) + c);
        koff[1][c] = box8_chunk<D>(g + 8, quad * (KW / 4) + c);
    }
    uint32_t voff[4];            // rows 2quad, 2quad+1, 2quad+8, 2quad+9 at byte g*D/8
    {
        const int rows[4] = {h0, h1, h0 + 8, h1 + 8};
#pragma unroll
        for (int r = 0; r < 4; r++)
            voff[r] = box8_chunk<D>(rows[r], (g * (D / 8)) >> 4) + ((g * (D / 8)) & 15);
    }

    uint32_t qh[KW], ql[KW];
    float f0 = 0.f, f0l = 0.f, f1 = 0.f, f1l = 0.f;
    float o[MT][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool whole = false;
#pragma unroll
    for (int j = 0; j < MT; j++)
        o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
#pragma unroll
    for (int w = 0; w < KW; w++)
        qh[w] = ql[w] = 0u;

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
            // q of head g, d in [quad*D/4, +D/4), split into E4M3 hi / lo
            const uint8_t *qs = smem + L.q + ((size_t)stage * NW + warp) * G * D * 2;
            float x[D / 4];
#pragma unroll
            for (int c = 0; c < D / 32; c++) {
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (g < G)
                    w = *reinterpret_cast<const uint4 *>(qs + (g * D + quad * (D / 4) + 8 * c) * 2);
                const float2 a = bf16x2_to_float2(w.x), b = bf16x2_to_float2(w.y);
                const float2 e = bf16x2_to_float2(w.z), f = bf16x2_to_float2(w.w);
                x[8 * c + 0] = a.x; x[8 * c + 1] = a.y; x[8 * c + 2] = b.x; x[8 * c + 3] = b.y;
                x[8 * c + 4] = e.x; x[8 * c + 5] = e.y; x[8 * c + 6] = f.x; x[8 * c + 7] = f.y;
            }
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < D / 4; i++)
                amax = fmaxf(amax, fabsf(x[i]));
            amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 2));
            // sq = 2^(E - 7) for amax in [2^E, 2^(E+1)): |q / sq| < 256 <= 448
            int ebits = (int)((__float_as_uint(amax) >> 23) & 0xFF);
            ebits = min(max(ebits, 8), 254);
            const float sq = __uint_as_float((uint32_t)(ebits - 7) << 23);
            const float inv = __uint_as_float((uint32_t)(261 - ebits) << 23);
#pragma unroll
            for (int w = 0; w < KW; w++) {
                float xs[4], rs[4];
#pragma unroll
                for (int i = 0; i < 4; i++)
                    xs[i] = x[4 * w + i] * inv;
                const uint32_t c01 = f32x2_to_e4m3x2(xs[0], xs[1]);
                const uint32_t c23 = f32x2_to_e4m3x2(xs[2], xs[3]);
                const float2 b01 = f16x2_to_float2(e4m3x2_to_f16x2(c01));
                const float2 b23 = f16x2_to_float2(e4m3x2_to_f16x2(c23));
                rs[0] = (xs[0] - b01.x) * 16.f;
                rs[1] = (xs[1] - b01.y) * 16.f;
                rs[2] = (xs[2] - b23.x) * 16.f;
                rs[3] = (xs[3] - b23.y) * 16.f;
                qh[w] = c01 | (c23 << 16);
                ql[w] = f32x2_to_e4m3x2(rs[0], rs[1]) | (f32x2_to_e4m3x2(rs[2], rs[3]) << 16);
            }
            const float sq0 = __shfl_sync(FULL, sq, 4 * h0);
            const float sq1 = __shfl_sync(FULL, sq, (4 * h1) & 31);
            f0 = p.scale_log2 * sq0;
            f1 = p.scale_log2 * sq1;
            f0l = f0 * 0.0625f;
            f1l = f1 * 0.0625f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
#pragma unroll
            for (int j = 0; j < MT; j++)
                o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
            whole = (bm.flags & kStreamFirst) != 0;
        }
        const int nvw = (bm.flags & kBoxLoaded) ? bm.nvalid : 0;
        // the stage goes back to the producer once the warp's last read of it
        // (the last V words it needs) is done, before the arithmetic on them
        bool released = false;
        auto release = [&]() {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[stage]);
            released = true;
        };
        if (nvw > 0) {
            const uint8_t *Ks = smem + L.kv + ((size_t)stage * 2 * NW + warp) * kBoxBytes;
            const uint8_t *Vs = Ks + (size_t)NW * kBoxBytes;
            // ---- scores S^T (tokens g, g+8 of each 16-token sub-box; heads h0, h1) ----
            // sub-box u holds tokens 16u .. 16u+15 of the box, 16 D bytes further
            // on (the swizzle pattern repeats every 8 rows)
            float sv[NSUB][4];
            uint32_t vw[NSUB][4][VW];  // V words of tokens 2quad, 2quad+1, 2quad+8, 2quad+9
            auto load_v = [&](int u, int nv) {
                const uint8_t *Vu = Vs + u * 16 * D;
#pragma unroll
                for (int r = 0; r < 4; r++) {
                    if constexpr (VW == 4) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(Vu + voff[r]);
                        vw[u][r][0] = w.x; vw[u][r][1] = w.y; vw[u][r][2] = w.z; vw[u][r][3] = w.w;
                    } else {
                        const uint2 w = *reinterpret_cast<const uint2 *>(Vu + voff[r]);
                        vw[u][r][0] = w.x; vw[u][r][1] = w.y;
                    }
                }
                if (nv < 16) {
                    // V of tokens past the context: 0 (0 * NaN is NaN)
                    const int rows[4] = {h0, h1, h0 + 8, h1 + 8};
#pragma unroll
                    for (int r = 0; r < 4; r++)
                        if (rows[r] >= nv) {
#pragma unroll
                            for (int w = 0; w < VW; w++)
                                vw[u][r][w] = 0u;
                        }
                }
            };
#pragma unroll
            for (int u = 0; u < NSUB; u++) {
                const int nv = nvw - 16 * u;  // valid tokens of the sub-box (warp-uniform)
                if (u > 0 && nv <= 0) {
                    sv[u][0] = sv[u][1] = sv[u][2] = sv[u][3] = -INFINITY;
                    continue;
                }
                const uint8_t *Ku = Ks + u * 16 * D;
                uint32_t ka[2][KW];
#pragma unroll
                for (int r = 0; r < 2; r++)
#pragma unroll
                    for (int c = 0; c < KW / 4; c++) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(Ku + koff[r][c]);
                        ka[r][4 * c + 0] = w.x;
                        ka[r][4 * c + 1] = w.y;
                        ka[r][4 * c + 2] = w.z;
                        ka[r][4 * c + 3] = w.w;
                    }
                float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k = 0; k < KS; k++) {
                    mma_e4m3_16832(sh, ka[0][2 * k], ka[1][2 * k], ka[0][2 * k + 1], ka[1][2 * k + 1],
                                   qh[2 * k], qh[2 * k + 1]);
                    mma_e4m3_16832(sl, ka[0][2 * k], ka[1][2 * k], ka[0][2 * k + 1], ka[1][2 * k + 1],
                                   ql[2 * k], ql[2 * k + 1]);
                }
                sv[u][0] = fmaf(sl[0], f0l, sh[0] * f0);
                sv[u][1] = fmaf(sl[1], f1l, sh[1] * f1);
                sv[u][2] = fmaf(sl[2], f0l, sh[2] * f0);
                sv[u][3] = fmaf(sl[3], f1l, sh[3] * f1);
                // with one sub-box, its V words are loaded before the softmax,
                // whose reductions cover their latency; with two, each after it
                // (registers)
                if (NSUB == 1) {
                    load_v(u, nv);
                    release();
                }
                if (nv < 16) {
                    // tokens past the context: scores -inf
                    if (g >= nv) { sv[u][0] = -INFINITY; sv[u][1] = -INFINITY; }
                    if (g + 8 >= nv) { sv[u][2] = -INFINITY; sv[u][3] = -INFINITY; }
                }
            }
            // ---- online softmax per head column (log2 domain) ----
            float b0 = fmaxf(sv[0][0], sv[0][2]), b1 = fmaxf(sv[0][1], sv[0][3]);
#pragma unroll
            for (int u = 1; u < NSUB; u++) {
                b0 = fmaxf(b0, fmaxf(sv[u][0], sv[u][2]));
                b1 = fmaxf(b1, fmaxf(sv[u][1], sv[u][3]));
            }
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                b0 = fmaxf(b0, __shfl_xor_sync(FULL, b0, x));
                b1 = fmaxf(b1, __shfl_xor_sync(FULL, b1, x));
            }
            if (__any_sync(FULL, b0 > m0 + kLazy || b1 > m1 + kLazy)) {
                const float n0 = fmaxf(m0, b0), n1 = fmaxf(m1, b1);
                const float a0 = fast_exp2(m0 - n0), a1 = fast_exp2(m1 - n1);
                m0 = n0;
                m1 = n1;
                l0 *= a0;
                l1 *= a1;
#pragma unroll
                for (int j = 0; j < MT; j++) {
                    o[j][0] *= a0;
                    o[j][1] *= a1;
                    o[j][2] *= a0;
                    o[j][3] *= a1;
                }
            }
#pragma unroll
            for (int u = 0; u < NSUB; u++) {
                const int nv = nvw - 16 * u;
                if (u > 0 && nv <= 0)
                    continue;  // no valid token: every weight is 0
                const float p0 = fast_exp2(sv[u][0] - m0), p1 = fast_exp2(sv[u][1] - m1);
                const float p2 = fast_exp2(sv[u][2] - m0), p3 = fast_exp2(sv[u][3] - m1);
                l0 += p0 + p2;
                l1 += p1 + p3;
                const uint32_t pb0 = movmatrix_trans(pack_f16x2(p0, p1));
                const uint32_t pb1 = movmatrix_trans(pack_f16x2(p2, p3));
                if (NSUB > 1) {
                    load_v(u, nv);
                    if (u == NSUB - 1 || nvw <= 16 * (u + 1))
                        release();
                }
                // ---- O^T += V^T P^T ----
#pragma unroll
                for (int w = 0; w < VW; w++) {
                    uint32_t a[2][4];  // [m-tile 2w + i][a0..a3]
#pragma unroll
                    for (int i = 0; i < 2; i++) {
                        const uint32_t sel = i == 0 ? 0x5140u : 0x7362u;
                        e4m3x4_to_f16x2x2(prmt(vw[u][0][w], vw[u][1][w], sel), a[i][0], a[i][1]);
                        e4m3x4_to_f16x2x2(prmt(vw[u][2][w], vw[u][3][w], sel), a[i][2], a[i][3]);
                        mma_f16_16816(o[2 * w + i], a[i][0], a[i][1], a[i][2], a[i][3], pb0, pb1);
                    }
                }
            }
        }
        if (!released)
            release();

        if (bm.flags & kPieceLast) {
            float t0 = l0, t1 = l1;
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                t0 += __shfl_xor_sync(FULL, t0, x);
                t1 += __shfl_xor_sync(FULL, t1, x);
            }
            const bool complete = whole && (bm.flags & kStreamLast);
            const size_t hq0 = (size_t)bm.b * p.Hq + (size_t)bm.h * G;
            // this lane owns d = g*D/8 + 0 .. D/8-1 of heads h0 (o[.][0], o[.][2]) and h1
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                const int head = hh == 0 ? h0 : h1;
                if (head >= G)
                    continue;
                const float lt = hh == 0 ? t0 : t1;
                const float mr = hh == 0 ? m0 : m1;
                if (complete) {
                    const float f = lt > 0.f ? p.v_scale / lt : 0.f;
                    uint16_t *dst = p.out + (hq0 + head) * D + g * (D / 8);
#pragma unroll
                    for (int c = 0; c < D / 64; c++) {
                        uint32_t pk[4];
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const int j = 4 * c + i;
                            pk[i] = pack_bf16x2(o[j][hh] * f, o[j][2 + hh] * f);
                        }
                        *reinterpret_cast<uint4 *>(dst + 8 * c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                } else {
                    float *pg = p.ws_part +
                                (((size_t)gw * 2 + ((bm.flags & kSlot1) ? 1 : 0)) * G + head) * (D + 4);
                    const float vs = p.v_scale;
#pragma unroll
                    for (int c = 0; c < D / 32; c++) {
                        const int j = 2 * c;
                        *reinterpret_cast<float4 *>(pg + g * (D / 8) + 4 * c) =
                            make_float4(o[j][hh] * vs, o[j][2 + hh] * vs, o[j + 1][hh] * vs,
                                        o[j + 1][2 + hh] * vs);
                    }
                    if (g == 0) {
                        pg[D] = mr;
                        pg[D + 1] = lt;
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
// counts (boxes of BT tokens per KV head before sequence b), b = 0..B.
template <int BT>
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
        local += (n + BT - 1) / BT;
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
        run += (len[b] + BT - 1) / BT;
    }
    if (tid == 0)
        pb[p.B] = wsum[nt / 32];
    __syncthreads();
}

// BT: tokens per box (16; 32 for FP8 caches whose block size is a multiple
// of 32, which halves the per-box work of the producer and the consumers).
template <int D, int G, int NW, bool F8, int BT>
__global__ void __launch_bounds__((NW + 1) * 32, NW == kPairWorkers ? (F8 ? 3 : 2) : 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const DecodeParams p)
{
    static_assert(BT == kBox || (F8 && BT == 2 * kBox), "32-token boxes on the FP8 path only");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const DecodeSmem L = decode_smem_layout(D, G, NW, p.stages, p.B, F8 ? 1 : 2, BT);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // No early launch of the dependent merge kernel: launched at this grid's
    // start, its CTAs would hold SM resources the decode CTAs need (measured:
    // 28% slower FP8 decode at three CTAs per SM).  It starts as CTAs exit.
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
    build_prefix<BT>(p, pb, len, reinterpret_cast<int *>(smem + L.scan));  // ends with __syncthreads()

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
        decode_producer<D, G, NW, F8, BT>(&tmk, &tmv, p, smem, L, lane, R, Tr, Wr, P);
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
            decode_consumer_fp8<D, G, NW, BT>(p, smem, L, warp, lane);
        else
            decode_consumer<D, G, NW>(p, smem, L, warp, lane);
    }
}

template <int D, int NW, bool F8, int BT = kBox>
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
    case 1: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 1, NW, F8, BT>, *tmk, *tmv, p);
    case 2: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 2, NW, F8, BT>, *tmk, *tmv, p);
    case 4: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 4, NW, F8, BT>, *tmk, *tmv, p);
    case 8: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 8, NW, F8, BT>, *tmk, *tmv, p);
    default: return cudaErrorInvalidValue;
    }
}

template <int D, int NW, bool F8, int BT = kBox> inline const void *decode_kernel_shape(int G)
{
    switch (G) {
    case 1: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 1, NW, F8, BT>);
    case 2: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 2, NW, F8, BT>);
    case 4: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 4, NW, F8, BT>);
    case 8: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 8, NW, F8, BT>);
    default: return nullptr;
    }
}

} // namespace pkv
