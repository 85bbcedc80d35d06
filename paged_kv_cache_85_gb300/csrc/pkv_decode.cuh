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
//  * Consumer warps (workers).  Scores: 8 lanes share a token (16-byte,
//    conflict-free reads of the K row); each lane dots its slice of d with
//    all G query rows in packed fp32 FMAs, and a reduce-scatter across the
//    8 lanes leaves one (token, head) score per lane.  Online softmax in fp32
//    (log2 domain, running max and sum per head); probabilities go through a
//    small per-warp buffer; P.V accumulates in packed fp32 FMAs with each
//    lane owning D/32 output columns of all G heads.  When a worker finishes
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
    size_t kv, q, pbuf, full, empty, meta, pb, len, scan, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline DecodeSmem decode_smem_layout(int D, int G, int NW, int stages, int B)
{
    DecodeSmem L;
    size_t o = 0;
    L.kv = o;  // per stage: K boxes [NW][16][D], then V boxes [NW][16][D]
    o += (size_t)stages * 2 * NW * kBox * D * 2;
    L.q = o;  // per stage and worker: G query rows
    o = align_up(o + (size_t)stages * NW * G * D * 2, 16);
    L.pbuf = o;  // per worker: probabilities [16 tokens][G] as (p, p) pairs
    o = align_up(o + (size_t)NW * kBox * G * 8, 16);
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
    L.total = o;
    return L;
}

// Deepest pipeline (2..max_stages) whose shared memory fits max_smem.
inline int decode_stages_for(int D, int G, int NW, int B, int max_stages, size_t max_smem)
{
    for (int s = max_stages; s >= kMinStages; s--)
        if (decode_smem_layout(D, G, NW, s, B).total <= max_smem)
            return s;
    return 0;
}

// Sum of G per-lane partial values over the 8 lanes of a token group, left
// as one (token, head) value per lane: halving exchanges while more than one
// head remains, plain butterflies after.  The head a lane ends with is
// (lane & 7) >> (3 - log2 G).
template <int N> __device__ __forceinline__ void halve(float *x, int lane, int mask)
{
    const bool upper = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; i++) {
        const float send = upper ? x[i] : x[i + N / 2];
        const float keep = upper ? x[i + N / 2] : x[i];
        x[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
    }
}

template <int G> __device__ __forceinline__ float reduce_scatter8(float (&x)[G], int lane)
{
    if constexpr (G == 8) {
        halve<8>(x, lane, 4);
        halve<4>(x, lane, 2);
        halve<2>(x, lane, 1);
    } else if constexpr (G == 4) {
        halve<4>(x, lane, 4);
        halve<2>(x, lane, 2);
        x[0] += __shfl_xor_sync(0xffffffffu, x[0], 1);
    } else if constexpr (G == 2) {
        halve<2>(x, lane, 4);
        x[0] += __shfl_xor_sync(0xffffffffu, x[0], 2);
        x[0] += __shfl_xor_sync(0xffffffffu, x[0], 1);
    } else {
        x[0] += __shfl_xor_sync(0xffffffffu, x[0], 4);
        x[0] += __shfl_xor_sync(0xffffffffu, x[0], 2);
        x[0] += __shfl_xor_sync(0xffffffffu, x[0], 1);
    }
    return x[0];
}

template <int G> struct GroupLog2;
template <> struct GroupLog2<1> { static constexpr int v = 0; };
template <> struct GroupLog2<2> { static constexpr int v = 1; };
template <> struct GroupLog2<4> { static constexpr int v = 2; };
template <> struct GroupLog2<8> { static constexpr int v = 3; };

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
template <int D, int G, int NW>
__device__ __forceinline__ void decode_producer(const CUtensorMap *tmk, const CUtensorMap *tmv,
                                                const DecodeParams &p, uint8_t *smem,
                                                const DecodeSmem &L, int lane, int R, int Tr,
                                                int Wr, int P)
{
    constexpr unsigned FULL = 0xffffffffu;
    constexpr int kBoxBytes = kBox * D * 2;
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
        if (flags & kBoxLoaded) {
            uint8_t *kd = smem + L.kv + ((size_t)stage * 2 * NW + lane) * kBoxBytes;
            tma_load_3d(kd, tmk, 0, h, row, &full[stage]);
            tma_load_3d(kd + (size_t)NW * kBoxBytes, tmv, 0, h, row, &full[stage]);
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

template <int D, int G, int NW>
__device__ __forceinline__ void decode_consumer(const DecodeParams &p, uint8_t *smem,
                                                const DecodeSmem &L, int warp, int lane)
{
    constexpr int NCH = D / 64;      // 16-byte K chunks per lane per token (2 or 1)
    constexpr int EP = NCH * 4;      // packed fp32 pairs of q per head per lane
    constexpr int DPL = D / 32;      // output columns per lane
    constexpr int VP = DPL / 2;      // packed pairs of output columns
    constexpr int HSHIFT = 3 - GroupLog2<G>::v;
    constexpr int kBoxBytes = kBox * D * 2;
    constexpr int kRowBytes = D * 2;
    constexpr unsigned FULL = 0xffffffffu;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    const BoxMeta *meta = reinterpret_cast<const BoxMeta *>(smem + L.meta);
    float2 *pbuf = reinterpret_cast<float2 *>(smem + L.pbuf) + warp * kBox * G;

    const int r = lane & 7;        // position within the 8-lane token group
    const int slot = lane >> 3;    // which of 4 tokens this lane scores per step
    const int hsel = r >> HSHIFT;  // head of this lane's score after the reduction
    const bool leader = (r & ((1 << HSHIFT) - 1)) == 0;
    const int gw = blockIdx.x * NW + warp;

    float2 qv[G][EP];
    float2 acc[G][VP];
    float m_run = -INFINITY, l_run = 0.f;
    bool whole = false;  // the current piece began at its stream's first box
#pragma unroll
    for (int g = 0; g < G; g++) {
#pragma unroll
        for (int i = 0; i < EP; i++)
            qv[g][i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < VP; i++)
            acc[g][i] = make_float2(0.f, 0.f);
    }

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
            const float2 sc = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
            for (int g = 0; g < G; g++)
#pragma unroll
                for (int ch = 0; ch < NCH; ch++) {
                    const uint4 w4 =
                        *reinterpret_cast<const uint4 *>(qs + (g * D + ch * 64 + r * 8) * 2);
                    qv[g][ch * 4 + 0] = __fmul2_rn(bf16x2_to_float2(w4.x), sc);
                    qv[g][ch * 4 + 1] = __fmul2_rn(bf16x2_to_float2(w4.y), sc);
                    qv[g][ch * 4 + 2] = __fmul2_rn(bf16x2_to_float2(w4.z), sc);
                    qv[g][ch * 4 + 3] = __fmul2_rn(bf16x2_to_float2(w4.w), sc);
                }
            m_run = -INFINITY;
            l_run = 0.f;
#pragma unroll
            for (int g = 0; g < G; g++)
#pragma unroll
                for (int i = 0; i < VP; i++)
                    acc[g][i] = make_float2(0.f, 0.f);
            whole = (bm.flags & kStreamFirst) != 0;
        }
        const int nvw = (bm.flags & kBoxLoaded) ? bm.nvalid : 0;
        if (nvw > 0) {
            const uint8_t *Ks = smem + L.kv + ((size_t)stage * 2 * NW + warp) * kBoxBytes;
            const uint8_t *Vs = Ks + (size_t)NW * kBoxBytes;
            // ---- scores for the box's 16 tokens (4 per step) ----
            float sv[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int tt = 4 * j + slot;
                const uint8_t *row = Ks + tt * kRowBytes;
                float2 kf[EP];
#pragma unroll
                for (int ch = 0; ch < NCH; ch++) {
                    const uint4 w4 = *reinterpret_cast<const uint4 *>(row + ch * 128 + r * 16);
                    kf[ch * 4 + 0] = bf16x2_to_float2(w4.x);
                    kf[ch * 4 + 1] = bf16x2_to_float2(w4.y);
                    kf[ch * 4 + 2] = bf16x2_to_float2(w4.z);
                    kf[ch * 4 + 3] = bf16x2_to_float2(w4.w);
                }
                float part[G];
#pragma unroll
                for (int g = 0; g < G; g++) {
                    float2 a = __fmul2_rn(qv[g][0], kf[0]);
#pragma unroll
                    for (int i = 1; i < EP; i++)
                        a = __ffma2_rn(qv[g][i], kf[i], a);
                    part[g] = a.x + a.y;
                }
                const float s = reduce_scatter8<G>(part, lane);
                sv[j] = tt < nvw ? s : -INFINITY;
            }
            // ---- online softmax (log2 domain) ----
            float mt = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
            mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 8));
            mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 16));
            const float m_new = fmaxf(m_run, mt);
            const float alpha = fast_exp2(m_run - m_new);
            m_run = m_new;
            float psum = 0.f;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const float pj = fast_exp2(sv[j] - m_new);
                psum += pj;
                if (leader)
                    pbuf[(4 * j + slot) * G + hsel] = make_float2(pj, pj);
            }
            l_run = l_run * alpha + psum;
#pragma unroll
            for (int g = 0; g < G; g++) {
                const float ag = __shfl_sync(FULL, alpha, g << HSHIFT);
                const float2 a2 = make_float2(ag, ag);
#pragma unroll
                for (int i = 0; i < VP; i++)
                    acc[g][i] = __fmul2_rn(acc[g][i], a2);
            }
            __syncwarp();
            // ---- P.V ----
            auto pv_step = [&](int t) {
                float2 pp[G];
                if constexpr (G == 1) {
                    pp[0] = pbuf[t];
                } else {
#pragma unroll
                    for (int g = 0; g < G; g += 2) {
                        const float4 x = *reinterpret_cast<const float4 *>(pbuf + t * G + g);
                        pp[g] = make_float2(x.x, x.y);
                        pp[g + 1] = make_float2(x.z, x.w);
                    }
                }
                float2 vf[VP];
                const uint8_t *vrow = Vs + t * kRowBytes + lane * DPL * 2;
                if constexpr (VP == 2) {
                    const uint2 w2 = *reinterpret_cast<const uint2 *>(vrow);
                    vf[0] = bf16x2_to_float2(w2.x);
                    vf[1] = bf16x2_to_float2(w2.y);
                } else {
                    vf[0] = bf16x2_to_float2(*reinterpret_cast<const uint32_t *>(vrow));
                }
#pragma unroll
                for (int g = 0; g < G; g++)
#pragma unroll
                    for (int i = 0; i < VP; i++)
                        acc[g][i] = __ffma2_rn(pp[g], vf[i], acc[g][i]);
            };
            if (nvw == kBox) {
#pragma unroll
                for (int t = 0; t < kBox; t++)
                    pv_step(t);
            } else {
                for (int t = 0; t < nvw; t++)
                    pv_step(t);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[stage]);

        if (bm.flags & kPieceLast) {
            // ---- finish this worker's piece of the stream ----
            float l_tot = l_run + __shfl_xor_sync(FULL, l_run, 8);
            l_tot += __shfl_xor_sync(FULL, l_tot, 16);
            const bool complete = whole && (bm.flags & kStreamLast);
            const size_t row0 = (size_t)bm.b * p.Hq + (size_t)bm.h * G;
            float *part = p.ws_part +
                          ((size_t)gw * 2 + ((bm.flags & kSlot1) ? 1 : 0)) * G * (D + 4);
#pragma unroll
            for (int g = 0; g < G; g++) {
                const float mg = __shfl_sync(FULL, m_run, g << HSHIFT);
                const float lg = __shfl_sync(FULL, l_tot, g << HSHIFT);
                if (complete) {
                    uint32_t pk[VP];
#pragma unroll
                    for (int i = 0; i < VP; i++) {
                        const float x0 = lg > 0.f ? acc[g][i].x / lg : 0.f;
                        const float x1 = lg > 0.f ? acc[g][i].y / lg : 0.f;
                        pk[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x0)) |
                                ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x1)) << 16);
                    }
                    uint16_t *o = p.out + (row0 + g) * D + lane * DPL;
                    if constexpr (VP == 2)
                        *reinterpret_cast<uint2 *>(o) = make_uint2(pk[0], pk[1]);
                    else
                        *reinterpret_cast<uint32_t *>(o) = pk[0];
                } else {
                    float *pg = part + (size_t)g * (D + 4);
                    if constexpr (VP == 2)
                        *reinterpret_cast<float4 *>(pg + lane * DPL) =
                            make_float4(acc[g][0].x, acc[g][0].y, acc[g][1].x, acc[g][1].y);
                    else
                        *reinterpret_cast<float2 *>(pg + lane * DPL) = acc[g][0];
                    if (lane == 0) {
                        pg[D] = mg;
                        pg[D + 1] = lg;
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

template <int D, int G, int NW>
__global__ void __launch_bounds__((NW + 1) * 32, NW == kPairWorkers ? 2 : 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const DecodeParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const DecodeSmem L = decode_smem_layout(D, G, NW, p.stages, p.B);
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
        decode_producer<D, G, NW>(&tmk, &tmv, p, smem, L, lane, R, Tr, Wr, P);
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
        decode_consumer<D, G, NW>(p, smem, L, warp, lane);
    }
}

template <int D, int NW>
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
    case 1: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 1, NW>, *tmk, *tmv, p);
    case 2: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 2, NW>, *tmk, *tmv, p);
    case 4: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 4, NW>, *tmk, *tmv, p);
    case 8: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 8, NW>, *tmk, *tmv, p);
    default: return cudaErrorInvalidValue;
    }
}

template <int D, int NW> inline const void *decode_kernel_shape(int G)
{
    switch (G) {
    case 1: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 1, NW>);
    case 2: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 2, NW>);
    case 4: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 4, NW>);
    case 8: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 8, NW>);
    default: return nullptr;
    }
}

} // namespace pkv
