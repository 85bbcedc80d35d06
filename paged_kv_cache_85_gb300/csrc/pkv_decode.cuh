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
//  * Split-K.  Each sequence's context is cut into partitions of `chunk`
//    tokens.  A work unit is one (partition, sequence, KV head); all G query
//    heads sharing that KV head are handled together, so every K/V byte is
//    read from HBM once.  Units are enumerated partition-major (all
//    sequences' first partitions, then the second ones, ...), which keeps
//    sequences that share prefix blocks reading them at the same time, and
//    they are dealt round-robin to a persistent grid of CTAs sized to fill
//    the 152 SMs.  Each CTA rebuilds the unit map from context_lens in
//    shared memory (a histogram + prefix sum), so the host never reads
//    context lengths and the call needs no host synchronisation.
//  * Producer warp.  One warp walks the CTA's units, resolves the block
//    table 32 boxes ahead (one coalesced load per 512 tokens, prefetched one
//    segment in advance), and issues TMA copies of 16-token boxes of K and V
//    ([16 tokens x D] bf16 from the [NB*bs, Hkv, D] cache view) into a ring
//    of shared-memory stages, each completed on an mbarrier with its byte
//    count.  The unit's G query rows come in with its first tile by a bulk
//    copy.
//  * Consumer warps (4).  Each takes one 16-token box of every 64-token
//    stage.  Scores: 8 lanes share a token (16 B vector loads of the K row,
//    conflict-free), each lane dots its slice of d with all G query rows in
//    packed fp32 FMAs, then a reduce-scatter across the 8 lanes leaves one
//    (token, head) score per lane.  Online softmax in fp32 (log2 domain,
//    running max and sum per head), probabilities go through a tiny shared
//    buffer, and P.V accumulates in packed fp32 FMAs with each lane owning
//    D/32 output columns of all G heads.  At the end of a unit the four
//    warps' partial states are merged (log-sum-exp) in shared memory; a
//    sequence with one partition is normalised and written as bf16, one
//    with several writes (acc, max, sum) to the workspace for the merge
//    kernel.
//  * Masking selects out tokens at or past context_len (scores -> -inf and
//    the P.V loop stops at the last valid token), so whatever the unused
//    slots of the last block hold (even NaN) never reaches the output.
#pragma once

#include <cuda_bf16.h>

#include "pkv_kernels.h"
#include "pkv_ptx.cuh"

namespace pkv {

template <int D> struct DecodeShape {
    static constexpr int kStages = D == 128 ? 3 : 6;
    static constexpr int kRowBytes = D * 2;
    static constexpr int kBoxBytes = kBox * kRowBytes;
    static constexpr int kTileBytes = kTile * kRowBytes;
};

// Per-stage descriptor written by the producer before it arms the stage.
struct __align__(16) StageMeta {
    int b, h, c, nvalid;
    int flags;
    int pad[3];
};
constexpr int kMetaFirst = 1;   // first tile of its unit (carries the q rows)
constexpr int kMetaLast = 2;    // last tile of its unit
constexpr int kMetaSingle = 4;  // the sequence has one partition: write bf16 out
constexpr int kMetaStop = 1 << 30;
constexpr int kMetaMaskShift = 8;  // bits 8..11: which 16-token boxes were loaded

struct DecodeSmem {
    size_t k, v, q, acc, ml, pbuf, full, empty, meta, prefix, hist, lens, nch, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline DecodeSmem decode_smem_layout(int D, int G, int stages, int B, int S)
{
    DecodeSmem L;
    size_t o = 0;
    const size_t tile = (size_t)kTile * D * 2;
    L.k = o;
    o += stages * tile;
    L.v = o;
    o += stages * tile;
    L.q = o;
    o = align_up(o + (size_t)stages * G * D * 2, 16);
    L.acc = o;
    o = align_up(o + (size_t)kConsumerWarps * G * D * 4, 16);
    L.ml = o;
    o = align_up(o + (size_t)kConsumerWarps * G * 2 * 4, 16);
    L.pbuf = o;
    o = align_up(o + (size_t)kConsumerWarps * kBox * G * 8, 16);
    L.full = o;
    o += stages * 8;
    L.empty = o;
    o += stages * 8;
    L.meta = o = align_up(o, 16);
    o += stages * sizeof(StageMeta);
    L.prefix = o;
    o = align_up(o + (size_t)(S + 1) * 4, 16);
    L.hist = o;
    o = align_up(o + (size_t)(S + 1) * 4, 16);
    L.lens = o;
    o = align_up(o + (size_t)B * 4, 16);
    L.nch = o;
    o = align_up(o + (size_t)B * 2, 16);
    L.total = o;
    return L;
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

// Work unit: (partition c, sequence b, KV head h) covering tokens [t0, t1).
struct Unit {
    int b, h, c, t0, t1, single;
};

// Map unit index u (partition-major order) to its unit; false past the end.
// Whole-warp call (ballot scan over the sequences).
__device__ __forceinline__ bool map_unit(int u, const DecodeParams &p, const int *sP,
                                         const int *sLen, const uint16_t *sN, int lane, Unit &U)
{
    const int total = sP[p.S] * p.Hkv;
    if (u >= total)
        return false;
    const int qi = u / p.Hkv;
    U.h = u - qi * p.Hkv;
    int lo = 0, hi = p.S - 1;  // largest c with sP[c] <= qi
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sP[mid] <= qi)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int c = lo;
    int k = qi - sP[c];  // k-th (0-based) sequence with more than c partitions
    int b = 0;
    for (int base = 0; base < p.B; base += 32) {
        const int bb = base + lane;
        const bool act = bb < p.B && sN[bb] > c;
        const unsigned m = __ballot_sync(0xffffffffu, act);
        const int cnt = __popc(m);
        if (k < cnt) {
            b = base + (int)__fns(m, 0, k + 1);
            break;
        }
        k -= cnt;
    }
    U.b = b;
    U.c = c;
    U.t0 = c * p.chunk;
    U.t1 = min(sLen[b], U.t0 + p.chunk);
    U.single = sN[b] == 1;
    return true;
}

// A stretch of <= kSegTokens tokens of one unit whose block ids are fetched
// by one load per lane (lane i holds the block of box i).
struct Seg {
    Unit U;
    int u, s0, s1;
    bool valid;
};

__device__ __forceinline__ void first_seg(int u, const DecodeParams &p, const int *sP,
                                          const int *sLen, const uint16_t *sN, int lane, Seg &s)
{
    s.u = u;
    s.valid = map_unit(u, p, sP, sLen, sN, lane, s.U);
    if (s.valid) {
        s.s0 = s.U.t0;
        s.s1 = min(s.U.t1, s.s0 + kSegTokens);
    }
}

__device__ __forceinline__ void next_seg(const Seg &cur, const DecodeParams &p, const int *sP,
                                         const int *sLen, const uint16_t *sN, int lane,
                                         Seg &n)
{
    if (cur.valid && cur.s1 < cur.U.t1) {
        n = cur;
        n.s0 = cur.s1;
        n.s1 = min(cur.U.t1, n.s0 + kSegTokens);
    } else {
        first_seg(cur.u + (int)gridDim.x, p, sP, sLen, sN, lane, n);
    }
}

__device__ __forceinline__ int load_seg_blocks(const Seg &s, const DecodeParams &p, int lane)
{
    const int tok = s.s0 + lane * kBox;
    if (!s.valid || tok >= s.s1)
        return -1;
    return __ldg(p.block_tables + (size_t)s.U.b * p.MBS + tok / p.bs);
}

template <int D, int G>
__device__ __forceinline__ void decode_producer(const CUtensorMap *tmk, const CUtensorMap *tmv,
                                                const DecodeParams &p, uint8_t *smem,
                                                const DecodeSmem &L, int lane)
{
    using Sh = DecodeShape<D>;
    constexpr int STAGES = Sh::kStages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    StageMeta *meta = reinterpret_cast<StageMeta *>(smem + L.meta);
    const int *sP = reinterpret_cast<const int *>(smem + L.prefix);
    const int *sLen = reinterpret_cast<const int *>(smem + L.lens);
    const uint16_t *sN = reinterpret_cast<const uint16_t *>(smem + L.nch);

    if (lane == 0) {
        prefetch_tensormap(tmk);
        prefetch_tensormap(tmv);
    }
    Seg cur, nxt;
    first_seg((int)blockIdx.x, p, sP, sLen, sN, lane, cur);
    int cur_blk = load_seg_blocks(cur, p, lane);
    next_seg(cur, p, sP, sLen, sN, lane, nxt);
    int nxt_blk = load_seg_blocks(nxt, p, lane);

    // K/V may have just been written by store_kvcache on this stream.
    grid_dependency_wait();

    int stage = 0;
    uint32_t phase = 0;
    while (cur.valid) {
        for (int ts = cur.s0; ts < cur.s1; ts += kTile) {
            const int nvalid = min(kTile, cur.U.t1 - ts);
            const int box0 = (ts - cur.s0) / kBox;
            int blk[4];
            int mask = 0;
            bool bad = false;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                blk[j] = __shfl_sync(0xffffffffu, cur_blk, (box0 + j) & 31);
                if (j * kBox < nvalid) {
                    if (blk[j] >= 0 && blk[j] < p.NB)
                        mask |= 1 << j;
                    else
                        bad = true;
                }
            }
            if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1))) {
                if (lane == 0)
                    flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
                return;
            }
            if (lane == 0) {
                if (bad)
                    flag_error(p.err_flag, 0x2 /* PKV_FLAG_BAD_BLOCK */);
                const bool first = ts == cur.U.t0;
                const bool last = ts + kTile >= cur.U.t1;
                StageMeta &m = meta[stage];
                m.b = cur.U.b;
                m.h = cur.U.h;
                m.c = cur.U.c;
                m.nvalid = nvalid;
                m.flags = (first ? kMetaFirst : 0) | (last ? kMetaLast : 0) |
                          (cur.U.single ? kMetaSingle : 0) | (mask << kMetaMaskShift);
                const uint32_t bytes = (uint32_t)__popc(mask) * 2u * Sh::kBoxBytes +
                                       (first ? (uint32_t)(G * D * 2) : 0u);
                mbar_arrive_expect_tx(&full[stage], bytes);
                if (first)
                    bulk_load(smem + L.q + (size_t)stage * G * D * 2,
                              p.q + ((size_t)cur.U.b * p.Hq + (size_t)cur.U.h * G) * D,
                              G * D * 2, &full[stage]);
                uint8_t *kd = smem + L.k + (size_t)stage * Sh::kTileBytes;
                uint8_t *vd = smem + L.v + (size_t)stage * Sh::kTileBytes;
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    if (mask & (1 << j)) {
                        const int tok = ts + j * kBox;
                        const int row = blk[j] * p.bs + tok % p.bs;
                        tma_load_3d(kd + j * Sh::kBoxBytes, tmk, 0, cur.U.h, row, &full[stage]);
                        tma_load_3d(vd + j * Sh::kBoxBytes, tmv, 0, cur.U.h, row, &full[stage]);
                    }
                }
            }
            __syncwarp();
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
        cur = nxt;
        cur_blk = nxt_blk;
        next_seg(cur, p, sP, sLen, sN, lane, nxt);
        nxt_blk = load_seg_blocks(nxt, p, lane);
    }
    // Tell the consumers there is no more work.
    if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1))) {
        if (lane == 0)
            flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
        return;
    }
    if (lane == 0) {
        meta[stage].flags = kMetaStop;
        mbar_arrive(&full[stage]);
    }
}

template <int D, int G>
__device__ __forceinline__ void decode_consumer(const DecodeParams &p, uint8_t *smem,
                                                const DecodeSmem &L, int warp, int lane)
{
    using Sh = DecodeShape<D>;
    constexpr int STAGES = Sh::kStages;
    constexpr int NCH = D / 64;      // 16-byte K chunks per lane per token (2 or 1)
    constexpr int EP = NCH * 4;      // packed fp32 pairs of q per head per lane
    constexpr int DPL = D / 32;      // output columns per lane
    constexpr int VP = DPL / 2;      // packed pairs of output columns
    constexpr int HSHIFT = 3 - GroupLog2<G>::v;
    constexpr unsigned FULL = 0xffffffffu;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    const StageMeta *meta = reinterpret_cast<const StageMeta *>(smem + L.meta);
    float2 *pbuf = reinterpret_cast<float2 *>(smem + L.pbuf) + warp * kBox * G;
    float *sAcc = reinterpret_cast<float *>(smem + L.acc);
    float *sML = reinterpret_cast<float *>(smem + L.ml);

    const int r = lane & 7;        // position within the 8-lane token group
    const int slot = lane >> 3;    // which of 4 tokens this lane scores per step
    const int hsel = r >> HSHIFT;  // head of this lane's score after the reduction
    const bool leader = (r & ((1 << HSHIFT) - 1)) == 0;

    float2 qv[G][EP];
    float2 acc[G][VP];
    float m_run = -INFINITY, l_run = 0.f;
#pragma unroll
    for (int g = 0; g < G; g++)
#pragma unroll
        for (int i = 0; i < VP; i++)
            acc[g][i] = make_float2(0.f, 0.f);

    int stage = 0;
    uint32_t phase = 0;
    for (;;) {
        if (!__all_sync(FULL, mbar_wait(&full[stage], phase))) {
            if (lane == 0)
                flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
            return;
        }
        const StageMeta m = meta[stage];
        if (m.flags & kMetaStop)
            break;
        const uint8_t *Ks = smem + L.k + (size_t)stage * Sh::kTileBytes + warp * Sh::kBoxBytes;
        const uint8_t *Vs = smem + L.v + (size_t)stage * Sh::kTileBytes + warp * Sh::kBoxBytes;

        if (m.flags & kMetaFirst) {
            const uint8_t *qs = smem + L.q + (size_t)stage * G * D * 2;
#pragma unroll
            for (int g = 0; g < G; g++)
#pragma unroll
                for (int ch = 0; ch < NCH; ch++) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(qs + (g * D + ch * 64 + r * 8) * 2);
                    const float2 sc = make_float2(p.scale_log2, p.scale_log2);
                    qv[g][ch * 4 + 0] = __fmul2_rn(bf16x2_to_float2(w.x), sc);
                    qv[g][ch * 4 + 1] = __fmul2_rn(bf16x2_to_float2(w.y), sc);
                    qv[g][ch * 4 + 2] = __fmul2_rn(bf16x2_to_float2(w.z), sc);
                    qv[g][ch * 4 + 3] = __fmul2_rn(bf16x2_to_float2(w.w), sc);
                }
        }

        int nvw = m.nvalid - warp * kBox;
        nvw = nvw < 0 ? 0 : (nvw > kBox ? kBox : nvw);
        if (!((m.flags >> (kMetaMaskShift + warp)) & 1))
            nvw = 0;

        if (nvw > 0) {
            // ---- scores for this warp's 16 tokens (4 per step) ----
            float sv[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int tt = 4 * j + slot;
                const uint8_t *row = Ks + tt * Sh::kRowBytes;
                float2 kf[EP];
#pragma unroll
                for (int ch = 0; ch < NCH; ch++) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(row + ch * 128 + r * 16);
                    kf[ch * 4 + 0] = bf16x2_to_float2(w.x);
                    kf[ch * 4 + 1] = bf16x2_to_float2(w.y);
                    kf[ch * 4 + 2] = bf16x2_to_float2(w.z);
                    kf[ch * 4 + 3] = bf16x2_to_float2(w.w);
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
                const uint8_t *vrow = Vs + t * Sh::kRowBytes + lane * DPL * 2;
                if constexpr (VP == 2) {
                    const uint2 w = *reinterpret_cast<const uint2 *>(vrow);
                    vf[0] = bf16x2_to_float2(w.x);
                    vf[1] = bf16x2_to_float2(w.y);
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

        if (m.flags & kMetaLast) {
            // ---- merge the four warps' partial states for this unit ----
            float l_tot = l_run + __shfl_xor_sync(FULL, l_run, 8);
            l_tot += __shfl_xor_sync(FULL, l_tot, 16);
            if (slot == 0 && leader) {
                sML[(warp * G + hsel) * 2 + 0] = m_run;
                sML[(warp * G + hsel) * 2 + 1] = l_tot;
            }
#pragma unroll
            for (int g = 0; g < G; g++)
#pragma unroll
                for (int i = 0; i < VP; i++)
                    *reinterpret_cast<float2 *>(sAcc + (warp * G + g) * D + lane * DPL + 2 * i) =
                        acc[g][i];
            named_barrier(1, kConsumerWarps * 32);
            const int ct = warp * 32 + lane;
            const bool single = (m.flags & kMetaSingle) != 0;
            for (int idx = ct; idx < G * D; idx += kConsumerWarps * 32) {
                const int g = idx / D;
                const int d = idx - g * D;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; w++)
                    M = fmaxf(M, sML[(w * G + g) * 2]);
                float Ls = 0.f, O = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; w++) {
                    const float e = fast_exp2(sML[(w * G + g) * 2] - M);
                    Ls += sML[(w * G + g) * 2 + 1] * e;
                    O += sAcc[(w * G + g) * D + d] * e;
                }
                const size_t rowi = (size_t)m.b * p.Hq + (size_t)m.h * G + g;
                if (single) {
                    p.out[rowi * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(O / Ls));
                } else {
                    const size_t pi = rowi * p.S + m.c;
                    p.ws_acc[pi * D + d] = O;
                    if (d == 0) {
                        p.ws_ml[pi * 2 + 0] = M;
                        p.ws_ml[pi * 2 + 1] = Ls;
                    }
                }
            }
            named_barrier(1, kConsumerWarps * 32);
            m_run = -INFINITY;
            l_run = 0.f;
#pragma unroll
            for (int g = 0; g < G; g++)
#pragma unroll
                for (int i = 0; i < VP; i++)
                    acc[g][i] = make_float2(0.f, 0.f);
        }
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
        }
    }
}

// Build the CTA's unit map: per sequence its clamped length and number of
// partitions, and sP[c] = number of (sequence, partition) pairs with
// partition index < c, for c = 0..S.
__device__ __forceinline__ void build_unit_map(const DecodeParams &p, uint8_t *smem,
                                               const DecodeSmem &L)
{
    int *sP = reinterpret_cast<int *>(smem + L.prefix);
    int *sH = reinterpret_cast<int *>(smem + L.hist);
    int *sLen = reinterpret_cast<int *>(smem + L.lens);
    uint16_t *sN = reinterpret_cast<uint16_t *>(smem + L.nch);
    const int tid = threadIdx.x;
    for (int i = tid; i <= p.S; i += blockDim.x)
        sH[i] = 0;
    __syncthreads();
    const int maxctx = p.MBS * p.bs;
    bool bad = false;
    for (int b = tid; b < p.B; b += blockDim.x) {
        int n = __ldg(p.context_lens + b);
        if (n < 0 || n > maxctx) {
            bad = true;
            n = n < 0 ? 0 : maxctx;
        }
        const int nc = (n + p.chunk - 1) / p.chunk;
        sLen[b] = n;
        sN[b] = (uint16_t)nc;
        atomicAdd(&sH[nc], 1);
    }
    if (bad && blockIdx.x == 0)
        flag_error(p.err_flag, 0x4 /* PKV_FLAG_BAD_CONTEXT_LEN */);
    __syncthreads();
    if (tid < 32) {
        const int lane = tid;
        // sH[i] <- number of sequences with at least i partitions (suffix sum)
        const int n = p.S + 1;
        const int per = (n + 31) / 32;
        const int lo = min(n, lane * per), hi = min(n, lo + per);
        int tot = 0;
        for (int i = lo; i < hi; i++)
            tot += sH[i];
        int incl = tot;  // sum over lanes >= this one
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_down_sync(0xffffffffu, incl, off);
            if (lane + off < 32)
                incl += t;
        }
        int run = incl - tot;
        for (int i = hi - 1; i >= lo; i--) {
            run += sH[i];
            sH[i] = run;
        }
        __syncwarp();
        // sP[c] = sum_{c' < c} (sequences with more than c' partitions) = sum_{c'<c} sH[c'+1]
        const int m = p.S;  // sP has S+1 entries; element c' contributes sH[c'+1]
        const int per2 = (m + 31) / 32;
        const int lo2 = min(m, lane * per2), hi2 = min(m, lo2 + per2);
        int tot2 = 0;
        for (int i = lo2; i < hi2; i++)
            tot2 += sH[i + 1];
        int inc2 = tot2;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, inc2, off);
            if (lane >= off)
                inc2 += t;
        }
        int run2 = inc2 - tot2;
        for (int i = lo2; i < hi2; i++) {
            sP[i] = run2;
            run2 += sH[i + 1];
        }
        if (lane == 31)
            sP[m] = inc2;
    }
    __syncthreads();
}

template <int D, int G>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const DecodeParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const DecodeSmem L = decode_smem_layout(D, G, DecodeShape<D>::kStages, p.B, p.S);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    grid_launch_dependents();
    if (threadIdx.x == 0) {
        uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
        uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
        for (int s = 0; s < DecodeShape<D>::kStages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbarrier_init();
    }
    build_unit_map(p, smem, L);  // ends with __syncthreads()

    if (warp == kConsumerWarps)
        decode_producer<D, G>(&tmk, &tmv, p, smem, L, lane);
    else
        decode_consumer<D, G>(p, smem, L, warp, lane);
}

template <int D, int G> struct DecodeLauncher {
    static void *fn() { return reinterpret_cast<void *>(&paged_decode_kernel<D, G>); }
};

template <int D>
inline cudaError_t launch_decode_dim(int G, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                     const DecodeParams &p, int grid, size_t smem,
                                     cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (G) {
    case 1: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 1>, *tmk, *tmv, p);
    case 2: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 2>, *tmk, *tmv, p);
    case 4: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 4>, *tmk, *tmv, p);
    case 8: return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, 8>, *tmk, *tmv, p);
    default: return cudaErrorInvalidValue;
    }
}

template <int D> inline const void *decode_kernel_ptr(int G)
{
    switch (G) {
    case 1: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 1>);
    case 2: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 2>);
    case 4: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 4>);
    case 8: return reinterpret_cast<const void *>(&paged_decode_kernel<D, 8>);
    default: return nullptr;
    }
}

} // namespace pkv
