// Paged prefill attention on the 5th-generation tensor cores (tcgen05/TMEM).
//
// What it computes (MinivLLM guide §4.5 prepare_prefill): the new tokens of
// all sequences are flattened; new token i of a sequence sits at position
// k_len - q_len + i and attends, causally, to positions 0 .. that one, K/V
// read through the sequence's block table.
//
// Persistent CTAs, two per SM (so one CTA's softmax overlaps the other's
// MMAs), each walking a list of work items: an item is a tile of 128 (token,
// head-in-group) rows of one sequence and KV head.  Items are ranked longest
// first and dealt to the CTAs back and forth (round k: CTA c takes position
// k nC + c, or k nC + nC - 1 - c for odd k).  The producer publishes each item
// to the other warps through a two-slot buffer; ring, S, P and P.V barrier
// phases run on over a CTA's items, so an item's Q and first K tiles load,
// and its first S runs, while the previous item drains.  Warps:
//   0..3  softmax: thread t owns row t (TMEM lane t) -- no shuffles.  Per
//         64-key tile: load S from TMEM and hand the S buffer back at once,
//         exponentiate, write P (f16) into one of two P buffers, and convert
//         the tile's V rows in shared memory from bf16 to f16 in place
//         (zeroing rows past k_len or of unloaded boxes)
//   4     producer: finds the next item, TMA of its Q tile, then 64-key K and
//         V tiles (four 16-token boxes each, resolved through the block
//         table) into two separate 2-stage rings: a K tile is released as
//         soon as its S MMA completes, so the next K tiles load while the
//         softmax runs, and V only has to arrive by its P.V
//   5     MMA: allocates 256 TMEM columns; one lane issues
//           S_j = Q K_j^T    (SS, bf16, K-major 128-byte-swizzled operands,
//                             M=128 N=64, into the single S buffer), and
//           O  += P_j V_j    (TS, f16: P from TMEM, V MN-major from shared
//                             memory, N=D)
// TMEM columns: O in [0, D); S at 128 (64 f32 columns); P buffers at 192 and
// 224 (64 f16 keys = 32 columns each, used by tile parity).  Because P does
// not live in the S buffer, S_{j+1} is issued as soon as the softmax has
// loaded S_j, and runs while the softmax works on S_j; the softmax writes
// P_j only after the P.V that read the same P buffer (P.V_{j-2}) has
// completed (MMAs are not ordered against each other's TMEM accesses).  An
// item's first P.V, which overwrites O, waits until the previous item's
// epilogue has read O out.
// P.V in f16: P = exp2(...) <= 2^8 is rounded to f16 (11 significant bits, 8x
// finer than bf16, so no hi + lo split is needed for the output tolerance), and
// V is converted to f16, exact for every bf16 value of magnitude in
// [2^-14, 65504]; smaller magnitudes round to f16 subnormals (absolute error
// <= 2^-25), larger finite values and infinities clamp to +-65504 and set
// PKV_FLAG_V_RANGE; NaN stays NaN.
// The running max moves only when a row's tile max exceeds it by more than
// 2^8 (then that warp rescales its O rows in TMEM after the previous P.V has
// completed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_kernels.h"
#include "pkv_prefill.h"
#include "pkv_ptx.cuh"
#include "pkv_tc.cuh"

namespace pkv {

constexpr int kTcRows = 128;            // query rows per CTA (MMA M)
constexpr int kTcKeys = 64;             // keys per K/V tile (MMA N of S)
constexpr int kTcKStages = 2;           // K ring depth
constexpr int kTcVStages = 2;           // V ring depth
constexpr int kTcThreads = 6 * 32;
constexpr uint32_t kTcCols = 256;       // TMEM columns per CTA
constexpr uint32_t kTcSCol = 128;       // the S buffer (64 f32 columns)
constexpr uint32_t kTcPCol = 192;       // P buffers at 192 and 224 (64 f16 keys each)
constexpr int kFlagVRange = 0x10;       // PKV_FLAG_V_RANGE (pkv.h)

struct TcSmem {
    size_t q, kv, bars, items, slot, total;
};

__host__ __device__ inline TcSmem tc_smem_layout(int D)
{
    TcSmem L;
    size_t o = 0;
    L.q = o;  // [D/64 halves][128 rows][128 B]
    o += (size_t)(D / 64) * kTcRows * 128;
    L.kv = o;  // K stages [D/64][64 keys][128 B], then V stages alike
    o += (size_t)(kTcKStages + kTcVStages) * (D / 64) * kTcKeys * 128;
    L.bars = o;  // q_full, q_empty, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full,
                 // s_free, pv_ready[2], pv_done[2], o_free, item_ready[2], item_free[2], mma_done
    o += 8 * (2 + 2 * kTcKStages + 2 * kTcVStages + 2 + 2 + 2 + 1 + 2 + 2 + 1);
    L.items = o;  // two published work items of 32 bytes
    o += 2 * 32;
    L.slot = o;
    o += 16;
    L.total = align_up(o, 16) + 1024;
    return L;
}

__device__ __forceinline__ bool prefill_seq_sane(const PrefillParams &p, int cq0, int cq1, int ck0,
                                                 int ck1)
{
    const int q_len = cq1 - cq0, k_len = ck1 - ck0;
    return cq0 >= 0 && q_len >= 0 && (long long)cq1 <= p.Tq && k_len >= q_len &&
           k_len <= p.MBS * p.bs && q_len <= p.max_q;
}

// Query tiles of one sequence whose causal key range spans at least c key
// tiles.  A tile's range grows with its index, so these are its last tiles.
template <int TPC>
__device__ __forceinline__ int tiles_at_least(int q_len, int base, int c)
{
    if (q_len <= 0)
        return 0;
    const int nt = (q_len + TPC - 1) / TPC;
    // tile t reaches key tile c-1 iff min(q_len, (t+1) TPC) >= need
    const int need = kTcKeys * (c - 1) - base + 1;
    if (need <= 0)
        return nt;
    if (need > q_len)
        return 0;
    return nt - ((need + TPC - 1) / TPC - 1);
}

struct PrefillWork {
    int b, kvh, tile;        // b < 0: nothing to do
    int cq0, cq1, ck0, ck1;  // sequence b's boundaries (cq0 == kNotLoaded: read them again)
};
constexpr int kNotLoaded = -2147483647 - 1;
constexpr int kSchedChunks = 8;  // sequences per lane in the longest-first schedule
constexpr int kSchedMaxSeqs = 32 * kSchedChunks;

// The (sequence, KV head, query tile) of work item `pos`, run by one warp.
// Items are handed out longest first (a tile's cost is its number of key
// tiles): with up to kSchedMaxSeqs sequences the item's rank r (its position
// over the KV heads) is mapped to the r-th tile in decreasing cost, found by
// a binary search over the cost with per-sequence closed-form counts, so
// every item after the first empty one is empty too.  Beyond that many
// sequences the last tile of every sequence goes first, then the
// second-to-last ones, and so on (empty items are then interleaved).  NCH
// chunks of 32 sequences are scanned (one lane per sequence).
template <int TPC, int NCH>
__device__ __forceinline__ PrefillWork prefill_schedule(const PrefillParams &p, int lane, int pos)
{
    constexpr unsigned FULL = 0xffffffffu;
    const int B = p.B, Hkv = p.Hkv, X = p.X;
    const int r = pos / Hkv;
    PrefillWork w{-1, pos % Hkv, 0, kNotLoaded, 0, 0, 0};
    if (B > kSchedMaxSeqs) {
        w.b = r % B;
        w.tile = X - 1 - r / B;
        return w;
    }
    int qv[NCH], bv[NCH], q0v[NCH], k0v[NCH];
    int cmax = 1;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < NCH; i++) {
        const int s = lane + 32 * i;
        qv[i] = 0;
        bv[i] = 0;
        q0v[i] = 0;
        k0v[i] = 0;
        if (s < B) {
            const int cq0 = __ldg(p.cu_q + s), cq1 = __ldg(p.cu_q + s + 1);
            const int ck0 = __ldg(p.cu_k + s), ck1 = __ldg(p.cu_k + s + 1);
            q0v[i] = cq0;
            k0v[i] = ck0;
            if (prefill_seq_sane(p, cq0, cq1, ck0, ck1)) {
                qv[i] = cq1 - cq0;
                bv[i] = (ck1 - ck0) - (cq1 - cq0);
                if (ck1 > ck0)
                    cmax = max(cmax, (ck1 - ck0 - 1) / kTcKeys + 1);
            } else {
                bad = true;
            }
        }
    }
    // sequences with bad lengths get no work; one CTA reports them
    if (bad && pos == 0)
        flag_error(p.err_flag, 0x4 /* PKV_FLAG_BAD_CONTEXT_LEN */);
    cmax = __reduce_max_sync(FULL, cmax);
    auto count = [&](int c) {
        int n = 0;
#pragma unroll
        for (int i = 0; i < NCH; i++)
            n += tiles_at_least<TPC>(qv[i], bv[i], c);
        return (int)__reduce_add_sync(FULL, (unsigned)n);
    };
    if (r >= count(1))
        return w;
    int lo = 1, hi = cmax + 1;  // count(lo) > r >= count(hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (count(mid) > r)
            lo = mid;
        else
            hi = mid;
    }
    // rank among the tiles costing exactly lo, in sequence order
    const int rp = r - count(lo + 1);
    int acc = 0;
#pragma unroll
    for (int i = 0; i < NCH; i++) {
        const int at = tiles_at_least<TPC>(qv[i], bv[i], lo);
        const int n = at - tiles_at_least<TPC>(qv[i], bv[i], lo + 1);
        int incl = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(FULL, incl, off);
            if (lane >= off)
                incl += y;
        }
        const int total = __shfl_sync(FULL, incl, 31);
        if (rp < acc + total) {
            const int ex = acc + incl - n;
            const bool mine = rp >= ex && rp < ex + n;
            const int src = __ffs(__ballot_sync(FULL, mine)) - 1;
            const int nt = (qv[i] + TPC - 1) / TPC;
            const int t = nt - at + (rp - ex);  // the first tile costing lo, plus the rank
            w.b = src + 32 * i;
            w.tile = __shfl_sync(FULL, t, src);
            // the winner lane's sequence passed on, so it is not read again
            w.cq0 = __shfl_sync(FULL, q0v[i], src);
            w.ck0 = __shfl_sync(FULL, k0v[i], src);
            w.cq1 = w.cq0 + __shfl_sync(FULL, qv[i], src);
            w.ck1 = w.ck0 + __shfl_sync(FULL, qv[i] + bv[i], src);
            return w;
        }
        acc += total;
    }
    return w;  // not reached: rp < count(lo) - count(lo + 1)
}

// One query tile's work, as the producer publishes it to the other warps.
struct PrefillItem {
    int b, kvh, tok0, cq0, q_len, k_len, nkt;  // b < 0: no more work for this CTA
    int pad;
};

template <int D, int G>
__global__ void __launch_bounds__(kTcThreads, 2)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq,
                            const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv, const PrefillParams p)
{
    constexpr int TPC = kTcRows / G;                  // query tokens per tile
    constexpr int HALVES = D / 64;
    constexpr uint32_t kQHalf = kTcRows * 128;        // 16 KB
    constexpr uint32_t kTileHalf = kTcKeys * 128;     // 8 KB
    constexpr uint32_t kTile = HALVES * kTileHalf;    // one K (or V) tile
    constexpr uint32_t kBoxBytes = kBox * D * 2;
    constexpr unsigned FULL = 0xffffffffu;
    constexpr float kLazy = 8.f;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const TcSmem L = tc_smem_layout(D);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *q_full = bars;                       // Q of the item landed (once per item)
    uint64_t *q_empty = q_full + 1;                // the item's last S completed: Q may be replaced
    uint64_t *k_full = q_empty + 1;
    uint64_t *k_empty = k_full + kTcKStages;
    uint64_t *v_full = k_empty + kTcKStages;
    uint64_t *v_empty = v_full + kTcVStages;
    uint64_t *s_full = v_empty + kTcVStages;       // S_g written (once per tile g)
    uint64_t *s_free = s_full + 1;                 // S_g loaded by all four softmax warps
    uint64_t *pv_ready = s_free + 1;               // [2] P_g written and V_g converted, by g & 1
    uint64_t *pv_done = pv_ready + 2;              // [2] P.V_g completed, by P buffer g & 1
    uint64_t *o_free = pv_done + 2;                // the item's O has been read out
    uint64_t *item_ready = o_free + 1;             // [2] item parameters published
    uint64_t *item_free = item_ready + 2;          // [2] item parameters no longer needed
    uint64_t *mma_done = item_free + 2;            // every MMA of the CTA completed
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem + L.slot);
    PrefillItem *items = reinterpret_cast<PrefillItem *>(smem + L.items);  // [2]
    uint8_t *sQ = smem + L.q;
    uint8_t *sK = smem + L.kv;                                         // kTcKStages K tiles
    uint8_t *sV = sK + (size_t)kTcKStages * (D / 64) * kTcKeys * 128;  // kTcVStages V tiles

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    grid_launch_dependents();
    if (warp == 4 && lane == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < kTcKStages; s++) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kTcVStages; s++) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, 4);  // one arrival per softmax warp
        for (int i = 0; i < 2; i++) {
            mbar_init(&pv_ready[i], 4);
            mbar_init(&pv_done[i], 1);
            mbar_init(&item_ready[i], 1);
            mbar_init(&item_free[i], 5);  // the MMA lane and the four softmax warps
        }
        mbar_init(o_free, 4);
        mbar_init(mma_done, 1);
        fence_mbarrier_init();
    } else if (warp == 5) {
        tc::alloc(smem_u32(slot), kTcCols);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *slot;
    const uint32_t tO = tmem, tS = tmem + kTcSCol, tP0 = tmem + kTcPCol;
    const int nC = (int)gridDim.x;
    const int c = (int)blockIdx.x;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        // Walks this CTA's items: round k takes position k nC + c (k even) or
        // k nC + nC - 1 - c (k odd), so the longest-first order is dealt out
        // back and forth over the CTAs.  For each item: publish it, load Q once
        // the previous item's last S has read the old Q, then its 64-key K and
        // V tiles through the two rings (tile counters gk, gv run over all of
        // this CTA's items).
        if (lane == 0) {
            prefetch_tensormap(&tmq);
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
        grid_dependency_wait();  // K/V may have just been written by store_kvcache
        int gk = 0, gv = 0;      // K and V tiles issued so far (all items)
        bool ok = true;
        int n = 0;               // items published
        int k = 0;               // walk rounds
        for (;;) {
            // ---- the next item with work, or the end
            PrefillItem it{-1, 0, 0, 0, 0, 0, 0, 0};
            for (; ok; k++) {
                const long long pos = (long long)k * nC + ((k & 1) ? nC - 1 - c : c);
                if (pos >= p.n_items)
                    break;
                const PrefillWork w = p.B <= 32 ? prefill_schedule<TPC, 1>(p, lane, (int)pos)
                                                : prefill_schedule<TPC, kSchedChunks>(p, lane, (int)pos);
                int cq0 = w.cq0, cq1 = w.cq1, ck0 = w.ck0, ck1 = w.ck1;
                if (w.b >= 0 && cq0 == kNotLoaded) {
                    cq0 = __ldg(p.cu_q + w.b);
                    cq1 = __ldg(p.cu_q + w.b + 1);
                    ck0 = __ldg(p.cu_k + w.b);
                    ck1 = __ldg(p.cu_k + w.b + 1);
                }
                const bool sane = w.b >= 0 && prefill_seq_sane(p, cq0, cq1, ck0, ck1);
                if (w.b >= 0 && !sane && lane == 0)
                    flag_error(p.err_flag, 0x4 /* PKV_FLAG_BAD_CONTEXT_LEN */);
                const int tok0 = w.tile * TPC;
                if (sane && tok0 < cq1 - cq0) {
                    it.b = w.b;
                    it.kvh = w.kvh;
                    it.tok0 = tok0;
                    it.cq0 = cq0;
                    it.q_len = cq1 - cq0;
                    it.k_len = ck1 - ck0;
                    const int last_pos = (it.k_len - it.q_len) + min(it.q_len, tok0 + TPC) - 1;
                    it.nkt = last_pos / kTcKeys + 1;
                    k++;
                    break;
                }
                // up to kSchedMaxSeqs sequences, ranks are longest first, so
                // the first empty item ends this CTA's work
                if (p.B <= kSchedMaxSeqs && w.b < 0) {
                    k = 0x3fffffff;
                    break;
                }
            }
            // ---- publish it in slot n & 1, once the item two back is done with it
            const int sl = n & 1;
            if (n >= 2 && !(ok = ok && __all_sync(FULL, mbar_wait(&item_free[sl], ((n >> 1) & 1) ^ 1)))) {
                break;  // the other warps time out on item_ready and stop
            }
            if (!ok)
                it.b = -1;
            if (lane == 0)
                items[sl] = it;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&item_ready[sl]);
            if (it.b < 0)
                break;
            // ---- Q, after the previous item's last S
            if (n >= 1 && !(ok = __all_sync(FULL, mbar_wait(q_empty, (n - 1) & 1))))
                break;
            if (lane == 0) {
                mbar_arrive_expect_tx(q_full, HALVES * kQHalf);
#pragma unroll
                for (int h = 0; h < HALVES; h++)
                    tma_load_4d(sQ + h * kQHalf, &tmq, 0, h, it.kvh * G, it.cq0 + it.tok0, q_full);
            }
            n++;
            // ---- K and V tiles.  One converged loop serves both rings: it
            // probes (without blocking) whether the next K stage and the next
            // V stage are free and issues whichever tile can go; lanes 0-3
            // resolve and copy one 16-token box each.  K runs ahead of V by up
            // to its ring depth.
            const int32_t *table = p.block_tables + (size_t)it.b * p.MBS;
            auto issue = [&](int j, int g, bool is_k) {
                uint64_t *fb = is_k ? k_full : v_full;
                const int nst = is_k ? kTcKStages : kTcVStages;
                const int s = g % nst;
                const int key0 = j * kTcKeys + lane * kBox;
                bool loaded = false;
                int row = 0;
                if (lane < kTcKeys / kBox && key0 < it.k_len) {
                    const int blk = __ldg(table + key0 / p.bs);
                    loaded = blk >= 0 && blk < p.NB;
                    if (!loaded && is_k)
                        flag_error(p.err_flag, 0x2 /* PKV_FLAG_BAD_BLOCK */);
                    row = blk * p.bs + key0 % p.bs;
                }
                const uint32_t mask = __ballot_sync(FULL, loaded);
                if (lane == 0)
                    mbar_arrive_expect_tx(&fb[s], (uint32_t)__popc(mask) * kBoxBytes);
                __syncwarp();
                if (loaded) {
                    uint8_t *dst = (is_k ? sK : sV) + (size_t)s * kTile + lane * (kBox * 128);
                    const CUtensorMap *map = is_k ? &tmk : &tmv;
#pragma unroll
                    for (int h = 0; h < HALVES; h++)
                        tma_load_4d(dst + h * kTileHalf, map, 0, h, it.kvh, row, &fb[s]);
                }
            };
            int jk = 0, jv = 0;
            uint64_t t_last = global_timer_ns();
            while (jk < it.nkt || jv < it.nkt) {
                bool prog = false;
                if (jk < it.nkt) {
                    const bool free_k = tc::test_wait(smem_u32(&k_empty[gk % kTcKStages]),
                                                      ((gk / kTcKStages) & 1) ^ 1);
                    if (__shfl_sync(FULL, free_k, 0)) {
                        issue(jk++, gk++, true);
                        prog = true;
                    }
                }
                if (jv < jk) {
                    const bool free_v = tc::test_wait(smem_u32(&v_empty[gv % kTcVStages]),
                                                      ((gv / kTcVStages) & 1) ^ 1);
                    if (__shfl_sync(FULL, free_v, 0)) {
                        issue(jv++, gv++, false);
                        prog = true;
                    }
                }
                if (prog) {
                    t_last = global_timer_ns();
                } else {
                    __nanosleep(32);
                    if (__shfl_sync(FULL, global_timer_ns() - t_last > 2000000000ull, 0)) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok)
                break;  // the other warps time out on their barriers and stop
        }
        if (lane == 0) {
            if (!ok)
                flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
            // copies still in flight land before the CTA may exit
            if (n >= 1)
                mbar_wait(q_full, (n - 1) & 1);
            for (int g = max(0, gk - kTcKStages); g < gk; g++)
                mbar_wait(&k_full[g % kTcKStages], (g / kTcKStages) & 1);
            for (int g = max(0, gv - kTcVStages); g < gv; g++)
                mbar_wait(&v_full[g % kTcVStages], (g / kTcVStages) & 1);
        }
        __syncwarp();
    } else if (warp == 5) {
        // ----------------------------------------------------------------- MMA
        // The whole warp runs the loop and waits on the barriers; one elected
        // lane issues the MMAs and their commits (issue from a converged warp
        // costs fewer cycles per MMA than from a lone lane).
        {
            bool ok = true;
            auto wait_all = [&](uint64_t *bar, uint32_t parity) {
                return __all_sync(FULL, mbar_wait(bar, parity));
            };
            const uint32_t qa = smem_u32(sQ);
            // a negative scale is applied by negating Q (bit 13 of the descriptor)
            const uint32_t idS = tc::idesc_bf16(kTcRows, kTcKeys, false) | (p.neg_scale ? 1u << 13 : 0u);
            const uint32_t idO = tc::idesc_f16(kTcRows, D, true);
            // S_g into the S buffer (the caller has seen K_g land and, for g >= 1,
            // the four softmax warps load S_{g-1} out of the buffer)
            auto issue_s_now = [&](int g, bool last_of_item) {
                const int s = g % kTcKStages;
                const uint32_t ka = smem_u32(sK + (size_t)s * kTile);
                if (tc::elect_one()) {
#pragma unroll
                    for (int kq = 0; kq < D / 16; kq++) {
                        const uint32_t off = (uint32_t)(kq >> 2) * kQHalf + (uint32_t)(kq & 3) * 32;
                        const uint32_t offk = (uint32_t)(kq >> 2) * kTileHalf + (uint32_t)(kq & 3) * 32;
                        tc::mma_ss(tS, tc::smem_desc(qa + off, 16, 1024),
                                   tc::smem_desc(ka + offk, 16, 1024), idS, kq > 0);
                    }
                    tc::commit(smem_u32(s_full));
                    tc::commit(smem_u32(&k_empty[s]));
                    if (last_of_item)
                        tc::commit(smem_u32(q_empty));
                }
                __syncwarp();
            };
            int g0 = 0;  // tiles of the previous items
            for (int n = 0; ok; n++) {
                if (!(ok = wait_all(&item_ready[n & 1], (n >> 1) & 1)))
                    break;
                const PrefillItem it = items[n & 1];
                if (it.b < 0)
                    break;
                if (!(ok = wait_all(q_full, n & 1)))
                    break;
                tc::fence_after();
                // Readiness-driven issue: the warp polls (never blocking) whether
                // the next P.V and the next S can go and issues P.V first, so V
                // stages return to the producer as early as possible; S needs its
                // K tile and the single S buffer back (s_free).  Every parity test
                // is at most one phase behind: pv_ready for g + 2 follows P_{g+2},
                // which the softmax writes only after P.V_g has completed; s_free
                // for g needs S_g, which is issued only after s_free for g - 1.
                const int gend = g0 + it.nkt;
                int ns = g0, np = g0;  // next S and next P.V (tile indices of this CTA)
                uint64_t t_last = global_timer_ns();
                while (np < gend) {
                    bool prog = false;
                    if (np < ns) {
                        bool rdy = tc::test_wait(smem_u32(&pv_ready[np & 1]), (np >> 1) & 1);
                        // the first P.V of an item overwrites O: the previous item's
                        // epilogue must have read it out
                        if (rdy && np == g0 && n >= 1)
                            rdy = tc::test_wait(smem_u32(o_free), (n - 1) & 1);
                        if (__shfl_sync(FULL, rdy, 0)) {
                            tc::fence_after();
                            const int s = np % kTcVStages;
                            const uint32_t va = smem_u32(sV + (size_t)s * kTile);
                            const uint32_t pP = tP0 + (uint32_t)(np & 1) * (kTcKeys / 2);
                            if (tc::elect_one()) {
#pragma unroll
                                for (int kk = 0; kk < kTcKeys / 16; kk++) {
                                    const uint64_t dv = tc::smem_desc(va + kk * 16 * 128, kTileHalf, 1024);
                                    tc::mma_ts(tO, pP + 8 * kk, dv, idO, (np > g0 || kk > 0) ? 1u : 0u);
                                }
                                tc::commit(smem_u32(&v_empty[s]));
                                tc::commit(smem_u32(&pv_done[np & 1]));
                            }
                            __syncwarp();
                            np++;
                            prog = true;
                        }
                    }
                    if (!prog && ns < gend) {
                        bool rdy = tc::test_wait(smem_u32(&k_full[ns % kTcKStages]),
                                                 (ns / kTcKStages) & 1);
                        if (rdy && ns >= 1)
                            rdy = tc::test_wait(smem_u32(s_free), (ns - 1) & 1);
                        if (__shfl_sync(FULL, rdy, 0)) {
                            tc::fence_after();
                            issue_s_now(ns, ns == gend - 1);
                            ns++;
                            prog = true;
                        }
                    }
                    if (prog) {
                        t_last = global_timer_ns();
                    } else {
                        __nanosleep(16);
                        if (__shfl_sync(FULL, global_timer_ns() - t_last > 2000000000ull, 0)) {
                            ok = false;
                            break;
                        }
                    }
                }
                if (!ok)
                    break;
                g0 += it.nkt;
                if (lane == 0)
                    mbar_arrive(&item_free[n & 1]);
            }
            if (!ok && lane == 0)
                flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
            // every MMA issued has completed before TMEM is released
            if (tc::elect_one())
                tc::commit(smem_u32(mma_done));
            __syncwarp();
            mbar_wait(mma_done, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax
        const int r = threadIdx.x;            // row = TMEM lane
        const uint32_t tl = (uint32_t)(32 * warp) << 16;
        bool ok = true;
        int g0 = 0;
        for (int n = 0; ok; n++) {
            ok = __all_sync(FULL, mbar_wait(&item_ready[n & 1], (n >> 1) & 1));
            if (!ok)
                break;
            const PrefillItem it = items[n & 1];
            if (it.b < 0)
                break;
            const int tok = it.tok0 + r / G, g = r % G;
            const bool valid = tok < it.q_len;
            const int pos = (it.k_len - it.q_len) + tok;
            const int32_t *table = p.block_tables + (size_t)it.b * p.MBS;
            const int nkt = it.nkt, k_len = it.k_len;
            float m = -INFINITY, l = 0.f;
            uint32_t vmax = 0;  // f16 magnitudes of the converted V rows, max per half
            // V_g in shared memory: bf16 -> f16 in place, rows past k_len or of
            // unloaded boxes zeroed (their weight is 0, and 0 * NaN would be NaN);
            // then P.V_g may be issued (P_g was written one tile earlier).  Done
            // while the warps work on tile g + 1, so V_g has a tile more to land.
            auto convert_v = [&](int gv, uint32_t vmask_bits, int kb) -> bool {
                const int sv = gv % kTcVStages;
                if (!__all_sync(FULL, mbar_wait(&v_full[sv], (gv / kTcVStages) & 1)))
                    return false;
                uint4 *vt = reinterpret_cast<uint4 *>(sV + (size_t)sv * kTile);
                const bool vmask = vmask_bits != 0xFu || kb + kTcKeys > k_len;
                // every load first, then the conversions, then every store: thread r
                // owns 16-byte chunks r + 128 u (chunk i: half i / 512, key row
                // (i / 8) % 64, one of the row's eight column groups)
                constexpr int NCH = HALVES * kTcKeys * 8 / 128;
                uint4 w[NCH];
#pragma unroll
                for (int u = 0; u < NCH; u++)
                    w[u] = vt[r + 128 * u];
#pragma unroll
                for (int u = 0; u < NCH; u++) {
                    w[u].x = bf16x2_to_f16x2_sat(w[u].x);
                    w[u].y = bf16x2_to_f16x2_sat(w[u].y);
                    w[u].z = bf16x2_to_f16x2_sat(w[u].z);
                    w[u].w = bf16x2_to_f16x2_sat(w[u].w);
                }
                if (vmask) {  // the same for the whole CTA: a tile with rows to clear
#pragma unroll
                    for (int u = 0; u < NCH; u++) {
                        const int kr = ((r + 128 * u) / 8) % kTcKeys;
                        if (kb + kr >= k_len || !((vmask_bits >> (kr / kBox)) & 1u))
                            w[u] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
#pragma unroll
                for (int u = 0; u < NCH; u++)
                    vmax = f16x2_absmax(vmax, f16x2_absmax(f16x2_absmax(w[u].x, w[u].y),
                                                           f16x2_absmax(w[u].z, w[u].w)));
#pragma unroll
                for (int u = 0; u < NCH; u++)
                    vt[r + 128 * u] = w[u];
                fence_proxy_async_smem();
                tc::fence_before();  // also orders this warp's tcgen05.st of P_g
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&pv_ready[gv & 1]);
                return true;
            };
            uint32_t prev_mask = 0;
            int prev_kb = 0;
            // boxes of a tile the producer loads (block ids in [0, NB)); read from
            // the table here, not from the producer, whose K stage may already hold
            // a later tile.  Lanes 0-3 read the entries of the next tile one tile
            // ahead, so the load's latency is off the softmax's path.
            auto table_entry = [&](int jt) -> int {
                const int key0 = jt * kTcKeys + (lane & 3) * kBox;
                return (lane < 4 && jt < nkt && key0 < k_len) ? __ldg(table + key0 / p.bs) : -1;
            };
            int blk_next = table_entry(0);
            for (int j = 0; j < nkt; j++) {
                const int gt = g0 + j;
                const int blk = blk_next;
                blk_next = table_entry(j + 1);
                const uint32_t mask = __ballot_sync(FULL, blk >= 0 && blk < p.NB) & 0xFu;
                ok = __all_sync(FULL, mbar_wait(s_full, gt & 1));
                if (!ok)
                    break;
                tc::fence_after();
                // raw scores of this row; the scale is applied inside the exp2
                // argument (p.scale_log2 >= 0: a negative scale negates Q in the MMA)
                float x[kTcKeys];
                {
                    uint32_t ra[32], rb[32];
                    tc::ld32(tS + tl, ra);
                    tc::ld32(tS + tl + 32, rb);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        x[i] = __uint_as_float(ra[i]);
                        x[32 + i] = __uint_as_float(rb[i]);
                    }
                }
                // S is in registers: the MMA warp may issue S_{g+1} into the buffer
                tc::fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(s_free);
                if (j > 0 && !(ok = convert_v(gt - 1, prev_mask, prev_kb)))
                    break;
                const int key_base = j * kTcKeys;
                // masked keys: past this row's position (the diagonal tiles) or in
                // an unloaded box.  Most tiles have none in the whole warp: they
                // take the paths without any per-key select.
                const bool masked = mask != 0xFu || key_base + kTcKeys - 1 > pos;
                const bool any_masked = __any_sync(FULL, masked);
                if (any_masked) {
                    const int lim = pos - key_base;  // keys i > lim are in the future
#pragma unroll
                    for (int i = 0; i < kTcKeys; i++)
                        x[i] = (i > lim || !((mask >> (i / kBox)) & 1u)) ? -INFINITY : x[i];
                }
                float mraw;
                {
                    float t[8];
#pragma unroll
                    for (int i = 0; i < 8; i++)
                        t[i] = x[i];
#pragma unroll
                    for (int i = 8; i < kTcKeys; i++)
                        t[i & 7] = fmaxf(t[i & 7], x[i]);
                    mraw = fmaxf(fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3])),
                                 fmaxf(fmaxf(t[4], t[5]), fmaxf(t[6], t[7])));
                }
                const float sl = p.scale_log2;
                const float mx = mraw == -INFINITY ? -INFINITY : mraw * sl;
                if (__any_sync(FULL, mx > m + kLazy)) {
                    const float mn = fmaxf(m, mx);
                    const float alpha = mn == -INFINITY ? 1.f : fast_exp2(m - mn);
                    if (j > 0) {
                        // O holds P_0..P_{j-1} V: rescale once the last P.V completed
                        // (its pv_ready was arrived above; pv_done of its P buffer is at
                        // most one phase behind: the buffer's previous P.V was awaited
                        // before P_{g-1} was written, and its next one needs this
                        // warp's next P)
                        if (!(ok = __all_sync(FULL, mbar_wait(&pv_done[(gt - 1) & 1],
                                                              ((gt - 1) >> 1) & 1))))
                            break;
                        tc::fence_after();
#pragma unroll 1
                        for (int cc = 0; cc < D / 32; cc++) {
                            uint32_t ro[32];
                            tc::ld32(tO + tl + 32 * cc, ro);
                            tc::wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; i++)
                                ro[i] = __float_as_uint(__uint_as_float(ro[i]) * alpha);
                            tc::st32(tO + tl + 32 * cc, ro);
                        }
                        tc::wait_st();
                    }
                    l *= alpha;
                    m = mn;
                }
                const float nmu = m == -INFINITY ? 0.f : -m;
                uint32_t pk[32];
                {
                    // p = exp2(x sl - m), two keys per packed f32x2 FMA and add
                    const float2 sl2 = make_float2(sl, sl), nm2 = make_float2(nmu, nmu);
                    float2 ls0 = make_float2(0.f, 0.f), ls1 = ls0;
                    if (!any_masked) {
#pragma unroll
                        for (int i = 0; i < 32; i++) {
                            const float2 a = ffma2(make_float2(x[2 * i], x[2 * i + 1]), sl2, nm2);
                            const float2 e = make_float2(fast_exp2(a.x), fast_exp2(a.y));
                            if (i & 1)
                                ls1 = fadd2(ls1, e);
                            else
                                ls0 = fadd2(ls0, e);
                            pk[i] = pack_f16x2(e.x, e.y);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i++) {
                            float2 a = ffma2(make_float2(x[2 * i], x[2 * i + 1]), sl2, nm2);
                            // exact zeros for masked keys (also when the scale is 0,
                            // where -inf * 0 would be NaN): exp2(-inf) = 0
                            a.x = x[2 * i] == -INFINITY ? -INFINITY : a.x;
                            a.y = x[2 * i + 1] == -INFINITY ? -INFINITY : a.y;
                            const float2 e = make_float2(fast_exp2(a.x), fast_exp2(a.y));
                            if (i & 1)
                                ls1 = fadd2(ls1, e);
                            else
                                ls0 = fadd2(ls0, e);
                            pk[i] = pack_f16x2(e.x, e.y);
                        }
                    }
                    l += (ls0.x + ls0.y) + (ls1.x + ls1.y);
                }
                // P buffer gt & 1 was last read by P.V_{gt-2}: wait for it.  At most
                // one phase behind: P.V_{gt-4} was awaited before P_{gt-2} was
                // written, and P.V_gt needs the V conversion of the next step.
                if (gt >= 2) {
                    if (!(ok = __all_sync(FULL, mbar_wait(&pv_done[gt & 1], ((gt - 2) >> 1) & 1))))
                        break;
                    tc::fence_after();
                }
                tc::st32(tP0 + (uint32_t)(gt & 1) * (kTcKeys / 2) + tl, pk);
                tc::wait_st();
                prev_mask = mask;
                prev_kb = key_base;
            }
            // the item's last V tile, after which its last P.V may run
            if (ok)
                ok = convert_v(g0 + nkt - 1, prev_mask, prev_kb);
            // a converted V value was clamped to +-65504 (beyond f16's range): bf16
            // values at or below 65280 convert exactly, so only a clamp gives 0x7bff
            if (ok && ((vmax & 0x7fffu) >= 0x7bffu || ((vmax >> 16) & 0x7fffu) >= 0x7bffu))
                flag_error(p.err_flag, kFlagVRange);
            if (!ok)
                break;
            // the item's last P.V done (its pv_done is at most one phase behind:
            // the next P.V in that buffer needs this warp's next P)
            const int gl = g0 + nkt - 1;
            ok = __all_sync(FULL, mbar_wait(&pv_done[gl & 1], (gl >> 1) & 1));
            if (!ok)
                break;
            tc::fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint16_t *dst = p.out + ((size_t)(it.cq0 + tok) * p.Hq + it.kvh * G + g) * D;
#pragma unroll 1
            for (int cc = 0; cc < D / 32; cc++) {
                uint32_t ro[32];
                tc::ld32(tO + tl + 32 * cc, ro);
                tc::wait_ld();
                if (valid) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; i++)
                        pk[i] = pack_bf16x2(__uint_as_float(ro[2 * i]) * inv,
                                            __uint_as_float(ro[2 * i + 1]) * inv);
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * cc);
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
            // O read out: the next item's first P.V may overwrite it
            tc::fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(o_free);
                mbar_arrive(&item_free[n & 1]);
            }
            g0 += nkt;
        }
        if (!ok && lane == 0)
            flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 5) {
        tc::fence_after();
        tc::dealloc(tmem, kTcCols);
    }
}

template <int D>
inline cudaError_t launch_prefill_tc_d(int G, const CUtensorMap *tmq, const CUtensorMap *tmk,
                                       const CUtensorMap *tmv, const PrefillParams &p, dim3 grid,
                                       size_t smem, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (G) {
    case 1: return cudaLaunchKernelEx(&cfg, paged_prefill_tc_kernel<D, 1>, *tmq, *tmk, *tmv, p);
    case 2: return cudaLaunchKernelEx(&cfg, paged_prefill_tc_kernel<D, 2>, *tmq, *tmk, *tmv, p);
    case 4: return cudaLaunchKernelEx(&cfg, paged_prefill_tc_kernel<D, 4>, *tmq, *tmk, *tmv, p);
    case 8: return cudaLaunchKernelEx(&cfg, paged_prefill_tc_kernel<D, 8>, *tmq, *tmk, *tmv, p);
    default: return cudaErrorInvalidValue;
    }
}

template <int D> inline const void *prefill_tc_kernel_d(int G)
{
    switch (G) {
    case 1: return reinterpret_cast<const void *>(&paged_prefill_tc_kernel<D, 1>);
    case 2: return reinterpret_cast<const void *>(&paged_prefill_tc_kernel<D, 2>);
    case 4: return reinterpret_cast<const void *>(&paged_prefill_tc_kernel<D, 4>);
    case 8: return reinterpret_cast<const void *>(&paged_prefill_tc_kernel<D, 8>);
    default: return nullptr;
    }
}

} // namespace pkv
