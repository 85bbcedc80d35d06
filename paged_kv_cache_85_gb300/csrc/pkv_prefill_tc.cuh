// Paged prefill attention on the 5th-generation tensor cores (tcgen05/TMEM).
//
// What it computes (MinivLLM guide §4.5 prepare_prefill): the new tokens of
// all sequences are flattened; new token i of a sequence sits at position
// k_len - q_len + i and attends, causally, to positions 0 .. that one, K/V
// read through the sequence's block table.
//
// One persistent CTA per SM.  A work item is a pair of adjacent query tiles
// (A and B, 128 (token, head-in-group) rows each) of one sequence and KV
// head, so every 64-key K/V tile loaded serves 256 query rows: half the load
// traffic per row of one tile per CTA, which leaves the shared memory for
// four-stage K and V rings that cover the copies' latency.  Items are ranked
// longest first and dealt to the CTAs back and forth (round k: CTA c takes
// position k nC + c, or k nC + nC - 1 - c for odd k); the producer publishes
// each item through a two-slot buffer, and every ring, S, P and P.V phase
// runs on over a CTA's items.  Warps:
//   0..3  softmax of tile A, 4..7 softmax of tile B: thread t of a group owns
//         row t (TMEM lane t).  Per 64-key tile: load S from TMEM, convert
//         the V tile in shared memory from bf16 to f16 (rows past k_len or of
//         unloaded boxes zeroed; tile A's group for the V tiles tile A reads,
//         tile B's for the rest), exponentiate, and write P (f16) over the
//         row's S
//   8     producer: finds the next item, TMA of its Q tiles, then 64-key K and
//         V tiles into separate 4-stage rings: one copy per tile where the
//         block size is a multiple of 64, else four 16-token boxes per tile
//         and half, each resolved through the block table
//   9, 10 MMA of tiles A and B (warp 9 allocates all 512 TMEM columns); per
//         key tile j, in order: S_t(j), then P.V_t(j - 1):
//           S_t = Q_t K_j^T   (SS, bf16, K-major 128-byte-swizzled, M=128 N=64)
//           O_t += P_t V_j    (TS, f16: P from TMEM, V MN-major, N=D)
// TMEM columns: O_A [0, D), O_B [128, 128 + D), two S buffers per tile (64
// f32 columns each) at 256 + 128 t + 64 b; P_t(j) (64 f16 keys, 32 columns)
// is written over S_t(j) once the row's S is in registers.  S_t(j + 1) goes
// into the other buffer and runs while the group works on S_t(j); S_t(j + 2)
// is issued only after P.V_t(j), which reads P_t(j) from its buffer, has
// completed (MMAs are not ordered against each other's TMEM accesses); an
// item's first P.V of a tile waits until that tile's previous epilogue has
// read O out.
// P.V in f16: P = exp2(...) <= 2^8 is rounded to f16 (11 significant bits),
// and V is converted to f16, exact for every bf16 value of magnitude in
// [2^-14, 65504] (and for any bf16 value >= 2^-17); smaller magnitudes round
// to f16 subnormals (absolute error <= 2^-25), larger finite values and
// infinities clamp to +-65504 and set PKV_FLAG_V_RANGE; NaN stays NaN.
// The running max moves only when a row's tile max exceeds it by more than
// 2^8 (then that group rescales its O rows in TMEM after the previous P.V has
// completed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "pkv_kernels.h"
#include "pkv_prefill.h"
#include "pkv_ptx.cuh"
#include "pkv_tc.cuh"

namespace pkv {

constexpr int kTcRows = 128;            // query rows per Q tile (MMA M)
constexpr int kTcKeys = 64;             // keys per K/V tile (MMA N of S)
constexpr int kTcKStages = 4;           // K ring depth
constexpr int kTcVStages = 4;           // V ring depth
constexpr int kTcThreads = kPrefillThreads;  // 8 softmax warps, producer, 2 MMA warps
constexpr int kTcProducerWarp = 8;
constexpr int kTcMmaWarp = 9;           // warps 9 and 10 issue the MMAs of tiles A and B
constexpr uint32_t kTcCols = 512;       // all of the SM's TMEM columns
constexpr uint32_t kTcSCol = 256;       // S_t buffers at 256 + 128 t + 64 b (64 f32 columns);
                                        // P_t(j) (64 f16 keys, 32 columns) over S_t(j)
constexpr int kFlagVRange = 0x10;       // PKV_FLAG_V_RANGE (pkv.h)
// More than half an SM's shared memory, so that one CTA (which holds every
// TMEM column) runs per SM.
constexpr size_t kTcMinSmem = kSmemPerSm / 2 + 4 * 1024;

struct TcSmem {
    size_t q, kv, bars, items, slot, total;
};

// Barriers: q_full[2], q_empty[2], k_full[KS], k_empty[KS], v_full[VS], v_empty[VS],
// v_conv[VS], then per Q tile: s_full[2], pv_ready[2], pv_done[2], o_free;
// then item_ready[2], item_free[2], mma_done.
constexpr int kTcTileBars = 7;
constexpr int kTcBars = 4 + 2 * kTcKStages + 3 * kTcVStages + 2 * kTcTileBars + 2 + 2 + 1;

__host__ __device__ inline TcSmem tc_smem_layout(int D)
{
    TcSmem L;
    size_t o = 0;
    L.q = o;  // [tile][D/64 halves][128 rows][128 B]
    o += (size_t)2 * (D / 64) * kTcRows * 128;
    L.kv = o;  // K stages [D/64][64 keys][128 B], then V stages alike
    o += (size_t)(kTcKStages + kTcVStages) * (D / 64) * kTcKeys * 128;
    L.bars = o;
    o += 8 * kTcBars;
    L.items = o;  // two published work items of 32 bytes
    o += 2 * 32;
    L.slot = o;
    o += 16;
    L.total = align_up(o, 16) + 1024;
    if (L.total < kTcMinSmem)
        L.total = kTcMinSmem;
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

// One item's work, as the producer publishes it to the other warps: a pair of
// adjacent query tiles of one sequence and KV head.
struct PrefillItem {
    int b, kvh, tok0, cq0, q_len, k_len;  // b < 0: no more work for this CTA
    int nkt[2];  // key tiles of tile A and tile B (0: tile B is past q_len)
};

template <int D, int G>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq,
                            const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv, const PrefillParams p)
{
    constexpr int TPC = kTcRows / G;                  // query tokens per tile
    constexpr int HALVES = D / 64;
    constexpr uint32_t kQHalf = kTcRows * 128;        // 16 KB
    constexpr uint32_t kQTile = HALVES * kQHalf;
    constexpr uint32_t kTileHalf = kTcKeys * 128;     // 8 KB
    constexpr uint32_t kTile = HALVES * kTileHalf;    // one K (or V) tile
    constexpr uint32_t kBoxBytes = kBox * D * 2;
    constexpr unsigned FULL = 0xffffffffu;
    constexpr float kLazy = 8.f;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const TcSmem L = tc_smem_layout(D);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *q_full = bars;                       // [2] Q tile t of the item landed
    uint64_t *q_empty = q_full + 2;                // [2] tile t's last S of the item completed
    uint64_t *k_full = q_empty + 2;
    uint64_t *k_empty = k_full + kTcKStages;       // both tiles' S of the K tile completed
    uint64_t *v_full = k_empty + kTcKStages;
    uint64_t *v_empty = v_full + kTcVStages;       // both tiles' P.V of the V tile completed
    uint64_t *v_conv = v_empty + kTcVStages;       // the V tile converted to f16 (8 warp shares)
    uint64_t *tbar = v_conv + kTcVStages;          // per Q tile: kTcTileBars barriers
    uint64_t *item_ready = tbar + 2 * kTcTileBars; // [2] item parameters published
    uint64_t *item_free = item_ready + 2;          // [2] item parameters no longer needed
    uint64_t *mma_done = item_free + 2;            // every MMA of the CTA completed
    // per Q tile t and S buffer b: s_full[b] (S_t written), pv_ready[b] (P_t
    // written over it), pv_done[b] (the P.V_t that read that P completed); and
    // o_free (the tile's O read out by its epilogue)
    auto s_full = [&](int t, int b) { return tbar + kTcTileBars * t + b; };
    auto pv_ready = [&](int t, int b) { return tbar + kTcTileBars * t + 2 + b; };
    auto pv_done = [&](int t, int b) { return tbar + kTcTileBars * t + 4 + b; };
    auto o_free = [&](int t) { return tbar + kTcTileBars * t + 6; };
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem + L.slot);
    PrefillItem *items = reinterpret_cast<PrefillItem *>(smem + L.items);  // [2]
    uint8_t *sQ = smem + L.q;                                          // [2] Q tiles
    uint8_t *sK = smem + L.kv;                                         // kTcKStages K tiles
    uint8_t *sV = sK + (size_t)kTcKStages * kTile;                     // kTcVStages V tiles

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_launch_dependents();
    if (warp == kTcProducerWarp && lane == 0) {
        // the Q, K and V stages are released by both MMA warps (one arrival each)
        for (int t = 0; t < 2; t++) {
            mbar_init(&q_full[t], 1);
            mbar_init(&q_empty[t], 1);  // the tile's MMA warp
        }
        for (int s = 0; s < kTcKStages; s++) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 2);
        }
        for (int s = 0; s < kTcVStages; s++) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 2);
            mbar_init(&v_conv[s], 8);  // one share per softmax warp
        }
        for (int t = 0; t < 2; t++) {
            for (int b = 0; b < 2; b++) {
                mbar_init(s_full(t, b), 1);
                mbar_init(pv_ready(t, b), 4);
                mbar_init(pv_done(t, b), 1);
            }
            mbar_init(o_free(t), 4);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&item_ready[i], 1);
            mbar_init(&item_free[i], 10);  // the two MMA warps and the eight softmax warps
        }
        mbar_init(mma_done, 2);
        fence_mbarrier_init();
    } else if (warp == kTcMmaWarp) {
        tc::alloc(smem_u32(slot), kTcCols);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *slot;
    const int nC = (int)gridDim.x;
    const int c = (int)blockIdx.x;

    if (warp == kTcProducerWarp) {
        // ------------------------------------------------------------ producer
        // Walks this CTA's items: round k takes position k nC + c (k even) or
        // k nC + nC - 1 - c (k odd).  For each item: publish it, load its Q
        // tiles once the previous item's last S has read the old ones, then
        // its 64-key K and V tiles through the two rings (tile counters gk, gv
        // run over all of this CTA's items).
        if (lane == 0) {
            prefetch_tensormap(&tmq);
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
        grid_dependency_wait();  // K/V may have just been written by store_kvcache
        int gk = 0, gv = 0;      // K and V tiles issued so far (all items)
        int q_loads[2] = {0, 0}; // Q tiles A and B loaded so far
        bool ok = true;
        int n = 0;               // items published
        int k = 0;               // walk rounds
        for (;;) {
            // ---- the next item with work, or the end
            PrefillItem it{-1, 0, 0, 0, 0, 0, {0, 0}};
            for (; ok; k++) {
                const long long pos = (long long)k * nC + ((k & 1) ? nC - 1 - c : c);
                if (pos >= p.n_items)
                    break;
                const PrefillWork w = p.B <= 32 ? prefill_schedule<2 * TPC, 1>(p, lane, (int)pos)
                                                : prefill_schedule<2 * TPC, kSchedChunks>(p, lane, (int)pos);
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
                const int tok0 = w.tile * 2 * TPC;
                if (sane && tok0 < cq1 - cq0) {
                    it.b = w.b;
                    it.kvh = w.kvh;
                    it.tok0 = tok0;
                    it.cq0 = cq0;
                    it.q_len = cq1 - cq0;
                    it.k_len = ck1 - ck0;
                    const int base = it.k_len - it.q_len;
                    it.nkt[0] = (base + min(it.q_len, tok0 + TPC) - 1) / kTcKeys + 1;
                    it.nkt[1] = tok0 + TPC < it.q_len
                                    ? (base + min(it.q_len, tok0 + 2 * TPC) - 1) / kTcKeys + 1
                                    : 0;
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
            // ---- Q tiles: tile t's once that tile's last S of the previous item
            // has completed (q_empty[t], one commit per item): tile A's is
            // usually done a key tile or two before tile B's.  Tile B's only
            // where it has work.
            for (int t = 0; t < (it.nkt[1] > 0 ? 2 : 1) && ok; t++) {
                if (n >= 1 && !(ok = __all_sync(FULL, mbar_wait(&q_empty[t], (n - 1) & 1))))
                    break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&q_full[t], HALVES * kQHalf);
#pragma unroll
                    for (int h = 0; h < HALVES; h++)
                        tma_load_4d(sQ + t * kQTile + h * kQHalf, &tmq, 0, h, it.kvh * G,
                                    it.cq0 + it.tok0 + t * TPC, &q_full[t]);
                }
                ++q_loads[t];
            }
            if (!ok)
                break;
            n++;
            // ---- K and V tiles.  One converged loop serves both rings: it
            // probes (without blocking) whether the next K stage and the next
            // V stage are free and issues whichever tile can go; lanes 0-3
            // resolve and copy one 16-token box each.  K runs ahead of V by up
            // to its ring depth.
            const int nkt = max(it.nkt[0], it.nkt[1]);
            const int32_t *table = p.block_tables + (size_t)it.b * p.MBS;
            // Lanes 0-3 resolve one 16-token box each.  A tile's block-table
            // entries are read once, one K tile ahead of its copy (so the load's
            // latency is off the producer's path), and kept for the V copy of the
            // same tile (V lags K by at most the ring depth, four tiles).
            auto entry = [&](int j) -> int {
                const int key0 = j * kTcKeys + lane * kBox;
                return (lane < kTcKeys / kBox && j < nkt && key0 < it.k_len) ? __ldg(table + key0 / p.bs) : -1;
            };
            int blk_next = entry(0);
            int row0 = -1, row1 = -1, row2 = -1, row3 = -1;  // box rows of tiles j % 4 (-1: not loaded)
            auto put_row = [&](int j, int v) {
                const int q = j & 3;
                row0 = q == 0 ? v : row0;
                row1 = q == 1 ? v : row1;
                row2 = q == 2 ? v : row2;
                row3 = q == 3 ? v : row3;
            };
            auto get_row = [&](int j) {
                const int q = j & 3;
                return q == 0 ? row0 : (q == 1 ? row1 : (q == 2 ? row2 : row3));
            };
            static_assert(kTcVStages <= 4 && kTcKStages <= 4, "V lags K by at most four tiles");
            auto issue = [&](int j, int g, bool is_k) {
                uint64_t *fb = is_k ? k_full : v_full;
                const int nst = is_k ? kTcKStages : kTcVStages;
                const int s = g % nst;
                int row = -1;
                if (is_k) {
                    const int blk = blk_next;
                    blk_next = entry(j + 1);
                    const int key0 = j * kTcKeys + lane * kBox;
                    if (lane < kTcKeys / kBox && key0 < it.k_len) {
                        if (blk >= 0 && blk < p.NB)
                            row = blk * p.bs + key0 % p.bs;
                        else
                            flag_error(p.err_flag, 0x2 /* PKV_FLAG_BAD_BLOCK */);
                    }
                    put_row(j, row);
                } else {
                    row = get_row(j);
                }
                const CUtensorMap *map = is_k ? &tmk : &tmv;
                uint8_t *dst = (is_k ? sK : sV) + (size_t)s * kTile;
                if (p.tile_copies) {
                    // the tile's 64 tokens lie in one block: one copy of the
                    // whole tile, both halves (rows past k_len included: the
                    // softmax masks their scores and zeroes their V rows)
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&fb[s], row >= 0 ? kTile : 0u);
                        if (row >= 0)
                            tma_load_4d(dst, map, 0, row, it.kvh, 0, &fb[s]);
                    }
                } else {
                    const bool loaded = row >= 0;
                    const uint32_t mask = __ballot_sync(FULL, loaded);
                    if (lane == 0)
                        mbar_arrive_expect_tx(&fb[s], (uint32_t)__popc(mask) * kBoxBytes);
                    __syncwarp();
                    if (loaded) {
                        if (is_k) {
                            // K: [half][64 rows], the layout the score MMA's
                            // descriptor walks with one stride along the keys
#pragma unroll
                            for (int h = 0; h < HALVES; h++)
                                tma_load_4d(dst + lane * (kBox * 128) + h * kTileHalf, map, 0, h, it.kvh,
                                            row, &fb[s]);
                        } else {
                            // V: one copy per box, both halves: [box][half][16 rows]
                            tma_load_4d(dst + lane * kBoxBytes, map, 0, row, it.kvh, 0, &fb[s]);
                        }
                    }
                }
            };
            int jk = 0, jv = 0;
            uint64_t t_last = sm_clock();
            while (jk < nkt || jv < nkt) {
                bool prog = false;
                // K at most four tiles ahead of the V copies (the kept box rows)
                if (jk < nkt && jk - jv < 4) {
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
                    t_last = sm_clock();
                } else {
                    __nanosleep(32);
                    if (__shfl_sync(FULL, sm_clock() - t_last > kPollLimitCycles, 0)) {
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
            for (int t = 0; t < 2; t++)
                if (q_loads[t] >= 1)
                    mbar_wait(&q_full[t], (q_loads[t] - 1) & 1);
            for (int g = max(0, gk - kTcKStages); g < gk; g++)
                mbar_wait(&k_full[g % kTcKStages], (g / kTcKStages) & 1);
            for (int g = max(0, gv - kTcVStages); g < gv; g++)
                mbar_wait(&v_full[g % kTcVStages], (g / kTcVStages) & 1);
        }
        __syncwarp();
    } else if (warp == kTcMmaWarp || warp == kTcMmaWarp + 1) {
        // ----------------------------------------------------------------- MMA
        // Warp 9 issues the MMAs of Q tile A, warp 10 those of tile B, so the two
        // tiles' issue and barrier waits run side by side.  Each warp walks the
        // item's key tiles in order with blocking waits: for key tile j, S_t(j);
        // then P.V_t(j - 1).  Lane 0 alone waits, issues the MMAs and commits.  A
        // K, V or Q stage is released by one arrival from each warp: the warp's
        // commit after its MMAs that read it, or, for a stage its tile does not
        // read, a commit once the stage's tile has landed (so the arrival always
        // counts towards that tile's phase: the stage is refilled only after both
        // warps arrived for its previous tile).
        const int t = warp - kTcMmaWarp;
        bool ok = true;
        const uint32_t qt = smem_u32(sQ) + (uint32_t)t * kQTile;
        // a negative scale is applied by negating Q (bit 13 of the descriptor)
        const uint32_t idS = tc::idesc_bf16(kTcRows, kTcKeys, false) | (p.neg_scale ? 1u << 13 : 0u);
        const uint32_t idO = tc::idesc_f16(kTcRows, D, true);
        const uint32_t dS0 = tmem + kTcSCol + 128u * (uint32_t)t, dO = tmem + 128u * (uint32_t)t;
        // V tile layout: whole-tile copies land as [half][64 rows]; per-box
        // copies as [16-token box][half][16 rows] (rows of 128 B).  A P.V MMA
        // takes 16 keys: one box; its halves are v_lbo apart
        const uint32_t v_lbo = p.tile_copies ? kTileHalf : (uint32_t)kBox * 128;
        const uint32_t v_kstep = p.tile_copies ? 16u * 128 : (uint32_t)kBoxBytes;
        uint64_t *my_o_free = o_free(t);
        int g0 = 0;    // K/V tiles of the previous items
        int gq = 0;    // S/P tiles of this Q tile over the previous items
        int used = 0;  // items in which this Q tile had work (its epilogues)
        // lane 0 alone waits, issues the MMAs and commits
        if (lane == 0) {
            for (int n = 0; ok; n++) {
                if (!(ok = mbar_wait(&item_ready[n & 1], (n >> 1) & 1)))
                    break;
                const PrefillItem it = items[n & 1];
                if (it.b < 0)
                    break;
                const int nk = it.nkt[t];
                const int nkt = max(it.nkt[0], it.nkt[1]);
                // this tile's Q of the item (loaded only where it has work)
                if (nk > 0 && !(ok = mbar_wait(&q_full[t], used & 1)))
                    break;
                tc::fence_after();
                if (nk == 0)
                    tc::commit(smem_u32(&q_empty[t]));  // this tile reads no Q this item
                for (int j = 0; j <= nkt && ok; j++) {
                    if (j < nkt) {
                        const int gkt = g0 + j, s = gkt % kTcKStages;
                        if (!(ok = mbar_wait(&k_full[s], (gkt / kTcKStages) & 1)))
                            break;
                        if (j < nk) {
                            // S_t(j) into S buffer gs & 1 once the P.V that read P_t(j - 2)
                            // from it completed (at most one phase behind: the next
                            // completion needs S_t(j), issued below; the one before was
                            // awaited before S_t(j - 2))
                            const int gs = gq + j;
                            if (gs >= 2 && !(ok = mbar_wait(pv_done(t, gs & 1), ((gs - 2) >> 1) & 1)))
                                break;
                            tc::fence_after();
                            const uint32_t ka = smem_u32(sK + (size_t)s * kTile);
                            const uint32_t dS = dS0 + 64u * (uint32_t)(gs & 1);
                            {
#pragma unroll
                                for (int kq = 0; kq < D / 16; kq++) {
                                    const uint32_t off = (uint32_t)(kq >> 2) * kQHalf + (uint32_t)(kq & 3) * 32;
                                    const uint32_t offk = (uint32_t)(kq >> 2) * kTileHalf + (uint32_t)(kq & 3) * 32;
                                    tc::mma_ss(dS, tc::smem_desc(qt + off, 16, 1024),
                                               tc::smem_desc(ka + offk, 16, 1024), idS, kq > 0);
                                }
                                tc::commit(smem_u32(s_full(t, gs & 1)));
                                tc::commit(smem_u32(&k_empty[s]));
                                if (j == nk - 1)
                                    tc::commit(smem_u32(&q_empty[t]));
                            }
                        } else {
                            tc::commit(smem_u32(&k_empty[s]));  // a K tile this Q tile does not read
                        }
                            }
                    if (j >= 1) {
                        const int jj = j - 1, gvt = g0 + jj, s = gvt % kTcVStages;
                        if (jj < nk) {
                            // P.V_t(jj) once P_t(jj) is written and both softmax groups
                            // converted their shares of V tile jj
                            const int gp = gq + jj;
                            if (!(ok = mbar_wait(pv_ready(t, gp & 1), (gp >> 1) & 1)))
                                break;
                            if (!(ok = mbar_wait(&v_conv[s], (gvt / kTcVStages) & 1)))
                                break;
                            // the item's first P.V overwrites O: the tile's previous
                            // epilogue must have read it out
                            if (jj == 0 && used >= 1 && !(ok = mbar_wait(my_o_free, (used - 1) & 1)))
                                break;
                            tc::fence_after();
                            const uint32_t va = smem_u32(sV + (size_t)s * kTile);
                            const uint32_t pP = dS0 + 64u * (uint32_t)(gp & 1);  // P_t(jj) over S_t(jj)
                            {
#pragma unroll
                                for (int kk = 0; kk < kTcKeys / 16; kk++) {
                                    const uint64_t dv = tc::smem_desc(va + kk * v_kstep, v_lbo, 1024);
                                    tc::mma_ts(dO, pP + 8 * kk, dv, idO, (jj > 0 || kk > 0) ? 1u : 0u);
                                }
                                tc::commit(smem_u32(pv_done(t, gp & 1)));
                                tc::commit(smem_u32(&v_empty[s]));
                            }
                        } else {
                            // a V tile this Q tile does not read: arrive once it is
                            // converted (so its tile has landed)
                            if (!(ok = mbar_wait(&v_conv[s], (gvt / kTcVStages) & 1)))
                                break;
                            tc::commit(smem_u32(&v_empty[s]));
                        }
                            }
                }
                if (!ok)
                    break;
                g0 += nkt;
                gq += nk;
                used += nk > 0 ? 1 : 0;
                mbar_arrive(&item_free[n & 1]);
            }
        }
        __syncwarp();
        if (!ok && lane == 0)
            flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
        // every MMA issued has completed before TMEM is released
        if (lane == 0)
            tc::commit(smem_u32(mma_done));
        __syncwarp();
        mbar_wait(mma_done, 0);
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax
        const int tq = warp >> 2;                       // Q tile of this group (A = 0, B = 1)
        const int r = threadIdx.x & 127;                // row = TMEM lane
        const uint32_t tl = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tO = tmem + 128u * tq, tS0 = tmem + kTcSCol + 128u * tq;
        bool ok = true;
        int g0 = 0, gq = 0;
        for (int n = 0; ok; n++) {
            ok = __all_sync(FULL, mbar_wait(&item_ready[n & 1], (n >> 1) & 1));
            if (!ok)
                break;
            const PrefillItem it = items[n & 1];
            if (it.b < 0)
                break;
            const int nkt = it.nkt[tq], nk_other = it.nkt[1 - tq];
            const int tok = it.tok0 + tq * TPC + r / G, g = r % G;
            const bool valid = tok < it.q_len;
            const int pos = (it.k_len - it.q_len) + tok;
            const int32_t *table = p.block_tables + (size_t)it.b * p.MBS;
            const int k_len = it.k_len;
            float m = -INFINITY, l = 0.f;
            uint32_t vmax = 0;  // f16 magnitudes of the converted V rows, max per half
            // V tile jv in shared memory: bf16 -> f16 in place, rows past k_len or
            // of unloaded boxes zeroed (their weight is 0, and 0 * NaN would be
            // NaN).  Every softmax warp takes part in every V tile, in order: it
            // waits for the tile to land, converts its share and arrives once on
            // the stage's v_conv (8 arrivals), so no group's parity wait on a V
            // stage can fall two phases behind.  Tile A's group converts every V
            // tile its tile reads, tile B's group only those tile A does not
            // read: B's group, with less to do per key tile, then runs behind
            // A's rather than in step with it, and the two tiles' MMAs queue
            // less behind each other.  A group converts V tile j right after
            // loading S of key tile j.
            auto convert_v = [&](int jv, uint32_t vmask_bits, bool convert) -> bool {
                const int gv = g0 + jv, sv = gv % kTcVStages, kb = jv * kTcKeys;
                if (!__all_sync(FULL, mbar_wait(&v_full[sv], (gv / kTcVStages) & 1)))
                    return false;
                uint4 *vt = reinterpret_cast<uint4 *>(sV + (size_t)sv * kTile);
                const bool vmask = vmask_bits != 0xFu || kb + kTcKeys > k_len;
                // thread r owns 16-byte chunks r + 128 u (chunk i: half i / 512,
                // key row (i / 8) % 64, one of the row's eight column groups)
                constexpr int NCH = HALVES * kTcKeys * 8 / 128;
                auto run = [&](int u0, auto nu_c) {
                    constexpr int NU = decltype(nu_c)::value;
                    uint4 w[NU];
#pragma unroll
                    for (int u = 0; u < NU; u++)
                        w[u] = vt[r + 128 * (u0 + u)];
#pragma unroll
                    for (int u = 0; u < NU; u++) {
                        w[u].x = bf16x2_to_f16x2_sat(w[u].x);
                        w[u].y = bf16x2_to_f16x2_sat(w[u].y);
                        w[u].z = bf16x2_to_f16x2_sat(w[u].z);
                        w[u].w = bf16x2_to_f16x2_sat(w[u].w);
                    }
                    if (vmask) {  // the same for the whole CTA: a tile with rows to clear
#pragma unroll
                        for (int u = 0; u < NU; u++) {
                            const int ci = r + 128 * (u0 + u);  // 16-byte chunk
                            const int kr = p.tile_copies ? (ci / 8) % kTcKeys
                                                         : (ci / (8 * kBox * HALVES)) * kBox + (ci / 8) % kBox;
                            if (kb + kr >= k_len || !((vmask_bits >> (kr / kBox)) & 1u))
                                w[u] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < NU; u++)
                        vmax = f16x2_absmax(vmax, f16x2_absmax(f16x2_absmax(w[u].x, w[u].y),
                                                               f16x2_absmax(w[u].z, w[u].w)));
#pragma unroll
                    for (int u = 0; u < NU; u++)
                        vt[r + 128 * (u0 + u)] = w[u];
                };
                if (convert)
                    run(0, std::integral_constant<int, NCH>());
                fence_proxy_async_smem();
                tc::fence_before();  // also orders this warp's tcgen05.st of P
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&v_conv[sv]);
                return true;
            };
            // whether this group converts V tile jv (its tile reads V tiles
            // 0 .. nkt - 1)
            auto share = [&](int jv) { return jv < nkt && (tq == 0 || jv >= nk_other); };
            if (nkt > 0) {
                // boxes of a tile the producer loads (block ids in [0, NB)); read
                // from the table here, not from the producer, whose K stage may
                // already hold a later tile.  Lanes 0-3 read the entries of the
                // next tile one tile ahead, so the load's latency is off the path.
                auto table_entry = [&](int jt) -> int {
                    const int key0 = jt * kTcKeys + (lane & 3) * kBox;
                    return (lane < 4 && jt < nkt && key0 < k_len) ? __ldg(table + key0 / p.bs) : -1;
                };
                int blk_next = table_entry(0);
                for (int j = 0; j < nkt; j++) {
                    const int gt = gq + j;
                    const int blk = blk_next;
                    blk_next = table_entry(j + 1);
                    const uint32_t mask = __ballot_sync(FULL, blk >= 0 && blk < p.NB) & 0xFu;
                    ok = __all_sync(FULL, mbar_wait(s_full(tq, gt & 1), (gt >> 1) & 1));
                    if (!ok)
                        break;
                    tc::fence_after();
                    const uint32_t tS = tS0 + 64u * (uint32_t)(gt & 1);
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
                    if (!(ok = convert_v(j, mask, share(j))))
                        break;
                    const int key_base = j * kTcKeys;
                    // masked keys: past this row's position (the diagonal tiles) or
                    // in an unloaded box.  Most tiles have none in the whole warp:
                    // they take the paths without any per-key select.
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
                        float t8[8];
#pragma unroll
                        for (int i = 0; i < 8; i++)
                            t8[i] = x[i];
#pragma unroll
                        for (int i = 8; i < kTcKeys; i++)
                            t8[i & 7] = fmaxf(t8[i & 7], x[i]);
                        mraw = fmaxf(fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3])),
                                     fmaxf(fmaxf(t8[4], t8[5]), fmaxf(t8[6], t8[7])));
                    }
                    const float sl = p.scale_log2;
                    const float mx = mraw == -INFINITY ? -INFINITY : mraw * sl;
                    if (__any_sync(FULL, mx > m + kLazy)) {
                        const float mn = fmaxf(m, mx);
                        const float alpha = mn == -INFINITY ? 1.f : fast_exp2(m - mn);
                        if (j > 0) {
                            // O holds P_0..P_{j-1} V: rescale once the last P.V
                            // completed (pv_done of its S buffer is at most one phase
                            // behind: the buffer's previous P.V completed before
                            // S_{j-1} was issued into it, and its next one needs this
                            // group's next P)
                            if (!(ok = __all_sync(FULL, mbar_wait(pv_done(tq, (gt - 1) & 1),
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
                    // P over this row's S (all of it is in registers; the next S
                    // into the buffer waits for the P.V that reads this P)
                    tc::st32(tS + tl, pk);
                    tc::wait_st();
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(pv_ready(tq, gt & 1));
                }
            }
            // V tiles of this item that only the other Q tile reads: no share to
            // convert, but this group arrives on them in order too
            for (int jv = nkt; ok && jv < max(it.nkt[0], it.nkt[1]); jv++)
                ok = convert_v(jv, 0xFu, false);
            if (!ok)
                break;
            if (nkt > 0) {
                // a converted V value was clamped to +-65504 (beyond f16's range):
                // bf16 values at or below 65280 convert exactly, so only a clamp
                // gives 0x7bff
                if ((vmax & 0x7fffu) >= 0x7bffu || ((vmax >> 16) & 0x7fffu) >= 0x7bffu)
                    flag_error(p.err_flag, kFlagVRange);
                // the tile's last P.V done (its pv_done is at most one phase
                // behind: the next P.V into that buffer needs this group's next P)
                const int gl = gq + nkt - 1;
                ok = __all_sync(FULL, mbar_wait(pv_done(tq, gl & 1), (gl >> 1) & 1));
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
                // O read out: the tile's next first P.V may overwrite it
                tc::fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(o_free(tq));
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&item_free[n & 1]);
            g0 += max(it.nkt[0], it.nkt[1]);
            gq += nkt;
        }
        if (!ok && lane == 0)
            flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
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
