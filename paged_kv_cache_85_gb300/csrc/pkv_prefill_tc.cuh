// Paged prefill attention on the 5th-generation tensor cores (tcgen05/TMEM).
//
// Same operation as paged_prefill_kernel (MinivLLM guide §4.5 prepare_prefill;
// causal: new token i of a sequence sits at position k_len - q_len + i and
// attends to positions 0 .. that one, K/V read through the block table).
//
// One CTA per (tile of 128 (token, head-in-group) rows, KV head, sequence);
// two CTAs per SM, so one CTA's softmax overlaps the other's MMAs.  Warps:
//   0..3  softmax: thread t owns row t (TMEM lane t) -- no shuffles
//   4     producer: TMA of the Q tile once, then 64-key K and V tiles (four
//         16-token boxes each, resolved through the block table) into two
//         separate 2-stage rings, lanes 0-3 for K and 4-7 for V: a K tile is
//         released as soon as its S MMA completes, so the next K tiles load
//         while the softmax runs, and V only has to arrive by its P.V
//   5     MMA: allocates 256 TMEM columns; one lane issues
//           S_j = Q K_j^T    (SS, K-major 128-byte-swizzled operands, M=128
//                             N=64, into one of two S buffers), and
//           O  += P_j V_j    (P from TMEM, V MN-major from shared memory,
//                             N=D), P split into bf16 hi + lo parts.
// TMEM columns: O in [0, D); S buffers at 128 and 192 (64 f32 columns each);
// P_j overwrites its S buffer (hi in the first 32 columns, lo in the next 32).
// An S MMA is issued into a buffer only after the P.V that read the P in it
// has completed (MMAs are not ordered against each other's TMEM accesses).
// The running max moves only when a row's tile max exceeds it by more than
// 2^8 (then that warp rescales its O rows in TMEM after the previous P.V has
// completed).  V rows past k_len or in unloaded boxes are zeroed in shared
// memory before P.V (their weight is 0, and 0 * NaN would be NaN).
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
constexpr uint32_t kTcSCol = 128;       // first S buffer column

struct TcSmem {
    size_t q, kv, bars, slot, total;
};

__host__ __device__ inline TcSmem tc_smem_layout(int D)
{
    TcSmem L;
    size_t o = 0;
    L.q = o;  // [D/64 halves][128 rows][128 B]
    o += (size_t)(D / 64) * kTcRows * 128;
    L.kv = o;  // K stages [D/64][64 keys][128 B], then V stages alike
    o += (size_t)(kTcKStages + kTcVStages) * (D / 64) * kTcKeys * 128;
    L.bars = o;  // q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2],
                 // o_done, mma_done
    o += 8 * (1 + 2 * kTcKStages + 2 * kTcVStages + 2 + 2 + 2);
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

// The (sequence, KV head, query tile) this CTA works on, run by one warp.
// CTAs start in launch order, so the work is handed out longest first (a
// tile's cost is its number of key tiles): with up to kSchedMaxSeqs
// sequences the CTA's rank r (its launch index over the KV heads) is mapped
// to the r-th tile in decreasing cost, found by a binary search over the
// cost with per-sequence closed-form counts.  Beyond that many sequences the
// last tile of every sequence goes first, then the second-to-last ones, and
// so on.  NCH chunks of 32 sequences are scanned (one lane per sequence).
template <int TPC, int NCH>
__device__ PrefillWork prefill_schedule(const PrefillParams &p, int lane)
{
    constexpr unsigned FULL = 0xffffffffu;
    const int B = (int)gridDim.z, Hkv = (int)gridDim.y, X = (int)gridDim.x;
    const unsigned lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    const int r = (int)(lin / (unsigned)Hkv);
    PrefillWork w{-1, (int)(lin % (unsigned)Hkv), 0, kNotLoaded, 0, 0, 0};
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
    if (bad && lin == 0)
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

template <int D, int G>
__global__ void __launch_bounds__(kTcThreads, 2)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq,
                            const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv, const PrefillParams p)
{
    constexpr int TPC = kTcRows / G;                  // query tokens per CTA
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
    uint64_t *q_full = bars;
    uint64_t *k_full = bars + 1;
    uint64_t *k_empty = k_full + kTcKStages;
    uint64_t *v_full = k_empty + kTcKStages;
    uint64_t *v_empty = v_full + kTcVStages;
    uint64_t *s_full = v_empty + kTcVStages;
    uint64_t *p_full = s_full + 2;
    uint64_t *o_done = p_full + 2;
    uint64_t *mma_done = o_done + 1;
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem + L.slot);
    uint8_t *sQ = smem + L.q;
    uint8_t *sK = smem + L.kv;                                   // kTcKStages K tiles
    uint8_t *sV = sK + (size_t)kTcKStages * (D / 64) * kTcKeys * 128;  // kTcVStages V tiles

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    grid_launch_dependents();
    // Prologue, in parallel: warp 0 finds this CTA's work, the producer warp
    // initialises the barriers, the MMA warp allocates TMEM; one barrier then
    // publishes all three.
    __shared__ int s_work[7];
    if (warp == 0) {
        const PrefillWork w = gridDim.z <= 32 ? prefill_schedule<TPC, 1>(p, lane)
                                              : prefill_schedule<TPC, kSchedChunks>(p, lane);
        if (lane == 0) {
            s_work[0] = w.b;
            s_work[1] = w.kvh;
            s_work[2] = w.tile;
            s_work[3] = w.cq0;
            s_work[4] = w.cq1;
            s_work[5] = w.ck0;
            s_work[6] = w.ck1;
        }
    } else if (warp == 4 && lane == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kTcKStages; s++) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kTcVStages; s++) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
        }
        mbar_init(o_done, 1);
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
    const int b = s_work[0], kvh = s_work[1], tile = s_work[2];
    int cq0 = s_work[3], cq1 = s_work[4], ck0 = s_work[5], ck1 = s_work[6];
    if (b >= 0 && cq0 == kNotLoaded) {
        cq0 = __ldg(p.cu_q + b);
        cq1 = __ldg(p.cu_q + b + 1);
        ck0 = __ldg(p.cu_k + b);
        ck1 = __ldg(p.cu_k + b + 1);
    }
    const int q_len = cq1 - cq0, k_len = ck1 - ck0;
    const int tok0 = tile * TPC;
    const bool sane = b >= 0 && prefill_seq_sane(p, cq0, cq1, ck0, ck1);
    if (!sane || tok0 >= q_len) {
        // nothing to do (or a bad sequence): release TMEM and leave
        if (b >= 0 && !sane && threadIdx.x == 0)
            flag_error(p.err_flag, 0x4 /* PKV_FLAG_BAD_CONTEXT_LEN */);
        if (warp == 5)
            tc::dealloc(tmem, kTcCols);
        return;
    }
    const int base = k_len - q_len;  // position of new token 0
    const int last_pos = base + min(q_len, tok0 + TPC) - 1;
    const int nkt = last_pos / kTcKeys + 1;
    const uint32_t tO = tmem, tS0 = tmem + kTcSCol;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&tmq);
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
        const int32_t *table = p.block_tables + (size_t)b * p.MBS;
        grid_dependency_wait();  // K/V may have just been written by store_kvcache
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, HALVES * kQHalf);
#pragma unroll
            for (int h = 0; h < HALVES; h++)
                tma_load_4d(sQ + h * kQHalf, &tmq, 0, h, kvh * G, cq0 + tok0, q_full);
        }
        // One converged loop serves both rings: it probes (without blocking)
        // whether the next K stage and the next V stage are free and issues
        // whichever tile can go; lanes 0-3 resolve and copy one 16-token box
        // each.  K runs ahead of V by up to its ring depth.
        auto issue = [&](int j, bool is_k) {
            uint64_t *fb = is_k ? k_full : v_full;
            const int nst = is_k ? kTcKStages : kTcVStages;
            const int s = j % nst;
            const int key0 = j * kTcKeys + lane * kBox;
            bool loaded = false;
            int row = 0;
            if (lane < kTcKeys / kBox && key0 < k_len) {
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
                    tma_load_4d(dst + h * kTileHalf, map, 0, h, kvh, row, &fb[s]);
            }
        };
        int jk = 0, jv = 0;
        bool ok = true;
        uint64_t t_last = global_timer_ns();
        while (jk < nkt || jv < nkt) {
            bool prog = false;
            if (jk < nkt) {
                const bool free_k = tc::test_wait(smem_u32(&k_empty[jk % kTcKStages]),
                                                  ((jk / kTcKStages) & 1) ^ 1);
                if (__shfl_sync(FULL, free_k, 0)) {
                    issue(jk++, true);
                    prog = true;
                }
            }
            if (jv < jk) {
                const bool free_v = tc::test_wait(smem_u32(&v_empty[jv % kTcVStages]),
                                                  ((jv / kTcVStages) & 1) ^ 1);
                if (__shfl_sync(FULL, free_v, 0)) {
                    issue(jv++, false);
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
        if (lane == 0) {
            if (!ok)
                flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
            // copies still in flight land before the CTA may exit
            mbar_wait(q_full, 0);
            for (int j = max(0, jk - kTcKStages); j < jk; j++)
                mbar_wait(&k_full[j % kTcKStages], (j / kTcKStages) & 1);
            for (int j = max(0, jv - kTcVStages); j < jv; j++)
                mbar_wait(&v_full[j % kTcVStages], (j / kTcVStages) & 1);
        }
        __syncwarp();
    } else if (warp == 5) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            bool ok = mbar_wait(q_full, 0);
            const uint32_t qa = smem_u32(sQ);
            // a negative scale is applied by negating Q (bit 13 of the descriptor)
            const uint32_t idS = tc::idesc_bf16(kTcRows, kTcKeys, false) | (p.neg_scale ? 1u << 13 : 0u);
            const uint32_t idO = tc::idesc_bf16(kTcRows, D, true);
            auto issue_s = [&](int j) {
                const int s = j % kTcKStages;
                const uint32_t ka = smem_u32(sK + (size_t)s * kTile);
                const uint32_t dst = tS0 + (uint32_t)(j & 1) * kTcKeys;
#pragma unroll
                for (int k = 0; k < D / 16; k++) {
                    const uint32_t off = (uint32_t)(k >> 2) * kQHalf + (uint32_t)(k & 3) * 32;
                    const uint32_t offk = (uint32_t)(k >> 2) * kTileHalf + (uint32_t)(k & 3) * 32;
                    tc::mma_ss(dst, tc::smem_desc(qa + off, 16, 1024),
                               tc::smem_desc(ka + offk, 16, 1024), idS, k > 0);
                }
                tc::commit(smem_u32(&s_full[j & 1]));
                tc::commit(smem_u32(&k_empty[s]));
            };
            if (ok && (ok = mbar_wait(&k_full[0], 0)))
                issue_s(0);
            for (int j = 0; j < nkt && ok; j++) {
                if (j + 1 < nkt) {
                    if (!(ok = mbar_wait(&k_full[(j + 1) % kTcKStages], ((j + 1) / kTcKStages) & 1)))
                        break;
                    // S_{j+1} overwrites the buffer P_{j-1} occupies: the tensor pipe
                    // does not order P.V_{j-1}'s TMEM reads before a later MMA's
                    // writes, so wait for P.V_{j-1} (long done, a softmax ago)
                    if (j >= 1) {
                        if (!(ok = mbar_wait(o_done, (j - 1) & 1)))
                            break;
                        tc::fence_after();
                    }
                    issue_s(j + 1);
                }
                if (!(ok = mbar_wait(&p_full[j & 1], (j >> 1) & 1)))
                    break;
                if (!(ok = mbar_wait(&v_full[j % kTcVStages], (j / kTcVStages) & 1)))
                    break;
                tc::fence_after();
                const int s = j % kTcVStages;
                const uint32_t va = smem_u32(sV + (size_t)s * kTile);
                const uint32_t pS = tS0 + (uint32_t)(j & 1) * kTcKeys;
#pragma unroll
                for (int kk = 0; kk < kTcKeys / 16; kk++) {
                    const uint64_t dv = tc::smem_desc(va + kk * 16 * 128, kTileHalf, 1024);
                    tc::mma_ts(tO, pS + 8 * kk, dv, idO, (j > 0 || kk > 0) ? 1u : 0u);
                    tc::mma_ts(tO, pS + 32 + 8 * kk, dv, idO, 1u);
                }
                tc::commit(smem_u32(&v_empty[s]));
                tc::commit(smem_u32(o_done));
            }
            if (!ok)
                flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
            // every MMA issued has completed before TMEM is released (and
            // before the softmax warps read O)
            tc::commit(smem_u32(mma_done));
            mbar_wait(mma_done, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax
        const int r = threadIdx.x;            // row = TMEM lane
        const int tok = tok0 + r / G, g = r % G;
        const bool valid = tok < q_len;
        const int pos = base + tok;
        const uint32_t tl = (uint32_t)(32 * warp) << 16;
        const int32_t *table = p.block_tables + (size_t)b * p.MBS;
        grid_dependency_wait();
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkt; j++) {
            const uint32_t tS = tS0 + (uint32_t)(j & 1) * kTcKeys;
            // boxes of this tile the producer loads (block ids in [0, NB)); read
            // from the table here, not from the producer, whose K stage may
            // already hold a later tile
            uint32_t mask;
            {
                const int key0 = j * kTcKeys + (lane & 3) * kBox;
                bool ld = false;
                if (lane < 4 && key0 < k_len) {
                    const int blk = __ldg(table + key0 / p.bs);
                    ld = blk >= 0 && blk < p.NB;
                }
                mask = __ballot_sync(FULL, ld) & 0xFu;
            }
            ok = __all_sync(FULL, mbar_wait(&s_full[j & 1], (j >> 1) & 1));
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
            const int key_base = j * kTcKeys;
            const bool masked = mask != 0xFu || key_base + kTcKeys - 1 > pos;
            if (masked) {
#pragma unroll
                for (int i = 0; i < kTcKeys; i++)
                    if (key_base + i > pos || !((mask >> (i / kBox)) & 1u))
                        x[i] = -INFINITY;
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
                    if (!(ok = __all_sync(FULL, mbar_wait(o_done, (j - 1) & 1))))
                        break;
                    tc::fence_after();
#pragma unroll 1
                    for (int c = 0; c < D / 32; c++) {
                        uint32_t ro[32];
                        tc::ld32(tO + tl + 32 * c, ro);
                        tc::wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i++)
                            ro[i] = __float_as_uint(__uint_as_float(ro[i]) * alpha);
                        tc::st32(tO + tl + 32 * c, ro);
                    }
                    tc::wait_st();
                }
                l *= alpha;
                m = mn;
            }
            const float nmu = m == -INFINITY ? 0.f : -m;
            {
                uint32_t hi[32], lo[32];
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    float p0 = fast_exp2(fmaf(x[2 * i], sl, nmu));
                    float p1 = fast_exp2(fmaf(x[2 * i + 1], sl, nmu));
                    if (masked) {  // exact zeros for masked keys (also when the scale is 0)
                        p0 = x[2 * i] == -INFINITY ? 0.f : p0;
                        p1 = x[2 * i + 1] == -INFINITY ? 0.f : p1;
                    }
                    ls[i & 3] += p0 + p1;
                    hi[i] = pack_bf16x2(p0, p1);
                    const float2 h = bf16x2_to_float2(hi[i]);
                    lo[i] = pack_bf16x2(p0 - h.x, p1 - h.y);
                }
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                tc::st32(tS + tl, hi);
                tc::st32(tS + tl + 32, lo);
                tc::wait_st();
            }
            // V rows past k_len or in unloaded boxes: zero them (all four warps)
            if (mask != 0xFu || key_base + kTcKeys > k_len) {
                // after the V copies of this tile have landed
                const int sv = j % kTcVStages;
                if (!(ok = __all_sync(FULL, mbar_wait(&v_full[sv], (j / kTcVStages) & 1))))
                    break;
                uint8_t *vt = sV + (size_t)sv * kTile;
                for (int it = r; it < HALVES * kTcKeys * 8; it += 128) {
                    const int h = it / (kTcKeys * 8), kr = (it / 8) % kTcKeys, c = it % 8;
                    if (key_base + kr >= k_len || !((mask >> (kr / kBox)) & 1u))
                        *reinterpret_cast<uint4 *>(vt + h * kTileHalf + kr * 128 + c * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&p_full[j & 1]);
        }
        // all P.V done: mma_done completes exactly once (o_done's parity is
        // ambiguous here, since P.V_{nkt-2} may still be running)
        if (ok)
            ok = __all_sync(FULL, mbar_wait(mma_done, 0));
        if (!ok) {
            if (lane == 0)
                flag_error(p.err_flag, 0x8 /* PKV_FLAG_TIMEOUT */);
        } else {
            tc::fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint16_t *dst = p.out + ((size_t)(cq0 + tok) * p.Hq + kvh * G + g) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; c++) {
                uint32_t ro[32];
                tc::ld32(tO + tl + 32 * c, ro);
                tc::wait_ld();
                if (valid) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; i++)
                        pk[i] = pack_bf16x2(__uint_as_float(ro[2 * i]) * inv,
                                            __uint_as_float(ro[2 * i + 1]) * inv);
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c);
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
        }
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
