// fa_bwd64.cu -- backward main kernel for d = 64: a persistent grid over
// (128-key tile, b*h) work items.
//
// The method is fa_bwd.cu's ("The Attention Matrix You Never Write Down",
// "Tiling forward, recomputing backward"; "FlashAttention: Mathematical
// Foundations ...", "Backward Pass and Activation Recomputation"): per key
// tile, for each 128-row query block that sees it, rebuild
// P^T = exp(scale k.q - LSE) on chip and form
//     dV += P^T dO,  dP^T = V dO^T,  dS^T = P^T o (dP^T - D),
//     dK += dS^T Q,  dQ = dS K (reduce-added into the fp32 accumulator).
//
// At d = 64 the products of a block take half as long as at d = 128 while
// the per-block softmax work stays the same, so fixed costs weigh twice as
// much.  This kernel keeps them off the compute warps' path:
//   - persistent grid, one CTA per SM: the set-up (barriers, TMEM, register
//     split) is paid once, work items (key tile, b*h) come from a counter in
//     the workspace (words 2 and 3, left at zero by every launch: the last
//     CTA to stop taking items resets it), head-major with the causally
//     heaviest key tile of a head first, or, when the items differ in length,
//     spread across the heads of a group (8 heads, or all of them: key tile 0
//     of every head in the group first) for a short tail;
//   - K and V double-buffered: the next item's tiles load while the current
//     item computes;
//   - a dQ-drain warpgroup of its own (TMEM -> swizzled staging -> TMA
//     reduce-add), as in fa_bwd128.cu, so the compute warps' chain per
//     block is P -> dS only;
//   - under a block mask the producer lists an item's query blocks once (a
//     ballot compaction of the mask column), so no role scans the mask in
//     global memory block by block.
// Roles (512 threads): warp 0 producer (items, TMA), warp 1 tcgen05 issuer,
// warp 2 LSE/D stager (a ring of four blocks), warps 4-11 two compute warpgroups (one key row per thread,
// warpgroup w on query columns [64w, 64w + 64); at the end of an item each
// converts half of dK * scale and dV to bf16), warps 12-15 the dQ drain
// (one query row per thread).  TMEM (512 columns): S^T (128), dP^T (128), dV
// (64), dK (64), two dQ buffers (64 each).  Every barrier phase (blocks,
// ring stages, K/V buffers, items) runs on across items.
#include <algorithm>
#include <climits>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

namespace {

struct Bwd64 {
    static constexpr int D = 64;
    static constexpr int BQ = 128;
    static constexpr int CW = 64;                          // query columns per compute warpgroup
    static constexpr int TILE = 128 * 128;                 // 128 rows x 64 bf16 (one 128-byte chunk)
    static constexpr int OFF_K = 0;                        // [2] buffers
    static constexpr int OFF_V = OFF_K + 2 * TILE;         // [2]
    static constexpr int OFF_Q = OFF_V + 2 * TILE;         // [2] stages
    static constexpr int OFF_DO = OFF_Q + 2 * TILE;        // [2] stages
    static constexpr int OFF_DS = OFF_DO + 2 * TILE;       // [query chunk 2][key 128][128 B]
    static constexpr int OFF_STG = OFF_DS + 2 * TILE;      // [column chunk 2][query 128][128 B] fp32
    static constexpr int LSE_BUFS = 4;                     // LSE/D ring depth (blocks staged ahead)
    static constexpr int OFF_LSE = OFF_STG + 2 * TILE;     // [LSE_BUFS][BQ] fp32 (log2 domain)
    static constexpr int OFF_DV = OFF_LSE + LSE_BUFS * BQ * 4;   // [LSE_BUFS][BQ] fp32
    static constexpr int OFF_BAR = OFF_DV + LSE_BUFS * BQ * 4;
    static constexpr int B_KVFULL = 0;                     // [2] per K/V buffer
    static constexpr int B_KVFREE = 2;                     // [2]
    static constexpr int B_QFULL = 4;                      // [2] per Q/dO stage
    static constexpr int B_QEMPTY = 6;                     // [2]
    static constexpr int B_SFULL = 8;
    static constexpr int B_DPFULL = 9;
    static constexpr int B_PFULL = 10;                     // 256
    static constexpr int B_DSFULL = 11;                    // 256
    static constexpr int B_SFREE = 12;                     // dV of a block done: S columns free
    static constexpr int B_DPFREE = 13;                    // dK of a block done: dP columns free
    static constexpr int B_DQFULL = 14;                    // [2]
    static constexpr int B_DQFREE = 16;                    // [2] 128 (drain warpgroup)
    static constexpr int B_ACC = 18;                       // an item's dK, dV complete
    static constexpr int B_FIN = 19;
    static constexpr int B_LSE = 20;                       // [LSE_BUFS] LSE/D block staged (32)
    static constexpr int B_LSEFREE = 24;                   // [LSE_BUFS] block's LSE/D read (8 compute warps)
    static constexpr int B_ITEM = 28;                      // [2] item slot published (32)
    static constexpr int B_ITEMFREE = 30;                  // [2] slot read by every consumer (1 + 1 + 8 + 4)
    static constexpr int NBAR = 32;
    static constexpr int OFF_SLOT = (OFF_BAR + NBAR * 8 + 127) & ~127;   // [2] item slots, 128 B each
    static constexpr int LIST_CAP = 2048;                  // query blocks listed per item under a block mask
    static constexpr int OFF_LIST = OFF_SLOT + 2 * 128;    // [2][LIST_CAP] uint16
    static constexpr int OFF_MISC = OFF_LIST + 2 * LIST_CAP * 2;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_S = 0;
    static constexpr uint32_t TM_DP = BQ;
    static constexpr uint32_t TM_DV = 2 * BQ;
    static constexpr uint32_t TM_DK = 2 * BQ + D;
    static constexpr uint32_t TM_DQ = 2 * BQ + 2 * D;      // 2 x 64 columns
    static constexpr int THREADS = 512;
    static constexpr int LAUNCH_REGS = 128;
    static constexpr int REGS_CTRL = 112;
    static constexpr int REGS_COMPUTE = 152;
    static constexpr int REGS_DRAIN = 96;
    static_assert(128 * REGS_CTRL + 256 * REGS_COMPUTE + 128 * REGS_DRAIN == THREADS * LAUNCH_REGS,
                  "register split");
};

// One work item as the producer publishes it to the other roles.
struct BwdItem {
    int item;          // work-item index, or -1: no more work
    int bh, h, kt;     // key tile kt of head bh (h = bh % H)
    int q_start, k_start;
    int Lq, Lk;        // the sequence's query and key rows
    int kvis, shift;   // keys < kvis visible; causal: key j <= query i + shift
    int qb_start;      // without a list: the query blocks seen are [qb_start, qb_start + count)
    int count;         // query blocks to visit
    int use_list;      // blocks come from the item's list (block mask)
};
static_assert(sizeof(BwdItem) <= 128, "item slot");

__device__ __forceinline__ void b64_drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > FA_WAIT_TIMEOUT_NS) break;
}

// P^T / dS^T as bf16 pairs inside the S / dP columns: queries [16k, 16k + 16)
// at column 64 (k / 4) + 8 (k mod 4), so each compute warpgroup stays inside
// its own 64-column half and never overwrites fp32 values the other reads.
__device__ __forceinline__ uint32_t packed_col64(int k) { return (uint32_t)((k >> 2) * 64 + 8 * (k & 3)); }

template <bool VARLEN, bool LIST>
__global__ void __launch_bounds__(512, 1) fa_bwd64_kernel(const __grid_constant__ BwdParams p) {
    grid_dep_wait();                                 // the previous kernel in the stream is done
    grid_dep_launch();
    using S = Bwd64;
    constexpr int BQ = S::BQ, CW = S::CW, D = S::D;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int n_items = p.Tk * p.BH;
    const int nb = (p.N + kTile - 1) / kTile;

    auto bar = [&](int i) -> uint32_t { return base + S::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + S::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sb + S::OFF_MISC + 4);
    const Guard g{p.status, p.status + 1, abort_flag};
    BwdItem *slots = reinterpret_cast<BwdItem *>(sb + S::OFF_SLOT);
    auto list_of = [&](int s) { return reinterpret_cast<uint16_t *>(sb + S::OFF_LIST) + s * S::LIST_CAP; };
    unsigned *sched = p.status + 2;                  // workspace words 2 (next item) and 3 (CTAs done)
    float *lse_s = reinterpret_cast<float *>(sb + S::OFF_LSE);   // [LSE_BUFS][BQ], log2 domain
    float *dv_s = reinterpret_cast<float *>(sb + S::OFF_DV);     // [LSE_BUFS][BQ]

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(S::B_KVFULL + s), 1);
            mbar_init(bar(S::B_KVFREE + s), 1);
            mbar_init(bar(S::B_QFULL + s), 1);
            mbar_init(bar(S::B_QEMPTY + s), 1);
            mbar_init(bar(S::B_DQFULL + s), 1);
            mbar_init(bar(S::B_DQFREE + s), 128);
            mbar_init(bar(S::B_ITEM + s), 32);
            mbar_init(bar(S::B_ITEMFREE + s), 14);
        }
        for (int s = 0; s < S::LSE_BUFS; ++s) {
            mbar_init(bar(S::B_LSE + s), 32);
            mbar_init(bar(S::B_LSEFREE + s), 8);
        }
        mbar_init(bar(S::B_SFULL), 1);
        mbar_init(bar(S::B_DPFULL), 1);
        mbar_init(bar(S::B_PFULL), 256);
        mbar_init(bar(S::B_DSFULL), 256);
        mbar_init(bar(S::B_SFREE), 1);
        mbar_init(bar(S::B_DPFREE), 1);
        mbar_init(bar(S::B_ACC), 1);
        mbar_init(bar(S::B_FIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&p.tmQ);
        tma_prefetch_desc(&p.tmdO);
        tma_prefetch_desc(&p.tmK);
        tma_prefetch_desc(&p.tmV);
        tma_prefetch_desc(&p.tmdQ);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), S::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // query block of entry e of an item
    auto entry_qb = [&](const BwdItem &it, const uint16_t *lst, int e) -> int {
        // LIST: a block mask may be given (query-block lists); without one the
        // kernel carries no list code
        if constexpr (!LIST) return it.qb_start + e;
        return it.use_list ? (int)lst[e] : it.qb_start + e;
    };
    // class of query block qb against the item's key tile (a listed block is
    // one the mask keeps)
    auto cls = [&](const BwdItem &it, int qb) -> unsigned {
        const int qa = qb * BQ, k0 = it.kt * kTile;
        if constexpr (VARLEN) return tile_class_shift(qa, min(BQ, it.Lq - qa), k0, kTile, it.kvis, p.causal, it.shift);
        return tile_class(qa, min(BQ, p.N - qa), k0, kTile, it.kvis, p.causal, 1);
    };

    // Register split (as in fa_bwd128.cu): warpgroup 0 and the drain give
    // registers back, the compute warpgroups take them; the pool is filled by
    // the unconditional decs, so the one inc never waits on a waiting warp.
    if (warp < 4) {
        setmaxnreg_dec<S::REGS_CTRL>();
        if (warp == 0) {
            // ---------------------------------------------------------- producer (whole warp)
            int k = 0, nkv = 0, i = 0;               // items published, items whose K/V were loaded, blocks
            bool ok = true;
            for (;; ++k) {
                const int s = k & 1;
                if (k >= 2 && !mbar_wait_warp(bar(S::B_ITEMFREE + s), (uint32_t)((k >> 1) - 1) & 1u, g, 0x130)) {
                    ok = false;
                    break;
                }
                BwdItem it;
                it.item = -1;
                for (;;) {
                    int j = 0;
                    if (lane == 0) j = (int)atomicAdd(sched, 1u);
                    j = __shfl_sync(0xffffffffu, j, 0);
                    if (j >= n_items) break;
                    // item j: head-major, the causally heaviest (lowest) key tile first;
                    // else groups of p.spread heads (every head: spread order), key
                    // tile 0 of a group's heads first, then key tile 1, the groups in order
                    int kt = j % p.Tk, bh = j / p.Tk;
                    if (p.spread > 0) {
                        const int per = p.Tk * p.spread;
                        const int gi = j / per, i = j - gi * per;
                        const int gs = min(p.spread, p.BH - gi * p.spread);
                        kt = i / gs;
                        bh = gi * p.spread + (i - kt * gs);
                    }
                    const int b = bh / p.H, h = bh % p.H;
                    int q_start = 0, k_start = 0, Lq = p.N, Lk = p.N;
                    bool bad = false;
                    if constexpr (VARLEN)
                        varlen_sequence(p.cu_q, p.cu_k, b, p.total_q, p.total_k, INT_MAX, p.Tk * kTile, &q_start, &Lq,
                                        &k_start, &Lk, &bad);
                    const int kvis = VARLEN ? Lk : key_visible_bound(p.key_len, b, p.N, &bad);
                    if (bad && lane == 0 && kt == 0 && h == 0) record_status(g, kStatusBadKeyLen, 0);
                    // a key tile past a ragged sequence's end has no row to write
                    if (VARLEN && kt * kTile >= Lk) continue;
                    const int Tqb = (Lq + BQ - 1) / BQ;
                    it.item = j;
                    it.bh = bh;
                    it.h = h;
                    it.kt = kt;
                    it.q_start = q_start;
                    it.k_start = k_start;
                    it.Lq = Lq;
                    it.Lk = Lk;
                    it.kvis = kvis;
                    it.shift = Lk - Lq;
                    it.qb_start = bwd_query_block_begin(kt * kTile, kvis, p.causal, it.shift, BQ, Tqb);
                    it.count = Tqb - it.qb_start;
                    it.use_list = (LIST && !VARLEN && p.block_mask) ? 1 : 0;
                    break;
                }
                uint16_t *lst = list_of(s);
                if (LIST && it.item >= 0 && it.use_list) {
                    // the query blocks that see this key tile, in order, compacted by the whole warp
                    const int Tqb = (it.Lq + BQ - 1) / BQ;
                    int n = 0;
                    for (int q0b = 0; q0b < Tqb; q0b += 32) {
                        const int qb = q0b + lane;
                        bool v = false;
                        if (qb < Tqb) {
                            const int qa = qb * BQ;
                            const int on = p.block_mask[(size_t)qb * nb + it.kt] != 0;
                            v = tile_class(qa, min(BQ, p.N - qa), it.kt * kTile, kTile, it.kvis, p.causal, on) !=
                                kTileSkip;
                        }
                        const unsigned ball = __ballot_sync(0xffffffffu, v);
                        if (v) lst[n + __popc(ball & ((1u << lane) - 1u))] = (uint16_t)qb;
                        n += __popc(ball);
                    }
                    it.count = n;
                }
                if (lane == 0) slots[s] = it;
                mbar_arrive(bar(S::B_ITEM + s));    // every lane, after its own list writes
                if (it.item < 0) break;
                if (it.count == 0) continue;        // no query block sees the tile: dK = dV = 0, no loads
                // K, V into buffer nkv & 1 once the item that last used it is done with it
                const int kb = nkv & 1;
                if (nkv >= 2 &&
                    !mbar_wait_warp(bar(S::B_KVFREE + kb), (uint32_t)((nkv >> 1) - 1) & 1u, g, 0x131)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_elect(bar(S::B_KVFULL + kb), 2 * S::TILE);
                const int k0 = it.kt * kTile;
                if constexpr (VARLEN) {
                    tma_load_3d_elect(base + S::OFF_K + kb * S::TILE, &p.tmK, bar(S::B_KVFULL + kb), 0, it.h,
                                      it.k_start + k0);
                    tma_load_3d_elect(base + S::OFF_V + kb * S::TILE, &p.tmV, bar(S::B_KVFULL + kb), 0, it.h,
                                      it.k_start + k0);
                } else {
                    tma_load_3d_elect(base + S::OFF_K + kb * S::TILE, &p.tmK, bar(S::B_KVFULL + kb), 0, k0, it.bh);
                    tma_load_3d_elect(base + S::OFF_V + kb * S::TILE, &p.tmV, bar(S::B_KVFULL + kb), 0, k0, it.bh);
                }
                ++nkv;
                for (int e = 0; e < it.count; ++e, ++i) {
                    const int qb = entry_qb(it, lst, e);
                    const int st = i & 1;
                    // Q, dO into stage st once dK(i - 2) has read it
                    if (!mbar_wait_warp(bar(S::B_QEMPTY + st), ((uint32_t)(i >> 1) & 1u) ^ 1u, g, 0x132)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_elect(bar(S::B_QFULL + st), 2 * S::TILE);
                    if constexpr (VARLEN) {
                        tma_load_3d_elect(base + S::OFF_Q + st * S::TILE, &p.tmQ, bar(S::B_QFULL + st), 0, it.h,
                                          it.q_start + qb * BQ);
                        tma_load_3d_elect(base + S::OFF_DO + st * S::TILE, &p.tmdO, bar(S::B_QFULL + st), 0, it.h,
                                          it.q_start + qb * BQ);
                    } else {
                        tma_load_3d_elect(base + S::OFF_Q + st * S::TILE, &p.tmQ, bar(S::B_QFULL + st), 0, qb * BQ,
                                          it.bh);
                        tma_load_3d_elect(base + S::OFF_DO + st * S::TILE, &p.tmdO, bar(S::B_QFULL + st), 0, qb * BQ,
                                          it.bh);
                    }
                }
                if (!ok) break;
            }
            // this CTA takes no more items; the last CTA to get here resets the counter
            if (lane == 0) {
                __threadfence();
                if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
                    atomicExch(sched, 0u);
                    atomicExch(sched + 1, 0u);
                }
            }
            __syncwarp();
            if (!ok && lane == 0) {
                // gave up: let every copy already issued land before the CTA exits
                if (nkv > 0) b64_drain_wait(bar(S::B_KVFULL + ((nkv - 1) & 1)), (uint32_t)((nkv - 1) >> 1) & 1u);
                for (int j = (i > 2 ? i - 2 : 0); j < i; ++j)
                    b64_drain_wait(bar(S::B_QFULL + (j & 1)), (uint32_t)(j >> 1) & 1u);
            }
        } else if (warp == 2) {
            // ---------------------------------------------------------- LSE / D stager (whole warp)
            // Stages each block's LSE (log2 domain; +inf past the sequence's
            // last query or for a row with no visible key, so that its P is 0)
            // and D into a ring of LSE_BUFS buffers, up to LSE_BUFS blocks ahead
            // of the compute warps and independent of the Q/dO ring: staged by
            // the producer behind each block's Q/dO slot, these global loads sat
            // on the compute warps' path.
            int i = 0;
            for (int k = 0;; ++k) {
                const int s = k & 1;
                if (!mbar_wait_warp(bar(S::B_ITEM + s), (uint32_t)(k >> 1) & 1u, g, 0x1b0)) break;
                const BwdItem it = slots[s];
                if (it.item < 0) break;
                const uint16_t *lst = list_of(s);
                bool ok = true;
                for (int e = 0; e < it.count; ++e, ++i) {
                    const int qb = entry_qb(it, lst, e);
                    const int lb = i % S::LSE_BUFS;
                    if (i >= S::LSE_BUFS && !mbar_wait_warp(bar(S::B_LSEFREE + lb),
                                                            (uint32_t)(i / S::LSE_BUFS - 1) & 1u, g, 0x1b1)) {
                        ok = false;
                        break;
                    }
                    // all eight loads of this lane first, then the stores
                    float v[BQ / 32], dd[BQ / 32];
#pragma unroll
                    for (int u = 0; u < BQ / 32; ++u) {
                        const int qq = qb * BQ + u * 32 + lane;
                        v[u] = INFINITY;
                        dd[u] = 0.f;
                        if (qq < it.Lq) {
                            const size_t li = VARLEN ? (size_t)it.h * p.total_q + it.q_start + qq
                                                     : (size_t)it.bh * p.N + qq;
                            const size_t di = VARLEN ? (size_t)(it.q_start + qq) * p.H + it.h : (size_t)it.bh * p.N + qq;
                            v[u] = p.LSE[li];
                            dd[u] = p.Dvec[di];
                        }
                    }
#pragma unroll
                    for (int u = 0; u < BQ / 32; ++u) {
                        lse_s[lb * BQ + u * 32 + lane] = (v[u] == -INFINITY) ? INFINITY : v[u] * 1.4426950408889634f;
                        dv_s[lb * BQ + u * 32 + lane] = dd[u];
                    }
                    mbar_arrive(bar(S::B_LSE + lb));
                }
                if (!ok) break;
                if (lane == 0) mbar_arrive(bar(S::B_ITEMFREE + s));
            }
        } else if (warp == 1) {
            // ---------------------------------------------------------- MMA issuer (whole warp)
            // Per block i: dV(i), S(i+1), dK(i), dQ(i), dP(i+1) within an item;
            // an item's first S and dP once the previous item's last dV and dK
            // have read the S and dP columns.
            constexpr uint32_t IDESC_S = idesc_bf16(128, BQ, false, false);   // S^T, dP^T
            constexpr uint32_t IDESC_ACC = idesc_bf16(128, D, false, true);   // dV, dK
            constexpr uint32_t IDESC_DQ = idesc_bf16(128, D, true, true);     // dQ = dS K
            bool ok = true;
            int k = 0, nkv = 0, i = 0;
            for (;; ++k) {
                const int s = k & 1;
                if (!mbar_wait_warp(bar(S::B_ITEM + s), (uint32_t)(k >> 1) & 1u, g, 0x230)) {
                    ok = false;
                    break;
                }
                const BwdItem it = slots[s];
                if (it.item < 0) break;
                if (it.count > 0) {
                    const int kb = nkv & 1;
                    const uint32_t ko = base + S::OFF_K + kb * S::TILE, vo = base + S::OFF_V + kb * S::TILE;
                    const uint64_t dK_kmaj = sdesc_sw128(ko, 16, 1024);           // K as A, K-major
                    const uint64_t dV_kmaj = sdesc_sw128(vo, 16, 1024);           // V as A, K-major
                    const uint64_t dK_mn = sdesc_sw128(ko, S::TILE, 1024);        // K as B, MN-major (dQ)
                    const uint64_t ddS_mn = sdesc_sw128(base + S::OFF_DS, S::TILE, 1024);   // dS as A, MN-major
                    auto issue_s = [&](int blk) {                                 // S^T = K Q^T
                        const uint64_t qd = sdesc_sw128(base + S::OFF_Q + (blk & 1) * S::TILE, 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss_elect(tmem + S::TM_S, sdesc_add(dK_kmaj, kk * 32), sdesc_add(qd, kk * 32), IDESC_S,
                                         kk > 0 ? 1u : 0u);
                        mma_commit_elect(bar(S::B_SFULL));
                    };
                    auto issue_dp = [&](int blk) {                                // dP^T = V dO^T
                        const uint64_t dd = sdesc_sw128(base + S::OFF_DO + (blk & 1) * S::TILE, 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss_elect(tmem + S::TM_DP, sdesc_add(dV_kmaj, kk * 32), sdesc_add(dd, kk * 32), IDESC_S,
                                         kk > 0 ? 1u : 0u);
                        mma_commit_elect(bar(S::B_DPFULL));
                    };
                    ok = mbar_wait_warp(bar(S::B_KVFULL + kb), (uint32_t)(nkv >> 1) & 1u, g, 0x231) &&
                         mbar_wait_warp(bar(S::B_QFULL + (i & 1)), (uint32_t)(i >> 1) & 1u, g, 0x232);
                    ++nkv;
                    // the item's first S and dP: the previous block's dV and dK must
                    // have read P^T and dS^T from those columns
                    if (ok && i > 0)
                        ok = mbar_wait_warp(bar(S::B_SFREE), (uint32_t)(i - 1) & 1u, g, 0x233);
                    if (ok) {
                        tc_fence_after();
                        issue_s(i);
                    }
                    if (ok && i > 0)
                        ok = mbar_wait_warp(bar(S::B_DPFREE), (uint32_t)(i - 1) & 1u, g, 0x234);
                    if (ok) {
                        tc_fence_after();
                        issue_dp(i);
                    }
                    for (int e = 0; ok && e < it.count; ++e, ++i) {
                        const int st = i & 1;
                        const uint64_t q_mn = sdesc_sw128(base + S::OFF_Q + st * S::TILE, S::TILE, 1024);
                        const uint64_t do_mn = sdesc_sw128(base + S::OFF_DO + st * S::TILE, S::TILE, 1024);
                        const uint32_t acc0 = e > 0 ? 1u : 0u;
                        const bool more = e + 1 < it.count;
                        // dV += P^T dO: A = P^T from TMEM, B = dO (N = D, K = queries, MN-major)
                        if (!mbar_wait_warp(bar(S::B_PFULL), (uint32_t)i & 1u, g, 0x235)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < BQ / 16; ++kk)
                            mma_ts_elect(tmem + S::TM_DV, tmem + S::TM_S + packed_col64(kk),
                                         sdesc_add(do_mn, (uint32_t)kk * 2048u), IDESC_ACC, kk > 0 ? 1u : acc0);
                        mma_commit_elect(bar(S::B_SFREE));
                        // S(i+1) once dV(i) has read P(i)
                        if (more) {
                            if (!mbar_wait_warp(bar(S::B_QFULL + (st ^ 1)), (uint32_t)((i + 1) >> 1) & 1u, g, 0x236) ||
                                !mbar_wait_warp(bar(S::B_SFREE), (uint32_t)i & 1u, g, 0x237)) { ok = false; break; }
                            tc_fence_after();
                            issue_s(i + 1);
                        }
                        // dK += dS^T Q: A = dS^T from TMEM, B = Q (MN-major)
                        if (!mbar_wait_warp(bar(S::B_DSFULL), (uint32_t)i & 1u, g, 0x238)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < BQ / 16; ++kk)
                            mma_ts_elect(tmem + S::TM_DK, tmem + S::TM_DP + packed_col64(kk),
                                         sdesc_add(q_mn, (uint32_t)kk * 2048u), IDESC_ACC, kk > 0 ? 1u : acc0);
                        mma_commit_elect(bar(S::B_DPFREE));
                        mma_commit_elect(bar(S::B_QEMPTY + st));
                        // dQ = dS K into TMEM buffer i % 2 once the drain has emptied it
                        if (i >= 2 &&
                            !mbar_wait_warp(bar(S::B_DQFREE + st), (uint32_t)((i - 2) >> 1) & 1u, g, 0x239)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t dq_tmem = tmem + S::TM_DQ + 64u * (uint32_t)st;
#pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk)
                            mma_ss_elect(dq_tmem, sdesc_add(ddS_mn, (uint32_t)kk * 2048u),
                                         sdesc_add(dK_mn, (uint32_t)kk * 2048u), IDESC_DQ, kk > 0 ? 1u : 0u);
                        mma_commit_elect(bar(S::B_DQFULL + st));
                        // dP(i+1) once dK(i) has read dS(i)
                        if (more) {
                            if (!mbar_wait_warp(bar(S::B_DPFREE), (uint32_t)i & 1u, g, 0x23a)) { ok = false; break; }
                            tc_fence_after();
                            issue_dp(i + 1);
                        }
                    }
                    if (!ok) break;
                    // the item's dK, dV are complete, and its K/V buffer is free, once these finish
                    mma_commit_elect(bar(S::B_ACC));
                    mma_commit_elect(bar(S::B_KVFREE + kb));
                }
                if (lane == 0) mbar_arrive(bar(S::B_ITEMFREE + s));
            }
            mma_commit_elect(bar(S::B_FIN));
            b64_drain_wait(bar(S::B_FIN), 0);
        }
    } else if (warp < 12) {
        setmaxnreg_inc<S::REGS_COMPUTE>();
        // ---------------------------------------------------------- compute (two warpgroups)
        const int wg = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;           // TMEM lane: key row of S^T, dP^T, dK, dV
        const int c0 = wg * CW;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const float c2 = p.scale_log2;
        bool ok = true;
        int i = 0, nacc = 0;
        for (int k = 0;; ++k) {
            const int s = k & 1;
            if (!mbar_wait_warp(bar(S::B_ITEM + s), (uint32_t)(k >> 1) & 1u, g, 0x430)) {
                ok = false;
                break;
            }
            const BwdItem &itr = slots[s];
            if (itr.item < 0) break;
            const BwdItem it = itr;
            const uint16_t *lst = list_of(s);
            const int key = it.kt * kTile + r;      // key row of the sequence
            for (int e = 0; e < it.count; ++e, ++i) {
                const int qb = entry_qb(it, lst, e);
                const unsigned klass = cls(it, qb);
                const int qa = qb * BQ;
                const int lb = i % S::LSE_BUFS;
                if (!mbar_wait_warp(bar(S::B_LSE + lb), (uint32_t)(i / S::LSE_BUFS) & 1u, g, 0x431)) {
                    ok = false;
                    break;
                }
                const float *ls = lse_s + lb * BQ;
                const float *dd = dv_s + lb * BQ;
                // P^T = 2^(s * c - LSE_q * log2 e), masked, for columns c0 .. c0 + CW
                if (!mbar_wait_warp(bar(S::B_SFULL), (uint32_t)i & 1u, g, 0x432)) { ok = false; break; }
                tc_fence_after();
                uint32_t pk[CW / 2];
                {
                    uint32_t sr[CW / 32][32];
#pragma unroll
                    for (int j = 0; j < CW / 32; ++j) tmem_ld32(tmem + lane_off + S::TM_S + c0 + 32u * j, sr[j]);
#pragma unroll
                    for (int j = 0; j < CW / 32; ++j) tmem_ld_wait(sr[j]);
                    if (klass == kTilePartial) {
                        // masked scores -> -inf, so that their p is exactly 0: this key
                        // row sees the columns from lo on (none past the visible keys),
                        // one compare against a constant per score
                        int lo = p.causal ? key - it.shift - qa - c0 : INT_MIN;
                        if (key >= it.kvis) lo = INT_MAX;
#pragma unroll
                        for (int j = 0; j < CW / 32; ++j)
#pragma unroll
                            for (int t = 0; t < 32; ++t)
                                if (32 * j + t < lo) sr[j][t] = __float_as_uint(-INFINITY);
                    }
#pragma unroll
                    for (int j = 0; j < CW / 32; ++j)
#pragma unroll
                        for (int t = 0; t < 32; t += 4) {
                            const float4 l4 = *reinterpret_cast<const float4 *>(ls + c0 + 32 * j + t);
                            float p0, p1, p2, p3;
                            fma2(p0, p1, __uint_as_float(sr[j][t]), __uint_as_float(sr[j][t + 1]), c2, c2, -l4.x, -l4.y);
                            fma2(p2, p3, __uint_as_float(sr[j][t + 2]), __uint_as_float(sr[j][t + 3]), c2, c2, -l4.z,
                                 -l4.w);
                            pk[16 * j + t / 2] = pack_bf16x2(ex2(p0), ex2(p1));
                            pk[16 * j + t / 2 + 1] = pack_bf16x2(ex2(p2), ex2(p3));
                        }
                }
#pragma unroll
                for (int j = 0; j < CW / 32; ++j) tmem_st16(tmem + lane_off + S::TM_S + c0 + 16u * j, pk + 16 * j);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(S::B_PFULL));

                // dS^T = P^T o (dP^T - D): bf16 into TMEM (for dK) and shared memory (for dQ)
                if (!mbar_wait_warp(bar(S::B_DPFULL), (uint32_t)i & 1u, g, 0x433)) { ok = false; break; }
                // the dQ product of the previous block must be done reading the shared dS tile
                if (i > 0 &&
                    !mbar_wait_warp(bar(S::B_DQFULL + ((i - 1) & 1)), (uint32_t)((i - 1) >> 1) & 1u, g, 0x434)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    uint32_t dp[CW / 32][32];
#pragma unroll
                    for (int j = 0; j < CW / 32; ++j) tmem_ld32(tmem + lane_off + S::TM_DP + c0 + 32u * j, dp[j]);
#pragma unroll
                    for (int j = 0; j < CW / 32; ++j) tmem_ld_wait(dp[j]);
#pragma unroll
                    for (int j = 0; j < CW / 32; ++j) {
                        uint32_t w[16];
#pragma unroll
                        for (int t = 0; t < 16; t += 2) {
                            const float4 d4 = *reinterpret_cast<const float4 *>(dd + c0 + 32 * j + 2 * t);
                            const uint32_t pa = pk[16 * j + t], pb = pk[16 * j + t + 1];
                            w[t] = pack_bf16x2(bf16lo(pa) * (__uint_as_float(dp[j][2 * t]) - d4.x),
                                               bf16hi(pa) * (__uint_as_float(dp[j][2 * t + 1]) - d4.y));
                            w[t + 1] = pack_bf16x2(bf16lo(pb) * (__uint_as_float(dp[j][2 * t + 2]) - d4.z),
                                                   bf16hi(pb) * (__uint_as_float(dp[j][2 * t + 3]) - d4.w));
                        }
                        tmem_st16(tmem + lane_off + S::TM_DP + c0 + 16u * j, w);
                        // shared dS tile, queries contiguous (MN-major, 128-byte swizzle):
                        // [query chunk of 64][key row 0..127][128 bytes]; this warpgroup's
                        // 64 queries are chunk wg
#pragma unroll
                        for (int u4 = 0; u4 < 4; ++u4) {
                            const int qo = 32 * j + 8 * u4;        // first query of this 16-byte piece, in the chunk
                            uint8_t *dst = sb + S::OFF_DS + wg * S::TILE + r * 128 + ((((qo >> 3)) ^ (r & 7)) << 4);
                            *reinterpret_cast<uint4 *>(dst) =
                                make_uint4(w[4 * u4], w[4 * u4 + 1], w[4 * u4 + 2], w[4 * u4 + 3]);
                        }
                    }
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(S::B_DSFULL));
                // this block's LSE and D have been read
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(S::B_LSEFREE + lb));
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue of the item: dK, dV
            // warpgroup wg converts head-dimension columns [32 wg, 32 wg + 32)
            if (it.count > 0) {
                if (!mbar_wait_warp(bar(S::B_ACC), (uint32_t)nacc & 1u, g, 0x435)) {
                    ok = false;
                    break;
                }
                ++nacc;
                tc_fence_after();
            }
            {
                uint32_t a[32], v[32];
                if (it.count > 0) {
                    tmem_ld32(tmem + lane_off + S::TM_DK + 32u * wg, a);
                    tmem_ld32(tmem + lane_off + S::TM_DV + 32u * wg, v);
                    tmem_ld_wait(a);
                    tmem_ld_wait(v);
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) a[t] = v[t] = 0u;
                }
                uint32_t wk[16], wv[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    wk[t] = pack_bf16x2(__uint_as_float(a[2 * t]) * p.scale, __uint_as_float(a[2 * t + 1]) * p.scale);
                    wv[t] = pack_bf16x2(__uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1]));
                }
                // Through this warp's own rows of the dS tile (free: the item's
                // products are complete, and only this warp writes these rows
                // again, in its next dS pass): 64 bytes of dK and of dV per row
                // (128-byte swizzle), then read back so that each store covers
                // 8 rows x 64 contiguous bytes.  Stored straight from registers,
                // each store touched 32 rows and the epilogue took ~4,000 cycles.
                uint8_t *stg = sb + S::OFF_DS + wg * S::TILE + wq * 32 * 128;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    *reinterpret_cast<uint4 *>(stg + lane * 128 + ((t ^ (lane & 7)) << 4)) =
                        make_uint4(wk[4 * t], wk[4 * t + 1], wk[4 * t + 2], wk[4 * t + 3]);
                    *reinterpret_cast<uint4 *>(stg + lane * 128 + (((4 + t) ^ (lane & 7)) << 4)) =
                        make_uint4(wv[4 * t], wv[4 * t + 1], wv[4 * t + 2], wv[4 * t + 3]);
                }
                __syncwarp();
                // all eight values first, then the stores: interleaved, each shared
                // load waited behind the previous global store (the compiler cannot
                // tell the two apart)
                const int u = lane & 3;
                uint4 kq[4], vq[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int rr = 8 * j + (lane >> 2);          // row of this warp's 32
                    kq[j] = *reinterpret_cast<const uint4 *>(stg + rr * 128 + ((u ^ (rr & 7)) << 4));
                    vq[j] = *reinterpret_cast<const uint4 *>(stg + rr * 128 + (((4 + u) ^ (rr & 7)) << 4));
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int rr = 8 * j + (lane >> 2);
                    const int keyr = it.kt * kTile + wq * 32 + rr;
                    if (keyr < it.Lk) {
                        const size_t krow =
                            VARLEN ? (size_t)(it.k_start + keyr) * p.H + it.h : (size_t)it.bh * p.N + keyr;
                        *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.dK) + krow * D + 32 * wg + 8 * u) =
                            kq[j];
                        *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.dV) + krow * D + 32 * wg + 8 * u) =
                            vq[j];
                    }
                }
                __syncwarp();
            }
            // (the next item's first dV and dK into these columns follow this
            // warpgroup's next P and dS arrivals, which follow these loads)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(S::B_ITEMFREE + s));
        }
        __syncwarp();
        setmaxnreg_dec<S::REGS_CTRL>();
    } else {
        setmaxnreg_dec<S::REGS_DRAIN>();
        // ---------------------------------------------------------- dQ drain (one warpgroup)
        // lane = query row 32 wq + lane of dQ(i) (64 columns): TMEM -> the
        // warp's 32 rows of both column chunks of the staging tile (128-byte
        // swizzle) -> two 32 x 32 fp32 TMA reduce-adds into the accumulator
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        int i = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int s = k & 1;
            if (!mbar_wait_warp(bar(S::B_ITEM + s), (uint32_t)(k >> 1) & 1u, g, 0x530)) break;
            const BwdItem &itr = slots[s];
            if (itr.item < 0) break;
            const BwdItem it = itr;
            const uint16_t *lst = list_of(s);
            for (int e = 0; e < it.count; ++e, ++i) {
                const int qb = entry_qb(it, lst, e);
                const int st = i & 1;
                if (!mbar_wait_warp(bar(S::B_DQFULL + st), (uint32_t)(i >> 1) & 1u, g, 0x531)) { ok = false; break; }
                tc_fence_after();
                uint32_t v[2][32];
                tmem_ld32(tmem + lane_off + S::TM_DQ + 64u * (uint32_t)st, v[0]);
                tmem_ld32(tmem + lane_off + S::TM_DQ + 64u * (uint32_t)st + 32u, v[1]);
                tmem_ld_wait(v[0]);
                tmem_ld_wait(v[1]);
                tc_fence_before();
                mbar_arrive(bar(S::B_DQFREE + st));
                // this warp's previous reduces must have read its rows of the staging tile
                if (lane == 0) bulk_wait_group_read<0>();
                __syncwarp();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint8_t *cb = sb + S::OFF_STG + c * S::TILE + r * 128;
#pragma unroll
                    for (int gq = 0; gq < 8; ++gq)
                        *reinterpret_cast<uint4 *>(cb + ((gq ^ (r & 7)) << 4)) =
                            make_uint4(v[c][4 * gq], v[c][4 * gq + 1], v[c][4 * gq + 2], v[c][4 * gq + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int q0 = qb * BQ + wq * 32;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t box = base + S::OFF_STG + c * S::TILE + wq * 32 * 128;
                        if constexpr (VARLEN)
                            tma_reduce_add_3d(&p.tmdQ, box, 32 * c, it.h, it.q_start + q0);
                        else
                            tma_reduce_add_3d(&p.tmdQ, box, 32 * c, q0, it.bh);
                    }
                    bulk_commit_group();
                }
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(S::B_ITEMFREE + s));
        }
        // the staged tiles must be fully reduced before shared memory goes away
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, S::TMEM_COLS);
}

template <bool VARLEN, bool LIST>
cudaError_t launch_bwd64_t(const BwdParams &p, cudaStream_t st) {
    const int smem = Bwd64::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(fa_bwd64_kernel<VARLEN, LIST>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)p.Tk * p.BH;
    const unsigned grid = (unsigned)std::min<int64_t>(items, device_sm_count());
    return launch_dep(fa_bwd64_kernel<VARLEN, LIST>, grid, Bwd64::THREADS, smem, st, p);
}

}  // namespace

int bwd64_smem_bytes() { return Bwd64::SMEM_BYTES; }

cudaError_t launch_bwd64_main(const BwdParams &p, cudaStream_t st) {
    return p.block_mask ? launch_bwd64_t<false, true>(p, st) : launch_bwd64_t<false, false>(p, st);
}

cudaError_t launch_bwd64_main_varlen(const BwdParams &p, cudaStream_t st) {
    return launch_bwd64_t<true, false>(p, st);
}

}  // namespace fa
