// fa_fwd.cu -- forward kernel: O and LSE of exact attention, tile by tile,
// never writing the score matrix.
//
// Method ("The Attention Matrix You Never Write Down", section "The
// running-statistics trick"; "FlashAttention: Mathematical Foundations ...",
// sections "Incremental Online Updates" and "IO-Aware Tiling Algorithm"):
// per query row keep a running maximum m and normaliser l; for each new key
// tile take m' = max(m, tile max), multiply l and the unnormalised output by
// exp(m - m'), add the tile's exp(s - m') and exp(s - m') V; divide by l at
// the end.  The tiling page prints the correction as diag(exp(m - m'))^-1;
// that contradicts the running-statistics page and its own final
// diag(l)^-1 normalisation, so the multiply-by-exp(m - m') reading is used.
// Everything is in base 2: x = s * scale * log2(e), p = 2^(x - m).
//
// The reference maximum is only moved when a row's tile maximum exceeds it
// by more than kRescaleLog2 (2^8): until then l, O and the new p all keep the
// old reference, which is the same identity with m' replaced by any common
// reference, so the result is unchanged and p stays <= 2^8.  This skips most
// O rescales (tcgen05.ld/st of the whole accumulator).
//
// GB300 design (not the A100 loop order the tiling page prints; the query
// tile is the outer loop, as in its "FlashAttention-2" section, so O stays
// on chip):
//   - a persistent grid, one CTA per SM; a work item is a pair of 128-row
//     query tiles of one b*h; the CTAs take items from a counter in the
//     workspace, head-major with the causally heaviest pair of a head first,
//     so the set-up (barriers, TMEM, register split) is paid once per SM and
//     the next item's Q load and first S product overlap the current item's
//     last tile and epilogue;
//   - warp 0: producer: takes the next item, describes it in a shared
//     slot for the other roles (under a block mask with the compacted list
//     of the key tiles the item sees, built once by the whole warp), then
//     TMA: both Q tiles once the previous item's S products are done with the
//     Q buffer; K and V tiles through a ring of shared-memory stages
//     (128-byte swizzle, 64-column boxes), over the union of the key tiles the
//     two query tiles see;
//   - warp 1: tcgen05 issuer: for each key tile and query tile x in turn,
//     O_x += P_x V with P_x read from TMEM (bf16, written over the first half
//     of S_x), then the next key tile's S_x = Q_x K^T as soon as that P.V
//     has read P_x, before the other query tile's P.V is waited for;
//   - warps 4-7 and 8-11: softmax of query tile 0 and 1, one row per thread
//     (TMEM lane = row, warp w reads lane quadrant w % 4), with 208 registers
//     each (setmaxnreg; warps 0-3 drop to 88).  The whole S row
//     is loaded with one wait, then max (3-input), 2^(x - m) with packed
//     f32x2 FMA/add, bf16 pack, store back; then the rare O rescale and, at
//     the end, the epilogue O / l -> bf16, LSE = (m + log2 l) * ln 2.
// Skipped tiles (block mask zero, all keys past key_len, above the causal
// diagonal) are never loaded; partial tiles get element masks.
//
// Ragged batches (VARLEN): sequences of different lengths packed one after
// another, [total][H][d]; the grid covers the longest sequence and CTAs past
// a shorter one's end have nothing to do.  A sequence's Lq queries are its
// last positions among its Lk keys (a cached prefix, or Lq = Lk for a plain
// prefill), so the causal diagonal is shifted by Lk - Lq.
#include <algorithm>
#include <climits>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

constexpr float kRescaleLog2 = 8.0f;

template <int D, int BC = 128>
struct FwdShape {
    static_assert(BC == 64 || BC == 128, "key tile width");
    static constexpr int KC = BC / 32;                  // 32-column chunks of an S row
    static constexpr int CHUNKS = D / 64;               // 64-element (128-byte) column chunks
    static constexpr int CHUNK_BYTES = 128 * 128;       // 128 query rows x 128 bytes
    static constexpr int TILE_BYTES = CHUNKS * CHUNK_BYTES;
    static constexpr int KV_CHUNK_BYTES = BC * 128;     // BC key rows x 128 bytes
    static constexpr int KV_TILE_BYTES = CHUNKS * KV_CHUNK_BYTES;
    static constexpr int STAGES = (D == 64 || BC == 64) ? 4 : 2;
    static constexpr int OFF_Q = 0;                     // [2] query tiles
    static constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
    static constexpr int OFF_V = OFF_K + STAGES * KV_TILE_BYTES;
    static constexpr int OFF_BAR = OFF_V + STAGES * KV_TILE_BYTES;
    static constexpr int B_QFULL = 0;
    static constexpr int B_QEMPTY = 1;                   // an item's S products are done: Q free
    static constexpr int B_KFULL = 2;
    static constexpr int B_VFULL = B_KFULL + STAGES;
    // a stage's K is free once the S products of its key tile are done, its V
    // once the P.V products are: released apart, the next K loads a step sooner
    static constexpr int B_KEMPTY = B_VFULL + STAGES;
    static constexpr int B_VEMPTY = B_KEMPTY + STAGES;
    static constexpr int B_SFULL = B_VEMPTY + STAGES;    // [2] one per query tile
    static constexpr int B_PFULL = B_SFULL + 2;          // [2]
    static constexpr int B_PVDONE = B_PFULL + 2;         // [2]
    static constexpr int B_SFREE = B_PVDONE + 2;         // [2] S_x loaded by its softmax (separate P only)
    static constexpr int B_ITEM = B_SFREE + 2;           // [2] work-item slot published (32 arrivals)
    static constexpr int B_ITEMFREE = B_ITEM + 2;        // [2] slot read by every consumer (1 + 8 arrivals)
    static constexpr int B_FIN = B_ITEMFREE + 2;
    static constexpr int NBAR = B_FIN + 1;
    static constexpr int OFF_SLOT = (OFF_BAR + NBAR * 8 + 127) & ~127;   // [2] FwdItem, 128 bytes each
    // key-tile list of an item under a block mask: entry = tile | visible to
    // query tile 0 << 14 | visible to query tile 1 << 15
    static constexpr int LIST_CAP = 2048;
    static constexpr int OFF_LIST = OFF_SLOT + 2 * 128;  // [2][LIST_CAP] uint16
    static constexpr int OFF_MISC = OFF_LIST + 2 * LIST_CAP * 2;   // tmem base (4 B), abort flag (4 B)
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1 KB
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static constexpr uint32_t TMEM_COLS = 512;
    // d = 64 leaves room for P in columns of its own (S_x 128, P_x 64, O_x 64
    // per query tile: 512 in all), so the next S_x need not wait for P_x V;
    // at d = 128 P overwrites the first half of S_x
    static constexpr bool SEP_P = (D == 64);
    static constexpr uint32_t TM_S = 0;                  // S_x at columns 128 x
    static constexpr uint32_t TM_P = SEP_P ? 256 : 0;    // P_x at TM_P + (BC / 2) x (separate), else over S_x
    static constexpr uint32_t TM_O = SEP_P ? 384 : 256;  // O_x at columns TM_O + D x
    static constexpr int THREADS = 384;
    // register split: launched at 168 per thread (384 x 168 = 64,512);
    // warpgroup 0 (producer, MMA, two idle warps) keeps 104, the two softmax
    // warpgroups get 200: 128 x 104 + 256 x 200 = 64,512.
    static constexpr int LAUNCH_REGS = 168;
    static constexpr int REGS_CTRL = 104;
    static constexpr int REGS_SOFTMAX = 200;
    static_assert(128 * REGS_CTRL + 256 * REGS_SOFTMAX == THREADS * LAUNCH_REGS, "register split");
};

// One work item as the producer publishes it to the other roles.
struct FwdItem {
    int item;          // work-item index, or -1: no more work
    int bh, h;
    int q_start, k_start;   // first row of the sequence in Q / K (0 unless ragged)
    int kvis, shift;        // keys < kvis are visible; causal: key j <= query i + shift
    int q0[2], qn[2];       // query tile x: rows [q0, q0 + qn) of the sequence (qn = 0: none)
    int kend[2];            // without a list: key tiles [0, kend[x]) are those query tile x sees
    int count;              // key-tile entries to visit (union of both query tiles)
    int use_list;           // entries come from the item's key-tile list (block mask)
    int nq;                 // query tiles with rows
};
static_assert(sizeof(FwdItem) <= 128, "item slot");

// Bounded wait used only while draining after an abort (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > FA_WAIT_TIMEOUT_NS) break;
}

// Persistent grid: one CTA per SM; each CTA takes work items (a pair of
// 128-row query tiles of one b*h) from a counter in the workspace until none
// is left.  The items are numbered head-major with the causally heaviest
// pair of each head first, and handed out in that order, so the CTAs at work
// at one time share one head's K and V in L2 and the longest items start
// first.  When the items differ in length (causal, key padding, block mask,
// ragged) the host asks for a spread order instead: the heads in groups (of
// 8, or all of them), the heaviest pair of every head in a group, then the
// next, so that the last items handed out are short (head-major would start
// the last head's heaviest pair near the end, where it runs alone) while the
// CTAs at work share the K and V of a few heads only.  The counter resets itself: the last CTA to finish taking items sets
// it back to zero, so the next launch on the same workspace starts from 0.
template <int D, bool VARLEN, int BC, int QPC, int MODE>
__global__ void __launch_bounds__(384, 1) fa_fwd_kernel(const __grid_constant__ FwdParams p) {
    grid_dep_wait();                                 // the previous kernel in the stream is done
    grid_dep_launch();
    // MODE 2 (plain): no causal mask, key padding or block mask, N a multiple
    // of the key tile: every visited tile is full.  MODE 1: no block mask.
    // MODE 0: a block mask may be given (key-tile lists).  Each kernel
    // carries only the code its mode needs.
    constexpr bool PLAIN = MODE == 2, LIST = MODE == 0;
    using S = FwdShape<D, BC>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    constexpr int qpc = QPC;                         // query tiles per item (1 or 2)
    const int Tp = (p.Tq + qpc - 1) / qpc;
    const int n_items = Tp * p.BH;
    const int nb = (p.N + kTile - 1) / kTile;

    auto bar = [&](int i) -> uint32_t { return base + S::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + S::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sb + S::OFF_MISC + 4);
    const Guard g{p.status, p.status + 1, abort_flag};
    FwdItem *slots = reinterpret_cast<FwdItem *>(sb + S::OFF_SLOT);
    auto list_of = [&](int s) { return reinterpret_cast<uint16_t *>(sb + S::OFF_LIST) + s * S::LIST_CAP; };
    unsigned *sched = p.status + 2;                  // workspace words 2 (next item) and 3 (CTAs done)

    if (threadIdx.x == 0) {
        mbar_init(bar(S::B_QFULL), 1);
        mbar_init(bar(S::B_QEMPTY), 1);
        for (int s = 0; s < S::STAGES; ++s) {
            mbar_init(bar(S::B_KFULL + s), 1);
            mbar_init(bar(S::B_VFULL + s), 1);
            mbar_init(bar(S::B_KEMPTY + s), 1);
            mbar_init(bar(S::B_VEMPTY + s), 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(bar(S::B_SFULL + j), 1);
            mbar_init(bar(S::B_PFULL + j), 128);
            mbar_init(bar(S::B_PVDONE + j), 1);
            mbar_init(bar(S::B_SFREE + j), 128);
            mbar_init(bar(S::B_ITEM + j), 32);
            mbar_init(bar(S::B_ITEMFREE + j), 9);
        }
        mbar_init(bar(S::B_FIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&p.tmQ);
        tma_prefetch_desc(&p.tmK);
        tma_prefetch_desc(&p.tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), S::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // entry e of an item: its key tile and whether query tile x sees it
    auto entry_kt = [&](const FwdItem &it, const uint16_t *lst, int e) -> int {
        if constexpr (!LIST) return e;
        return it.use_list ? (int)(lst[e] & 0x3FFFu) : e;
    };
    auto entry_vis = [&](const FwdItem &it, const uint16_t *lst, int x, int e) -> bool {
        if (LIST && it.use_list) return (lst[e] >> (14 + x)) & 1u;
        return e < (x ? it.kend[1] : it.kend[0]);
    };

    // Register split.  Warpgroup 0 gives registers back once, here, and
    // keeps REGS_CTRL to the end; the softmax warpgroups take them, here, and
    // give them back at the end of their branch, so the shared teardown below
    // runs with REGS_CTRL everywhere.  The only setmaxnreg.inc (which blocks
    // until the pool holds enough) is the softmax one at the start, and the
    // pool is filled by warpgroup 0's unconditional dec: no inc ever waits on
    // a warp that is itself waiting.
    if (warp < 4) {
        setmaxnreg_dec<S::REGS_CTRL>();
        if (warp == 0) {
            // ---------------------------------------------------------- producer (whole warp)
            // Takes the items, describes each one in a slot for the other
            // roles (and, under a block mask, lists its key tiles), loads the
            // item's Q tiles once the previous item's S products are done with
            // the Q buffer, and streams K and V through the ring.
            int k = 0, m = 0, u = 0;                 // items published, items with Q loaded, ring uses
            int k_only = -1;                         // a use whose K was loaded but not its V (on giving up)
            bool ok = true;
            for (;; ++k) {
                const int s = k & 1;
                if (k >= 2 && !mbar_wait_warp(bar(S::B_ITEMFREE + s), (uint32_t)((k >> 1) - 1) & 1u, g, 0x100)) {
                    ok = false;
                    break;
                }
                FwdItem it;
                it.item = -1;
                for (;;) {
                    int j = 0;
                    if (lane == 0) j = (int)atomicAdd(sched, 1u);
                    j = __shfl_sync(0xffffffffu, j, 0);
                    if (j >= n_items) break;
                    // item j: head-major, the causally heaviest pair of the head first
                    int pqi = j % Tp, bh = j / Tp;
                    if (p.spread > 0) {
                        // groups of p.spread heads (every head: spread order), items
                        // spread across a group's heads, the groups in order
                        const int per = Tp * p.spread;
                        const int gi = j / per, i = j - gi * per;
                        const int gs = min(p.spread, p.BH - gi * p.spread);
                        pqi = i / gs;
                        bh = gi * p.spread + (i - pqi * gs);
                    }
                    const int pq = Tp - 1 - pqi;
                    const int b = bh / p.H, h = bh % p.H;
                    int q_start = 0, k_start = 0, Lq = p.N, Lk = p.N;
                    bool bad = false;
                    if constexpr (VARLEN)
                        varlen_sequence(p.cu_q, p.cu_k, b, p.total_q, p.total_k, p.Tq * kTile, INT_MAX, &q_start,
                                        &Lq, &k_start, &Lk, &bad);
                    const int kvis = VARLEN ? Lk : key_visible_bound(p.key_len, b, p.N, &bad);
                    if (bad && lane == 0 && pq == 0 && h == 0) record_status(g, kStatusBadKeyLen, 0);
                    it.item = j;
                    it.bh = bh;
                    it.h = h;
                    it.q_start = q_start;
                    it.k_start = k_start;
                    it.kvis = kvis;
                    it.shift = Lk - Lq;
                    it.nq = 0;
                    for (int x = 0; x < 2; ++x) {
                        it.q0[x] = (qpc * pq + x) * kTile;
                        it.qn[x] = x < qpc ? max(0, min(kTile, Lq - it.q0[x])) : 0;
                        it.kend[x] = fwd_key_tile_end(it.q0[x], it.qn[x], kvis, p.causal, it.shift, BC);
                        it.nq += it.qn[x] > 0 ? 1 : 0;
                    }
                    it.use_list = (LIST && !VARLEN && p.block_mask) ? 1 : 0;
                    it.count = max(it.kend[0], it.kend[1]);
                    // an item with no query row (past a ragged sequence's end) is not published
                    if (it.nq > 0) break;
                    it.item = -1;
                }
                uint16_t *lst = list_of(s);
                if (LIST && it.item >= 0 && it.use_list) {
                    // the key tiles either query tile sees, in order, compacted by the whole warp
                    const int Tk = p.Tk;
                    int n = 0;
                    for (int t0 = 0; t0 < Tk; t0 += 32) {
                        const int kt = t0 + lane;
                        bool v[2] = {false, false};
                        if (kt < Tk)
                            for (int x = 0; x < 2; ++x) {
                                if (it.qn[x] <= 0) continue;
                                const int mb = BC == kTile ? kt : kt / (kTile / BC);
                                const int on = p.block_mask[(size_t)(it.q0[x] / kTile) * nb + mb] != 0;
                                v[x] = tile_class(it.q0[x], it.qn[x], kt * BC, BC, it.kvis, p.causal, on) != kTileSkip;
                            }
                        const unsigned ball = __ballot_sync(0xffffffffu, v[0] || v[1]);
                        if (v[0] || v[1])
                            lst[n + __popc(ball & ((1u << lane) - 1u))] =
                                (uint16_t)(kt | (v[0] ? 1u << 14 : 0u) | (v[1] ? 1u << 15 : 0u));
                        n += __popc(ball);
                    }
                    it.count = n;
                }
                if (lane == 0) slots[s] = it;
                mbar_arrive(bar(S::B_ITEM + s));    // every lane, after its own list writes
                if (it.item < 0) break;
                if (it.count == 0) continue;        // every row sees no key: no loads
                // Q tiles, once the previous item's S products no longer read the buffer
                if (m > 0 && !mbar_wait_warp(bar(S::B_QEMPTY), (uint32_t)(m - 1) & 1u, g, 0x101)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_elect(bar(S::B_QFULL), (uint32_t)it.nq * S::TILE_BYTES);
                for (int x = 0; x < 2; ++x)
                    if (it.qn[x] > 0)
                        for (int c = 0; c < S::CHUNKS; ++c) {
                            const uint32_t dst = base + S::OFF_Q + x * S::TILE_BYTES + c * S::CHUNK_BYTES;
                            if constexpr (VARLEN)
                                tma_load_3d_elect(dst, &p.tmQ, bar(S::B_QFULL), c * 64, it.h, it.q_start + it.q0[x]);
                            else
                                tma_load_3d_elect(dst, &p.tmQ, bar(S::B_QFULL), c * 64, it.q0[x], it.bh);
                        }
                ++m;
                for (int e = 0; e < it.count; ++e, ++u) {
                    const int kt = entry_kt(it, lst, e);
                    const int st = u % S::STAGES;
                    const uint32_t ph = (uint32_t)(u / S::STAGES) & 1u;
                    // K of stage st once the S products of its previous key tile
                    // are done, V once that tile's P.V products are
                    if (!mbar_wait_warp(bar(S::B_KEMPTY + st), ph ^ 1u, g, 0x102)) {
                        ok = false;
                        break;
                    }
                    const uint32_t koff = base + S::OFF_K + st * S::KV_TILE_BYTES;
                    const uint32_t voff = base + S::OFF_V + st * S::KV_TILE_BYTES;
                    mbar_arrive_expect_tx_elect(bar(S::B_KFULL + st), S::KV_TILE_BYTES);
                    for (int c = 0; c < S::CHUNKS; ++c) {
                        if constexpr (VARLEN)
                            tma_load_3d_elect(koff + c * S::KV_CHUNK_BYTES, &p.tmK, bar(S::B_KFULL + st), c * 64, it.h,
                                              it.k_start + kt * BC);
                        else
                            tma_load_3d_elect(koff + c * S::KV_CHUNK_BYTES, &p.tmK, bar(S::B_KFULL + st), c * 64,
                                              kt * BC, it.bh);
                    }
                    if (!mbar_wait_warp(bar(S::B_VEMPTY + st), ph ^ 1u, g, 0x103)) {
                        k_only = u;                 // this use's K load is on its way, its V not
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_elect(bar(S::B_VFULL + st), S::KV_TILE_BYTES);
                    for (int c = 0; c < S::CHUNKS; ++c) {
                        if constexpr (VARLEN)
                            tma_load_3d_elect(voff + c * S::KV_CHUNK_BYTES, &p.tmV, bar(S::B_VFULL + st), c * 64, it.h,
                                              it.k_start + kt * BC);
                        else
                            tma_load_3d_elect(voff + c * S::KV_CHUNK_BYTES, &p.tmV, bar(S::B_VFULL + st), c * 64,
                                              kt * BC, it.bh);
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
                if (m > 0) drain_wait(bar(S::B_QFULL), (uint32_t)(m - 1) & 1u);
                for (int i = (u > S::STAGES ? u - S::STAGES : 0); i < u; ++i) {
                    const int st = i % S::STAGES;
                    const uint32_t ph = (uint32_t)(i / S::STAGES) & 1u;
                    drain_wait(bar(S::B_KFULL + st), ph);
                    drain_wait(bar(S::B_VFULL + st), ph);
                }
                if (k_only >= 0)
                    drain_wait(bar(S::B_KFULL + k_only % S::STAGES), (uint32_t)(k_only / S::STAGES) & 1u);
            }
        } else if (warp == 1) {
            // ---------------------------------------------------------- MMA issuer (whole warp)
            constexpr uint32_t IDESC_S = idesc_bf16(128, BC, false, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
            // shared-memory descriptors built once; per MMA only the start
            // address moves (K-major: 32 bytes per 16-wide K step inside a
            // 128-byte row, then the next 64-column chunk; MN-major V: 16 rows)
            const uint64_t dq0 = sdesc_sw128(base + S::OFF_Q, 16, 1024);
            const uint64_t dk0 = sdesc_sw128(base + S::OFF_K, 16, 1024);
            const uint64_t dv0 = sdesc_sw128(base + S::OFF_V, S::KV_CHUNK_BYTES, 1024);
            // S_x = Q_x K^T for the key tile in stage st (the x-th S buffer)
            auto issue_s = [&](int x, int st) {
                const uint32_t d_tmem = tmem + S::TM_S + 128u * (uint32_t)x;
                const uint64_t qd = sdesc_add(dq0, (uint32_t)(x * S::TILE_BYTES));
                const uint64_t kd = sdesc_add(dk0, (uint32_t)(st * S::KV_TILE_BYTES));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * S::CHUNK_BYTES + (kk & 3) * 32;
                    const uint32_t koff = (kk >> 2) * S::KV_CHUNK_BYTES + (kk & 3) * 32;
                    mma_ss_elect(d_tmem, sdesc_add(qd, off), sdesc_add(kd, koff), IDESC_S, kk > 0 ? 1u : 0u);
                }
                mma_commit_elect(bar(S::B_SFULL + x));
            };
            bool ok = true;
            int k = 0, m = 0, u = 0;
            int nv[2] = {0, 0};      // P.V products issued so far for query tile x (all items)
            int ns[2] = {0, 0};      // S products issued so far for query tile x (all items)
            auto p_tmem_of = [&](int x) -> uint32_t {
                return S::SEP_P ? tmem + S::TM_P + (uint32_t)(BC / 2 * x) : tmem + S::TM_S + 128u * (uint32_t)x;
            };
            // S_x into its columns: with P aliasing S, once the previous P_x V
            // has read P_x; with P apart, once softmax x has loaded S_x
            auto s_ready = [&](int x, unsigned site) -> bool {
                if (ns[x] == 0) return true;
                if constexpr (S::SEP_P)
                    return mbar_wait_warp(bar(S::B_SFREE + x), (uint32_t)(ns[x] - 1) & 1u, g, site);
                return nv[x] == 0 || mbar_wait_warp(bar(S::B_PVDONE + x), (uint32_t)(nv[x] - 1) & 1u, g, site);
            };
            for (;; ++k) {
                const int s = k & 1;
                if (!mbar_wait_warp(bar(S::B_ITEM + s), (uint32_t)(k >> 1) & 1u, g, 0x200)) {
                    ok = false;
                    break;
                }
                const FwdItem it = slots[s];
                const uint16_t *lst = list_of(s);
                if (it.item < 0) break;
                if (it.count > 0) {
                    int nvi[2] = {0, 0};     // this item's P.V products for query tile x
                    // first entry: S_x for each query tile that sees it, once the
                    // previous item's last P_x has been read (P_x aliases S_x)
                    ok = mbar_wait_warp(bar(S::B_QFULL), (uint32_t)m & 1u, g, 0x201) &&
                         mbar_wait_warp(bar(S::B_KFULL + u % S::STAGES), (uint32_t)(u / S::STAGES) & 1u, g, 0x202);
                    ++m;
                    if (ok) {
                        tc_fence_after();
#pragma unroll
                        for (int x = 0; x < 2 && ok; ++x)
                            if (entry_vis(it, lst, x, 0)) {
                                if (!s_ready(x, 0x207)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                issue_s(x, u % S::STAGES);
                                ++ns[x];
                            }
                        // the first key tile's S products are issued: its K is free once they finish
                        if (ok) mma_commit_elect(bar(S::B_KEMPTY + u % S::STAGES));
                        // the item's S products are all issued: Q is free once they finish
                        if (ok && it.count == 1) mma_commit_elect(bar(S::B_QEMPTY));
                    }
                    for (int e = 0; ok && e < it.count; ++e, ++u) {
                        const int st = u % S::STAGES;
                        const int st2 = (u + 1) % S::STAGES;
                        const bool more = e + 1 < it.count;
                        bool vwaited = false, kwaited = false;
                        if constexpr (S::SEP_P) {
                            // both query tiles' next S first (each needs only its
                            // softmax to have loaded the current S), then this
                            // entry's P V products as the P tiles arrive
#pragma unroll
                            for (int x = 0; x < 2 && ok && more; ++x)
                                if (entry_vis(it, lst, x, e + 1)) {
                                    if ((!kwaited && !mbar_wait_warp(bar(S::B_KFULL + st2),
                                                                     (uint32_t)((u + 1) / S::STAGES) & 1u, g, 0x208)) ||
                                        !s_ready(x, 0x209)) {
                                        ok = false;
                                        break;
                                    }
                                    kwaited = true;
                                    tc_fence_after();
                                    issue_s(x, st2);
                                    ++ns[x];
                                }
                            if (!ok) break;
                            if (more) mma_commit_elect(bar(S::B_KEMPTY + st2));
                            if (e + 2 == it.count) mma_commit_elect(bar(S::B_QEMPTY));
#pragma unroll
                            for (int x = 0; x < 2 && ok; ++x)
                                if (entry_vis(it, lst, x, e)) {
                                    if (!mbar_wait_warp(bar(S::B_PFULL + x), (uint32_t)nv[x] & 1u, g, 0x20a) ||
                                        (!vwaited && !mbar_wait_warp(bar(S::B_VFULL + st), (uint32_t)(u / S::STAGES) & 1u,
                                                                     g, 0x20b))) {
                                        ok = false;
                                        break;
                                    }
                                    vwaited = true;
                                    tc_fence_after();
                                    const uint32_t o_tmem = tmem + S::TM_O + (uint32_t)(D * x);
                                    const uint64_t vd = sdesc_add(dv0, (uint32_t)(st * S::KV_TILE_BYTES));
                                    const uint32_t acc0 = nvi[x] > 0 ? 1u : 0u;
#pragma unroll
                                    for (int kk = 0; kk < BC / 16; ++kk)
                                        mma_ts_elect(o_tmem, p_tmem_of(x) + (uint32_t)kk * 8u,
                                                     sdesc_add(vd, (uint32_t)kk * 2048u), IDESC_PV, kk > 0 ? 1u : acc0);
                                    mma_commit_elect(bar(S::B_PVDONE + x));
                                    ++nv[x];
                                    ++nvi[x];
                                }
                            if (!ok) break;
                            mma_commit_elect(bar(S::B_VEMPTY + st));
                            continue;
                        }
                        // per query tile: O_x += P_x V, then at once the next key
                        // tile's S_x (it overwrites P_x, so it waits for that P.V),
                        // so that each tile's chain S -> softmax -> P.V -> S moves
                        // on without waiting for the other tile's P
#pragma unroll
                        for (int x = 0; x < 2 && ok; ++x) {
                            if (entry_vis(it, lst, x, e)) {
                                if (!mbar_wait_warp(bar(S::B_PFULL + x), (uint32_t)nv[x] & 1u, g, 0x203) ||
                                    (!vwaited &&
                                     !mbar_wait_warp(bar(S::B_VFULL + st), (uint32_t)(u / S::STAGES) & 1u, g, 0x204))) {
                                    ok = false;
                                    break;
                                }
                                vwaited = true;
                                tc_fence_after();
                                const uint32_t p_tmem = tmem + S::TM_S + 128u * (uint32_t)x;
                                const uint32_t o_tmem = tmem + S::TM_O + (uint32_t)(D * x);
                                const uint64_t vd = sdesc_add(dv0, (uint32_t)(st * S::KV_TILE_BYTES));
                                const uint32_t acc0 = nvi[x] > 0 ? 1u : 0u;
#pragma unroll
                                for (int kk = 0; kk < BC / 16; ++kk)
                                    mma_ts_elect(o_tmem, p_tmem + (uint32_t)kk * 8u, sdesc_add(vd, (uint32_t)kk * 2048u),
                                                 IDESC_PV, kk > 0 ? 1u : acc0);
                                mma_commit_elect(bar(S::B_PVDONE + x));
                                ++nv[x];
                                ++nvi[x];
                            }
                            // V of stage st is free once both P.V products (its last readers)
                            // are done: released before the second query tile's next S
                            if (x == 1) mma_commit_elect(bar(S::B_VEMPTY + st));
                            if (more && entry_vis(it, lst, x, e + 1)) {
                                if (!kwaited && !mbar_wait_warp(bar(S::B_KFULL + st2), (uint32_t)((u + 1) / S::STAGES) & 1u,
                                                                g, 0x205)) {
                                    ok = false;
                                    break;
                                }
                                kwaited = true;
                                if (!s_ready(x, 0x206)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                issue_s(x, st2);
                                ++ns[x];
                            }
                        }
                        if (!ok) break;
                        // the next key tile's S products are issued: its K is free once they finish
                        if (more) mma_commit_elect(bar(S::B_KEMPTY + st2));
                        // the item's last S products were issued just now: Q is free once they finish
                        if (e + 2 == it.count) mma_commit_elect(bar(S::B_QEMPTY));
                    }
                }
                if (!ok) break;
                // every field of the slot has been read
                if (lane == 0) mbar_arrive(bar(S::B_ITEMFREE + s));
            }
            // every MMA this thread issued must finish before TMEM is freed
            mma_commit_elect(bar(S::B_FIN));
            drain_wait(bar(S::B_FIN), 0);
        }
    } else {
        setmaxnreg_inc<S::REGS_SOFTMAX>();
        // ---------------------------------------------------------- softmax of query tile x
        const int x = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t s_tmem = tmem + lane_off + S::TM_S + 128u * (uint32_t)x;
        const uint32_t p_tmem = S::SEP_P ? tmem + lane_off + S::TM_P + (uint32_t)(BC / 2 * x) : s_tmem;
        const uint32_t o_tmem = tmem + lane_off + S::TM_O + (uint32_t)(D * x);
        const float c2 = p.scale_log2;
        bool ok = true;
        int ns = 0;                                  // S tiles of query tile x so far (all items)
        for (int k = 0;; ++k) {
            const int s = k & 1;
            if (!mbar_wait_warp(bar(S::B_ITEM + s), (uint32_t)(k >> 1) & 1u, g, 0x400)) {
                ok = false;
                break;
            }
            const FwdItem &itr = slots[s];
            const int item = itr.item;
            if (item < 0) break;
            const uint16_t *lst = list_of(s);
            const int q0x = x ? itr.q0[1] : itr.q0[0], qnx = x ? itr.qn[1] : itr.qn[0];
            const int kvis = itr.kvis, shift = itr.shift, count = itr.count, bh = itr.bh, h = itr.h;
            const int q_start = itr.q_start;
            const int use_list = itr.use_list, kendx = x ? itr.kend[1] : itr.kend[0];
            const int q = q0x + r;
            float m_ref = -INFINITY, l = 0.f;
            int it = 0;                              // this item's tiles
            for (int e = 0; e < count; ++e) {
                const bool vis = (LIST && use_list) ? ((lst[e] >> (14 + x)) & 1u) : (e < kendx);
                if (!vis) continue;
                const int kt = (LIST && use_list) ? (int)(lst[e] & 0x3FFFu) : e;
                const int k0 = kt * BC;
                unsigned klass = kTileFull;
                if constexpr (VARLEN)
                    klass = tile_class_shift(q0x, qnx, k0, BC, kvis, p.causal, shift);
                else if constexpr (!PLAIN)
                    klass = tile_class(q0x, qnx, k0, BC, kvis, p.causal, 1);
                const bool partial = !PLAIN && klass == kTilePartial;
                if (!mbar_wait_warp(bar(S::B_SFULL + x), (uint32_t)ns & 1u, g, 0x401)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[S::KC][32];
#pragma unroll
                for (int j = 0; j < S::KC; ++j) tmem_ld32(s_tmem + 32u * j, sr[j]);
#pragma unroll
                for (int j = 0; j < S::KC; ++j) tmem_ld_wait(sr[j]);
                if constexpr (S::SEP_P) {
                    // S_x is in registers: the next S_x may overwrite its columns
                    tc_fence_before();
                    mbar_arrive(bar(S::B_SFREE + x));
                }
                if (partial) {
                    // this row sees keys k0 .. k0 + lim - 1 of the tile: one compare
                    // against a constant per score
                    int lim = kvis - k0;
                    if (p.causal) lim = min(lim, q + shift + 1 - k0);
#pragma unroll
                    for (int j = 0; j < S::KC; ++j)
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (32 * j + t >= lim) sr[j][t] = __float_as_uint(-INFINITY);
                }
                // row maximum as eight independent 3-input chains, then a tree:
                // one warp per sub-partition runs this, so the latency of a single
                // 64-deep chain would sit on the critical path
                float pm[8];
#pragma unroll
                for (int uu = 0; uu < 8; ++uu) pm[uu] = -INFINITY;
#pragma unroll
                for (int j = 0; j < S::KC; ++j)
#pragma unroll
                    for (int t = 0; t < 32; t += 4) {
                        const int uu = (j * 8 + t / 4) & 7;
                        pm[uu] = fmax3(pm[uu], __uint_as_float(sr[j][t]), __uint_as_float(sr[j][t + 1]));
                        pm[uu] = fmax3(pm[uu], __uint_as_float(sr[j][t + 2]), __uint_as_float(sr[j][t + 3]));
                    }
                const float mx = fmaxf(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], fmax3(pm[5], pm[6], pm[7])));
                // move the reference maximum only when the row outgrew it by 2^8
                const float m_tile = mx * c2;
                const bool grow = m_tile > m_ref + kRescaleLog2;
                float alpha = 1.f;
                const bool rescale = __any_sync(0xffffffffu, grow);
                if (rescale) {
                    const float m_new = fmaxf(m_ref, m_tile);
                    alpha = (m_new == -INFINITY) ? 1.f : ex2(m_ref - m_new);
                    l *= alpha;
                    m_ref = m_new;
                }
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                // p = 2^(s * c - m), bf16; the row sum in four independent
                // packed accumulators.  With P apart from S, P_x is written only
                // once the previous P_x V has read it (the first tile of an item
                // included: the buffer serves every item); with P over S, S_x's
                // columns are already this tile's.
                float ps[8];
#pragma unroll
                for (int uu = 0; uu < 8; ++uu) ps[uu] = 0.f;
                uint32_t pk[S::KC][16];
#pragma unroll
                for (int j = 0; j < S::KC; ++j) {
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        float a, bb;
                        fma2(a, bb, __uint_as_float(sr[j][2 * t]), __uint_as_float(sr[j][2 * t + 1]), c2, c2, -m_use,
                             -m_use);
                        a = ex2(a);
                        bb = ex2(bb);
                        const int uu = 2 * (t & 3);
                        add2(ps[uu], ps[uu + 1], a, bb);
                        pk[j][t] = pack_bf16x2(a, bb);
                    }
                    if constexpr (!S::SEP_P) tmem_st16(p_tmem + 16u * j, pk[j]);
                }
                bool pv_waited = false;
                if constexpr (S::SEP_P) {
                    if (ns > 0 && !mbar_wait_warp(bar(S::B_PVDONE + x), (uint32_t)(ns - 1) & 1u, g, 0x404)) {
                        ok = false;
                        break;
                    }
                    pv_waited = true;
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < S::KC; ++j) tmem_st16(p_tmem + 16u * j, pk[j]);
                }
                l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
                tmem_st_wait();
                if (rescale && it > 0) {
                    // O_x may be rescaled only once the previous P_x V has landed
                    if (!pv_waited && !mbar_wait_warp(bar(S::B_PVDONE + x), (uint32_t)(ns - 1) & 1u, g, 0x402)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // O_x is D columns: D / 32 chunks of 32, loaded up to four at a time
                    constexpr int RC = (D / 32 < 4) ? D / 32 : 4;
#pragma unroll
                    for (int j0 = 0; j0 < D / 32; j0 += RC) {
                        uint32_t o[RC][32];
#pragma unroll
                        for (int j = 0; j < RC; ++j) tmem_ld32(o_tmem + 32u * (j0 + j), o[j]);
#pragma unroll
                        for (int j = 0; j < RC; ++j) tmem_ld_wait(o[j]);
#pragma unroll
                        for (int j = 0; j < RC; ++j) {
#pragma unroll
                            for (int t = 0; t < 32; t += 2) {
                                float a, bb;
                                fma2(a, bb, __uint_as_float(o[j][t]), __uint_as_float(o[j][t + 1]), alpha, alpha, 0.f,
                                     0.f);
                                o[j][t] = __float_as_uint(a);
                                o[j][t + 1] = __float_as_uint(bb);
                            }
                            tmem_st32(o_tmem + 32u * (j0 + j), o[j]);
                        }
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(bar(S::B_PFULL + x));
                ++ns;
                ++it;
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue of the item
            // (the next item's first P.V into O_x is issued only after this
            // warpgroup's next P arrival, which follows these loads)
            if (it > 0) {
                if (!mbar_wait_warp(bar(S::B_PVDONE + x), (uint32_t)(ns - 1) & 1u, g, 0x403)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (qnx > 0) {
                const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
                const size_t orow_idx = VARLEN ? (size_t)(q_start + q) * p.H + h : (size_t)bh * p.N + q;
                __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.O) + orow_idx * D;
#pragma unroll 1
                for (int j = 0; j < D / 32; ++j) {
                    uint32_t o[32];
                    if (it > 0) {
                        tmem_ld32(o_tmem + 32u * j, o);
                        tmem_ld_wait(o);
                    } else {
#pragma unroll
                        for (int t = 0; t < 32; ++t) o[t] = 0u;
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        w[t] = pack_bf16x2(__uint_as_float(o[2 * t]) * inv_l, __uint_as_float(o[2 * t + 1]) * inv_l);
                    if (r < qnx) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * j);
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            dst[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
                    }
                }
                if (r < qnx)
                    p.LSE[VARLEN ? (size_t)h * p.total_q + q_start + q : (size_t)bh * p.N + q] =
                        (l > 0.f) ? (m_ref + log2f(l)) * 0.69314718055994530942f : -INFINITY;
            }
            tc_fence_before();
            __syncwarp();
            // every field of the slot has been read
            if (lane == 0) mbar_arrive(bar(S::B_ITEMFREE + s));
        }
        __syncwarp();
        setmaxnreg_dec<S::REGS_CTRL>();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, S::TMEM_COLS);
}

int device_sm_count() {
    constexpr int kMaxDev = 64;
    static int cached[kMaxDev] = {};
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < kMaxDev && cached[dev] > 0) return cached[dev];
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    if (dev >= 0 && dev < kMaxDev) cached[dev] = n;
    return n;
}

int fwd_smem_bytes(int d) { return d == 64 ? FwdShape<64>::SMEM_BYTES : FwdShape<128>::SMEM_BYTES; }

template <int D, bool VARLEN, int BC, int QPC, int MODE = 0>
static cudaError_t launch_fwd_t(const FwdParams &p, cudaStream_t st) {
    using S = FwdShape<D, BC>;
    const int smem = S::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D, VARLEN, BC, QPC, MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM (the shared-memory footprint allows one),
    // never more CTAs than work items
    const int64_t items = (int64_t)((p.Tq + QPC - 1) / QPC) * p.BH;
    const unsigned grid = (unsigned)std::min<int64_t>(items, device_sm_count());
    return launch_dep(fa_fwd_kernel<D, VARLEN, BC, QPC, MODE>, grid, S::THREADS, smem, st, p);
}

cudaError_t launch_fwd(int d, const FwdParams &p, cudaStream_t st) {
    const int mode = p.block_mask ? 0 : (!p.causal && !p.key_len && p.N % 128 == 0) ? 2 : 1;
    if (d == 64)
        return mode == 2 ? launch_fwd_t<64, false, 128, 2, 2>(p, st)
             : mode == 1 ? launch_fwd_t<64, false, 128, 2, 1>(p, st) : launch_fwd_t<64, false, 128, 2, 0>(p, st);
    return mode == 2 ? launch_fwd_t<128, false, 128, 2, 2>(p, st)
         : mode == 1 ? launch_fwd_t<128, false, 128, 2, 1>(p, st) : launch_fwd_t<128, false, 128, 2, 0>(p, st);
}

cudaError_t launch_fwd_varlen(int d, const FwdParams &p, cudaStream_t st) {
    return d == 64 ? launch_fwd_t<64, true, 128, 2, 1>(p, st) : launch_fwd_t<128, true, 128, 2, 1>(p, st);
}

template <int D>
static cudaError_t launch_fwd_tiles_d(int block_k, const FwdParams &p, cudaStream_t st) {
    if (p.qpc == 1)
        return block_k == 64 ? launch_fwd_t<D, false, 64, 1>(p, st) : launch_fwd_t<D, false, 128, 1>(p, st);
    return block_k == 64 ? launch_fwd_t<D, false, 64, 2>(p, st) : launch_fwd_t<D, false, 128, 2>(p, st);
}

cudaError_t launch_fwd_tiles(int d, int block_k, const FwdParams &p, cudaStream_t st) {
    return d == 64 ? launch_fwd_tiles_d<64>(block_k, p, st) : launch_fwd_tiles_d<128>(block_k, p, st);
}

}  // namespace fa
