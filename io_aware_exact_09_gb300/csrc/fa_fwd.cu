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
//   - one CTA per (pair of 128-row query tiles, b*h), head-major, causally
//     heaviest pairs first within a head;
//   - warp 0: TMA producer: both Q tiles once; K and V tiles through a ring
//     of shared-memory stages (128-byte swizzle, 64-column boxes), over the
//     union of the key tiles the two query tiles see;
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
    static constexpr int B_KFULL = 1;
    static constexpr int B_VFULL = B_KFULL + STAGES;
    static constexpr int B_KVEMPTY = B_VFULL + STAGES;
    static constexpr int B_SFULL = B_KVEMPTY + STAGES;   // [2] one per query tile
    static constexpr int B_PFULL = B_SFULL + 2;          // [2]
    static constexpr int B_PVDONE = B_PFULL + 2;         // [2]
    static constexpr int B_FIN = B_PVDONE + 2;
    static constexpr int NBAR = B_FIN + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem base (4 B), abort flag (4 B)
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1 KB
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_S = 0;                  // S_x at columns 128 x
    static constexpr uint32_t TM_O = 256;                // O_x at columns 256 + D x
    static constexpr int THREADS = 384;
    // register split: launched at 168 per thread (384 x 168 = 64,512);
    // warpgroup 0 (producer, MMA, two idle warps) keeps 88, the two softmax
    // warpgroups get 208: 128 x 88 + 256 x 208 = 64,512.
    static constexpr int LAUNCH_REGS = 168;
    static constexpr int REGS_CTRL = 104;
    static constexpr int REGS_SOFTMAX = 200;
    static_assert(128 * REGS_CTRL + 256 * REGS_SOFTMAX == THREADS * LAUNCH_REGS, "register split");
};

// Bounded wait used only while draining after an abort (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > FA_WAIT_TIMEOUT_NS) break;
}

template <int D, bool VARLEN, int BC, int QPC>
__global__ void __launch_bounds__(384, 1) fa_fwd_kernel(const __grid_constant__ FwdParams p) {
    using S = FwdShape<D, BC>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Work item, head-major: the CTAs resident at one time share one head's K
    // and V in L2; within a head the causally heaviest pairs start first.
    constexpr int qpc = QPC;                         // query tiles per CTA (1 or 2)
    const int Tp = (p.Tq + qpc - 1) / qpc;
    const int pq = Tp - 1 - (int)(blockIdx.x % Tp);
    const int bh = (int)(blockIdx.x / Tp);
    const int b = bh / p.H, h = bh % p.H;
    const int nb = (p.N + kTile - 1) / kTile;
    // the sequence this CTA works on: rows [q_start, q_start + Lq) of Q and
    // [k_start, k_start + Lk) of K, V.  Its queries are its last Lq
    // positions: under the causal mask query i sees key j iff j <= i + shift
    // (shift = Lk - Lq; 0 for the square [B, H, N, d] case).
    int q_start = 0, k_start = 0, Lq = p.N, Lk = p.N, Tk = p.Tk;
    bool bad_len = false;
    if constexpr (VARLEN) {
        q_start = p.cu_q[b];
        Lq = p.cu_q[b + 1] - q_start;
        k_start = p.cu_k[b];
        Lk = p.cu_k[b + 1] - k_start;
        if (q_start < 0 || Lq < 0 || q_start + Lq > p.total_q || k_start < 0 || Lk < 0 ||
            k_start + Lk > p.total_k || Lq > p.Tq * kTile) {
            bad_len = true;
            Lq = Lk = 0;
        }
        Tk = (Lk + BC - 1) / BC;
    }
    const int shift = Lk - Lq;
    int q0[2], qn[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        q0[x] = (qpc * pq + x) * kTile;
        qn[x] = x < qpc ? max(0, min(kTile, Lq - q0[x])) : 0;
    }
    // TMA coordinates of row `row` of a sequence starting at `start`:
    // [B*H][N][d] view, or the [total][H][d] view of a ragged batch
    // warp-collective (the producer warp calls it with uniform arguments)
    auto tload = [&](uint32_t dst, const CUtensorMap *m, uint32_t mbar, int c, int row, int start) {
        if constexpr (VARLEN)
            tma_load_3d_elect(dst, m, mbar, c * 64, h, start + row);
        else
            tma_load_3d_elect(dst, m, mbar, c * 64, row, bh);
    };

    auto bar = [&](int i) -> uint32_t { return base + S::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + S::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sb + S::OFF_MISC + 4);
    const Guard g{p.status, p.status + 1, abort_flag};

    bool bad = bad_len;
    const int kvis = VARLEN ? Lk : key_visible_bound(p.key_len, b, p.N, &bad);
    if (bad && threadIdx.x == 0 && pq == 0 && (bh % p.H) == 0) record_status(g, kStatusBadKeyLen, 0);
    // In a ragged batch the grid covers the longest sequence: a CTA whose
    // query tiles both lie past its own sequence's end has no row to write and
    // leaves before any set-up (the whole CTA takes this branch together)
    if (qn[0] <= 0 && qn[1] <= 0) return;

    // Without a block mask the key tiles query tile x sees are exactly
    // [0, kend[x]): keys below key_len and, under the causal mask, not past
    // its last row.  (tile_class below takes the same decision per tile.)
    int kend[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) kend[x] = fwd_key_tile_end(q0[x], qn[x], kvis, p.causal, shift, BC);
    const int kend_union = max(kend[0], kend[1]);
    // per-query-tile values by selection, so that the arrays stay in registers
    auto q0_of = [&](int x) { return x ? q0[1] : q0[0]; };
    auto qn_of = [&](int x) { return x ? qn[1] : qn[0]; };
    auto kend_of = [&](int x) { return x ? kend[1] : kend[0]; };
    // class of key tile kt for query tile x of the pair
    auto cls = [&](int x, int kt) -> unsigned {
        if (qn_of(x) <= 0) return kTileSkip;
        if constexpr (VARLEN) return tile_class_shift(q0_of(x), qn_of(x), kt * BC, BC, kvis, p.causal, shift);
        // a key tile of BC <= 128 columns lies inside one 128-wide mask block
        const int on =
            p.block_mask ? (p.block_mask[(size_t)(QPC * pq + x) * nb + (BC == kTile ? kt : kt / (kTile / BC))] != 0) : 1;
        return tile_class(q0_of(x), qn_of(x), kt * BC, BC, kvis, p.causal, on);
    };
    // next key tile after kt seen by query tile x (x = 2: by either)
    auto next_tile = [&](int x, int kt) -> int {
        if (!p.block_mask) {
            const int lim = x == 2 ? kend_union : kend_of(x);
            return kt + 1 < lim ? kt + 1 : Tk;
        }
        for (int k = kt + 1; k < Tk; ++k) {
            const bool v0 = (x != 1) && cls(0, k) != kTileSkip;
            const bool v1 = (x != 0) && cls(1, k) != kTileSkip;
            if (v0 || v1) return k;
        }
        return Tk;
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(S::B_QFULL), 1);
        for (int s = 0; s < S::STAGES; ++s) {
            mbar_init(bar(S::B_KFULL + s), 1);
            mbar_init(bar(S::B_VFULL + s), 1);
            mbar_init(bar(S::B_KVEMPTY + s), 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(bar(S::B_SFULL + j), 1);
            mbar_init(bar(S::B_PFULL + j), 128);
            mbar_init(bar(S::B_PVDONE + j), 1);
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

    // Register split.  Warpgroup 0 gives registers back once, here, and
    // keeps 88 to the end; the softmax warpgroups take them, here, and give
    // them back at the end of their branch, so the shared teardown below runs
    // with 88 everywhere.  The only setmaxnreg.inc (which blocks until the
    // pool holds enough) is the softmax one at the start, and the pool is
    // filled by warpgroup 0's unconditional dec: no inc ever waits on a warp
    // that is itself waiting.
    if (warp < 4) {
        setmaxnreg_dec<S::REGS_CTRL>();
        if (warp == 0) {
            // ---------------------------------------------------------- producer
            {
                int u = 0;
                bool ok = true;
                int kt = next_tile(2, -1);
                if (kt < Tk) {
                    const uint32_t nq = (qn[0] > 0 ? 1u : 0u) + (qn[1] > 0 ? 1u : 0u);
                    mbar_arrive_expect_tx_elect(bar(S::B_QFULL), nq * S::TILE_BYTES);
                    #pragma unroll
                    for (int x = 0; x < 2; ++x)
                        if (qn[x] > 0)
                            for (int c = 0; c < S::CHUNKS; ++c)
                                tload(base + S::OFF_Q + x * S::TILE_BYTES + c * S::CHUNK_BYTES, &p.tmQ,
                                      bar(S::B_QFULL), c, q0[x], q_start);
                }
                for (; kt < Tk; kt = next_tile(2, kt), ++u) {
                    const int s = u % S::STAGES;
                    const uint32_t ph = (uint32_t)(u / S::STAGES) & 1u;
                    if (!mbar_wait_warp(bar(S::B_KVEMPTY + s), ph ^ 1u, g, 0x101)) {
                        ok = false;
                        break;
                    }
                    const uint32_t koff = base + S::OFF_K + s * S::KV_TILE_BYTES;
                    const uint32_t voff = base + S::OFF_V + s * S::KV_TILE_BYTES;
                    mbar_arrive_expect_tx_elect(bar(S::B_KFULL + s), S::KV_TILE_BYTES);
                    for (int c = 0; c < S::CHUNKS; ++c)
                        tload(koff + c * S::KV_CHUNK_BYTES, &p.tmK, bar(S::B_KFULL + s), c, kt * BC, k_start);
                    mbar_arrive_expect_tx_elect(bar(S::B_VFULL + s), S::KV_TILE_BYTES);
                    for (int c = 0; c < S::CHUNKS; ++c)
                        tload(voff + c * S::KV_CHUNK_BYTES, &p.tmV, bar(S::B_VFULL + s), c, kt * BC, k_start);
                }
                if (!ok) {
                    // gave up: let every copy already issued land before the CTA exits
                    if (next_tile(2, -1) < Tk) drain_wait(bar(S::B_QFULL), 0);
                    for (int i = (u > S::STAGES ? u - S::STAGES : 0); i < u; ++i) {
                        const int s = i % S::STAGES;
                        const uint32_t ph = (uint32_t)(i / S::STAGES) & 1u;
                        drain_wait(bar(S::B_KFULL + s), ph);
                        drain_wait(bar(S::B_VFULL + s), ph);
                    }
                }
            }
        } else if (warp == 1) {
            // ---------------------------------------------------------- MMA issuer
            {
                constexpr uint32_t IDESC_S = idesc_bf16(128, BC, false, false);
                constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
                int kt = next_tile(2, -1);
                bool ok = true;
                int nv[2] = {0, 0};      // key tiles processed so far by query tile x
                // shared-memory descriptors built once; per MMA only the start
                // address moves (K-major: 32 bytes per 16-wide K step inside a
                // 128-byte row, then the next 64-column chunk; MN-major V: 16 rows)
                const uint64_t dq0 = sdesc_sw128(base + S::OFF_Q, 16, 1024);
                const uint64_t dk0 = sdesc_sw128(base + S::OFF_K, 16, 1024);
                const uint64_t dv0 = sdesc_sw128(base + S::OFF_V, S::KV_CHUNK_BYTES, 1024);
                // S_x = Q_x K^T for the key tile in stage s (the x-th S buffer)
                auto issue_s = [&](int x, int s) {
                    const uint32_t d_tmem = tmem + S::TM_S + 128u * (uint32_t)x;
                    const uint64_t qd = sdesc_add(dq0, (uint32_t)(x * S::TILE_BYTES));
                    const uint64_t kd = sdesc_add(dk0, (uint32_t)(s * S::KV_TILE_BYTES));
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = (k >> 2) * S::CHUNK_BYTES + (k & 3) * 32;
                        const uint32_t koff = (k >> 2) * S::KV_CHUNK_BYTES + (k & 3) * 32;
                        mma_ss_elect(d_tmem, sdesc_add(qd, off), sdesc_add(kd, koff), IDESC_S, k > 0 ? 1u : 0u);
                    }
                    mma_commit_elect(bar(S::B_SFULL + x));
                };
                if (kt < Tk) {
                    ok = mbar_wait_warp(bar(S::B_QFULL), 0, g, 0x201) && mbar_wait_warp(bar(S::B_KFULL + 0), 0, g, 0x202);
                    if (ok) {
                        tc_fence_after();
                        #pragma unroll
                        for (int x = 0; x < 2; ++x)
                            if (cls(x, kt) != kTileSkip) issue_s(x, 0);
                    }
                    int u = 0;
                    while (ok && kt < Tk) {
                        const int s = u % S::STAGES;
                        const int kt_next = next_tile(2, kt);
                        const int s2 = (u + 1) % S::STAGES;
                        bool vwaited = false, kwaited = false;
                        // per query tile: O_x += P_x V, then at once the next key
                        // tile's S_x (it overwrites P_x, so it waits for that P.V),
                        // so that each tile's chain S -> softmax -> P.V -> S moves
                        // on without waiting for the other tile's P
                        #pragma unroll
                        for (int x = 0; x < 2 && ok; ++x) {
                            if (cls(x, kt) != kTileSkip) {
                                if (!mbar_wait_warp(bar(S::B_PFULL + x), (uint32_t)nv[x] & 1u, g, 0x203) ||
                                    (!vwaited &&
                                     !mbar_wait_warp(bar(S::B_VFULL + s), (uint32_t)(u / S::STAGES) & 1u, g, 0x204))) {
                                    ok = false;
                                    break;
                                }
                                vwaited = true;
                                tc_fence_after();
                                const uint32_t p_tmem = tmem + S::TM_S + 128u * (uint32_t)x;
                                const uint32_t o_tmem = tmem + S::TM_O + (uint32_t)(D * x);
                                const uint64_t vd = sdesc_add(dv0, (uint32_t)(s * S::KV_TILE_BYTES));
                                const uint32_t acc0 = nv[x] > 0 ? 1u : 0u;
#pragma unroll
                                for (int k = 0; k < BC / 16; ++k)
                                    mma_ts_elect(o_tmem, p_tmem + (uint32_t)k * 8u, sdesc_add(vd, (uint32_t)k * 2048u),
                                           IDESC_PV, k > 0 ? 1u : acc0);
                                mma_commit_elect(bar(S::B_PVDONE + x));
                                ++nv[x];
                            }
                            if (kt_next < Tk && cls(x, kt_next) != kTileSkip) {
                                if (!kwaited && !mbar_wait_warp(bar(S::B_KFULL + s2), (uint32_t)((u + 1) / S::STAGES) & 1u,
                                                           g, 0x205)) {
                                    ok = false;
                                    break;
                                }
                                kwaited = true;
                                if (nv[x] > 0 && !mbar_wait_warp(bar(S::B_PVDONE + x), (uint32_t)(nv[x] - 1) & 1u, g, 0x206)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                issue_s(x, s2);
                            }
                        }
                        if (!ok) break;
                        // K and V of stage s are free once this tile's products are done
                        mma_commit_elect(bar(S::B_KVEMPTY + s));
                        kt = kt_next;
                        ++u;
                    }
                }
                // every MMA this thread issued must finish before TMEM is freed
                mma_commit_elect(bar(S::B_FIN));
                drain_wait(bar(S::B_FIN), 0);
            }
        }
    } else {
        setmaxnreg_inc<S::REGS_SOFTMAX>();
        // ---------------------------------------------------------- softmax of query tile x
        const int x = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const int q0x = q0_of(x), qnx = qn_of(x);
        const int q = q0x + r;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t s_tmem = tmem + lane_off + S::TM_S + 128u * (uint32_t)x;
        const uint32_t o_tmem = tmem + lane_off + S::TM_O + (uint32_t)(D * x);
        const float c2 = p.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        int it = 0;
        bool ok = true;
        for (int kt = next_tile(x, -1); kt < Tk; kt = next_tile(x, kt), ++it) {
            const bool partial = cls(x, kt) == kTilePartial;
            const int k0 = kt * BC;
            if (!mbar_wait_warp(bar(S::B_SFULL + x), (uint32_t)it & 1u, g, 0x401)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[S::KC][32];
#pragma unroll
            for (int j = 0; j < S::KC; ++j) tmem_ld32(s_tmem + 32u * j, sr[j]);
#pragma unroll
            for (int j = 0; j < S::KC; ++j) tmem_ld_wait(sr[j]);
            if (partial) {
#pragma unroll
                for (int j = 0; j < S::KC; ++j)
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const int key = k0 + 32 * j + t;
                        if (key >= kvis || (p.causal && key > q + shift)) sr[j][t] = __float_as_uint(-INFINITY);
                    }
            }
            // row maximum as eight independent 3-input chains, then a tree:
            // one warp per sub-partition runs this, so the latency of a single
            // 64-deep chain would sit on the critical path
            float pm[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) pm[u] = -INFINITY;
#pragma unroll
            for (int j = 0; j < S::KC; ++j)
#pragma unroll
                for (int t = 0; t < 32; t += 4) {
                    const int u = (j * 8 + t / 4) & 7;
                    pm[u] = fmax3(pm[u], __uint_as_float(sr[j][t]), __uint_as_float(sr[j][t + 1]));
                    pm[u] = fmax3(pm[u], __uint_as_float(sr[j][t + 2]), __uint_as_float(sr[j][t + 3]));
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
            // p = 2^(s * c - m), bf16 into the first 64 columns of S_x; the row
            // sum in four independent packed accumulators
            float ps[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) ps[u] = 0.f;
#pragma unroll
            for (int j = 0; j < S::KC; ++j) {
                uint32_t pk[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    float a, bb;
                    fma2(a, bb, __uint_as_float(sr[j][2 * t]), __uint_as_float(sr[j][2 * t + 1]), c2, c2, -m_use, -m_use);
                    a = ex2(a);
                    bb = ex2(bb);
                    const int u = 2 * (t & 3);
                    add2(ps[u], ps[u + 1], a, bb);
                    pk[t] = pack_bf16x2(a, bb);
                }
                tmem_st16(s_tmem + 16u * j, pk);
            }
            l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
            tmem_st_wait();
            if (rescale && it > 0) {
                // O_x may be rescaled only once the previous P_x V has landed
                if (!mbar_wait_warp(bar(S::B_PVDONE + x), (uint32_t)(it - 1) & 1u, g, 0x402)) {
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
                            fma2(a, bb, __uint_as_float(o[j][t]), __uint_as_float(o[j][t + 1]), alpha, alpha, 0.f, 0.f);
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
        }
        // ---------------------------------------------------------- epilogue
        if (ok && it > 0) {
            ok = mbar_wait_warp(bar(S::B_PVDONE + x), (uint32_t)(it - 1) & 1u, g, 0x403);
            tc_fence_after();
        }
        if (ok) {
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
                    for (int t = 0; t < 4; ++t) dst[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
                }
            }
            if (r < qnx)
                p.LSE[VARLEN ? (size_t)h * p.total_q + q_start + q : (size_t)bh * p.N + q] =
                    (l > 0.f) ? (m_ref + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        }
        __syncwarp();
        setmaxnreg_dec<S::REGS_CTRL>();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, S::TMEM_COLS);
}

int fwd_smem_bytes(int d) { return d == 64 ? FwdShape<64>::SMEM_BYTES : FwdShape<128>::SMEM_BYTES; }

template <int D, bool VARLEN, int BC, int QPC>
static cudaError_t launch_fwd_t(const FwdParams &p, cudaStream_t st) {
    using S = FwdShape<D, BC>;
    const int smem = S::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D, VARLEN, BC, QPC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((p.Tq + QPC - 1) / QPC) * (unsigned)p.BH;
    fa_fwd_kernel<D, VARLEN, BC, QPC><<<grid, S::THREADS, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_fwd(int d, const FwdParams &p, cudaStream_t st) {
    return d == 64 ? launch_fwd_t<64, false, 128, 2>(p, st) : launch_fwd_t<128, false, 128, 2>(p, st);
}

cudaError_t launch_fwd_varlen(int d, const FwdParams &p, cudaStream_t st) {
    return d == 64 ? launch_fwd_t<64, true, 128, 2>(p, st) : launch_fwd_t<128, true, 128, 2>(p, st);
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
