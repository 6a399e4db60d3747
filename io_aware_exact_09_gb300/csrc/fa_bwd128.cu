// fa_bwd128.cu -- backward main kernel for d = 128 with 128-row query blocks.
//
// The same method as fa_bwd.cu ("The Attention Matrix You Never Write Down",
// "Tiling forward, recomputing backward"; "FlashAttention: Mathematical
// Foundations ...", "Backward Pass and Activation Recomputation"): per
// 128-key tile, for each query block rebuild P^T = exp(scale k.q - LSE),
//     dV += P^T dO,  dP^T = V dO^T,  dS^T = P^T o (dP^T - D),
//     dK += dS^T Q,  dQ^T = K^T dS^T (reduce-added into the fp32 accumulator).
//
// Why a second kernel: with 64-row query blocks every S^T, dP^T and dQ^T MMA
// is N = 64, and an N = 64 MMA reads nearly as many shared-memory operand
// bytes as an N = 128 one for half the work, so the tensor pipe waits on
// shared memory.  128-row blocks make every MMA N = 128, but S^T, dP^T, dV,
// dK and dQ^T would need 640 TMEM columns.  They fit in 512 because the
// blocks alternate two 128-column regions:
//     block i:  S^T(i) -> region a, dP^T(i) -> region b (a, b swap each block)
//               P^T(i) (bf16, packed) stays in region a until dV(i) reads it,
//               dS^T(i) (packed) in region b until dK(i) reads it;
//               dQ^T(i) -> region a once dV(i) is done;
//     block i+1: S^T(i+1) -> region b once dK(i) is done,
//                dP^T(i+1) -> region a once dQ^T(i) has been drained.
// Shared memory (224 KB): K, V; Q double-buffered, dO single; the dS^T tile
// (the dQ MMA's B operand); 32 KB of dQ staging.
//
// Roles (512 threads): warp 0 TMA producer (under the causal mask also the
// LSE/D staging); warp 1 tcgen05 issuer; warp 2 the LSE/D stager
// (non-causal); warps 4-7 and 8-11 two compute warpgroups,
// one key row per thread, warpgroup w on query columns [64w, 64w + 64);
// warps 12-15 the dQ drain, one head-dimension row of dQ^T per thread: TMEM
// -> swizzled shared staging (two halves of 64 query columns, 8 KB per warp)
// -> TMA reduce-add into the fp32 accumulator.  The drain has its own
// warpgroup because on the compute warps it cost ~45 % of every block (a
// clock64 trace: staging stores queue behind the SS MMAs' operand reads, and
// the staging area shared with the dS^T tile made them wait for the previous
// reduce); off their path, the compute chain per block is P -> dS only.
#include <algorithm>
#include <climits>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

namespace {

struct Bwd128 {
    static constexpr int BQ = 128;
    static constexpr int CW = 64;                          // query columns per compute warpgroup
    static constexpr int CHUNK = 128 * 128;                // 128 rows x 128 bytes (64 bf16 columns)
    static constexpr int TILE = 2 * CHUNK;                 // 128 rows x 128 bf16
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + TILE;
    static constexpr int OFF_Q = OFF_V + TILE;             // [2]
    static constexpr int OFF_DO = OFF_Q + 2 * TILE;
    static constexpr int OFF_DS = OFF_DO + TILE;           // [query chunk 2][key 128][128 B]
    static constexpr int OFF_STG = OFF_DS + TILE;          // [4 drain warps][2 boxes][32 queries][128 B]
    static constexpr int OFF_LSE = OFF_STG + 8 * 4096;     // [BQ] fp32, log2 domain
    static constexpr int OFF_DV = OFF_LSE + BQ * 4;        // [BQ] fp32
    static constexpr int OFF_BAR = OFF_DV + BQ * 4;
    static constexpr int B_KV = 0;
    static constexpr int B_QFULL = 1;                      // [2]
    static constexpr int B_QEMPTY = 3;                     // [2]
    static constexpr int B_DOFULL = 5;
    static constexpr int B_LSE = 7;                        // LSE of a block staged (32 arrivals)
    static constexpr int B_LSEFREE = 8;                    // LSE read by the P pass (256)
    static constexpr int B_SFULL = 9;
    static constexpr int B_DPFULL = 10;
    static constexpr int B_PFULL = 11;                     // 256
    static constexpr int B_DSFULL = 12;                    // 256
    static constexpr int B_DVDONE = 13;                    // dV(i) done: dO free, region a readable
    static constexpr int B_DQFULL = 15;
    static constexpr int B_DQFREE = 16;                    // 128 (drain warpgroup)
    static constexpr int B_ACC = 17;
    static constexpr int B_FIN = 18;
    static constexpr int B_D = 19;                         // D of a block staged (32)
    static constexpr int B_DFREE = 20;                     // D read by the dS pass (256)
    static constexpr int NBAR = 21;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_R0 = 0;                   // regions a / b: 128 columns each
    static constexpr uint32_t TM_DV = 256;
    static constexpr uint32_t TM_DK = 384;
    static constexpr int THREADS = 512;
    static constexpr int LAUNCH_REGS = 128;
    static constexpr int REGS_CTRL = 112;
    static constexpr int REGS_COMPUTE = 152;
    static constexpr int REGS_DRAIN = 96;
    static_assert(128 * REGS_CTRL + 256 * REGS_COMPUTE + 128 * REGS_DRAIN == THREADS * LAUNCH_REGS,
                  "register split");
};

__device__ __forceinline__ void b128_drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > FA_WAIT_TIMEOUT_NS) break;
}

// P^T / dS^T packed (bf16 pairs) inside a region: queries [16k, 16k + 16)
// at column 64 (k / 4) + 8 (k mod 4): each warpgroup stays inside its own
// 64-column half, so neither overwrites fp32 values the other still reads.
__device__ __forceinline__ uint32_t packed_col128(int k) { return (uint32_t)((k >> 2) * 64 + 8 * (k & 3)); }

template <bool VARLEN, bool STAGER, bool PLAIN>
__global__ void __launch_bounds__(512, 1) fa_bwd128_kernel(const __grid_constant__ BwdParams p) {
    grid_dep_wait();                                 // the previous kernel in the stream is done
    grid_dep_launch();
    using S = Bwd128;
    constexpr int BQ = S::BQ, CW = S::CW;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the item (key tile, b*h) of this CTA; from split_from on (every tile
    // full), part `part` of an item run as split_f CTAs, each over its own
    // range of query blocks (the last wave's items, so that it fills the SMs)
    // (split_part: -1 for a whole item, else the part; *sidx: the split item's
    // index past split_from.  Recomputed where needed rather than kept live.)
    auto split_part = [&](int *sidx) -> int {
        const int j = (int)blockIdx.x - p.split_from;
        if (!PLAIN || p.split_f < 2 || j < 0) return -1;
        *sidx = j / p.split_f;
        return j - *sidx * p.split_f;
    };
    int item = (int)blockIdx.x;
    {
        int si = 0;
        if (split_part(&si) >= 0) item = p.split_from + si;
    }
    // Block order.  Every tile full (PLAIN): head-major, every key tile of a
    // head, then the next head.  Under a mask the items differ in length (the
    // causal mask gives key tile kt T - kt query blocks), and head-major would
    // dispatch the last head's longest near the end; so the heads go in groups
    // of kGroup, key-tile-major inside a group (key tile 0 of the group's heads,
    // then key tile 1, ...): the last blocks dispatched are the last group's
    // shortest, and the CTAs at work at one time touch about kGroup heads, so
    // their Q, dO, LSE and D stay shared in L2 as in head-major order.
    constexpr int kGroup = 8;
    int kt = item % p.Tk, bh = item / p.Tk;
    if (!VARLEN && !PLAIN) {
        const int per = p.Tk * kGroup;
        const int gi = item / per, i = item - gi * per;
        const int gs = min(kGroup, p.BH - gi * kGroup);      // the last group may be smaller
        kt = i / gs;
        bh = gi * kGroup + (i - kt * gs);
    }
    const int b = bh / p.H, h = bh % p.H;
    const int k0 = kt * kTile;
    const int nb = (p.N + kTile - 1) / kTile;

    auto bar = [&](int i) -> uint32_t { return base + S::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + S::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sb + S::OFF_MISC + 4);
    const Guard g{p.status, p.status + 1, abort_flag};

    // the sequence (as in fa_bwd.cu): queries [q_start, q_start + Lq), keys
    // [k_start, k_start + Lk), bottom-right causal shift Lk - Lq (0 if square)
    int q_start = 0, k_start = 0, Lq = p.N, Lk = p.N, Tqb = p.Tqb;
    bool bad = false;
    if constexpr (VARLEN) {
        varlen_sequence(p.cu_q, p.cu_k, b, p.total_q, p.total_k, INT_MAX, p.Tk * kTile, &q_start, &Lq, &k_start,
                        &Lk, &bad);
        Tqb = (Lq + BQ - 1) / BQ;
    }
    int qb_lo = 0;                      // a part's first query block (its range ends at Tqb)
    if constexpr (PLAIN) {
        int si = 0;
        const int part = split_part(&si);
        if (part >= 0) {
            qb_lo = part * Tqb / p.split_f;
            Tqb = (part + 1) * Tqb / p.split_f;
        }
    }
    const int shift = Lk - Lq;
    const int kvis = VARLEN ? Lk : key_visible_bound(p.key_len, b, p.N, &bad);
    if (bad && threadIdx.x == 0 && kt == 0 && h == 0) record_status(g, kStatusBadKeyLen, 0);
    // a key tile past a ragged sequence's end has nothing to write: the whole
    // CTA leaves before any set-up
    if (VARLEN && k0 >= Lk) return;

    // query block qb (128 rows = one mask block) against this key tile
    auto cls = [&](int qb) -> unsigned {
        const int qa = qb * BQ;
        if constexpr (VARLEN) return tile_class_shift(qa, min(BQ, Lq - qa), k0, kTile, kvis, p.causal, shift);
        const int on = p.block_mask ? (p.block_mask[(size_t)qb * nb + kt] != 0) : 1;
        return tile_class(qa, min(BQ, p.N - qa), k0, kTile, kvis, p.causal, on);
    };
    const int qb_start = PLAIN ? qb_lo : bwd_query_block_begin(k0, kvis, p.causal, shift, BQ, Tqb);
    auto next_qb = [&](int qb) -> int {
        if (PLAIN || VARLEN || !p.block_mask) {
            const int nq = qb < qb_start ? qb_start : qb + 1;
            return nq < Tqb ? nq : Tqb;
        }
        for (int x = qb + 1; x < Tqb; ++x)
            if (cls(x) != kTileSkip) return x;
        return Tqb;
    };
    // TMA coordinates: [B*H][N][d] view, or the ragged [total][H][d] view
    auto tload = [&](uint32_t dst, const CUtensorMap *m, uint32_t mbar, int c, int row, int start) {
        if constexpr (VARLEN)
            tma_load_3d(dst, m, mbar, c * 64, h, start + row);
        else
            tma_load_3d(dst, m, mbar, c * 64, row, bh);
    };
    auto lse_index = [&](int qq) -> size_t {
        return VARLEN ? (size_t)h * p.total_q + q_start + qq : (size_t)bh * p.N + qq;
    };
    auto d_index = [&](int qq) -> size_t {
        return VARLEN ? (size_t)(q_start + qq) * p.H + h : (size_t)bh * p.N + qq;
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(S::B_KV), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(S::B_QFULL + s), 1);
            mbar_init(bar(S::B_QEMPTY + s), 1);
        }
        mbar_init(bar(S::B_DOFULL), 1);
        mbar_init(bar(S::B_LSE), 32);
        mbar_init(bar(S::B_LSEFREE), 256);
        mbar_init(bar(S::B_D), 32);
        mbar_init(bar(S::B_DFREE), 256);
        mbar_init(bar(S::B_SFULL), 1);
        mbar_init(bar(S::B_DPFULL), 1);
        mbar_init(bar(S::B_PFULL), 256);
        mbar_init(bar(S::B_DSFULL), 256);
        mbar_init(bar(S::B_DVDONE), 1);
        mbar_init(bar(S::B_DQFULL), 1);
        mbar_init(bar(S::B_DQFREE), 128);
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
    const int first = next_qb(-1);
    float *lse_s = reinterpret_cast<float *>(sb + S::OFF_LSE);   // log2 domain
    float *dv_s = reinterpret_cast<float *>(sb + S::OFF_DV);
    // LSE and D of a block, raw, for lane `lane`'s four rows (row >= Lq: LSE
    // -inf, D 0), and their conversion into the staging buffers: LSE into the
    // log2 domain, +inf for a row past the sequence's end or with no visible
    // key (its P is then 0)
    auto fetch_lse = [&](int qb, float (&rl)[BQ / 32], float (&rd)[BQ / 32]) {
#pragma unroll
        for (int u = 0; u < BQ / 32; ++u) {
            const int qq = qb * BQ + u * 32 + lane;
            rl[u] = -INFINITY;
            rd[u] = 0.f;
            if (qq < Lq) {
                rl[u] = p.LSE[lse_index(qq)];
                rd[u] = p.Dvec[d_index(qq)];
            }
        }
    };
    auto store_lse = [&](const float (&rl)[BQ / 32]) {
#pragma unroll
        for (int u = 0; u < BQ / 32; ++u)
            lse_s[u * 32 + lane] = (rl[u] == -INFINITY) ? INFINITY : rl[u] * 1.4426950408889634f;
    };
    auto store_d = [&](const float (&rd)[BQ / 32]) {
#pragma unroll
        for (int u = 0; u < BQ / 32; ++u) dv_s[u * 32 + lane] = rd[u];
    };
    // Who stages them: without the causal mask a warp of its own (warp 2),
    // which loads the next block's values while the current one computes and
    // stores each buffer as soon as its pass has read it; under the causal
    // mask the producer, behind the previous block's dS pass.  Measured on
    // the long-context shapes: the stager warp takes the non-causal backward
    // from 4.95 to 4.74 ms but the causal one from 2.36 to 2.50 ms (same
    // GPU, several variants of the stager alike), so each mode keeps the
    // faster one.  The mode is a template parameter (STAGER = !causal), so
    // that each kernel carries only its own staging code.
    constexpr bool stager = STAGER;

    if (warp < 4) {
        setmaxnreg_dec<S::REGS_CTRL>();
        if (warp == 0 && first < Tqb) {
            // ---------------------------------------------------------- producer
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(S::B_KV), 2 * S::TILE);
                for (int c = 0; c < 2; ++c) {
                    tload(base + S::OFF_K + c * S::CHUNK, &p.tmK, bar(S::B_KV), c, k0, k_start);
                    tload(base + S::OFF_V + c * S::CHUNK, &p.tmV, bar(S::B_KV), c, k0, k_start);
                }
            }
            int i = 0, nq = 0, nl = 0;  // blocks seen, blocks whose Q / dO loads were issued
            bool ok = true;
            for (int qb = first; qb < Tqb; qb = next_qb(qb), ++i) {
                const int s = i & 1;
                // Q(i) into stage s once dK(i - 2) has read it, then dO(i) once dV(i - 1)
                // has read the single dO buffer: each load waits for its own buffer only
                // (Q used to wait for dV(i - 1) too, a block later than its stage was free)
                if (!mbar_wait_warp(bar(S::B_QEMPTY + s), ((uint32_t)(i >> 1) & 1u) ^ 1u, g, 0x121)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(S::B_QFULL + s), S::TILE);
                    for (int c = 0; c < 2; ++c)
                        tload(base + S::OFF_Q + s * S::TILE + c * S::CHUNK, &p.tmQ, bar(S::B_QFULL + s), c, qb * BQ,
                              q_start);
                }
                nq = i + 1;
                if (!mbar_wait_warp(bar(S::B_DVDONE), ((uint32_t)i & 1u) ^ 1u, g, 0x122)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(S::B_DOFULL), S::TILE);
                    for (int c = 0; c < 2; ++c)
                        tload(base + S::OFF_DO + c * S::CHUNK, &p.tmdO, bar(S::B_DOFULL), c, qb * BQ, q_start);
                }
                nl = i + 1;
                if (!stager) {
                    // LSE and D of block i once the dS pass has read block i - 1's
                    if (!mbar_wait_warp(bar(S::B_DFREE), ((uint32_t)i & 1u) ^ 1u, g, 0x123)) {
                        ok = false;
                        break;
                    }
                    float rl[BQ / 32], rd[BQ / 32];
                    fetch_lse(qb, rl, rd);
                    store_lse(rl);
                    store_d(rd);
                    mbar_arrive(bar(S::B_LSE));
                    mbar_arrive(bar(S::B_D));
                }
            }
            if (!ok && lane == 0) {
                // gave up: let every copy already issued land before the CTA exits
                b128_drain_wait(bar(S::B_KV), 0);
                for (int j = (nq > 2 ? nq - 2 : 0); j < nq; ++j)
                    b128_drain_wait(bar(S::B_QFULL + (j & 1)), (uint32_t)(j >> 1) & 1u);
                if (nl > 0) b128_drain_wait(bar(S::B_DOFULL), (uint32_t)(nl - 1) & 1u);
            }
        } else if (warp == 2 && stager && first < Tqb) {
            // ---------------------------------------------------------- LSE / D stager (non-causal)
            // The next block's values are loaded into registers while the
            // current block computes; LSE is stored as soon as the P pass has
            // read the previous block's, D as soon as the dS pass has read the
            // previous D, so that no global-load latency falls between two
            // blocks (staged by the producer behind the previous block's
            // release, the compute warps waited ~3,500 cycles per block for them
            // on the non-causal long-context shape).
            float rl[BQ / 32], rd[BQ / 32];
            int i = 0;
            fetch_lse(first, rl, rd);
            for (int qb = first; qb < Tqb; ++i) {
                if (i > 0 && !mbar_wait_warp(bar(S::B_LSEFREE), (uint32_t)(i - 1) & 1u, g, 0x124)) break;
                store_lse(rl);
                mbar_arrive(bar(S::B_LSE));
                if (i > 0 && !mbar_wait_warp(bar(S::B_DFREE), (uint32_t)(i - 1) & 1u, g, 0x125)) break;
                store_d(rd);
                mbar_arrive(bar(S::B_D));
                qb = next_qb(qb);
                if (qb < Tqb) fetch_lse(qb, rl, rd);
            }
        } else if (warp == 1) {
            // ---------------------------------------------------------- MMA issuer
            // Order per block i: dV(i), dQ^T(i), dK(i), S^T(i+1), dP^T(i+1).
            constexpr uint32_t IDESC_S = idesc_bf16(128, BQ, false, false);   // S^T, dP^T
            constexpr uint32_t IDESC_ACC = idesc_bf16(128, 128, false, true); // dV, dK: B MN-major
            constexpr uint32_t IDESC_DQ = idesc_bf16(128, BQ, true, true);    // dQ^T = K^T dS^T
            const uint64_t dK_kmaj = sdesc_sw128(base + S::OFF_K, 16, 1024);
            const uint64_t dV_kmaj = sdesc_sw128(base + S::OFF_V, 16, 1024);
            const uint64_t dQ_kmaj = sdesc_sw128(base + S::OFF_Q, 16, 1024);
            const uint64_t ddO_kmaj = sdesc_sw128(base + S::OFF_DO, 16, 1024);
            const uint64_t dQ_mn = sdesc_sw128(base + S::OFF_Q, S::CHUNK, 1024);
            const uint64_t ddO_mn = sdesc_sw128(base + S::OFF_DO, S::CHUNK, 1024);
            const uint64_t dK_mn = sdesc_sw128(base + S::OFF_K, S::CHUNK, 1024);
            const uint64_t ddS_mn = sdesc_sw128(base + S::OFF_DS, S::CHUNK, 1024);
            auto region = [&](int r) -> uint32_t { return tmem + S::TM_R0 + 128u * (uint32_t)r; };
            // S^T(i) = K Q^T into region (i & 1)
            auto issue_s = [&](int i) {
                const uint64_t qd = sdesc_add(dQ_kmaj, (uint32_t)((i & 1) * S::TILE));
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * S::CHUNK + (k & 3) * 32;
                    mma_ss_elect(region(i & 1), sdesc_add(dK_kmaj, off), sdesc_add(qd, off), IDESC_S, k > 0 ? 1u : 0u);
                }
                mma_commit_elect(bar(S::B_SFULL));
            };
            // dP^T(i) = V dO^T into region (i & 1) ^ 1
            auto issue_dp = [&](int i) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * S::CHUNK + (k & 3) * 32;
                    mma_ss_elect(region((i & 1) ^ 1), sdesc_add(dV_kmaj, off), sdesc_add(ddO_kmaj, off), IDESC_S,
                           k > 0 ? 1u : 0u);
                }
                mma_commit_elect(bar(S::B_DPFULL));
            };
            bool ok = true;
            int i = 0;
            if (first < Tqb) {
                ok = mbar_wait_warp(bar(S::B_KV), 0, g, 0x221) && mbar_wait_warp(bar(S::B_QFULL), 0, g, 0x222) &&
                     mbar_wait_warp(bar(S::B_DOFULL), 0, g, 0x223);
                if (ok) {
                    tc_fence_after();
                    issue_s(0);
                    issue_dp(0);
                }
                for (int qb = first; ok && qb < Tqb; ++i) {
                    const int s = i & 1;
                    const uint32_t ra = region(s), rb = region(s ^ 1);
                    const uint32_t acc0 = i > 0 ? 1u : 0u;
                    const int qb_next = next_qb(qb);
                    // dV += P^T dO: A = P^T (region a, packed), B = dO (MN-major)
                    if (!mbar_wait_warp(bar(S::B_PFULL), (uint32_t)i & 1u, g, 0x224)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < BQ / 16; ++k)
                        mma_ts_elect(tmem + S::TM_DV, ra + packed_col128(k), sdesc_add(ddO_mn, (uint32_t)k * 2048u),
                               IDESC_ACC, k > 0 ? 1u : acc0);
                    mma_commit_elect(bar(S::B_DVDONE));
                    // dQ^T = K^T dS^T into region a (once dV has read P^T there), first:
                    // the sooner it is drained, the sooner dP^T(i+1) can use region a;
                    // dK follows
                    if (!mbar_wait_warp(bar(S::B_DSFULL), (uint32_t)i & 1u, g, 0x225) ||
                        !mbar_wait_warp(bar(S::B_DVDONE), (uint32_t)i & 1u, g, 0x226)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < kTile / 16; ++k)
                        mma_ss_elect(ra, sdesc_add(dK_mn, (uint32_t)k * 2048u), sdesc_add(ddS_mn, (uint32_t)k * 2048u),
                               IDESC_DQ, k > 0 ? 1u : 0u);
                    mma_commit_elect(bar(S::B_DQFULL));
                    // dK += dS^T Q: A = dS^T (region b, packed), B = Q (MN-major)
                    const uint64_t q_mn = sdesc_add(dQ_mn, (uint32_t)(s * S::TILE));
#pragma unroll
                    for (int k = 0; k < BQ / 16; ++k)
                        mma_ts_elect(tmem + S::TM_DK, rb + packed_col128(k), sdesc_add(q_mn, (uint32_t)k * 2048u),
                               IDESC_ACC, k > 0 ? 1u : acc0);
                    mma_commit_elect(bar(S::B_QEMPTY + s));       // dK(i) done
                    if (qb_next < Tqb) {
                        // S^T(i+1) into region b once dK has read dS^T there
                        if (!mbar_wait_warp(bar(S::B_QFULL + (s ^ 1)), (uint32_t)((i + 1) >> 1) & 1u, g, 0x227) ||
                            !mbar_wait_warp(bar(S::B_QEMPTY + s), (uint32_t)(i >> 1) & 1u, g, 0x228)) { ok = false; break; }
                        tc_fence_after();
                        issue_s(i + 1);
                        // dP^T(i+1) into region a once dQ^T(i) has been drained
                        if (!mbar_wait_warp(bar(S::B_DOFULL), (uint32_t)(i + 1) & 1u, g, 0x229) ||
                            !mbar_wait_warp(bar(S::B_DQFREE), (uint32_t)i & 1u, g, 0x22a)) { ok = false; break; }
                        tc_fence_after();
                        issue_dp(i + 1);
                    }
                    qb = qb_next;
                }
                if (ok) mma_commit_elect(bar(S::B_ACC));
            }
            mma_commit_elect(bar(S::B_FIN));
            b128_drain_wait(bar(S::B_FIN), 0);
        }
    } else if (warp < 12) {
        setmaxnreg_inc<S::REGS_COMPUTE>();
        // ---------------------------------------------------------- compute (two warpgroups)
        const int wg = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;           // TMEM lane: key row (S^T, dP^T, dK, dV), head dim (dQ^T)
        const int key = k0 + r;
        const int c0 = wg * CW;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const float c2 = p.scale_log2;
        bool ok = true;
        int i = 0;

        for (int qb = first; qb < Tqb; qb = next_qb(qb), ++i) {
            // PLAIN: no causal mask, key padding or block mask, N a multiple of
            // 128: every block is full and the masking code is not compiled
            const unsigned klass = PLAIN ? kTileFull : cls(qb);
            const int qa = qb * BQ;
            const uint32_t ra = tmem + lane_off + S::TM_R0 + 128u * (uint32_t)(i & 1);
            const uint32_t rb = tmem + lane_off + S::TM_R0 + 128u * (uint32_t)((i & 1) ^ 1);
            if (!mbar_wait_warp(bar(S::B_LSE), (uint32_t)i & 1u, g, 0x421)) { ok = false; break; }

            // P^T = 2^(s * c - LSE_q * log2 e), masked, for columns c0 .. c0 + 63.
            // The block's LSE values go to registers before the wait: shared-memory
            // loads inside the loop would queue behind the MMAs' operand reads.
            if (!mbar_wait_warp(bar(S::B_SFULL), (uint32_t)i & 1u, g, 0x422)) { ok = false; break; }
            tc_fence_after();
            uint32_t pk[CW / 2];
            {
                uint32_t sr[2][32];
                tmem_ld32(ra + c0, sr[0]);
                tmem_ld32(ra + c0 + 32, sr[1]);
                tmem_ld_wait(sr[0]);
                tmem_ld_wait(sr[1]);
                if (!PLAIN && klass == kTilePartial) {
                    // masked scores -> -inf, so that their p is exactly 0 (a mask
                    // test inside the exp loop below made that loop several times slower)
                    // this key row sees the columns from lo on (none past the visible
                    // keys): one compare against a constant per score
                    int lo = p.causal ? key - shift - qa - c0 : INT_MIN;
                    if (key >= kvis) lo = INT_MAX;
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (32 * j + t < lo) sr[j][t] = __float_as_uint(-INFINITY);
                }
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int t = 0; t < 32; t += 4) {
                        const float4 l4 = *reinterpret_cast<const float4 *>(lse_s + c0 + 32 * j + t);
                        float p0, p1, p2, p3;
                        fma2(p0, p1, __uint_as_float(sr[j][t]), __uint_as_float(sr[j][t + 1]), c2, c2, -l4.x, -l4.y);
                        fma2(p2, p3, __uint_as_float(sr[j][t + 2]), __uint_as_float(sr[j][t + 3]), c2, c2, -l4.z,
                             -l4.w);
                        pk[16 * j + t / 2] = pack_bf16x2(ex2(p0), ex2(p1));
                        pk[16 * j + t / 2 + 1] = pack_bf16x2(ex2(p2), ex2(p3));
                    }
            }
            tmem_st16(ra + c0, pk);
            tmem_st16(ra + c0 + 16, pk + 16);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(S::B_PFULL));
            mbar_arrive(bar(S::B_LSEFREE));           // this block's LSE has been read

            // dS^T = P^T o (dP^T - D): bf16 into region b (for dK) and the shared dS^T tile (for dQ);
            // D to registers before the wait, as LSE above
            if (!mbar_wait_warp(bar(S::B_DPFULL), (uint32_t)i & 1u, g, 0x423) ||
                !mbar_wait_warp(bar(S::B_D), (uint32_t)i & 1u, g, 0x424)) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t dp[2][32];
                tmem_ld32(rb + c0, dp[0]);
                tmem_ld32(rb + c0 + 32, dp[1]);
                tmem_ld_wait(dp[0]);
                tmem_ld_wait(dp[1]);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    uint32_t w[16];
#pragma unroll
                    for (int t = 0; t < 16; t += 2) {
                        const float4 d4 = *reinterpret_cast<const float4 *>(dv_s + c0 + 32 * j + 2 * t);
                        const uint32_t pa = pk[16 * j + t], pb = pk[16 * j + t + 1];
                        w[t] = pack_bf16x2(bf16lo(pa) * (__uint_as_float(dp[j][2 * t]) - d4.x),
                                           bf16hi(pa) * (__uint_as_float(dp[j][2 * t + 1]) - d4.y));
                        w[t + 1] = pack_bf16x2(bf16lo(pb) * (__uint_as_float(dp[j][2 * t + 2]) - d4.z),
                                               bf16hi(pb) * (__uint_as_float(dp[j][2 * t + 3]) - d4.w));
                    }
                    tmem_st16(rb + c0 + 16u * j, w);
                    // shared dS^T tile, queries contiguous (MN-major, 128-byte swizzle):
                    // [query chunk of 64][key row 0..127][128 bytes]; this warpgroup's
                    // 64 queries are chunk wg
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int qo = 32 * j + 8 * u;              // first query of this 16-byte piece, in the chunk
                        uint8_t *dst = sb + S::OFF_DS + wg * S::CHUNK + r * 128 + ((((qo >> 3)) ^ (r & 7)) << 4);
                        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                    }
                }
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(S::B_DSFULL));
            mbar_arrive(bar(S::B_DFREE));             // this block's D has been read
        }

        // ---------------------------------------------------------- epilogue: dK, dV
        if (ok && i > 0) {
            ok = mbar_wait_warp(bar(S::B_ACC), 0, g, 0x425);
            tc_fence_after();
        }
        if constexpr (!STAGER) {
        if (ok) {
            // causal mode: dK (* scale) and dV, this warp's 32 rows x 64 columns
            // (128 bytes) of each through its own 8 KB of the query tiles (free:
            // every product is complete and no further block is loaded), read
            // back so that each store covers 4 whole 128-byte rows (stored
            // straight from registers, every store touched 32 rows: measured
            // 2-8 % slower on causal shapes; the non-causal kernel, whose speed
            // changed with its code rather than with this work, keeps that)
            uint8_t *stg = sb + S::OFF_Q + (warp - 4) * 8192;
#pragma unroll 1
            for (int jh = 0; jh < 2; ++jh) {
                uint32_t a[32], vv[32];
                if (i > 0) {
                    tmem_ld32(tmem + lane_off + S::TM_DK + 32u * (wg * 2 + jh), a);
                    tmem_ld32(tmem + lane_off + S::TM_DV + 32u * (wg * 2 + jh), vv);
                    tmem_ld_wait(a);
                    tmem_ld_wait(vv);
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) a[t] = vv[t] = 0u;
                }
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int off = lane * 128 + (((4 * jh + t) ^ (lane & 7)) << 4);
                    *reinterpret_cast<uint4 *>(stg + off) = make_uint4(
                        pack_bf16x2(__uint_as_float(a[8 * t]) * p.scale, __uint_as_float(a[8 * t + 1]) * p.scale),
                        pack_bf16x2(__uint_as_float(a[8 * t + 2]) * p.scale, __uint_as_float(a[8 * t + 3]) * p.scale),
                        pack_bf16x2(__uint_as_float(a[8 * t + 4]) * p.scale, __uint_as_float(a[8 * t + 5]) * p.scale),
                        pack_bf16x2(__uint_as_float(a[8 * t + 6]) * p.scale, __uint_as_float(a[8 * t + 7]) * p.scale));
                    *reinterpret_cast<uint4 *>(stg + 4096 + off) = make_uint4(
                        pack_bf16x2(__uint_as_float(vv[8 * t]), __uint_as_float(vv[8 * t + 1])),
                        pack_bf16x2(__uint_as_float(vv[8 * t + 2]), __uint_as_float(vv[8 * t + 3])),
                        pack_bf16x2(__uint_as_float(vv[8 * t + 4]), __uint_as_float(vv[8 * t + 5])),
                        pack_bf16x2(__uint_as_float(vv[8 * t + 6]), __uint_as_float(vv[8 * t + 7])));
                }
            }
            __syncwarp();
            const int u = lane & 7;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int rr = 4 * jj + (lane >> 3);                // row of this warp's 32
                const int off = rr * 128 + ((u ^ (rr & 7)) << 4);
                const uint4 kq = *reinterpret_cast<const uint4 *>(stg + off);
                const uint4 vq = *reinterpret_cast<const uint4 *>(stg + 4096 + off);
                const int keyr = k0 + wq * 32 + rr;
                if (keyr < Lk) {
                    const size_t krow = VARLEN ? (size_t)(k_start + keyr) * p.H + h : (size_t)bh * p.N + keyr;
                    *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.dK) + krow * 128 + 64 * wg + 8 * u) = kq;
                    *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.dV) + krow * 128 + 64 * wg + 8 * u) = vq;
                }
            }
        }
        } else {
            // An item split over several CTAs: each part stores its fp32 dK
            // (unscaled) and dV in its own slot, then counts itself; the part
            // that counts last sums the slots in part order (its own from
            // TMEM), so the result does not depend on which part that is, and
            // writes dK, dV.  Slot layout: float4 (c, key row) at c * 128 + row,
            // c = 8 j + t for dK columns 32 j + 4 t .. + 3, 32 + 8 j + t for dV,
            // so that a warp's store covers 512 contiguous bytes.  The stores
            // are published by one thread (CTA barrier, release fence, count)
            // and the counter read the same way (count, acquire fence, barrier);
            // all 256 compute threads take both barriers on every path.
            bool write = ok;
            const float4 *slots = nullptr;           // part 0's slot of this item
            int sidx = 0;
            const int part = split_part(&sidx);
            if constexpr (PLAIN) {
                if (part >= 0) {
                    slots = reinterpret_cast<const float4 *>(p.split_buf) + (size_t)sidx * p.split_f * 8192;
                    if (ok) {
                        float4 *mine = const_cast<float4 *>(slots) + (size_t)part * 8192 + r;
    #pragma unroll 1
                        for (int j = wg * 2; j < wg * 2 + 2; ++j) {
                            uint32_t a[32], vv[32];
                            tmem_ld32(tmem + lane_off + S::TM_DK + 32u * j, a);
                            tmem_ld32(tmem + lane_off + S::TM_DV + 32u * j, vv);
                            tmem_ld_wait(a);
                            tmem_ld_wait(vv);
    #pragma unroll
                            for (int t = 0; t < 8; ++t) {
                                mine[(8 * j + t) * 128] = make_float4(__uint_as_float(a[4 * t]), __uint_as_float(a[4 * t + 1]),
                                                                      __uint_as_float(a[4 * t + 2]), __uint_as_float(a[4 * t + 3]));
                                mine[(32 + 8 * j + t) * 128] =
                                    make_float4(__uint_as_float(vv[4 * t]), __uint_as_float(vv[4 * t + 1]),
                                                __uint_as_float(vv[4 * t + 2]), __uint_as_float(vv[4 * t + 3]));
                            }
                        }
                    }
                    named_bar_sync(1, 256);
                    volatile int *last = reinterpret_cast<volatile int *>(sb + S::OFF_MISC + 8);
                    if (threadIdx.x == 128) {
                        // byte counter sidx % 4 of word sidx / 4 (it never exceeds split_f <= 4)
                        unsigned *w = p.split_cnt + (sidx >> 2);
                        const unsigned sh = 8u * (unsigned)(sidx & 3);
                        fence_acq_rel_gpu();
                        const unsigned n = ((atomicAdd(w, 1u << sh) >> sh) & 0xFFu) + 1u;
                        const int l = n == (unsigned)p.split_f ? 1 : 0;
                        if (l) {
                            atomicAnd(w, ~(0xFFu << sh));   // every part has counted: zero for the next launch
                            fence_acq_rel_gpu();
                        }
                        *last = l;
                    }
                    named_bar_sync(1, 256);
                    write = ok && *last != 0;
                }
            }
            if (write) {
                const size_t krow = VARLEN ? (size_t)(k_start + key) * p.H + h : (size_t)bh * p.N + key;
                __nv_bfloat16 *dkrow = reinterpret_cast<__nv_bfloat16 *>(p.dK) + krow * 128;
                __nv_bfloat16 *dvrow = reinterpret_cast<__nv_bfloat16 *>(p.dV) + krow * 128;
                // one half (dK columns 32 j .. 32 j + 31, scaled, or dV's) of
                // this thread's key row: TMEM, for a split item summed with the
                // other parts' slots, to bf16 and global memory
                auto write_half = [&](uint32_t tm_col, int grp0, float sc, __nv_bfloat16 *dst) {
                    uint32_t a[32];
                    if (i > 0) {
                        tmem_ld32(tmem + lane_off + tm_col, a);
                        tmem_ld_wait(a);
                    } else {
    #pragma unroll
                        for (int t = 0; t < 32; ++t) a[t] = 0u;
                    }
                    if constexpr (PLAIN) {
                        if (part >= 0) {
                            // sum over the parts in order 0, 1, ...: slot o (its eight
                            // float4 loads issued together) or, for o = part, own
                            auto load_slot = [&](int o, float (&x)[32]) {
                                const float4 *src = slots + (size_t)o * 8192 + (size_t)grp0 * 128 + r;
    #pragma unroll
                                for (int t = 0; t < 8; ++t) {
                                    const float4 q = __ldcg(src + t * 128);
                                    x[4 * t] = q.x;
                                    x[4 * t + 1] = q.y;
                                    x[4 * t + 2] = q.z;
                                    x[4 * t + 3] = q.w;
                                }
                            };
                            float sum[32];
                            if (part == 0) {
    #pragma unroll
                                for (int t = 0; t < 32; ++t) sum[t] = __uint_as_float(a[t]);
                            } else {
                                load_slot(0, sum);
                            }
                            for (int o = 1; o < p.split_f; ++o) {
                                if (o == part) {
    #pragma unroll
                                    for (int t = 0; t < 32; ++t) sum[t] += __uint_as_float(a[t]);
                                } else {
                                    float x[32];
                                    load_slot(o, x);
    #pragma unroll
                                    for (int t = 0; t < 32; ++t) sum[t] += x[t];
                                }
                            }
    #pragma unroll
                            for (int t = 0; t < 32; ++t) a[t] = __float_as_uint(sum[t]);
                        }
                    }
                    uint32_t w[16];
    #pragma unroll
                    for (int t = 0; t < 16; ++t)
                        w[t] = pack_bf16x2(__uint_as_float(a[2 * t]) * sc, __uint_as_float(a[2 * t + 1]) * sc);
                    if (key < Lk) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    #pragma unroll
                        for (int t = 0; t < 4; ++t) d4[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
                    }
                };
    #pragma unroll 1
                for (int j = wg * 2; j < wg * 2 + 2; ++j) {
                    write_half(S::TM_DK + 32u * j, 8 * j, p.scale, dkrow + 32 * j);
                    write_half(S::TM_DV + 32u * j, 32 + 8 * j, 1.f, dvrow + 32 * j);
                }
            }
        }
        __syncwarp();
        setmaxnreg_dec<S::REGS_CTRL>();
    } else {
        setmaxnreg_dec<S::REGS_DRAIN>();
        // ---------------------------------------------------------- dQ drain (one warpgroup)
        // lane = head dimension 32 wq + lane of dQ^T(i); 128 query columns in two
        // halves through this warp's two staging boxes (32 queries x 32 fp32,
        // 128-byte swizzle)
        const int wq = warp & 3;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        uint8_t *stg = sb + S::OFF_STG + wq * 8192;
        const int grp = lane >> 2;
        int i = 0;
        for (int qb = first; qb < Tqb; qb = next_qb(qb), ++i) {
            const uint32_t ra = tmem + lane_off + S::TM_R0 + 128u * (uint32_t)(i & 1);
            if (!mbar_wait_warp(bar(S::B_DQFULL), (uint32_t)i & 1u, g, 0x426)) break;
            tc_fence_after();
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t v[2][32];
                tmem_ld32(ra + 64u * hf, v[0]);
                tmem_ld32(ra + 64u * hf + 32, v[1]);
                tmem_ld_wait(v[0]);
                tmem_ld_wait(v[1]);
                if (hf == 1) {
                    // all of dQ^T(i) is in registers or staged: region a is free
                    tc_fence_before();
                    mbar_arrive(bar(S::B_DQFREE));
                }
                // the boxes' previous reduce must have read them
                if (lane == 0) bulk_wait_group_read<0>();
                __syncwarp();
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    uint8_t *cb = stg + u * 4096 + (lane & 3) * 4;
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        *reinterpret_cast<uint32_t *>(cb + t * 128 + ((grp ^ (t & 7)) << 4)) = v[u][t];
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int q0 = qb * BQ + 64 * hf;
                    if constexpr (VARLEN) {
                        tma_reduce_add_3d(&p.tmdQ, smem_u32(stg), wq * 32, h, q_start + q0);
                        tma_reduce_add_3d(&p.tmdQ, smem_u32(stg + 4096), wq * 32, h, q_start + q0 + 32);
                    } else {
                        tma_reduce_add_3d(&p.tmdQ, smem_u32(stg), wq * 32, q0, bh);
                        tma_reduce_add_3d(&p.tmdQ, smem_u32(stg + 4096), wq * 32, q0 + 32, bh);
                    }
                    bulk_commit_group();
                }
            }
        }
        // the staged boxes must be fully reduced before shared memory goes away
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, S::TMEM_COLS);
}

}  // namespace

int bwd128_smem_bytes() { return Bwd128::SMEM_BYTES; }

template <bool VARLEN, bool STAGER, bool PLAIN = false>
static cudaError_t launch_bwd128_t(const BwdParams &p, cudaStream_t st) {
    const int smem = Bwd128::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(fa_bwd128_kernel<VARLEN, STAGER, PLAIN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)p.Tk * p.BH;
    const int64_t grid = p.split_f > 1 ? p.split_from + (items - p.split_from) * p.split_f : items;
    return launch_dep(fa_bwd128_kernel<VARLEN, STAGER, PLAIN>, (unsigned)grid, Bwd128::THREADS, smem, st, p);
}

// Split plan of the plain instantiation, whose items all take the same time:
// one CTA per SM at a time, so the items past the last full wave (rem of
// them) would run on rem SMs while the others idle.  Each of those runs as
// f = SMs / rem parts instead (at most 4, at least two query blocks per part,
// at most what the buffer holds), so that the last wave is about 1/f as long.
// A part costs a few microseconds more than its share of the blocks (the
// slots' stores and loads): with one query block per part that was more
// than the split saved.
static void plan_split(BwdParams &q) {
    q.split_from = 0;
    q.split_f = 0;
    if (!q.split_buf || !q.split_cnt || q.split_cap < 2) return;
    const int64_t items = (int64_t)q.Tk * q.BH;
    const int64_t sms = device_sm_count();
    const int64_t rem = items % sms;
    if (rem == 0) return;
    if (rem > kSplitMaxItems) return;
    int64_t f = std::min<int64_t>(std::min<int64_t>(sms / rem, 4), q.Tqb / 2);
    if (f * rem > q.split_cap) f = q.split_cap / rem;
    if (f < 2) return;
    q.split_from = (int)(items - rem);
    q.split_f = (int)f;
}

cudaError_t launch_bwd128_main(const BwdParams &p, cudaStream_t st) {
    BwdParams q = p;
    q.split_from = 0;
    q.split_f = 0;
    if (q.causal) return launch_bwd128_t<false, false>(q, st);
    const bool plain = !q.key_len && !q.block_mask && q.N % 128 == 0;
    if (!plain) return launch_bwd128_t<false, true>(q, st);
    plan_split(q);
    return launch_bwd128_t<false, true, true>(q, st);
}

cudaError_t launch_bwd128_main_varlen(const BwdParams &p, cudaStream_t st) {
    BwdParams q = p;
    q.split_from = 0;
    q.split_f = 0;
    return q.causal ? launch_bwd128_t<true, false>(q, st) : launch_bwd128_t<true, true>(q, st);
}

}  // namespace fa
