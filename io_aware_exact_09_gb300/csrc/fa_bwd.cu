// fa_bwd.cu -- backward kernels: gradients of exact attention by recomputing
// the score and probability tiles on chip.
//
// Method ("The Attention Matrix You Never Write Down", section "Tiling
// forward, recomputing backward"; "FlashAttention: Mathematical Foundations
// ...", section "Backward Pass and Activation Recomputation"): the forward
// kept only O and the per-row statistic LSE; the backward rebuilds each tile
// P_ij = exp(scale * q_i.k_j - LSE_i) from Q_i, K_j and LSE_i instead of
// reading a stored N x N matrix.  The gradient formulas themselves are the
// chain rule through O = P V and the row softmax (the pages give none):
//     dV = P^T dO,  dP = dO V^T,  D_i = sum_k dO_ik O_ik,
//     dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// Three kernels:
//   1. fa_bwd_pre:     D = rowsum(dO * O) (fp32) and dQacc = 0      (HBM-bound)
//   2. fa_bwd_kernel:  one CTA per (128-key tile, b*h); loop over the query
//      blocks that see the tile:
//        warp 0  TMA: K_j, V_j once; Q_i, dO_i through a 2-stage ring; the
//                whole warp stages LSE_i and D_i into shared memory with them
//        warp 1  tcgen05: S^T = K Q^T, dP^T = V dO^T, dV += P^T dO,
//                dK += dS^T Q (P^T, dS^T read from TMEM), and the dQ
//                contribution into one of two TMEM buffers
//        warps 4-7 and 8-11  two compute warpgroups, one key row per thread,
//                each on half of the query columns (the backward has no row
//                reduction): P^T = 2^(s*c - LSE*log2 e), masks,
//                dS^T = P^T o (dP^T - D) -> bf16 into TMEM and into shared
//                memory (the dQ MMA's operand); each drains half of the
//                previous dQ contribution through a swizzled shared tile and
//                per-warp TMA reduce-adds into the fp32 accumulator; at the
//                end each converts half of dK * scale and dV to bf16.
//      This kernel is the d = 64 one: 128-row query blocks and dQ = dS K
//      (TMEM lane = query), so that S, dP (128 columns each), dV, dK and two
//      dQ buffers (64 each) fit in the 512 TMEM columns.  d = 128 has its own
//      kernel, fa_bwd128.cu.
//   3. fa_bwd_convert: dQ = bf16(scale * dQacc)                        (HBM-bound)
// The preprocessing and conversion kernels serve both head dimensions.
#include <climits>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

template <int D>
struct BwdShape {
    static_assert(D == 64, "d = 128 has its own kernel (fa_bwd128.cu)");
    static constexpr int BQ = 128;                        // query rows per inner step
    static constexpr int CHUNKS = D / 64;
    static constexpr int KV_CHUNK = 128 * 128;            // 128 keys x 128 bytes
    static constexpr int KV_BYTES = CHUNKS * KV_CHUNK;
    static constexpr int Q_CHUNK = BQ * 128;              // BQ rows x 128 bytes
    static constexpr int Q_BYTES = CHUNKS * Q_CHUNK;
    static constexpr int STAGES = 2;
    static constexpr int DS_BYTES = BQ * 128 * 2;         // BQ queries x 128 keys, bf16
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KV_BYTES;
    static constexpr int OFF_Q = OFF_V + KV_BYTES;        // [STAGES]
    static constexpr int OFF_DO = OFF_Q + STAGES * Q_BYTES;
    static constexpr int OFF_DS = OFF_DO + STAGES * Q_BYTES;
    // dQ staging for the TMA reduce-add: [D/32 chunks][BQ rows][128 bytes]
    // fp32, 128-byte swizzled, two buffers
    static constexpr int STG_BYTES = D * BQ * 4;
    static constexpr int OFF_DQS = OFF_DS + DS_BYTES;
    static constexpr int DQ_BOX_ROWS = 32;                // one warp's reduce box: 32 x 32 fp32
    static constexpr int OFF_LSE = OFF_DQS + 2 * STG_BYTES;  // [2][BQ] fp32 (log2 domain)
    static constexpr int OFF_DV = OFF_LSE + 2 * BQ * 4;   // [2][BQ] fp32
    static constexpr int OFF_BAR = OFF_DV + 2 * BQ * 4;
    static constexpr int B_KV = 0;
    static constexpr int B_QFULL = 1;                     // [2]
    static constexpr int B_QEMPTY = 3;                    // [2]
    static constexpr int B_SFULL = 5;
    static constexpr int B_DPFULL = 6;
    static constexpr int B_PFULL = 7;
    static constexpr int B_DSFULL = 8;
    static constexpr int B_SFREE = 9;                     // dV of a step done: S columns free
    static constexpr int B_DQFULL = 10;                   // [2]
    static constexpr int B_DQFREE = 12;                   // [2]
    static constexpr int B_ACC = 14;
    static constexpr int B_FIN = 15;
    static constexpr int B_LSE = 16;                      // [2] LSE/D block staged (32 arrivals)
    static constexpr int B_DPFREE = 18;                   // dK of a step done: dP columns free
    static constexpr int NBAR = 19;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_S = 0;                   // BQ columns (P^T as bf16: see packed_col)
    static constexpr uint32_t TM_DP = BQ;                 // BQ columns (dS^T as bf16: see packed_col)
    static constexpr uint32_t TM_DV = 2 * BQ;             // D columns
    static constexpr uint32_t TM_DK = 2 * BQ + D;         // D columns
    static constexpr uint32_t TM_DQ = 2 * BQ + 2 * D;     // 2 x 64 columns
};

__device__ __forceinline__ void drain_wait_b(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > FA_WAIT_TIMEOUT_NS) break;
}

template <int D, bool VARLEN>
__global__ void __launch_bounds__(384, 1) fa_bwd_kernel(const __grid_constant__ BwdParams p) {
    using S = BwdShape<D>;
    constexpr int BQ = S::BQ;
    constexpr int CW = BQ / 2;                  // query columns per compute warpgroup
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // head-major order: the CTAs resident at one time share one head's Q, dO
    // and dQ accumulator in L2; within a head the causally heaviest key
    // tiles (lowest index) start first
    const int kt = (int)(blockIdx.x % p.Tk);
    const int bh = (int)(blockIdx.x / p.Tk);
    const int b = bh / p.H, h = bh % p.H;
    const int k0 = kt * kTile;
    const int nb = (p.N + kTile - 1) / kTile;

    auto bar = [&](int i) -> uint32_t { return base + S::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + S::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sb + S::OFF_MISC + 4);
    const Guard g{p.status, p.status + 1, abort_flag};

    // the sequence: query rows [q_start, q_start + Lq), key rows [k_start,
    // k_start + Lk); in the square [B, H, N, d] case both are [0, N).  Under
    // the causal mask query i sees key j iff j <= i + shift (shift = Lk - Lq,
    // 0 for the square case: a ragged sequence's queries are its last ones).
    int q_start = 0, k_start = 0, Lq = p.N, Lk = p.N, Tqb = p.Tqb;
    bool bad = false;
    if constexpr (VARLEN) {
        varlen_sequence(p.cu_q, p.cu_k, b, p.total_q, p.total_k, INT_MAX, p.Tk * kTile, &q_start, &Lq, &k_start,
                        &Lk, &bad);
        Tqb = (Lq + BQ - 1) / BQ;
    }
    const int shift = Lk - Lq;
    const int kvis = VARLEN ? Lk : key_visible_bound(p.key_len, b, p.N, &bad);
    if (bad && threadIdx.x == 0 && kt == 0 && h == 0) record_status(g, kStatusBadKeyLen, 0);
    // a ragged batch's grid covers its longest key sequence: a key tile past
    // this sequence's end has no dK, dV row to write and leaves before any
    // set-up (the whole CTA takes this branch together)
    if (VARLEN && k0 >= Lk) return;

    // class of query block qb (BQ rows) against this key tile
    auto cls = [&](int qb) -> unsigned {
        const int qa = qb * BQ;
        if constexpr (VARLEN) return tile_class_shift(qa, min(BQ, Lq - qa), k0, kTile, kvis, p.causal, shift);
        const int on = p.block_mask ? (p.block_mask[(size_t)(qa / kTile) * nb + kt] != 0) : 1;
        return tile_class(qa, min(BQ, p.N - qa), k0, kTile, kvis, p.causal, on);
    };
    // Without a block mask the query blocks that see this key tile are
    // exactly [qb_start, Tqb) (none when the tile lies past key_len): under
    // the causal mask the first block whose last row reaches k0 - shift.
    const int qb_start = bwd_query_block_begin(k0, kvis, p.causal, shift, BQ, Tqb);
    auto next_qb = [&](int qb) -> int {
        if (VARLEN || !p.block_mask) {
            const int nq = qb < qb_start ? qb_start : qb + 1;
            return nq < Tqb ? nq : Tqb;
        }
        for (int x = qb + 1; x < Tqb; ++x)
            if (cls(x) != kTileSkip) return x;
        return Tqb;
    };
    // TMA coordinates: the [B*H][N][d] view, or the [total][H][d] view of a
    // ragged batch (warp-collective: the producer warp calls it uniformly)
    auto tload = [&](uint32_t dst, const CUtensorMap *m, uint32_t mbar, int c, int row, int start) {
        if constexpr (VARLEN)
            tma_load_3d_elect(dst, m, mbar, c * 64, h, start + row);
        else
            tma_load_3d_elect(dst, m, mbar, c * 64, row, bh);
    };
    // index of query row qq of this sequence in LSE ([BH][N] or [H][total_q])
    // and in D ([BH][N] or [total_q][H])
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
            mbar_init(bar(S::B_DQFULL + s), 1);
            mbar_init(bar(S::B_DQFREE + s), 256);
            mbar_init(bar(S::B_LSE + s), 32);
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
    const int first = next_qb(-1);
    float *lse_s = reinterpret_cast<float *>(sb + S::OFF_LSE);   // [2][BQ], log2 domain
    float *dv_s = reinterpret_cast<float *>(sb + S::OFF_DV);     // [2][BQ]

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        // one elected lane issues the TMA copies; the whole warp stages LSE
        // and D of the same query block into shared memory one stage ahead.
        if (first < Tqb) {
            mbar_arrive_expect_tx_elect(bar(S::B_KV), 2 * S::KV_BYTES);
            for (int c = 0; c < S::CHUNKS; ++c) {
                tload(base + S::OFF_K + c * S::KV_CHUNK, &p.tmK, bar(S::B_KV), c, k0, k_start);
                tload(base + S::OFF_V + c * S::KV_CHUNK, &p.tmV, bar(S::B_KV), c, k0, k_start);
            }
            int i = 0;
            bool ok = true;
            for (int qb = first; qb < Tqb; qb = next_qb(qb), ++i) {
                const int s = i & 1;
                if (!mbar_wait_warp(bar(S::B_QEMPTY + s), ((uint32_t)(i >> 1) & 1u) ^ 1u, g, 0x111)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_elect(bar(S::B_QFULL + s), 2 * S::Q_BYTES);
                for (int c = 0; c < S::CHUNKS; ++c) {
                    tload(base + S::OFF_Q + s * S::Q_BYTES + c * S::Q_CHUNK, &p.tmQ, bar(S::B_QFULL + s), c, qb * BQ,
                          q_start);
                    tload(base + S::OFF_DO + s * S::Q_BYTES + c * S::Q_CHUNK, &p.tmdO, bar(S::B_QFULL + s), c,
                          qb * BQ, q_start);
                }
                // LSE in the log2 domain (+inf past the sequence's last query
                // or for a row with no visible key: its P is 0) and D for the
                // block's rows
                const int qa = qb * BQ;
                for (int t = lane; t < BQ; t += 32) {
                    const int qq = qa + t;
                    float v = INFINITY, dd = 0.f;
                    if (qq < Lq) {
                        const float L = p.LSE[lse_index(qq)];
                        v = (L == -INFINITY) ? INFINITY : L * 1.4426950408889634f;
                        dd = p.Dvec[d_index(qq)];
                    }
                    lse_s[s * BQ + t] = v;
                    dv_s[s * BQ + t] = dd;
                }
                mbar_arrive(bar(S::B_LSE + s));
            }
            if (!ok && lane == 0) {
                drain_wait_b(bar(S::B_KV), 0);
                for (int j = (i > 2 ? i - 2 : 0); j < i; ++j)
                    drain_wait_b(bar(S::B_QFULL + (j & 1)), (uint32_t)(j >> 1) & 1u);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        // Issue order, step i:  dV(i), S(i+1), dK(i), dQ(i), dP(i+1).
        // S(i+1) only needs dV(i) to have read P(i) from the S columns, and
        // dP(i+1) only needs dK(i) to have read dS(i) from the dP columns,
        // so the next step's scores are ready while the compute warps are
        // still on this step, and the tensor pipe keeps a queue.
        {
            constexpr uint32_t IDESC_S = idesc_bf16(128, BQ, false, false);   // S^T, dP^T
            constexpr uint32_t IDESC_ACC = idesc_bf16(128, D, false, true);   // dV, dK
            constexpr uint32_t IDESC_DQ = idesc_bf16(128, 64, true, true);    // dQ or dQ^T
            // shared-memory descriptors built once; per MMA only the start
            // address moves (sdesc_add)
            const uint64_t dK_kmaj = sdesc_sw128(base + S::OFF_K, 16, 1024);          // K as A, K-major
            const uint64_t dV_kmaj = sdesc_sw128(base + S::OFF_V, 16, 1024);          // V as A, K-major
            const uint64_t dQ_kmaj = sdesc_sw128(base + S::OFF_Q, 16, 1024);          // Q as B, K-major
            const uint64_t ddO_kmaj = sdesc_sw128(base + S::OFF_DO, 16, 1024);        // dO as B, K-major
            const uint64_t dQ_mn = sdesc_sw128(base + S::OFF_Q, S::Q_CHUNK, 1024);    // Q as B, MN-major
            const uint64_t ddO_mn = sdesc_sw128(base + S::OFF_DO, S::Q_CHUNK, 1024);  // dO as B, MN-major
            const uint64_t dK_mn = sdesc_sw128(base + S::OFF_K, S::KV_CHUNK, 1024);   // K (A or B), MN-major
            const uint64_t ddS_mn = sdesc_sw128(base + S::OFF_DS, 128 * 128, 1024);   // dS (A or B), MN-major
            auto issue_s = [&](int step) {       // S^T = K Q^T: M = 128 keys, N = BQ, K = D
                const uint64_t qd = sdesc_add(dQ_kmaj, (uint32_t)((step & 1) * S::Q_BYTES));
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_ss_elect(tmem + S::TM_S, sdesc_add(dK_kmaj, (k >> 2) * S::KV_CHUNK + (k & 3) * 32),
                           sdesc_add(qd, (k >> 2) * S::Q_CHUNK + (k & 3) * 32), IDESC_S, k > 0 ? 1u : 0u);
                mma_commit_elect(bar(S::B_SFULL));
            };
            auto issue_dp = [&](int step) {      // dP^T = V dO^T
                const uint64_t dd = sdesc_add(ddO_kmaj, (uint32_t)((step & 1) * S::Q_BYTES));
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_ss_elect(tmem + S::TM_DP, sdesc_add(dV_kmaj, (k >> 2) * S::KV_CHUNK + (k & 3) * 32),
                           sdesc_add(dd, (k >> 2) * S::Q_CHUNK + (k & 3) * 32), IDESC_S, k > 0 ? 1u : 0u);
                mma_commit_elect(bar(S::B_DPFULL));
            };
            // P^T and dS^T are stored as bf16 pairs by the two compute
            // warpgroups, each inside its own half of the columns (so that
            // neither overwrites fp32 values the other is still reading):
            // queries [16k, 16k + 16) sit at column (16k / CW) CW + 8 (k mod CW/16).
            auto packed_col = [](int k) -> uint32_t {
                constexpr int KW = (BQ / 2) / 16;
                return (uint32_t)((k / KW) * (BQ / 2) + 8 * (k % KW));
            };
            bool ok = true;
            int i = 0;
            if (first < Tqb) {
                ok = mbar_wait_warp(bar(S::B_KV), 0, g, 0x211) && mbar_wait_warp(bar(S::B_QFULL), 0, g, 0x212);
                if (ok) {
                    tc_fence_after();
                    issue_s(0);
                    issue_dp(0);
                }
                for (int qb = first; ok && qb < Tqb; ++i) {
                    const int s = i & 1;
                    const uint64_t q_mn = sdesc_add(dQ_mn, (uint32_t)(s * S::Q_BYTES));
                    const uint64_t do_mn = sdesc_add(ddO_mn, (uint32_t)(s * S::Q_BYTES));
                    const uint32_t acc0 = i > 0 ? 1u : 0u;
                    const int qb_next = next_qb(qb);
                    const bool more = qb_next < Tqb;
                    // dV += P^T dO: A = P^T from TMEM, B = dO (N = D, K = queries, MN-major)
                    if (!mbar_wait_warp(bar(S::B_PFULL), (uint32_t)i & 1u, g, 0x214)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < BQ / 16; ++k)
                        mma_ts_elect(tmem + S::TM_DV, tmem + S::TM_S + packed_col(k), sdesc_add(do_mn, (uint32_t)k * 2048u),
                               IDESC_ACC, k > 0 ? 1u : acc0);
                    mma_commit_elect(bar(S::B_SFREE));
                    // S(i+1) once dV(i) has read P(i)
                    if (more) {
                        if (!mbar_wait_warp(bar(S::B_QFULL + (s ^ 1)), (uint32_t)((i + 1) >> 1) & 1u, g, 0x217) ||
                            !mbar_wait_warp(bar(S::B_SFREE), (uint32_t)i & 1u, g, 0x213)) { ok = false; break; }
                        tc_fence_after();
                        issue_s(i + 1);
                    }
                    // dK += dS^T Q: A = dS^T from TMEM, B = Q (MN-major)
                    if (!mbar_wait_warp(bar(S::B_DSFULL), (uint32_t)i & 1u, g, 0x215)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < BQ / 16; ++k)
                        mma_ts_elect(tmem + S::TM_DK, tmem + S::TM_DP + packed_col(k), sdesc_add(q_mn, (uint32_t)k * 2048u),
                               IDESC_ACC, k > 0 ? 1u : acc0);
                    mma_commit_elect(bar(S::B_DPFREE));
                    mma_commit_elect(bar(S::B_QEMPTY + s));
                    // dQ contribution into TMEM buffer i % 2 (drained by the compute warps)
                    if (i >= 2 &&
                        !mbar_wait_warp(bar(S::B_DQFREE + s), (uint32_t)((i - 2) >> 1) & 1u, g, 0x216)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t dq_tmem = tmem + S::TM_DQ + 64u * (uint32_t)s;
#pragma unroll
                    for (int k = 0; k < kTile / 16; ++k) {
                        const uint64_t kk = sdesc_add(dK_mn, (uint32_t)k * 2048u);
                        const uint64_t dd = sdesc_add(ddS_mn, (uint32_t)k * 2048u);
                        // dQ = dS K: A = dS (M = queries), B = K (N = d)
                        mma_ss_elect(dq_tmem, dd, kk, IDESC_DQ, k > 0 ? 1u : 0u);
                    }
                    mma_commit_elect(bar(S::B_DQFULL + s));
                    // dP(i+1) once dK(i) has read dS(i)
                    if (more) {
                        if (!mbar_wait_warp(bar(S::B_DPFREE), (uint32_t)i & 1u, g, 0x218)) { ok = false; break; }
                        tc_fence_after();
                        issue_dp(i + 1);
                    }
                    qb = qb_next;
                }
                if (ok) mma_commit_elect(bar(S::B_ACC));
            }
            mma_commit_elect(bar(S::B_FIN));
            drain_wait_b(bar(S::B_FIN), 0);
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------- compute (two warpgroups)
        // Warpgroup wg handles query columns [wg*CW, wg*CW + CW) of S^T and
        // dP^T (the backward needs no row reduction, so the halves are
        // independent), half of the dQ drain and half of the dK/dV columns.
        const int wg = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;           // TMEM lane: key row (S^T, dP^T, dK, dV), query/dim row (dQ)
        const int key = k0 + r;
        const int c0 = wg * CW;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const float c2 = p.scale_log2;
        bool ok = true;
        int i = 0, prev_qb = -1;

        // drain this warpgroup's half of step j's dQ contribution (query
        // block qb): TMEM -> swizzled shared staging -> per-warp TMA
        // reduce-add (box 32 x 32) into the fp32 accumulator
        auto drain_dq = [&](int j, int qb) -> bool {
            if (!mbar_wait_warp(bar(S::B_DQFULL + (j & 1)), (uint32_t)(j >> 1) & 1u, g, 0x411)) return false;
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + S::TM_DQ + 64u * (uint32_t)(j & 1) + 32u * wg, v);
            tmem_ld_wait(v);
            tc_fence_before();
            mbar_arrive(bar(S::B_DQFREE + (j & 1)));
            uint8_t *stg = sb + S::OFF_DQS + (j & 1) * S::STG_BYTES;
            // the reduce issued from this buffer two drains ago must have read it
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            uint32_t box;             // shared address of this warp's 32 x 32 box
            int cx, cy;               // its coordinates (head dimension, query)
            {
                // lane = query row r of the block, columns = head dimensions 32*wg .. 32*wg + 31
                uint8_t *cb = stg + wg * (BQ * 128) + r * 128;
#pragma unroll
                for (int gq = 0; gq < 8; ++gq)
                    *reinterpret_cast<uint4 *>(cb + ((gq ^ (r & 7)) << 4)) =
                        make_uint4(v[4 * gq], v[4 * gq + 1], v[4 * gq + 2], v[4 * gq + 3]);
                box = smem_u32(stg + wg * (BQ * 128) + wq * 32 * 128);
                cx = wg * 32;
                cy = qb * BQ + wq * 32;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if constexpr (VARLEN)
                    tma_reduce_add_3d(&p.tmdQ, box, cx, h, q_start + cy);
                else
                    tma_reduce_add_3d(&p.tmdQ, box, cx, cy, bh);
                bulk_commit_group();
            }
            return true;
        };

        for (int qb = first; qb < Tqb; qb = next_qb(qb), ++i) {
            const unsigned klass = cls(qb);
            const int qa = qb * BQ;
            if (!mbar_wait_warp(bar(S::B_LSE + (i & 1)), (uint32_t)(i >> 1) & 1u, g, 0x410)) { ok = false; break; }
            const float *ls = lse_s + (i & 1) * BQ;
            const float *dd = dv_s + (i & 1) * BQ;

            // P^T = 2^(s * c - LSE_q * log2 e), masked, for columns c0 .. c0 + CW
            if (!mbar_wait_warp(bar(S::B_SFULL), (uint32_t)i & 1u, g, 0x412)) { ok = false; break; }
            tc_fence_after();
            uint32_t pk[CW / 2];
            {
                uint32_t sr[CW / 32][32];
#pragma unroll
                for (int j = 0; j < CW / 32; ++j) tmem_ld32(tmem + lane_off + S::TM_S + c0 + 32u * j, sr[j]);
#pragma unroll
                for (int j = 0; j < CW / 32; ++j) tmem_ld_wait(sr[j]);
                if (klass == kTilePartial) {
                    // masked scores -> -inf, so that their p is exactly 0 (a mask
                    // test inside the exp loop below made that loop several times slower)
#pragma unroll
                    for (int j = 0; j < CW / 32; ++j)
#pragma unroll
                        for (int t = 0; t < 32; ++t) {
                            const int qq = qa + c0 + 32 * j + t;
                            if (key >= kvis || (p.causal && key > qq + shift)) sr[j][t] = __float_as_uint(-INFINITY);
                        }
                }
#pragma unroll
                for (int j = 0; j < CW / 32; ++j)
#pragma unroll
                    for (int t = 0; t < 32; t += 2) {
                        const int cq = c0 + 32 * j + t;          // query column within the block
                        const float2 l2 = *reinterpret_cast<const float2 *>(ls + cq);
                        float p0, p1;
                        fma2(p0, p1, __uint_as_float(sr[j][t]), __uint_as_float(sr[j][t + 1]), c2, c2, -l2.x, -l2.y);
                        pk[16 * j + t / 2] = pack_bf16x2(ex2(p0), ex2(p1));
                    }
            }
#pragma unroll
            for (int j = 0; j < CW / 32; ++j) tmem_st16(tmem + lane_off + S::TM_S + c0 + 16u * j, pk + 16 * j);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(S::B_PFULL));

            // dS^T = P^T o (dP^T - D): bf16 into TMEM (for dK) and shared memory (for dQ)
            if (!mbar_wait_warp(bar(S::B_DPFULL), (uint32_t)i & 1u, g, 0x413)) { ok = false; break; }
            // the dQ MMA of the previous step must be done reading the shared dS tile
            if (i > 0 && !mbar_wait_warp(bar(S::B_DQFULL + ((i - 1) & 1)), (uint32_t)((i - 1) >> 1) & 1u, g, 0x414)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint8_t *ds_smem = sb + S::OFF_DS;
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
                    for (int t = 0; t < 16; ++t) {
                        const int cq = c0 + 32 * j + 2 * t;
                        const uint32_t pp = pk[16 * j + t];
                        const float2 d2 = *reinterpret_cast<const float2 *>(dd + cq);
                        const float d0 = __uint_as_float(dp[j][2 * t]) - d2.x;
                        const float d1 = __uint_as_float(dp[j][2 * t + 1]) - d2.y;
                        w[t] = pack_bf16x2(bf16lo(pp) * d0, bf16hi(pp) * d1);
                    }
                    tmem_st16(tmem + lane_off + S::TM_DP + c0 + 16u * j, w);
                    // shared dS tile, queries contiguous (MN-major, 128-byte swizzle):
                    // [query chunk of 64][key row 0..127][128 bytes]
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int qo = c0 + 32 * j + 8 * u;        // first query of this 16-byte piece
                        const int grp = (qo & 63) >> 3;
                        uint8_t *dst = ds_smem + (qo >> 6) * (128 * 128) + r * 128 + ((grp ^ (r & 7)) << 4);
                        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                    }
                }
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(S::B_DSFULL));

            // drain the previous step's dQ while the tensor cores work on this one
            if (i > 0 && !drain_dq(i - 1, prev_qb)) { ok = false; break; }
            prev_qb = qb;
        }
        if (ok && i > 0) ok = drain_dq(i - 1, prev_qb);
        // the staged dQ tiles must be fully reduced before shared memory goes away
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();

        // ---------------------------------------------------------- epilogue: dK, dV
        // warpgroup wg converts head-dimension columns [wg*D/2, wg*D/2 + D/2)
        if (ok && i > 0) {
            ok = mbar_wait_warp(bar(S::B_ACC), 0, g, 0x415);
            tc_fence_after();
        }
        if (ok) {
            // the TMEM loads are warp-collective: every lane loads, only rows < N store
            const size_t krow = VARLEN ? (size_t)(k_start + key) * p.H + h : (size_t)bh * p.N + key;
            __nv_bfloat16 *dkrow = reinterpret_cast<__nv_bfloat16 *>(p.dK) + krow * D;
            __nv_bfloat16 *dvrow = reinterpret_cast<__nv_bfloat16 *>(p.dV) + krow * D;
#pragma unroll 1
            for (int j = wg * (D / 64); j < (wg + 1) * (D / 64); ++j) {
                uint32_t a[32], v[32];
                if (i > 0) {
                    tmem_ld32(tmem + lane_off + S::TM_DK + 32u * j, a);
                    tmem_ld32(tmem + lane_off + S::TM_DV + 32u * j, v);
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
                if (key < Lk) {
                    uint4 *dk4 = reinterpret_cast<uint4 *>(dkrow + 32 * j);
                    uint4 *dv4 = reinterpret_cast<uint4 *>(dvrow + 32 * j);
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        dk4[t] = make_uint4(wk[4 * t], wk[4 * t + 1], wk[4 * t + 2], wk[4 * t + 3]);
                        dv4[t] = make_uint4(wv[4 * t], wv[4 * t + 1], wv[4 * t + 2], wv[4 * t + 3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, S::TMEM_COLS);
}

// D = rowsum(dO * O) in fp32 and dQacc = 0, one warp per row.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const __nv_bfloat16 *__restrict__ O,
                                                         const __nv_bfloat16 *__restrict__ dO,
                                                         float *__restrict__ Dvec, float *__restrict__ dQacc,
                                                         int64_t rows) {
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    constexpr int PER = D / 32;   // elements per lane: 2 or 4
    float acc = 0.f;
    if (PER == 4) {
        const uint2 o = reinterpret_cast<const uint2 *>(O + row * D)[lane];
        const uint2 g = reinterpret_cast<const uint2 *>(dO + row * D)[lane];
        acc = bf16lo(o.x) * bf16lo(g.x) + bf16hi(o.x) * bf16hi(g.x) + bf16lo(o.y) * bf16lo(g.y) +
              bf16hi(o.y) * bf16hi(g.y);
        reinterpret_cast<float4 *>(dQacc + row * D)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        const uint32_t o = reinterpret_cast<const uint32_t *>(O + row * D)[lane];
        const uint32_t g = reinterpret_cast<const uint32_t *>(dO + row * D)[lane];
        acc = bf16lo(o) * bf16lo(g) + bf16hi(o) * bf16hi(g);
        reinterpret_cast<float2 *>(dQacc + row * D)[lane] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) Dvec[row] = acc;
}

// dQ = bf16(scale * dQacc), 8 elements per thread.
__global__ void __launch_bounds__(256) fa_bwd_convert_kernel(const float *__restrict__ acc,
                                                             __nv_bfloat16 *__restrict__ dQ, int64_t n8,
                                                             float scale) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = reinterpret_cast<const float4 *>(acc)[2 * i];
        const float4 c = reinterpret_cast<const float4 *>(acc)[2 * i + 1];
        reinterpret_cast<uint4 *>(dQ)[i] =
            make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                       pack_bf16x2(c.x * scale, c.y * scale), pack_bf16x2(c.z * scale, c.w * scale));
    }
}

// Tile plan export: the tile_class the attention kernels take their full /
// partial decisions with, checked against the visit rules the kernels skip
// tiles with.  With a block mask the kernels visit exactly the tiles whose
// class is not skip; without one the forward visits the key tiles below
// fwd_key_tile_end and the backward the query blocks from
// bwd_query_block_begin.  A tile on which either rule disagrees with its
// class is exported as kTileRuleMismatch, which no correct plan contains.
__global__ void fa_plan_kernel(int B, int N, int T, int causal, const int32_t *key_len,
                               const uint8_t *block_mask, uint8_t *plan, unsigned *status) {
    const int64_t n = (int64_t)B * T * T;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int kt = (int)(idx % T);
        const int qt = (int)((idx / T) % T);
        const int b = (int)(idx / ((int64_t)T * T));
        bool bad = false;
        const int kvis = key_visible_bound(key_len, b, N, &bad);
        if (bad && qt == 0 && kt == 0 && atomicCAS(status, 0u, kStatusBadKeyLen) == 0u) atomicExch(status + 1, 0u);
        const int on = block_mask ? (block_mask[(size_t)qt * T + kt] != 0) : 1;
        const int q0 = qt * kTile, qn = min(kTile, N - q0);
        const unsigned c = tile_class(q0, qn, kt * kTile, kTile, kvis, causal, on);
        bool fwd_visits = c != kTileSkip, bwd_visits = c != kTileSkip;
        if (!block_mask) {
            fwd_visits = kt < fwd_key_tile_end(q0, qn, kvis, causal, 0, kTile);
            bwd_visits = qt >= bwd_query_block_begin(kt * kTile, kvis, causal, 0, kTile, T);
        }
        const bool agree = fwd_visits == (c != kTileSkip) && bwd_visits == (c != kTileSkip);
        plan[idx] = (uint8_t)(agree ? c : kTileRuleMismatch);
    }
}

// d = 128 runs fa_bwd128_kernel (128-row query blocks)
int bwd_query_block(int d) { return d == 64 ? BwdShape<64>::BQ : 128; }
int bwd_dq_box_rows(int) { return BwdShape<64>::DQ_BOX_ROWS; }   // fa_bwd128.cu uses the same 32 x 32 boxes
int bwd_smem_bytes(int d) { return d == 64 ? BwdShape<64>::SMEM_BYTES : bwd128_smem_bytes(); }

template <int D, bool VARLEN>
static cudaError_t launch_bwd_main_t(const BwdParams &p, cudaStream_t st) {
    const int smem = BwdShape<D>::SMEM_BYTES;
    cudaError_t e =
        cudaFuncSetAttribute(fa_bwd_kernel<D, VARLEN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    fa_bwd_kernel<D, VARLEN><<<(unsigned)p.Tk * (unsigned)p.BH, 384, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_main(int d, const BwdParams &p, cudaStream_t st) {
    return d == 64 ? launch_bwd_main_t<64, false>(p, st) : launch_bwd128_main(p, st);
}

cudaError_t launch_bwd_main_varlen(int d, const BwdParams &p, cudaStream_t st) {
    return d == 64 ? launch_bwd_main_t<64, true>(p, st) : launch_bwd128_main_varlen(p, st);
}

cudaError_t launch_bwd_pre(int d, const void *O, const void *dO, float *Dvec, float *dQacc, int64_t rows,
                           cudaStream_t st) {
    const unsigned grid = (unsigned)((rows + 7) / 8);
    if (d == 64)
        fa_bwd_pre_kernel<64><<<grid, 256, 0, st>>>((const __nv_bfloat16 *)O, (const __nv_bfloat16 *)dO, Dvec,
                                                    dQacc, rows);
    else
        fa_bwd_pre_kernel<128><<<grid, 256, 0, st>>>((const __nv_bfloat16 *)O, (const __nv_bfloat16 *)dO, Dvec,
                                                     dQacc, rows);
    return cudaGetLastError();
}

cudaError_t launch_bwd_convert(int d, const float *dQacc, void *dQ, int64_t elems, float scale,
                               cudaStream_t st) {
    (void)d;
    const int64_t n8 = elems / 8;
    int64_t blocks = (n8 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    fa_bwd_convert_kernel<<<(unsigned)blocks, 256, 0, st>>>(dQacc, (__nv_bfloat16 *)dQ, n8, scale);
    return cudaGetLastError();
}

cudaError_t launch_plan(int B, int N, int causal, const int32_t *key_len, const uint8_t *block_mask,
                        uint8_t *plan, unsigned *status, cudaStream_t st) {
    const int T = (N + kTile - 1) / kTile;
    const int64_t n = (int64_t)B * T * T;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    fa_plan_kernel<<<(unsigned)blocks, 256, 0, st>>>(B, N, T, causal, key_len, block_mask, plan, status);
    return cudaGetLastError();
}

}  // namespace fa
