// fa_fwd_fp8.cu -- FP8 forward (d = 128): exact attention of block-quantised
// e4m3 Q, K, V with both products on the FP8 tensor cores.
//
// "FlashAttention: Mathematical Foundations ...", section "Architectural
// Evolution" (FlashAttention-3 paragraph): block-quantised FP8 matmuls with
// dynamic scaling.  Q, K and V^T arrive as e4m3 codes with one fp32 scale per
// 128-row block (fa_quant.cu).  The score of the (query block i, key block
// j) tile is scale * sQ_i * sK_j * (q8 . k8): the softmax multiplier becomes
// c * sQ_i * sK_j per tile.  The online softmax is the forward kernel's
// ("The Attention Matrix You Never Write Down", "The running-statistics
// trick"; base 2; reference maximum moved only when a row outgrows it by
// 2^8).  P is rounded to e4m3 for the P.V product; V's block scale sV_j is
// folded into it as P * (sV_j / max_j sV_j) (at most 1, so P stays <= 2^8,
// inside e4m3's range; the factor goes into the exponent) and the head's
// max_j sV_j multiplies O in the epilogue; l sums the unrounded p.
//
// What differs from the bf16 forward: with e4m3 operands the two MMAs of a
// tile take half as long, so the per-tile chain S -> softmax -> P -> P.V
// would leave the tensor pipe idle most of the time if P overwrote S in
// TMEM (the next S could only start once P.V had read P).  Here P goes to
// shared memory instead (16 KB per tile in e4m3, double-buffered per query
// tile), and the softmax warps release S as soon as they have loaded it into
// registers, so the next tile's S = Q K^T runs while they compute:
//   - one CTA per (pair of 128-row query tiles, b*h), head-major;
//   - warp 0: TMA of both Q tiles once, K and V^T tiles through a 3-stage
//     ring;
//   - warps 1 and 2: tcgen05 issuers, one per query tile x, so that one
//     tile's chain never waits on the other's softmax.  Per key tile i:
//     S_x(i+1) = Q_x K(i+1)^T as soon as softmax x has loaded S_x(i)
//     (SFREE), then O_x += P_x(i) V(i) (A = P_x from shared memory, B = V^T,
//     both K-major) once P_x(i) is written (PFULL).  A K/V stage is free
//     once both issuers are done with it (two arrivals);
//   - warps 4-7 and 8-11: softmax of query tile 0 and 1, one row per
//     thread; P rows go to shared memory in the 128-byte-swizzled K-major
//     layout the MMA reads.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

namespace {

constexpr float kRescaleLog2F8 = 8.0f;

struct F8Shape {
    static constexpr int D = 128;
    static constexpr int TILE_BYTES = 128 * 128;            // 128 rows x 128 bytes (e4m3)
    static constexpr int STAGES = 3;
    static constexpr int OFF_Q = 0;                         // [2] query tiles
    static constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;    // [STAGES]
    static constexpr int OFF_V = OFF_K + STAGES * TILE_BYTES;
    static constexpr int OFF_P = OFF_V + STAGES * TILE_BYTES;  // [2 query tiles][2 buffers]
    static constexpr int OFF_BAR = OFF_P + 4 * TILE_BYTES;
    static constexpr int B_QFULL = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_VFULL = B_KFULL + STAGES;
    static constexpr int B_KVEMPTY = B_VFULL + STAGES;
    static constexpr int B_SFULL = B_KVEMPTY + STAGES;      // [2] per query tile
    static constexpr int B_SFREE = B_SFULL + 2;             // [2]
    // P_x is written ahead of the P.V products, so its ready barrier is kept
    // per P buffer: a softmax warp refills a buffer only after the product
    // that read it, so the issuer is never two phases behind on one barrier
    static constexpr int B_PFULL = B_SFREE + 2;             // [2][2] per query tile and P buffer
    static constexpr int B_PFREE = B_PFULL + 4;             // [2][2]
    static constexpr int B_OFULL = B_PFREE + 4;             // [2] every product done (single use)
    static constexpr int B_FIN = B_OFULL + 2;               // [2] per issuer
    static constexpr int NBAR = B_FIN + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_S = 0;                     // S_x at columns 128 x
    static constexpr uint32_t TM_O = 256;                   // O_x at columns 256 + 128 x
    static constexpr int THREADS = 384;
    static constexpr int LAUNCH_REGS = 168;
    static constexpr int REGS_CTRL = 104;
    static constexpr int REGS_SOFTMAX = 200;
    static_assert(128 * REGS_CTRL + 256 * REGS_SOFTMAX == THREADS * LAUNCH_REGS, "register split");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ void f8_drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > FA_WAIT_TIMEOUT_NS) break;
}

template <bool PLAIN>
__global__ void __launch_bounds__(384, 1) fa_fwd_fp8_kernel(const __grid_constant__ FwdParams p) {
    grid_dep_wait();                                 // the previous kernel in the stream is done
    grid_dep_launch();
    using S = F8Shape;
    constexpr int D = S::D;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int Tp = (p.Tq + 1) / 2;
    const int nb = (p.N + kTile - 1) / kTile;
    // the item (query-tile pair, b*h) of this CTA; from split_from on (every
    // tile full), part `part` of an item run as split_f CTAs, each over its own
    // range of key tiles (the last wave's items, so that it fills the SMs).
    // split_part: -1 for a whole item, else the part; *sidx: the split item's
    // index past split_from.  Recomputed where needed rather than kept live.
    auto split_part = [&](int *sidx) -> int {
        const int j = (int)blockIdx.x - p.split_from;
        if (!PLAIN || p.split_f < 2 || j < 0) return -1;
        *sidx = j / p.split_f;
        return j - *sidx * p.split_f;
    };
    int item = (int)blockIdx.x;
    int khi = 0;                                     // a part's key tiles end here (0: whole item)
    {
        int si = 0;
        const int part = split_part(&si);
        if (part >= 0) {
            item = p.split_from + si;
            khi = (part + 1) * nb / p.split_f;
        }
    }
    const int pq = Tp - 1 - item % Tp;
    const int bh = item / Tp;
    const int b = bh / p.H;
    int q0[2], qn[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        q0[x] = (2 * pq + x) * kTile;
        qn[x] = max(0, min(kTile, p.N - q0[x]));
    }

    auto bar = [&](int i) -> uint32_t { return base + S::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + S::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sb + S::OFF_MISC + 4);
    const Guard g{p.status, p.status + 1, abort_flag};

    bool bad = false;
    const int kvis = key_visible_bound(p.key_len, b, p.N, &bad);
    if (bad && threadIdx.x == 0 && pq == 0 && (bh % p.H) == 0) record_status(g, kStatusBadKeyLen, 0);

    int kend[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        int lim = kvis;
        if (p.causal) lim = min(lim, q0[x] + qn[x]);
        kend[x] = qn[x] > 0 ? (lim + kTile - 1) / kTile : 0;
        // a split part's key tiles end at khi; an empty query tile (the
        // second of the last pair when the tile count is odd) keeps none
        if (PLAIN && khi > 0 && qn[x] > 0) kend[x] = khi;
    }
    const int kend_union = max(kend[0], kend[1]);
    // per-query-tile values by selection, so that the arrays stay in registers
    auto q0_of = [&](int x) { return x ? q0[1] : q0[0]; };
    auto qn_of = [&](int x) { return x ? qn[1] : qn[0]; };
    auto kend_of = [&](int x) { return x ? kend[1] : kend[0]; };
    // PLAIN: no causal mask, key padding or block mask, N a multiple of 128:
    // every visible tile is full and the masking code is not compiled
    auto cls = [&](int x, int kt) -> unsigned {
        if (qn_of(x) <= 0) return kTileSkip;
        if constexpr (PLAIN) return kTileFull;
        const int on = p.block_mask ? (p.block_mask[(size_t)(2 * pq + x) * nb + kt] != 0) : 1;
        return tile_class(q0_of(x), qn_of(x), kt * kTile, kTile, kvis, p.causal, on);
    };
    // without a block mask the visible tiles of query tile x are 0 .. kend[x]-1
    auto skip = [&](int x, int kt) -> bool {
        return (!PLAIN && p.block_mask) ? cls(x, kt) == kTileSkip : kt >= kend_of(x);
    };
    auto next_tile = [&](int x, int kt) -> int {
        if (PLAIN || !p.block_mask) {
            const int lim = x == 2 ? kend_union : kend_of(x);
            return kt + 1 < lim ? kt + 1 : p.Tk;
        }
        for (int k = kt + 1; k < p.Tk; ++k) {
            const bool v0 = (x != 1) && cls(0, k) != kTileSkip;
            const bool v1 = (x != 0) && cls(1, k) != kTileSkip;
            if (v0 || v1) return k;
        }
        return p.Tk;
    };
    // the first tile of query tile x (x = 2: of either): a split part starts
    // at its own first key tile (computed here, at the loops' entry, so that
    // the per-tile next_tile keeps no extra value live)
    auto first_tile = [&](int x) -> int {
        if constexpr (PLAIN) {
            int si = 0;
            const int part = split_part(&si);
            if (part >= 0) {
                const int k = part * nb / p.split_f;
                return k < (x == 2 ? kend_union : kend_of(x)) ? k : p.Tk;
            }
        }
        return next_tile(x, -1);
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(S::B_QFULL), 1);
        for (int s = 0; s < S::STAGES; ++s) {
            mbar_init(bar(S::B_KFULL + s), 1);
            mbar_init(bar(S::B_VFULL + s), 1);
            mbar_init(bar(S::B_KVEMPTY + s), 2);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(bar(S::B_SFULL + j), 1);
            mbar_init(bar(S::B_SFREE + j), 128);
        }
        for (int j = 0; j < 4; ++j) {
            mbar_init(bar(S::B_PFULL + j), 128);
            mbar_init(bar(S::B_PFREE + j), 1);
        }
        mbar_init(bar(S::B_OFULL + 0), 1);
        mbar_init(bar(S::B_OFULL + 1), 1);
        mbar_init(bar(S::B_FIN + 0), 1);
        mbar_init(bar(S::B_FIN + 1), 1);
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

    if (warp < 4) {
        setmaxnreg_dec<S::REGS_CTRL>();
        if (warp == 0) {
            // ---------------------------------------------------------- producer
            {
                int u = 0;
                bool ok = true;
                int kt = first_tile(2);
                if (kt < p.Tk) {
                    const uint32_t nq = (qn[0] > 0 ? 1u : 0u) + (qn[1] > 0 ? 1u : 0u);
                    mbar_arrive_expect_tx_elect(bar(S::B_QFULL), nq * S::TILE_BYTES);
#pragma unroll
                    for (int x = 0; x < 2; ++x)
                        if (qn[x] > 0)
                            tma_load_3d_elect(base + S::OFF_Q + x * S::TILE_BYTES, &p.tmQ, bar(S::B_QFULL), 0, q0[x], bh);
                }
                for (; kt < p.Tk; kt = next_tile(2, kt), ++u) {
                    const int s = u % S::STAGES;
                    const uint32_t ph = (uint32_t)(u / S::STAGES) & 1u;
                    if (!mbar_wait_warp(bar(S::B_KVEMPTY + s), ph ^ 1u, g, 0x111)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_elect(bar(S::B_KFULL + s), S::TILE_BYTES);
                    tma_load_3d_elect(base + S::OFF_K + s * S::TILE_BYTES, &p.tmK, bar(S::B_KFULL + s), 0, kt * kTile, bh);
                    mbar_arrive_expect_tx_elect(bar(S::B_VFULL + s), S::TILE_BYTES);
                    tma_load_3d_elect(base + S::OFF_V + s * S::TILE_BYTES, &p.tmV, bar(S::B_VFULL + s), kt * kTile, 0, bh);
                }
                if (!ok) {
                    if (first_tile(2) < p.Tk) f8_drain_wait(bar(S::B_QFULL), 0);
                    for (int i = (u > S::STAGES ? u - S::STAGES : 0); i < u; ++i) {
                        const int s = i % S::STAGES;
                        const uint32_t ph = (uint32_t)(i / S::STAGES) & 1u;
                        f8_drain_wait(bar(S::B_KFULL + s), ph);
                        f8_drain_wait(bar(S::B_VFULL + s), ph);
                    }
                }
            }
        } else if (warp == 1 || warp == 2) {
            // ---------------------------------------------------------- MMA issuer of query tile x
            {
                const int x = warp - 1;
                constexpr uint32_t IDESC_S = idesc_e4m3(128, 128);
                constexpr uint32_t IDESC_PV = idesc_e4m3(128, D);
                const uint64_t dq = sdesc_add(sdesc_sw128(base + S::OFF_Q, 16, 1024), (uint32_t)(x * S::TILE_BYTES));
                const uint64_t dk0 = sdesc_sw128(base + S::OFF_K, 16, 1024);
                const uint64_t dv0 = sdesc_sw128(base + S::OFF_V, 16, 1024);
                const uint64_t dp = sdesc_add(sdesc_sw128(base + S::OFF_P, 16, 1024), (uint32_t)(2 * x * S::TILE_BYTES));
                const uint32_t s_tm = tmem + S::TM_S + 128u * (uint32_t)x;
                const uint32_t o_tm = tmem + S::TM_O + (uint32_t)(D * x);
                int nv = 0, ns = 0;
                bool ok = true;
                auto issue_s = [&](int s) {
                    const uint64_t kd = sdesc_add(dk0, (uint32_t)(s * S::TILE_BYTES));
#pragma unroll
                    for (int k = 0; k < D / 32; ++k)
                        mma_ss_f8_elect(s_tm, sdesc_add(dq, 32u * k), sdesc_add(kd, 32u * k), IDESC_S, k > 0 ? 1u : 0u);
                    mma_commit_elect(bar(S::B_SFULL + x));
                    ++ns;
                };
                int kt = first_tile(2);
                if (kt < p.Tk) {
                    ok = mbar_wait_warp(bar(S::B_QFULL), 0, g, 0x211) && mbar_wait_warp(bar(S::B_KFULL + 0), 0, g, 0x212);
                    if (ok && !skip(x, kt)) {
                        tc_fence_after();
                        issue_s(0);
                    }
                }
                int u = 0;
                while (ok && kt < p.Tk) {
                    const int s = u % S::STAGES;
                    const int kt_next = next_tile(2, kt);
                    if (kt_next < p.Tk && !skip(x, kt_next)) {
                        const int s2 = (u + 1) % S::STAGES;
                        if (!mbar_wait_warp(bar(S::B_KFULL + s2), (uint32_t)((u + 1) / S::STAGES) & 1u, g, 0x213) ||
                            (ns > 0 && !mbar_wait_warp(bar(S::B_SFREE + x), (uint32_t)(ns - 1) & 1u, g, 0x214))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_s(s2);
                    }
                    if (!skip(x, kt)) {
                        if (!mbar_wait_warp(bar(S::B_PFULL + 2 * x + (nv & 1)), (uint32_t)(nv >> 1) & 1u, g, 0x215) ||
                            !mbar_wait_warp(bar(S::B_VFULL + s), (uint32_t)(u / S::STAGES) & 1u, g, 0x216)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const int pb = nv & 1;
                        const uint64_t pd = sdesc_add(dp, (uint32_t)(pb * S::TILE_BYTES));
                        const uint64_t vd = sdesc_add(dv0, (uint32_t)(s * S::TILE_BYTES));
                        const uint32_t acc0 = nv > 0 ? 1u : 0u;
#pragma unroll
                        for (int k = 0; k < kTile / 32; ++k)
                            mma_ss_f8_elect(o_tm, sdesc_add(pd, 32u * k), sdesc_add(vd, 32u * k), IDESC_PV,
                                            k > 0 ? 1u : acc0);
                        mma_commit_elect(bar(S::B_PFREE + 2 * x + pb));
                        ++nv;
                        mma_commit_elect(bar(S::B_KVEMPTY + s));
                    } else {
                        // no product of this query tile reads the stage: release it, but
                        // only once the stage holds this use, so that the arrival counts
                        // towards this use's phase and not an earlier one
                        if (!mbar_wait_warp(bar(S::B_KFULL + s), (uint32_t)(u / S::STAGES) & 1u, g, 0x217)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) mbar_arrive(bar(S::B_KVEMPTY + s));
                        __syncwarp();
                    }
                    kt = kt_next;
                    ++u;
                }
                if (ok) mma_commit_elect(bar(S::B_OFULL + x));
                mma_commit_elect(bar(S::B_FIN + x));
                f8_drain_wait(bar(S::B_FIN + x), 0);
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
        // this thread's row of the P buffers (128-byte swizzle: 16-byte unit
        // c of row r sits at unit c ^ (r % 8))
        uint8_t *prow = sb + S::OFF_P + (2 * x) * S::TILE_BYTES + (r >> 3) * 1024 + (r & 7) * 128;
        const int sw = r & 7;
        const float c2 = p.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        float sq = 1.f;
        if (qnx > 0) sq = p.sQ[(size_t)bh * p.Tq + 2 * pq + x];
        float mv = 0.f;
        for (int k = lane; k < p.Tk; k += 32) mv = fmaxf(mv, p.sV[(size_t)bh * p.Tk + k]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
        const float sv_max = mv, inv_sv_max = mv > 0.f ? 1.f / mv : 0.f;
        int it = 0;
        bool ok = true;
        // per-tile block scales, loaded one tile ahead so their latency hides
        // behind the previous tile's work
        const float *sKh = p.sK + (size_t)bh * p.Tk, *sVh = p.sV + (size_t)bh * p.Tk;
        int kt = first_tile(x);
        float sk_n = 0.f, sv_n = 0.f;
        if (kt < p.Tk) {
            sk_n = sKh[kt];
            sv_n = sVh[kt];
        }
        for (; kt < p.Tk; ++it) {
            const bool partial = !PLAIN && cls(x, kt) == kTilePartial;
            const int k0 = kt * kTile;
            const int kt_next = next_tile(x, kt);
            // multiplier of this tile's scores; V-scale ratio rt folded into
            // the exponent (p * rt = 2^(x - m + log2 rt)), and l takes the
            // tile's sum back divided by rt.  rt = 0 only for an all-zero V
            // block, whose codes make P irrelevant: there p itself is stored.
            const float ct = c2 * sq * sk_n;
            const float rt = sv_n * inv_sv_max;
            const float lg = rt > 0.f ? __log2f(rt) : 0.f;
            const float inv_rt = rt > 0.f ? 1.f / rt : 1.f;
            if (kt_next < p.Tk) {
                sk_n = sKh[kt_next];
                sv_n = sVh[kt_next];
            }
            if (!mbar_wait_warp(bar(S::B_SFULL + x), (uint32_t)it & 1u, g, 0x411)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_ld32(s_tmem + 32u * j, sr[j]);
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_ld_wait(sr[j]);
            // S_x is in registers: the next tile's S_x may overwrite it
            tc_fence_before();
            mbar_arrive(bar(S::B_SFREE + x));
            if (partial) {
                // this row sees keys k0 .. k0 + lim - 1: one compare against a
                // constant per score
                int lim = kvis - k0;
                if (p.causal) lim = min(lim, q + 1 - k0);
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        if (32 * j + t >= lim) sr[j][t] = __float_as_uint(-INFINITY);
            }
            float pm[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) pm[u] = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int t = 0; t < 32; t += 4) {
                    const int u = (j * 8 + t / 4) & 7;
                    pm[u] = fmax3(pm[u], __uint_as_float(sr[j][t]), __uint_as_float(sr[j][t + 1]));
                    pm[u] = fmax3(pm[u], __uint_as_float(sr[j][t + 2]), __uint_as_float(sr[j][t + 3]));
                }
            const float mx = fmaxf(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], fmax3(pm[5], pm[6], pm[7])));
            const float m_tile = mx * ct;
            const bool grow = m_tile > m_ref + kRescaleLog2F8;
            float alpha = 1.f;
            const bool rescale = __any_sync(0xffffffffu, grow);
            if (rescale) {
                const float m_new = fmaxf(m_ref, m_tile);
                alpha = (m_new == -INFINITY) ? 1.f : ex2(m_ref - m_new);
                l *= alpha;
                m_ref = m_new;
            }
            const float m_use = ((m_ref == -INFINITY) ? 0.f : m_ref) - lg;
            // the P buffer of this tile was last read by the P.V two tiles back
            const int pb = it & 1;
            if (it >= 2 &&
                !mbar_wait_warp(bar(S::B_PFREE + 2 * x + pb), (uint32_t)((it >> 1) - 1) & 1u, g, 0x412)) {
                ok = false;
                break;
            }
            uint8_t *pdst = prow + pb * S::TILE_BYTES;
            float ps[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) ps[u] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t pk[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    float a0, a1, a2, a3;
                    fma2(a0, a1, __uint_as_float(sr[j][4 * t]), __uint_as_float(sr[j][4 * t + 1]), ct, ct, -m_use,
                         -m_use);
                    fma2(a2, a3, __uint_as_float(sr[j][4 * t + 2]), __uint_as_float(sr[j][4 * t + 3]), ct, ct, -m_use,
                         -m_use);
                    a0 = ex2(a0);
                    a1 = ex2(a1);
                    a2 = ex2(a2);
                    a3 = ex2(a3);
                    add2(ps[2 * (t & 3)], ps[2 * (t & 3) + 1], a0, a1);
                    add2(ps[2 * ((t + 2) & 3)], ps[2 * ((t + 2) & 3) + 1], a2, a3);
                    pk[t] = pack_e4m3x4(a0, a1, a2, a3);
                }
                // keys 32j .. 32j+31 are 16-byte units 2j and 2j+1 of the row
                *reinterpret_cast<uint4 *>(pdst + (((2 * j) ^ sw) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4 *>(pdst + (((2 * j + 1) ^ sw) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
            l += (((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]))) * inv_rt;
            if (rescale && it > 0) {
                // O_x may be rescaled only once the previous P.V has landed:
                // that product freed P buffer (it - 1) & 1
                if (!mbar_wait_warp(bar(S::B_PFREE + 2 * x + ((it - 1) & 1)), (uint32_t)((it - 1) >> 1) & 1u, g,
                                    0x413)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int j0 = 0; j0 < D / 32; j0 += 4) {
                    uint32_t o[4][32];
#pragma unroll
                    for (int j = 0; j < 4; ++j) tmem_ld32(o_tmem + 32u * (j0 + j), o[j]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) tmem_ld_wait(o[j]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
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
            // P rows (generic-proxy stores) must be visible to the tensor core
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(S::B_PFULL + 2 * x + pb));
            kt = kt_next;
        }
        // ---------------------------------------------------------- epilogue
        if (ok && it > 0) {
            ok = mbar_wait_warp(bar(S::B_OFULL + x), 0u, g, 0x414);
            tc_fence_after();
        }
        // An item split over several CTAs: each part stores its row of O
        // (unnormalised fp32, relative to its m_ref) and (m_ref, l) in its slot,
        // then counts itself; the part that counts last merges the parts in part
        // order (its own from TMEM and registers), O = sum_j w_j O_j * sv_max /
        // sum_j w_j l_j with w_j = 2^(m_j - max m), so the result does not depend
        // on which part that is.  O in the slot is [query tile][column group of
        // 4][row] float4, so that a warp's store covers 512 contiguous bytes.
        // The stores are published by one thread (CTA barrier, release fence,
        // count) and the counter read the same way (count, acquire fence,
        // barrier); all 256 softmax threads take both barriers on every path.
        constexpr int kSlotF4 = (int)(kFwdSplitSlotBytes / 16);
        bool write = ok;
        const float4 *slots = nullptr;               // part 0's slot of this item
        int sidx = 0;
        const int part = split_part(&sidx);
        if constexpr (PLAIN) {
            if (part >= 0) {
                slots = reinterpret_cast<const float4 *>(p.split_buf) + (size_t)sidx * p.split_f * kSlotF4;
                if (ok) {
                    float4 *mine = const_cast<float4 *>(slots) + (size_t)part * kSlotF4;
#pragma unroll 1
                    for (int j = 0; j < D / 32; ++j) {
                        uint32_t o[32];
                        tmem_ld32(o_tmem + 32u * j, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int t = 0; t < 8; ++t)
                            mine[(x * 32 + 8 * j + t) * 128 + r] =
                                make_float4(__uint_as_float(o[4 * t]), __uint_as_float(o[4 * t + 1]),
                                            __uint_as_float(o[4 * t + 2]), __uint_as_float(o[4 * t + 3]));
                    }
                    reinterpret_cast<float2 *>(mine + 2 * 32 * 128)[x * 128 + r] = make_float2(m_ref, l);
                }
                named_bar_sync(1, 256);
                volatile int *last = reinterpret_cast<volatile int *>(sb + S::OFF_MISC + 8);
                if (threadIdx.x == 128) {
                    // byte counter sidx % 4 of word sidx / 4 (it never exceeds split_f <= 4)
                    unsigned *w = p.split_cnt + (sidx >> 2);
                    const unsigned sh = 8u * (unsigned)(sidx & 3);
                    fence_acq_rel_gpu();
                    const unsigned n = ((atomicAdd(w, 1u << sh) >> sh) & 0xFFu) + 1u;
                    const int lst = n == (unsigned)p.split_f ? 1 : 0;
                    if (lst) {
                        atomicAnd(w, ~(0xFFu << sh));    // every part has counted: zero for the next launch
                        fence_acq_rel_gpu();
                    }
                    *last = lst;
                }
                named_bar_sync(1, 256);
                write = ok && *last != 0;
            }
        }
        if (write) {
            float inv_l = (l > 0.f) ? sv_max / l : 0.f;
            float lse2 = (l > 0.f) ? m_ref + log2f(l) : -INFINITY;     // log2 domain
            float wgt[4] = {1.f, 1.f, 1.f, 1.f};                       // the parts' weights (split items)
            if constexpr (PLAIN) {
                if (part >= 0) {
                    float mm[4], ll[4];
                    float M = -INFINITY;
#pragma unroll
                    for (int o = 0; o < 4; ++o) {
                        mm[o] = -INFINITY;
                        ll[o] = 0.f;
                        if (o < p.split_f) {
                            if (o == part) {
                                mm[o] = m_ref;
                                ll[o] = l;
                            } else {
                                const float2 v = __ldcg(reinterpret_cast<const float2 *>(
                                                            slots + (size_t)o * kSlotF4 + 2 * 32 * 128) + x * 128 + r);
                                mm[o] = v.x;
                                ll[o] = v.y;
                            }
                            M = fmaxf(M, mm[o]);
                        }
                    }
                    float L = 0.f;
#pragma unroll
                    for (int o = 0; o < 4; ++o) {
                        wgt[o] = (o < p.split_f && mm[o] != -INFINITY) ? ex2(mm[o] - M) : 0.f;
                        L += wgt[o] * ll[o];
                    }
                    inv_l = (L > 0.f) ? sv_max / L : 0.f;
                    lse2 = (L > 0.f) ? M + log2f(L) : -INFINITY;
                }
            }
            __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.O) + ((size_t)bh * p.N + q) * D;
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
                if constexpr (PLAIN) {
                    if (part >= 0) {
                        // sum over the parts in order 0, 1, ...: slot oo (its eight
                        // float4 loads issued together) or, for oo = part, own
                        float acc[32];
#pragma unroll
                        for (int t = 0; t < 32; ++t) acc[t] = 0.f;
#pragma unroll
                        for (int oo = 0; oo < 4; ++oo) {
                            if (oo >= p.split_f) break;
                            float xv[32];
                            if (oo == part) {
#pragma unroll
                                for (int t = 0; t < 32; ++t) xv[t] = __uint_as_float(o[t]);
                            } else {
                                const float4 *src = slots + (size_t)oo * kSlotF4 + (size_t)(x * 32 + 8 * j) * 128 + r;
#pragma unroll
                                for (int t = 0; t < 8; ++t) {
                                    const float4 v = __ldcg(src + t * 128);
                                    xv[4 * t] = v.x;
                                    xv[4 * t + 1] = v.y;
                                    xv[4 * t + 2] = v.z;
                                    xv[4 * t + 3] = v.w;
                                }
                            }
#pragma unroll
                            for (int t = 0; t < 32; ++t) acc[t] = fmaf(wgt[oo], xv[t], acc[t]);
                        }
#pragma unroll
                        for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(acc[t]);
                    }
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
            if (r < qnx) p.LSE[(size_t)bh * p.N + q] = lse2 * 0.69314718055994530942f;
        }
        __syncwarp();
        setmaxnreg_dec<S::REGS_CTRL>();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, S::TMEM_COLS);
}

}  // namespace

// Split plan of the plain instantiation, whose items all take the same time:
// one CTA per SM, so the items past the last full wave (rem of them) would run
// on rem SMs while the others idle.  Each of those runs as f parts over
// consecutive key-tile ranges instead, f in 2..4 chosen so that the parts'
// waves, ceil(rem f / SMs) of them, each 1/f long, end soonest; none if no f
// beats a whole wave.  A part costs ~5-10 us beyond its share of the tiles
// (the slot's stores, the count, the last part's merge), paid once per wave of
// parts, so a part gets 16 key tiles at least: with 8 (B4 H16 N4096, f = 4)
// the split was 7 % slower.  Long-context shape: 1,024 items, 112 past six
// waves of 152, f = 4 (1.158 -> 1.139 ms).
static void plan_fwd_split(FwdParams &q) {
    q.split_from = 0;
    q.split_f = 0;
    if (!q.split_buf || !q.split_cnt || q.split_cap < 2) return;
    const int64_t items = (int64_t)((q.Tq + 1) / 2) * q.BH;
    const int64_t sms = device_sm_count();
    const int64_t rem = items % sms;
    if (rem == 0 || rem > kSplitMaxItems) return;
    int64_t best = 1, best_num = 1, best_den = 1;          // last wave's length best_num / best_den
    for (int64_t f = 2; f <= 4 && f <= q.Tk / 16 && rem * f <= q.split_cap; ++f) {
        const int64_t num = (rem * f + sms - 1) / sms;
        if (num * best_den < best_num * f) {
            best = f;
            best_num = num;
            best_den = f;
        }
    }
    if (best < 2) return;
    q.split_from = (int)(items - rem);
    q.split_f = (int)best;
}

cudaError_t launch_fwd_fp8(const FwdParams &p, cudaStream_t st) {
    const int smem = F8Shape::SMEM_BYTES;
    const bool plain = !p.causal && !p.key_len && !p.block_mask && p.N % 128 == 0;
    cudaError_t e = cudaFuncSetAttribute(plain ? fa_fwd_fp8_kernel<true> : fa_fwd_fp8_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    FwdParams q = p;
    q.split_from = 0;
    q.split_f = 0;
    if (plain) plan_fwd_split(q);
    const int64_t items = (int64_t)((q.Tq + 1) / 2) * q.BH;
    const int64_t grid = q.split_f > 1 ? q.split_from + (items - q.split_from) * q.split_f : items;
    if (plain)
        return launch_dep(fa_fwd_fp8_kernel<true>, (unsigned)grid, F8Shape::THREADS, smem, st, q);
    else
        return launch_dep(fa_fwd_fp8_kernel<false>, (unsigned)grid, F8Shape::THREADS, smem, st, q);
}

}  // namespace fa
