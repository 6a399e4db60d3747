// fa_decode.cu -- decode-time attention: a few query rows (the newest tokens)
// against a long key/value cache, with the cache split across CTAs.
//
// The pages say decoding needs the same IO-aware framing applied to a much
// smaller, much more frequent product ("Attention" chapter, decoding
// paragraph).  With Nq << Nk one query tile per (b, h) would leave most SMs
// idle, so the key tiles of each (query tile, b, h) are split over several
// CTAs; each computes exact attention over its own key range with the
// running statistics of "The Attention Matrix You Never Write Down" ("The
// running-statistics trick") and writes a normalised partial output O_s and
// its log-sum-exp L_s.  A second kernel combines the splits with the
// block-merge identity of "FlashAttention: Mathematical Foundations ...",
// section "Incremental Online Updates", generalised to k blocks:
//     L = log sum_s exp(L_s),   O = sum_s exp(L_s - L) O_s.
//
// Kernel 1 (one CTA per (128-row query tile, b*h, split), 256 threads):
//   warp 0  TMA: the query tile once, K and V tiles of the split through a
//           3-stage (d = 128) / 6-stage (d = 64) ring;
//   warp 1  tcgen05: S = Q K^T into one of two TMEM buffers, O += P V with P
//           read from TMEM;
//   warps 4-7  softmax, one query row per thread, reference maximum moved
//           only when a row outgrows it by 2^8; epilogue O / l (fp32) and
//           L_s = (m + log2 l) ln 2 -- or, when there is one split, the final
//           bf16 O and LSE, and kernel 2 is not launched.
// It is HBM-bound (each K/V element is read once); query rows past Nq are
// zero-filled by TMA and never stored.
// Kernel 2: one warp per (b, h, query row) merges the splits, O -> bf16.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

namespace {

constexpr float kDecRescaleLog2 = 8.0f;

template <int D>
struct DecShape {
    static constexpr int CHUNKS = D / 64;
    static constexpr int CHUNK_BYTES = 128 * 128;
    static constexpr int TILE_BYTES = CHUNKS * CHUNK_BYTES;
    static constexpr int STAGES = (D == 64) ? 6 : 3;   // deep ring: the kernel streams K/V from HBM
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + TILE_BYTES;
    static constexpr int OFF_V = OFF_K + STAGES * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_V + STAGES * TILE_BYTES;
    static constexpr int B_QFULL = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_VFULL = B_KFULL + STAGES;
    static constexpr int B_KVEMPTY = B_VFULL + STAGES;
    static constexpr int B_SFULL = B_KVEMPTY + STAGES;   // [2]
    static constexpr int B_PFULL = B_SFULL + 2;          // [2]
    static constexpr int B_PVDONE = B_PFULL + 2;         // [2]
    static constexpr int B_FIN = B_PVDONE + 2;
    static constexpr int NBAR = B_FIN + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_S = 0;                  // S buffers at columns 0 and 128
    static constexpr uint32_t TM_O = 256;                // O accumulator, D columns
};

__device__ __forceinline__ void dec_drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > FA_WAIT_TIMEOUT_NS) break;
}

}  // namespace

// QTR (2 <= Nq <= 32, one query tile): the query rows are loaded into all four
// 32-row quarters of the tile, and softmax warp k takes key columns
// [32 k, 32 k + 32) of every key tile for its copy, with running statistics
// of its own; the epilogue merges the four partial rows of each query
// (the block-merge identity of "FlashAttention: Mathematical Foundations
// ...", "Incremental Online Updates").  One warp's softmax over whole
// 128-key rows, four of them real, was the chain each key tile waited on.
template <int D, bool QTR>
__global__ void __launch_bounds__(256, 1) fa_decode_kernel(const __grid_constant__ DecParams p) {
    grid_dep_wait();                                 // the previous kernel in the stream is done
    grid_dep_launch();
    using S = DecShape<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // work item: (split, b*h, query tile), splits of one (b, h) adjacent
    const int sp = (int)(blockIdx.x % p.splits);
    const int rest = (int)(blockIdx.x / p.splits);
    const int qt = rest % p.Tq;
    const int bh = rest / p.Tq;
    const int b = bh / p.H;
    const int q0 = qt * kTile;
    const int qn = min(kTile, p.Nq - q0);
    const int kt_begin = sp * p.tiles_per_split;
    const int kt_end = min(p.Tk, kt_begin + p.tiles_per_split);

    auto bar = [&](int i) -> uint32_t { return base + S::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + S::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sb + S::OFF_MISC + 4);
    const Guard g{p.status, p.status + 1, abort_flag};

    int kvis = p.Nk;
    if (p.kv_len) {
        kvis = p.kv_len[b];
        if (kvis < 0 || kvis > p.Nk) {
            if (threadIdx.x == 0 && qt == 0 && sp == 0 && (bh % p.H) == 0) record_status(g, kStatusBadKeyLen, 0);
            kvis = kvis < 0 ? 0 : p.Nk;
        }
    }
    const int shift = kvis - p.Nq;       // causal: query i sees keys j <= i + shift
    auto cls = [&](int kt) -> unsigned {
        return tile_class_shift(q0, qn, kt * kTile, kTile, kvis, p.causal, shift);
    };
    auto next_tile = [&](int kt) -> int {
        for (int k = kt + 1; k < kt_end; ++k)
            if (cls(k) != kTileSkip) return k;
        return kt_end;
    };
    const int first = next_tile(kt_begin - 1);

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

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (first < kt_end) {
            int it = 0;
            bool ok = true;
            mbar_arrive_expect_tx_elect(bar(S::B_QFULL), S::TILE_BYTES);
            if constexpr (QTR) {
                // rows 0..31 of the queries into each quarter (a 32-row offset keeps the 128-byte swizzle)
                for (int cp = 0; cp < 4; ++cp)
                    for (int c = 0; c < S::CHUNKS; ++c)
                        tma_load_3d_elect(base + S::OFF_Q + c * S::CHUNK_BYTES + cp * 32 * 128, &p.tmQs,
                                          bar(S::B_QFULL), c * 64, 0, bh);
            } else {
                for (int c = 0; c < S::CHUNKS; ++c)
                    tma_load_3d_elect(base + S::OFF_Q + c * S::CHUNK_BYTES, &p.tmQ, bar(S::B_QFULL), c * 64, q0, bh);
            }
            for (int kt = first; kt < kt_end; kt = next_tile(kt), ++it) {
                const int s = it % S::STAGES;
                const uint32_t ph = (uint32_t)(it / S::STAGES) & 1u;
                if (!mbar_wait_warp(bar(S::B_KVEMPTY + s), ph ^ 1u, g, 0x501)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_elect(bar(S::B_KFULL + s), S::TILE_BYTES);
                for (int c = 0; c < S::CHUNKS; ++c)
                    tma_load_3d_elect(base + S::OFF_K + s * S::TILE_BYTES + c * S::CHUNK_BYTES, &p.tmK, bar(S::B_KFULL + s),
                                c * 64, kt * kTile, bh);
                mbar_arrive_expect_tx_elect(bar(S::B_VFULL + s), S::TILE_BYTES);
                for (int c = 0; c < S::CHUNKS; ++c)
                    tma_load_3d_elect(base + S::OFF_V + s * S::TILE_BYTES + c * S::CHUNK_BYTES, &p.tmV, bar(S::B_VFULL + s),
                                c * 64, kt * kTile, bh);
            }
            if (!ok) {
                dec_drain_wait(bar(S::B_QFULL), 0);
                for (int i = (it > S::STAGES ? it - S::STAGES : 0); i < it; ++i) {
                    const int s = i % S::STAGES;
                    const uint32_t ph = (uint32_t)(i / S::STAGES) & 1u;
                    dec_drain_wait(bar(S::B_KFULL + s), ph);
                    dec_drain_wait(bar(S::B_VFULL + s), ph);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        {
            constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
            const uint64_t dq0 = sdesc_sw128(base + S::OFF_Q, 16, 1024);
            const uint64_t dk0 = sdesc_sw128(base + S::OFF_K, 16, 1024);
            const uint64_t dv0 = sdesc_sw128(base + S::OFF_V, S::CHUNK_BYTES, 1024);
            bool ok = true;
            if (first < kt_end) {
                ok = mbar_wait_warp(bar(S::B_QFULL), 0, g, 0x511);
                // S_i = Q K_i^T into TMEM buffer i % 2
                auto issue_s = [&](int i) -> bool {
                    const int s = i % S::STAGES;
                    if (!mbar_wait_warp(bar(S::B_KFULL + s), (uint32_t)(i / S::STAGES) & 1u, g, 0x512)) return false;
                    // buffer i % 2 last held P_{i-2}: its P.V must have finished
                    if (i >= 2 && !mbar_wait_warp(bar(S::B_PVDONE + (i & 1)), (uint32_t)((i - 2) >> 1) & 1u, g, 0x513))
                        return false;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + S::TM_S + (uint32_t)(i & 1) * 128u;
                    const uint64_t kd = sdesc_add(dk0, (uint32_t)(s * S::TILE_BYTES));
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = (k >> 2) * S::CHUNK_BYTES + (k & 3) * 32;
                        mma_ss_elect(d_tmem, sdesc_add(dq0, off), sdesc_add(kd, off), IDESC_S, k > 0 ? 1u : 0u);
                    }
                    mma_commit_elect(bar(S::B_SFULL + (i & 1)));
                    return true;
                };
                if (ok) ok = issue_s(0);
                int it = 0;
                for (int kt = first; ok && kt < kt_end; ++it) {
                    const int kt_next = next_tile(kt);
                    if (kt_next < kt_end && !(ok = issue_s(it + 1))) break;
                    const int s = it % S::STAGES;
                    if (!mbar_wait_warp(bar(S::B_PFULL + (it & 1)), (uint32_t)(it >> 1) & 1u, g, 0x514) ||
                        !mbar_wait_warp(bar(S::B_VFULL + s), (uint32_t)(it / S::STAGES) & 1u, g, 0x515)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t p_tmem = tmem + S::TM_S + (uint32_t)(it & 1) * 128u;
                    const uint64_t vd = sdesc_add(dv0, (uint32_t)(s * S::TILE_BYTES));
                    const uint32_t acc0 = it > 0 ? 1u : 0u;
#pragma unroll
                    for (int k = 0; k < kTile / 16; ++k)
                        mma_ts_elect(tmem + S::TM_O, p_tmem + (uint32_t)k * 8u, sdesc_add(vd, (uint32_t)k * 2048u), IDESC_PV,
                               k > 0 ? 1u : acc0);
                    mma_commit_elect(bar(S::B_KVEMPTY + s));
                    mma_commit_elect(bar(S::B_PVDONE + (it & 1)));
                    kt = kt_next;
                }
            }
            mma_commit_elect(bar(S::B_FIN));
            dec_drain_wait(bar(S::B_FIN), 0);
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------- softmax
        const int wq = warp & 3;
        const int r = wq * 32 + lane;                // TMEM lane / tile row
        const int q = QTR ? lane : q0 + r;           // the query row (QTR: copy wq of query `lane`)
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t o_tmem = tmem + lane_off + S::TM_O;
        const float c2 = p.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        int it = 0;
        bool ok = true;
        // a warp whose 32 rows all lie past Nq has nothing to compute: its P
        // rows only feed output rows that are never stored
        const bool active = QTR || q0 + wq * 32 < p.Nq;
        for (int kt = first; kt < kt_end; kt = next_tile(kt), ++it) {
            if (!active) {
                if (!mbar_wait_warp(bar(S::B_SFULL + (it & 1)), (uint32_t)(it >> 1) & 1u, g, 0x521)) {
                    ok = false;
                    break;
                }
                mbar_arrive(bar(S::B_PFULL + (it & 1)));
                continue;
            }
            const bool partial = cls(kt) == kTilePartial;
            const int k0 = kt * kTile;
            if (!mbar_wait_warp(bar(S::B_SFULL + (it & 1)), (uint32_t)(it >> 1) & 1u, g, 0x521)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t s_tmem = tmem + lane_off + S::TM_S + (uint32_t)(it & 1) * 128u;
            if constexpr (QTR) {
                // key columns [32 wq, 32 wq + 32) of this tile for query `lane`
                uint32_t sr[32];
                tmem_ld32(s_tmem + 32u * wq, sr);
                tmem_ld_wait(sr);
                if (partial) {
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const int key = k0 + 32 * wq + t;
                        if (key >= kvis || (p.causal && key > q + shift)) sr[t] = __float_as_uint(-INFINITY);
                    }
                }
                float pm[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) pm[u] = -INFINITY;
#pragma unroll
                for (int t = 0; t < 32; t += 8) {
                    const int u = t / 8;
                    pm[u] = fmax3(pm[u], __uint_as_float(sr[t]), __uint_as_float(sr[t + 1]));
                    pm[u] = fmax3(pm[u], __uint_as_float(sr[t + 2]), __uint_as_float(sr[t + 3]));
                    pm[u] = fmax3(pm[u], __uint_as_float(sr[t + 4]), __uint_as_float(sr[t + 5]));
                    pm[u] = fmax3(pm[u], __uint_as_float(sr[t + 6]), __uint_as_float(sr[t + 7]));
                }
                const float m_tile = c2 * fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
                const bool rescale = __any_sync(0xffffffffu, m_tile > m_ref + kDecRescaleLog2);
                float alpha = 1.f;
                if (rescale) {
                    const float m_new = fmaxf(m_ref, m_tile);
                    alpha = (m_new == -INFINITY) ? 1.f : ex2(m_ref - m_new);
                    l *= alpha;
                    m_ref = m_new;
                }
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                float ps[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[16], zero[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    float a, bb;
                    fma2(a, bb, __uint_as_float(sr[2 * t]), __uint_as_float(sr[2 * t + 1]), c2, c2, -m_use, -m_use);
                    a = ex2(a);
                    bb = ex2(bb);
                    const int u = 2 * (t & 1);
                    add2(ps[u], ps[u + 1], a, bb);
                    pk[t] = pack_bf16x2(a, bb);
                    zero[t] = 0u;
                }
                // this row's P: its own 32 keys, zero for the other quarters' keys
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j == wq)                     // warp-uniform
                        tmem_st16(s_tmem + 16u * j, pk);
                    else
                        tmem_st16(s_tmem + 16u * j, zero);
                }
                l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
                tmem_st_wait();
                if (rescale && it > 0) {
                    if (!mbar_wait_warp(bar(S::B_PVDONE + ((it - 1) & 1)), (uint32_t)((it - 1) >> 1) & 1u, g, 0x522)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int j = 0; j < D / 32; ++j) {
                        uint32_t o[32];
                        tmem_ld32(o_tmem + 32u * j, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
                        tmem_st32(o_tmem + 32u * j, o);
                    }
                    tmem_st_wait();
                }
            } else {
                uint32_t sr[4][32];
    #pragma unroll
                for (int j = 0; j < 4; ++j) tmem_ld32(s_tmem + 32u * j, sr[j]);
    #pragma unroll
                for (int j = 0; j < 4; ++j) tmem_ld_wait(sr[j]);
                if (partial) {
    #pragma unroll
                    for (int j = 0; j < 4; ++j)
    #pragma unroll
                        for (int t = 0; t < 32; ++t) {
                            const int key = k0 + 32 * j + t;
                            if (key >= kvis || (p.causal && key > q + shift)) sr[j][t] = __float_as_uint(-INFINITY);
                        }
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
                const float m_tile = c2 * fmaxf(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], fmax3(pm[5], pm[6], pm[7])));
                const bool rescale = __any_sync(0xffffffffu, m_tile > m_ref + kDecRescaleLog2);
                float alpha = 1.f;
                if (rescale) {
                    const float m_new = fmaxf(m_ref, m_tile);
                    alpha = (m_new == -INFINITY) ? 1.f : ex2(m_ref - m_new);
                    l *= alpha;
                    m_ref = m_new;
                }
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                float ps[8];
    #pragma unroll
                for (int u = 0; u < 8; ++u) ps[u] = 0.f;
    #pragma unroll
                for (int j = 0; j < 4; ++j) {
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
                    if (!mbar_wait_warp(bar(S::B_PVDONE + ((it - 1) & 1)), (uint32_t)((it - 1) >> 1) & 1u, g, 0x522)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
    #pragma unroll 1
                    for (int j = 0; j < D / 32; ++j) {
                        uint32_t o[32];
                        tmem_ld32(o_tmem + 32u * j, o);
                        tmem_ld_wait(o);
    #pragma unroll
                        for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
                        tmem_st32(o_tmem + 32u * j, o);
                    }
                    tmem_st_wait();
                }
            }
            tc_fence_before();
            mbar_arrive(bar(S::B_PFULL + (it & 1)));
        }
        // ---------------------------------------------------------- epilogue: this split's partial
        // (or, with a single split, the final bf16 output and LSE)
        if (ok && it > 0) {
            ok = mbar_wait_warp(bar(S::B_PVDONE + ((it - 1) & 1)), (uint32_t)((it - 1) >> 1) & 1u, g, 0x523);
            tc_fence_after();
        }
        if constexpr (QTR) {
            // merge the four copies of each query row: every softmax thread
            // stages (m_ref, l) and its unnormalised O row in the K stages'
            // shared memory (free: every product is done), O as [copy][column
            // group of 4][row] float4 so that a warp's store covers 512
            // contiguous bytes; the copy-0 warp then sums the copies in copy
            // order with weights 2^(m_k - max m).  All 128 softmax threads take
            // the barrier on every path.
            float4 *ostg = reinterpret_cast<float4 *>(sb + S::OFF_K);
            float2 *mstg = reinterpret_cast<float2 *>(sb + S::OFF_K + 4 * (D / 4) * 32 * 16);
            if (ok) {
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
#pragma unroll
                    for (int t = 0; t < 8; ++t)
                        ostg[(wq * (D / 4) + 8 * j + t) * 32 + lane] =
                            make_float4(__uint_as_float(o[4 * t]), __uint_as_float(o[4 * t + 1]),
                                        __uint_as_float(o[4 * t + 2]), __uint_as_float(o[4 * t + 3]));
                }
                mstg[wq * 32 + lane] = make_float2(m_ref, l);
            }
            named_bar_sync(1, 128);
            if (ok && wq == 0 && lane < qn) {
                float mm[4], ll[4], wk[4];
                float M = -INFINITY;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 v = mstg[k * 32 + lane];
                    mm[k] = v.x;
                    ll[k] = v.y;
                    M = fmaxf(M, mm[k]);
                }
                float L = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    wk[k] = (mm[k] == -INFINITY) ? 0.f : ex2(mm[k] - M);
                    L += wk[k] * ll[k];
                }
                const float inv_l = (L > 0.f) ? 1.f / L : 0.f;
                const size_t row = ((size_t)sp * p.BH + bh) * p.Nq + q;
#pragma unroll 1
                for (int c = 0; c < D / 4; ++c) {
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float4 v = ostg[(k * (D / 4) + c) * 32 + lane];
                        acc.x = fmaf(wk[k], v.x, acc.x);
                        acc.y = fmaf(wk[k], v.y, acc.y);
                        acc.z = fmaf(wk[k], v.z, acc.z);
                        acc.w = fmaf(wk[k], v.w, acc.w);
                    }
                    if (p.O) {
                        uint2 *dst = reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.O) + row * D + 4 * c);
                        *dst = make_uint2(pack_bf16x2(acc.x * inv_l, acc.y * inv_l), pack_bf16x2(acc.z * inv_l, acc.w * inv_l));
                    } else {
                        reinterpret_cast<float4 *>(p.Opart + row * D)[c] =
                            make_float4(acc.x * inv_l, acc.y * inv_l, acc.z * inv_l, acc.w * inv_l);
                    }
                }
                (p.LSE ? p.LSE : p.Lpart)[row] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
            }
        } else if (ok && active) {
            const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
            const size_t row = ((size_t)sp * p.BH + bh) * p.Nq + q;
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
                if (r < qn && p.O) {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.O) + row * D + 32 * j);
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        dst[t] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * t]) * inv_l, __uint_as_float(o[8 * t + 1]) * inv_l),
                                            pack_bf16x2(__uint_as_float(o[8 * t + 2]) * inv_l, __uint_as_float(o[8 * t + 3]) * inv_l),
                                            pack_bf16x2(__uint_as_float(o[8 * t + 4]) * inv_l, __uint_as_float(o[8 * t + 5]) * inv_l),
                                            pack_bf16x2(__uint_as_float(o[8 * t + 6]) * inv_l, __uint_as_float(o[8 * t + 7]) * inv_l));
                } else if (r < qn) {
                    float4 *dst = reinterpret_cast<float4 *>(p.Opart + row * D + 32 * j);
#pragma unroll
                    for (int t = 0; t < 8; ++t)
                        dst[t] = make_float4(__uint_as_float(o[4 * t]) * inv_l, __uint_as_float(o[4 * t + 1]) * inv_l,
                                             __uint_as_float(o[4 * t + 2]) * inv_l, __uint_as_float(o[4 * t + 3]) * inv_l);
                }
            }
            if (r < qn) (p.LSE ? p.LSE : p.Lpart)[row] = (l > 0.f) ? (m_ref + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, S::TMEM_COLS);
}

// Merge the splits of one (b, h, query row) per warp:
//   L = log sum_s exp(L_s),  O = sum_s exp(L_s - L) O_s  (bf16 out).
template <int D>
__global__ void __launch_bounds__(256) fa_decode_merge_kernel(const float *__restrict__ Opart,
                                                              const float *__restrict__ Lpart,
                                                              __nv_bfloat16 *__restrict__ O, float *__restrict__ LSE,
                                                              int64_t rows, int splits) {
    grid_dep_wait();                                 // the previous kernel in the stream is done
    grid_dep_launch();
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    constexpr int PER = D / 32;   // columns per lane
    float lmax = -INFINITY;
    for (int s = 0; s < splits; ++s) lmax = fmaxf(lmax, Lpart[(int64_t)s * rows + row]);
    float acc[PER];
#pragma unroll
    for (int t = 0; t < PER; ++t) acc[t] = 0.f;
    float wsum = 0.f;
    if (lmax != -INFINITY) {
        for (int s = 0; s < splits; ++s) {
            const float ls = Lpart[(int64_t)s * rows + row];
            if (ls == -INFINITY) continue;
            const float w = __expf(ls - lmax);
            wsum += w;
            const float *src = Opart + ((int64_t)s * rows + row) * D + lane * PER;
            if (PER == 4) {
                const float4 v = *reinterpret_cast<const float4 *>(src);
                acc[0] += w * v.x;
                acc[1] += w * v.y;
                acc[2] += w * v.z;
                acc[3] += w * v.w;
            } else {
                const float2 v = *reinterpret_cast<const float2 *>(src);
                acc[0] += w * v.x;
                acc[1] += w * v.y;
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16 *dst = O + row * D + lane * PER;
    if (PER == 4) {
        reinterpret_cast<uint2 *>(dst)[0] = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                       pack_bf16x2(acc[2] * inv, acc[3] * inv));
    } else {
        reinterpret_cast<uint32_t *>(dst)[0] = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0) LSE[row] = wsum > 0.f ? lmax + logf(wsum) : -INFINITY;
}

template <int D, bool QTR>
static cudaError_t launch_decode_t(const DecParams &p, cudaStream_t st) {
    const int smem = DecShape<D>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(fa_decode_kernel<D, QTR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)p.Tq * (unsigned)p.BH * (unsigned)p.splits;
    return launch_dep(fa_decode_kernel<D, QTR>, grid, 256, smem, st, p);
}

cudaError_t launch_decode(int d, const DecParams &p, cudaStream_t st) {
    // 2..32 query rows: the quartered softmax (the host encoded tmQs).  One
    // query row: the whole-row softmax of one warp, which keeps up with HBM
    // there (the quartered form measured 0.7 % slower: four warps' TMEM traffic)
    if (p.Nq >= 2 && p.Nq <= 32)
        return d == 64 ? launch_decode_t<64, true>(p, st) : launch_decode_t<128, true>(p, st);
    return d == 64 ? launch_decode_t<64, false>(p, st) : launch_decode_t<128, false>(p, st);
}

cudaError_t launch_decode_merge(int d, const float *Opart, const float *Lpart, void *O, float *LSE, int64_t rows,
                                int splits, cudaStream_t st) {
    const unsigned grid = (unsigned)((rows + 7) / 8);
    if (d == 64)
        return launch_dep(fa_decode_merge_kernel<64>, grid, 256, 0, st, Opart, Lpart, (__nv_bfloat16 *)O, LSE, rows,
                          splits);
    else
        return launch_dep(fa_decode_merge_kernel<128>, grid, 256, 0, st, Opart, Lpart, (__nv_bfloat16 *)O, LSE, rows,
                          splits);
}

}  // namespace fa
