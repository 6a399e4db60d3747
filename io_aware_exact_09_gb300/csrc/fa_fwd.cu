// fa_fwd.cu -- forward kernel: O and LSE of exact attention, tile by tile,
// never writing the score matrix.
//
// Method ("The Attention Matrix You Never Write Down", section "The
// running-statistics trick"; "FlashAttention: Mathematical Foundations ...",
// sections "Incremental Online Updates" and "IO-Aware Tiling Algorithm"):
// per query row keep the running maximum m and normaliser l; for each new key
// tile take m' = max(m, tile max), multiply l and the unnormalised output by
// exp(m - m'), add the tile's exp(s - m') and exp(s - m') V; divide by l at
// the end.  The tiling page prints the correction as diag(exp(m - m'))^-1;
// that contradicts the running-statistics page and its own final
// diag(l)^-1 normalisation, so the multiply-by-exp(m - m') reading is used.
// Everything is in base 2: x = s * scale * log2(e), p = 2^(x - m).
//
// GB300 design (not the A100 loop order the tiling page prints; the query
// tile is the outer loop, as in its "FlashAttention-2" section, so O stays on
// chip):
//   - one CTA per (128-row query tile, b*h); heavier causal tiles first;
//   - warp 0: TMA producer.  Q tile once; K and V tiles through a ring of
//     shared-memory stages (128-byte swizzle, 64-column boxes);
//   - warp 1: tcgen05 issuer.  S = Q K^T into one of two TMEM buffers (so the
//     next tile's S overlaps this tile's softmax), then O += P V with P read
//     from TMEM (it overwrites the first half of its S buffer as bf16);
//   - warps 4-7: softmax, one query row per thread (TMEM lane = row), the
//     O rescale (only when a row's maximum moved), and the epilogue
//     O / l -> bf16, LSE = (m + log2 l) * ln 2.
// Skipped tiles (block mask zero, all keys past key_len, above the causal
// diagonal) are never loaded; partial tiles get element masks.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

template <int D>
struct FwdShape {
    static constexpr int CHUNKS = D / 64;               // 64-element (128-byte) column chunks
    static constexpr int CHUNK_BYTES = 128 * 128;       // 128 rows x 128 bytes
    static constexpr int TILE_BYTES = CHUNKS * CHUNK_BYTES;
    static constexpr int STAGES = (D == 64) ? 4 : 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + TILE_BYTES;
    static constexpr int OFF_V = OFF_K + STAGES * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_V + STAGES * TILE_BYTES;
    // barrier indices
    static constexpr int B_QFULL = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_VFULL = B_KFULL + STAGES;
    static constexpr int B_KVEMPTY = B_VFULL + STAGES;
    static constexpr int B_SFULL = B_KVEMPTY + STAGES;   // [2]
    static constexpr int B_PFULL = B_SFULL + 2;          // [2]
    static constexpr int B_PVDONE = B_PFULL + 2;         // [2]
    static constexpr int B_FIN = B_PVDONE + 2;
    static constexpr int NBAR = B_FIN + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem base (4 B), abort flag (4 B)
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1 KB
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_S = 0;                  // S buffers at columns 0 and 128
    static constexpr uint32_t TM_O = 256;                // O accumulator, D columns
};

// Bounded wait used only while draining after an abort (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > FA_WAIT_TIMEOUT_NS) break;
}

template <int D>
__global__ void __launch_bounds__(256, 1) fa_fwd_kernel(const __grid_constant__ FwdParams p) {
    using S = FwdShape<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Work item, head-major: the CTAs resident at one time share one head's K
    // and V in L2; within a head the causally heaviest query tiles (highest
    // index, most key tiles) start first.
    const int qt = p.Tq - 1 - (int)(blockIdx.x % p.Tq);
    const int bh = (int)(blockIdx.x / p.Tq);
    const int b = bh / p.H;
    const int q0 = qt * kTile;
    const int qn = min(kTile, p.N - q0);
    const int nb = (p.N + kTile - 1) / kTile;

    auto bar = [&](int i) -> uint32_t { return base + S::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + S::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sb + S::OFF_MISC + 4);
    const Guard g{p.status, p.status + 1, abort_flag};

    bool bad = false;
    const int kvis = key_visible_bound(p.key_len, b, p.N, &bad);
    if (bad && threadIdx.x == 0 && qt == 0 && (bh % p.H) == 0) record_status(g, kStatusBadKeyLen, 0);

    auto cls = [&](int kt) -> unsigned {
        const int on = p.block_mask ? (p.block_mask[(size_t)qt * nb + kt] != 0) : 1;
        return tile_class(q0, qn, kt * kTile, kTile, kvis, p.causal, on);
    };
    auto next_tile = [&](int kt) -> int {
        for (int k = kt + 1; k < p.Tk; ++k)
            if (cls(k) != kTileSkip) return k;
        return p.Tk;
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

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            int kt = next_tile(-1);
            if (kt < p.Tk) {
                mbar_arrive_expect_tx(bar(S::B_QFULL), S::TILE_BYTES);
                for (int c = 0; c < S::CHUNKS; ++c)
                    tma_load_3d(base + S::OFF_Q + c * S::CHUNK_BYTES, &p.tmQ, bar(S::B_QFULL), c * 64,
                                q0, bh);
            }
            for (; kt < p.Tk; kt = next_tile(kt), ++it) {
                const int s = it % S::STAGES;
                const uint32_t ph = (uint32_t)(it / S::STAGES) & 1u;
                if (!mbar_wait(bar(S::B_KVEMPTY + s), ph ^ 1u, g, 0x101)) {
                    ok = false;
                    break;
                }
                const uint32_t koff = base + S::OFF_K + s * S::TILE_BYTES;
                const uint32_t voff = base + S::OFF_V + s * S::TILE_BYTES;
                mbar_arrive_expect_tx(bar(S::B_KFULL + s), S::TILE_BYTES);
                for (int c = 0; c < S::CHUNKS; ++c)
                    tma_load_3d(koff + c * S::CHUNK_BYTES, &p.tmK, bar(S::B_KFULL + s), c * 64,
                                kt * kTile, bh);
                mbar_arrive_expect_tx(bar(S::B_VFULL + s), S::TILE_BYTES);
                for (int c = 0; c < S::CHUNKS; ++c)
                    tma_load_3d(voff + c * S::CHUNK_BYTES, &p.tmV, bar(S::B_VFULL + s), c * 64,
                                kt * kTile, bh);
            }
            if (!ok) {
                // gave up: let every copy already issued land before the CTA exits
                if (next_tile(-1) < p.Tk) drain_wait(bar(S::B_QFULL), 0);
                for (int i = (it > S::STAGES ? it - S::STAGES : 0); i < it; ++i) {
                    const int s = i % S::STAGES;
                    const uint32_t ph = (uint32_t)(i / S::STAGES) & 1u;
                    drain_wait(bar(S::B_KFULL + s), ph);
                    drain_wait(bar(S::B_VFULL + s), ph);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
            int kt = next_tile(-1);
            bool ok = true;
            if (kt < p.Tk) {
                ok = mbar_wait(bar(S::B_QFULL), 0, g, 0x201);
                // S_i = Q K_i^T into TMEM buffer i % 2
                auto issue_s = [&](int i) -> bool {
                    const int s = i % S::STAGES;
                    if (!mbar_wait(bar(S::B_KFULL + s), (uint32_t)(i / S::STAGES) & 1u, g, 0x202))
                        return false;
                    // buffer i%2 last held P_{i-2}: its P.V must have finished
                    if (i >= 2 &&
                        !mbar_wait(bar(S::B_PVDONE + (i & 1)), (uint32_t)((i - 2) >> 1) & 1u, g, 0x203))
                        return false;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + S::TM_S + (uint32_t)(i & 1) * 128u;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t qa = base + S::OFF_Q + (k >> 2) * S::CHUNK_BYTES + (k & 3) * 32;
                        const uint32_t ka = base + S::OFF_K + s * S::TILE_BYTES +
                                            (k >> 2) * S::CHUNK_BYTES + (k & 3) * 32;
                        mma_ss(d_tmem, sdesc_sw128(qa, 16, 1024), sdesc_sw128(ka, 16, 1024), IDESC_S,
                               k > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(S::B_SFULL + (i & 1)));
                    return true;
                };
                if (ok) ok = issue_s(0);
                int it = 0;
                while (ok && kt < p.Tk) {
                    const int kt_next = next_tile(kt);
                    if (kt_next < p.Tk && !(ok = issue_s(it + 1))) break;
                    const int s = it % S::STAGES;
                    if (!mbar_wait(bar(S::B_PFULL + (it & 1)), (uint32_t)(it >> 1) & 1u, g, 0x204) ||
                        !mbar_wait(bar(S::B_VFULL + s), (uint32_t)(it / S::STAGES) & 1u, g, 0x205)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t p_tmem = tmem + S::TM_S + (uint32_t)(it & 1) * 128u;
                    const uint32_t voff = base + S::OFF_V + s * S::TILE_BYTES;
#pragma unroll
                    for (int k = 0; k < kTile / 16; ++k) {
                        // A = P (bf16 pairs, 8 columns per 16 keys); B = V, MN-major
                        mma_ts(tmem + S::TM_O, p_tmem + (uint32_t)k * 8u,
                               sdesc_sw128(voff + k * 2048, S::CHUNK_BYTES, 1024), IDESC_PV,
                               (it > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(S::B_KVEMPTY + s));
                    mma_commit(bar(S::B_PVDONE + (it & 1)));
                    kt = kt_next;
                    ++it;
                }
            }
            // every MMA this thread issued must finish before TMEM is freed
            mma_commit(bar(S::B_FIN));
            drain_wait(bar(S::B_FIN), 0);
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------- softmax
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const int q = q0 + r;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const float c2 = p.scale_log2;
        float m = -INFINITY, l = 0.f;
        int it = 0;
        bool ok = true;
        for (int kt = next_tile(-1); kt < p.Tk; kt = next_tile(kt), ++it) {
            const unsigned klass = cls(kt);
            if (!mbar_wait_warp(bar(S::B_SFULL + (it & 1)), (uint32_t)(it >> 1) & 1u, g, 0x401)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t s_tmem = tmem + lane_off + S::TM_S + (uint32_t)(it & 1) * 128u;
            uint32_t sr[4][32];
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_ld32(s_tmem + 32u * j, sr[j]);
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_ld_wait(sr[j]);
            if (klass == kTilePartial) {
                const int k0 = kt * kTile;
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const int key = k0 + 32 * j + t;
                        if (key >= kvis || (p.causal && key > q)) sr[j][t] = __float_as_uint(-INFINITY);
                    }
            }
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int t = 0; t < 32; ++t) mx = fmaxf(mx, __uint_as_float(sr[j][t]));
            const float m_new = fmaxf(m, mx * c2);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2(m - m_use);
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t pk[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const float a = ex2(fmaf(__uint_as_float(sr[j][2 * t]), c2, -m_use));
                    const float bb = ex2(fmaf(__uint_as_float(sr[j][2 * t + 1]), c2, -m_use));
                    sum += a + bb;
                    pk[t] = pack_bf16x2(a, bb);
                }
                // P (bf16) overwrites the first 64 columns of this S buffer
                tmem_st16(s_tmem + 16u * j, pk);
            }
            l = l * alpha + sum;
            m = m_new;
            tmem_st_wait();
            if (it > 0) {
                // O may be rescaled only once the previous P.V has landed
                if (!mbar_wait_warp(bar(S::B_PVDONE + ((it - 1) & 1)), (uint32_t)((it - 1) >> 1) & 1u, g,
                                    0x402)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int j = 0; j < D / 32; ++j) {
                        uint32_t o[32];
                        const uint32_t oa = tmem + lane_off + S::TM_O + 32u * j;
                        tmem_ld32(oa, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
                        tmem_st32(oa, o);
                    }
                    tmem_st_wait();
                }
            }
            tc_fence_before();
            mbar_arrive(bar(S::B_PFULL + (it & 1)));
        }
        // ---------------------------------------------------------- epilogue
        if (ok && it > 0) {
            ok = mbar_wait_warp(bar(S::B_PVDONE + ((it - 1) & 1)), (uint32_t)((it - 1) >> 1) & 1u, g,
                                0x403);
            tc_fence_after();
        }
        if (ok) {
            const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
            __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.O) + ((size_t)bh * p.N + q) * D;
#pragma unroll 1
            for (int j = 0; j < D / 32; ++j) {
                uint32_t o[32];
                if (it > 0) {
                    tmem_ld32(tmem + lane_off + S::TM_O + 32u * j, o);
                    tmem_ld_wait(o);
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) o[t] = 0u;
                }
                uint32_t w[16];
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    w[t] = pack_bf16x2(__uint_as_float(o[2 * t]) * inv_l, __uint_as_float(o[2 * t + 1]) * inv_l);
                if (q < p.N) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * j);
#pragma unroll
                    for (int t = 0; t < 4; ++t) dst[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
                }
            }
            if (q < p.N)
                p.LSE[(size_t)bh * p.N + q] = (l > 0.f) ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, S::TMEM_COLS);
}

int fwd_smem_bytes(int d) { return d == 64 ? FwdShape<64>::SMEM_BYTES : FwdShape<128>::SMEM_BYTES; }

template <int D>
static cudaError_t launch_fwd_t(const FwdParams &p, cudaStream_t st) {
    const int smem = FwdShape<D>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)p.Tq * (unsigned)p.BH;
    fa_fwd_kernel<D><<<grid, 256, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_fwd(int d, const FwdParams &p, cudaStream_t st) {
    return d == 64 ? launch_fwd_t<64>(p, st) : launch_fwd_t<128>(p, st);
}

}  // namespace fa
