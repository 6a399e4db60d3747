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
// This file holds the two HBM-bound kernels around the main one and the
// tile-plan export:
//   1. fa_bwd_pre:     D = rowsum(dO * O) (fp32) and dQacc = 0
//   2. the main kernel: fa_bwd64.cu (d = 64, persistent) or fa_bwd128.cu
//      (d = 128): one key tile per CTA or work item, recomputing S and P
//      tile by tile, dQ reduce-added into dQacc
//   3. fa_bwd_convert: dQ = bf16(scale * dQacc)
#include <algorithm>
#include <climits>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

// D = rowsum(dO * O) in fp32 and dQacc = 0.  Each thread takes 8 consecutive
// elements of a row (16-byte loads; D / 8 threads per row, reduced with
// shuffles inside an aligned group of lanes) and four rows a grid stride
// apart at once, so that enough bytes are in flight to keep HBM busy.  The
// loop bound is uniform over the block, so every lane reaches the shuffles.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const __nv_bfloat16 *__restrict__ O,
                                                         const __nv_bfloat16 *__restrict__ dO,
                                                         float *__restrict__ Dvec, float *__restrict__ dQacc,
                                                         int64_t rows) {
    grid_dep_wait();                                 // the previous kernel in the stream is done
    grid_dep_launch();
    constexpr int TPR = D / 8;                 // threads per row
    constexpr int RPB = 256 / TPR;             // rows per block and pass
    constexpr int U = 4;                       // passes in flight per thread
    const int sub = threadIdx.x % TPR;
    const int64_t stride = (int64_t)gridDim.x * RPB;
    for (int64_t b0 = (int64_t)blockIdx.x * RPB; b0 < rows; b0 += stride * U) {
        uint4 o[U], g[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = b0 + threadIdx.x / TPR + u * stride;
            if (row < rows) {
                o[u] = __ldg(reinterpret_cast<const uint4 *>(O + row * D) + sub);
                g[u] = __ldg(reinterpret_cast<const uint4 *>(dO + row * D) + sub);
            } else {
                o[u] = g[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = b0 + threadIdx.x / TPR + u * stride;
            float acc = bf16lo(o[u].x) * bf16lo(g[u].x) + bf16hi(o[u].x) * bf16hi(g[u].x) +
                        bf16lo(o[u].y) * bf16lo(g[u].y) + bf16hi(o[u].y) * bf16hi(g[u].y) +
                        bf16lo(o[u].z) * bf16lo(g[u].z) + bf16hi(o[u].z) * bf16hi(g[u].z) +
                        bf16lo(o[u].w) * bf16lo(g[u].w) + bf16hi(o[u].w) * bf16hi(g[u].w);
#pragma unroll
            for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (row < rows) {
                float4 *z = reinterpret_cast<float4 *>(dQacc + row * D) + 2 * sub;
                z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (sub == 0) Dvec[row] = acc;
            }
        }
    }
}

// dQ = bf16(scale * dQacc), 8 elements per thread.
__global__ void __launch_bounds__(256) fa_bwd_convert_kernel(const float *__restrict__ acc,
                                                             __nv_bfloat16 *__restrict__ dQ, int64_t n8,
                                                             float scale) {
    grid_dep_wait();                                 // the previous kernel in the stream is done
    grid_dep_launch();
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

// Both main kernels use 128-row query blocks and 32 x 32 dQ reduce boxes.
int bwd_query_block(int) { return 128; }
int bwd_dq_box_rows(int) { return 32; }
int bwd_smem_bytes(int d) { return d == 64 ? bwd64_smem_bytes() : bwd128_smem_bytes(); }

cudaError_t launch_bwd_main(int d, const BwdParams &p, cudaStream_t st) {
    return d == 64 ? launch_bwd64_main(p, st) : launch_bwd128_main(p, st);
}

cudaError_t launch_bwd_main_varlen(int d, const BwdParams &p, cudaStream_t st) {
    return d == 64 ? launch_bwd64_main_varlen(p, st) : launch_bwd128_main_varlen(p, st);
}

cudaError_t launch_bwd_pre(int d, const void *O, const void *dO, float *Dvec, float *dQacc, int64_t rows,
                           cudaStream_t st) {
    // rows per block and pass: 256 / (d / 8); four passes per thread
    const int64_t per_block = (int64_t)(256 / (d / 8)) * 4;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>((rows + per_block - 1) / per_block,
                                                                           (int64_t)device_sm_count() * 16));
    // A plain launch (the kernel's wait is then a no-op; its trigger still lets
    // the main kernel be scheduled early).  Launched to overlap the forward's
    // last CTAs, it made the step after it slower: long-context step 5.74 ->
    // 5.81 ms (the main kernel's CTAs then also scheduled early; either
    // plain launch alone removes the loss), GPT-2-medium shape unchanged.
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
    return launch_dep(fa_bwd_convert_kernel, (unsigned)blocks, 256, 0, st, dQacc, (__nv_bfloat16 *)dQ, n8, scale);
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
