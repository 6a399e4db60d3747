// fa_quant.cu -- FP8 block quantisation of Q, K or V for the FP8 forward.
//
// "FlashAttention: Mathematical Foundations ...", section "Architectural
// Evolution" (FlashAttention-3 paragraph): the FP8 matmuls are
// block-quantised with dynamic scaling.  A block is 128 consecutive rows
// (tokens) x all d columns of one (b, h); its scale is amax / 448 (the
// largest finite e4m3 magnitude), taken from the data, and 0 for an all-zero
// block; each element becomes e4m3(x / scale) (fp32 division, nearest-even,
// saturating).  V is written transposed, [BH][d][Np] with Np = ceil(N/16)*16,
// so that it is the K-major operand of the P.V product.
//
// One CTA per (b*h, block): 256 threads load the block with 16-byte loads,
// reduce amax, and write the codes (row layout: 8 bytes per thread per
// vector; transposed: through a shared-memory tile, 128-byte rows out).
// HBM-bound: 2 bytes read and 1 written per element.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

namespace {

template <int D>
__global__ void __launch_bounds__(256) fa_quant_fp8_kernel(const __nv_bfloat16 *__restrict__ X,
                                                           uint8_t *__restrict__ Y, float *__restrict__ scales,
                                                           int N, int T, int Np, int transpose) {
    constexpr int VPR = D / 8;                 // 16-byte vectors per row
    constexpr int NV = 128 * VPR / 256;        // vectors per thread
    constexpr int TS = 128 + 16;               // transposed staging row stride (bytes)
    __shared__ float red[8];
    __shared__ __align__(16) uint8_t tr[D * TS];
    const int bh = (int)(blockIdx.x / T), t = (int)(blockIdx.x % T);
    const int r0 = t * 128;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const __nv_bfloat16 *xb = X + ((size_t)bh * N + r0) * D;

    uint4 v[NV];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int idx = tid + 256 * i, row = idx / VPR, cv = idx % VPR;
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (r0 + row < N) v[i] = __ldg(reinterpret_cast<const uint4 *>(xb + (size_t)row * D) + cv);
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(w[k])), fabsf(bf16hi(w[k]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int k = 1; k < 8; ++k) amax = fmaxf(amax, red[k]);
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
    if (tid == 0) scales[blockIdx.x] = scale;

#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int idx = tid + 256 * i, row = idx / VPR, cv = idx % VPR;
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        float f[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            f[2 * k] = scale > 0.f ? __fdiv_rn(bf16lo(w[k]), scale) : 0.f;
            f[2 * k + 1] = scale > 0.f ? __fdiv_rn(bf16hi(w[k]), scale) : 0.f;
        }
        const uint32_t c0 = pack_e4m3x4(f[0], f[1], f[2], f[3]);
        const uint32_t c1 = pack_e4m3x4(f[4], f[5], f[6], f[7]);
        if (!transpose) {
            if (r0 + row < N)
                *reinterpret_cast<uint2 *>(Y + ((size_t)bh * N + r0 + row) * D + cv * 8) = make_uint2(c0, c1);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                tr[(cv * 8 + k) * TS + row] = (uint8_t)(c0 >> (8 * k));
                tr[(cv * 8 + 4 + k) * TS + row] = (uint8_t)(c1 >> (8 * k));
            }
        }
    }
    if (transpose) {
        __syncthreads();
        // column c of the block -> 128 bytes of row c of V^T, in 16-byte pieces
        for (int idx = tid; idx < D * 8; idx += 256) {
            const int c = idx >> 3, piece = idx & 7;
            const int col = r0 + piece * 16;
            if (col < Np)
                *reinterpret_cast<uint4 *>(Y + ((size_t)bh * D + c) * Np + col) =
                    *reinterpret_cast<const uint4 *>(tr + c * TS + piece * 16);
        }
    }
}

}  // namespace

cudaError_t launch_quant_fp8(int d, const void *X, void *Y, float *scales, int BH, int N, int transpose,
                             cudaStream_t st) {
    const int T = (N + 127) / 128;
    const int Np = (N + 15) / 16 * 16;
    const unsigned grid = (unsigned)BH * (unsigned)T;
    if (d == 64)
        fa_quant_fp8_kernel<64><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(X),
                                                      static_cast<uint8_t *>(Y), scales, N, T, Np, transpose);
    else
        fa_quant_fp8_kernel<128><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(X),
                                                       static_cast<uint8_t *>(Y), scales, N, T, Np, transpose);
    return cudaGetLastError();
}

}  // namespace fa
