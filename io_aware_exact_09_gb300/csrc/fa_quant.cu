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
// vector; transposed: the block is staged in shared memory and each thread
// writes 32 consecutive codes of one row of V^T).
// HBM-bound: 2 bytes read and 1 written per element.
//
// Incoherent processing (same chapter's FlashAttention-3 paragraph: "block
// quantization with incoherent processing"), for Q and K: before the block
// amax, each row x becomes (x * s) H, s a caller-given vector of random
// signs and H the unnormalised d x d Sylvester-Hadamard matrix, so that
// (Q s H)(K s H)^T = d Q K^T and a few large channels are spread over all d.
// The fast Walsh-Hadamard transform runs in fp32, stage h = 1, 2, 4, ...,
// d/2 turning each pair (i, i + h) into (x_i + x_{i+h}, x_i - x_{i+h}): the
// first three stages inside a thread's 8 values, the rest across the lanes
// that hold the row (its 16-byte vectors sit in consecutive lanes).
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

namespace {

template <int D, bool TRANSPOSE, bool ROTATE>
__global__ void __launch_bounds__(256) fa_quant_fp8_kernel(const __nv_bfloat16 *__restrict__ X,
                                                           uint8_t *__restrict__ Y, float *__restrict__ scales,
                                                           const int8_t *__restrict__ signs, int N, int T, int Np) {
    static_assert(!(ROTATE && TRANSPOSE), "the rotation is for Q and K (row layout)");
    constexpr int VPR = D / 8;                 // 16-byte vectors per row
    constexpr int NV = 128 * VPR / 256;        // vectors per thread
    __shared__ float red[8];
    // transposed path: the bf16 block, read back column by column
    __shared__ __align__(16) __nv_bfloat16 blk[TRANSPOSE ? 128 * D : 8];
    const int bh = (int)(blockIdx.x / T), t = (int)(blockIdx.x % T);
    const int r0 = t * 128;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const __nv_bfloat16 *xb = X + ((size_t)bh * N + r0) * D;

    uint4 v[NV];
    // rotated path: the thread's 8 values of each of its rows, in fp32
    float f[ROTATE ? NV : 1][8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int idx = tid + 256 * i, row = idx / VPR, cv = idx % VPR;
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (r0 + row < N) v[i] = __ldg(reinterpret_cast<const uint4 *>(xb + (size_t)row * D) + cv);
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        if constexpr (ROTATE) {
            // columns 8 cv .. 8 cv + 7 (cv is the same for all i: 256 is a
            // multiple of VPR)
            const uint2 sg = __ldg(reinterpret_cast<const uint2 *>(signs) + cv);
            const uint32_t sb[2] = {sg.x, sg.y};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float x = (k & 1) ? bf16hi(w[k >> 1]) : bf16lo(w[k >> 1]);
                const int8_t s = (int8_t)((sb[k >> 2] >> (8 * (k & 3))) & 0xFFu);
                f[i][k] = s < 0 ? -x : x;
            }
#pragma unroll
            for (int h = 1; h < 8; h <<= 1)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (!(k & h)) {
                        const float a = f[i][k], b = f[i][k + h];
                        f[i][k] = a + b;
                        f[i][k + h] = a - b;
                    }
#pragma unroll
            for (int j = 1; j < VPR; j <<= 1)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float pv = __shfl_xor_sync(0xffffffffu, f[i][k], j);
                    f[i][k] = (cv & j) ? pv - f[i][k] : f[i][k] + pv;
                }
#pragma unroll
            for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(f[i][k]));
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(w[k])), fabsf(bf16hi(w[k]))));
        }
        if constexpr (TRANSPOSE) reinterpret_cast<uint4 *>(blk)[idx] = v[i];
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
    auto q = [&](float x) { return scale > 0.f ? __fdiv_rn(x, scale) : 0.f; };

    if constexpr (!TRANSPOSE) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int idx = tid + 256 * i, row = idx / VPR, cv = idx % VPR;
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            float e[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if constexpr (ROTATE)
                    e[k] = f[i][k];
                else
                    e[k] = (k & 1) ? bf16hi(w[k >> 1]) : bf16lo(w[k >> 1]);
            }
            const uint32_t c0 = pack_e4m3x4(q(e[0]), q(e[1]), q(e[2]), q(e[3]));
            const uint32_t c1 = pack_e4m3x4(q(e[4]), q(e[5]), q(e[6]), q(e[7]));
            if (r0 + row < N)
                *reinterpret_cast<uint2 *>(Y + ((size_t)bh * N + r0 + row) * D + cv * 8) = make_uint2(c0, c1);
        }
    } else {
        // task (column c, 32-row segment): 32 codes = 32 contiguous bytes of
        // row c of V^T; a warp covers 32 consecutive columns, so its shared
        // reads are 64 contiguous bytes per row
        constexpr int TASKS = D * 4;
#pragma unroll 1
        for (int task = tid; task < TASKS; task += 256) {
            const int c = task % D, seg = task / D;
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int rr = seg * 32 + 4 * k;
                w[k] = pack_e4m3x4(q(__bfloat162float(blk[(rr + 0) * D + c])), q(__bfloat162float(blk[(rr + 1) * D + c])),
                                   q(__bfloat162float(blk[(rr + 2) * D + c])), q(__bfloat162float(blk[(rr + 3) * D + c])));
            }
            const int col = r0 + seg * 32;
            uint8_t *dst = Y + ((size_t)bh * D + c) * Np + col;
            if (col < Np) *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            if (col + 16 < Np) *reinterpret_cast<uint4 *>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
        }
    }
}

}  // namespace

cudaError_t launch_quant_fp8(int d, const void *X, void *Y, float *scales, int BH, int N, int transpose,
                             const int8_t *signs, cudaStream_t st) {
    const int T = (N + 127) / 128;
    const int Np = (N + 15) / 16 * 16;
    const unsigned grid = (unsigned)BH * (unsigned)T;
    const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(X);
    uint8_t *y = static_cast<uint8_t *>(Y);
    if (d == 64) {
        if (transpose)
            fa_quant_fp8_kernel<64, true, false><<<grid, 256, 0, st>>>(x, y, scales, nullptr, N, T, Np);
        else if (signs)
            fa_quant_fp8_kernel<64, false, true><<<grid, 256, 0, st>>>(x, y, scales, signs, N, T, Np);
        else
            fa_quant_fp8_kernel<64, false, false><<<grid, 256, 0, st>>>(x, y, scales, nullptr, N, T, Np);
    } else {
        if (transpose)
            fa_quant_fp8_kernel<128, true, false><<<grid, 256, 0, st>>>(x, y, scales, nullptr, N, T, Np);
        else if (signs)
            fa_quant_fp8_kernel<128, false, true><<<grid, 256, 0, st>>>(x, y, scales, signs, N, T, Np);
        else
            fa_quant_fp8_kernel<128, false, false><<<grid, 256, 0, st>>>(x, y, scales, nullptr, N, T, Np);
    }
    return cudaGetLastError();
}

}  // namespace fa
