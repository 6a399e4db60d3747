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
// Persistent CTAs of 256 threads loop over the blocks; each block is copied
// into shared memory (cp.async, 16 bytes per thread and copy, rows past N
// zero-filled) while the previous one is quantised: block amax, then the codes
// (row layout: 8 bytes per thread per vector; transposed: each thread writes
// 32 consecutive codes of one row of V^T, read column-wise from the staged
// block).  2 bytes read and 1 written per element.
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

#include <algorithm>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

namespace {

template <int D>
struct QuantShape {
    static constexpr int VPR = D / 8;                  // 16-byte vectors per row
    static constexpr int NV = 128 * VPR / 256;         // vectors per thread per block
    static constexpr int BUF = 128 * VPR;              // one block in shared memory, in 16-byte vectors
    static constexpr int SMEM_BYTES = 2 * BUF * 16;    // two blocks: the one in work, the next in flight
};

// Persistent: CTA c quantises blocks c, c + gridDim.x, ...  The next block
// is copied into the other shared buffer (cp.async, rows past N zero-filled)
// while this one is worked on, so the load latency is hidden behind the
// arithmetic (the block amax, the exact fp32 divisions, the conversions).
template <int D, bool TRANSPOSE, bool ROTATE>
__global__ void __launch_bounds__(256) fa_quant_fp8_kernel(const __nv_bfloat16 *__restrict__ X,
                                                           uint8_t *__restrict__ Y, float *__restrict__ scales,
                                                           const int8_t *__restrict__ signs, int N, int T, int Np,
                                                           int nblk) {
    grid_dep_wait();                                 // the previous kernel in the stream is done
    grid_dep_launch();
    static_assert(!(ROTATE && TRANSPOSE), "the rotation is for Q and K (row layout)");
    using Q = QuantShape<D>;
    constexpr int VPR = Q::VPR, NV = Q::NV;
    extern __shared__ __align__(16) uint4 qbuf[];      // [2][128 rows x VPR vectors]
    __shared__ float red[2][8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t qbase = smem_u32(qbuf);

    auto load = [&](int blk, int s) {
        const int bh = blk / T, r0 = (blk % T) * 128;
        const __nv_bfloat16 *xb = X + ((size_t)bh * N + r0) * D;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int idx = tid + 256 * i, row = idx / VPR, cv = idx % VPR;
            const bool in = r0 + row < N;
            cp_async16_zfill(qbase + (uint32_t)(s * Q::BUF + idx) * 16u,
                             in ? static_cast<const void *>(xb + (size_t)row * D + cv * 8) : static_cast<const void *>(X),
                             in ? 16u : 0u);
        }
        cp_async_commit();
    };

    int k = 0;
    if ((int)blockIdx.x < nblk) load(blockIdx.x, 0);
    for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x, ++k) {
        const int s = k & 1;
        if (blk + (int)gridDim.x < nblk) {
            load(blk + gridDim.x, s ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();                                // this block's data is in buffer s
        const uint4 *bb = qbuf + s * Q::BUF;
        const int bh = blk / T, r0 = (blk % T) * 128;

        // rotated path: the thread's 8 values of each of its rows, in fp32
        float f[ROTATE ? NV : 1][8];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int idx = tid + 256 * i, cv = idx % VPR;
            const uint4 v = bb[idx];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            if constexpr (ROTATE) {
                // columns 8 cv .. 8 cv + 7 (cv is the same for all i: 256 is a
                // multiple of VPR)
                const uint2 sg = __ldg(reinterpret_cast<const uint2 *>(signs) + cv);
                const uint32_t sb[2] = {sg.x, sg.y};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float x = (e & 1) ? bf16hi(w[e >> 1]) : bf16lo(w[e >> 1]);
                    const int8_t sgn = (int8_t)((sb[e >> 2] >> (8 * (e & 3))) & 0xFFu);
                    f[i][e] = sgn < 0 ? -x : x;
                }
#pragma unroll
                for (int h = 1; h < 8; h <<= 1)
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (!(e & h)) {
                            const float a = f[i][e], b = f[i][e + h];
                            f[i][e] = a + b;
                            f[i][e + h] = a - b;
                        }
#pragma unroll
                for (int j = 1; j < VPR; j <<= 1)
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float pv = __shfl_xor_sync(0xffffffffu, f[i][e], j);
                        f[i][e] = (cv & j) ? pv - f[i][e] : f[i][e] + pv;
                    }
#pragma unroll
                for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[i][e]));
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(w[e])), fabsf(bf16hi(w[e]))));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) red[s][warp] = amax;
        __syncthreads();
        amax = red[s][0];
#pragma unroll
        for (int w8 = 1; w8 < 8; ++w8) amax = fmaxf(amax, red[s][w8]);
        const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
        if (tid == 0) scales[blk] = scale;
        auto q = [&](float x) { return scale > 0.f ? __fdiv_rn(x, scale) : 0.f; };

        if constexpr (!TRANSPOSE) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int idx = tid + 256 * i, row = idx / VPR, cv = idx % VPR;
                float e[8];
                if constexpr (ROTATE) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) e[j] = f[i][j];
                } else {
                    const uint4 v = bb[idx];
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) e[j] = (j & 1) ? bf16hi(w[j >> 1]) : bf16lo(w[j >> 1]);
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
            const __nv_bfloat16 *blkv = reinterpret_cast<const __nv_bfloat16 *>(bb);
            constexpr int TASKS = D * 4;
#pragma unroll 1
            for (int task = tid; task < TASKS; task += 256) {
                const int c = task % D, seg = task / D;
                uint32_t w[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int rr = seg * 32 + 4 * j;
                    w[j] = pack_e4m3x4(q(__bfloat162float(blkv[(rr + 0) * D + c])),
                                       q(__bfloat162float(blkv[(rr + 1) * D + c])),
                                       q(__bfloat162float(blkv[(rr + 2) * D + c])),
                                       q(__bfloat162float(blkv[(rr + 3) * D + c])));
                }
                const int col = r0 + seg * 32;
                uint8_t *dst = Y + ((size_t)bh * D + c) * Np + col;
                if (col < Np) *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
                if (col + 16 < Np) *reinterpret_cast<uint4 *>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
        __syncthreads();                                // buffer s is refilled two blocks later
    }
}

template <int D, bool TRANSPOSE, bool ROTATE>
cudaError_t launch_quant_t(const __nv_bfloat16 *x, uint8_t *y, float *scales, const int8_t *signs, int N, int T,
                           int Np, int nblk, cudaStream_t st) {
    constexpr int smem = QuantShape<D>::SMEM_BYTES;
    auto kern = fa_quant_fp8_kernel<D, TRANSPOSE, ROTATE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem)) != cudaSuccess)
        return e;
    const int grid = std::max(1, std::min(nblk, sms * std::max(per_sm, 1)));
    return launch_dep(kern, grid, 256, smem, st, x, y, scales, signs, N, T, Np, nblk);
}

}  // namespace

cudaError_t launch_quant_fp8(int d, const void *X, void *Y, float *scales, int BH, int N, int transpose,
                             const int8_t *signs, cudaStream_t st) {
    const int T = (N + 127) / 128;
    const int Np = (N + 15) / 16 * 16;
    const int nblk = BH * T;
    const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(X);
    uint8_t *y = static_cast<uint8_t *>(Y);
    if (nblk == 0) return cudaSuccess;
    if (d == 64) {
        if (transpose) return launch_quant_t<64, true, false>(x, y, scales, nullptr, N, T, Np, nblk, st);
        if (signs) return launch_quant_t<64, false, true>(x, y, scales, signs, N, T, Np, nblk, st);
        return launch_quant_t<64, false, false>(x, y, scales, nullptr, N, T, Np, nblk, st);
    }
    if (transpose) return launch_quant_t<128, true, false>(x, y, scales, nullptr, N, T, Np, nblk, st);
    if (signs) return launch_quant_t<128, false, true>(x, y, scales, signs, N, T, Np, nblk, st);
    return launch_quant_t<128, false, false>(x, y, scales, nullptr, N, T, Np, nblk, st);
}

}  // namespace fa
