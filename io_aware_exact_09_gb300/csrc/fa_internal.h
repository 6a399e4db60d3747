// fa_internal.h -- host-side launchers shared by the API translation unit and
// the kernel translation units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_tiles.cuh"

namespace fa {

// Multiprocessor count of the current device (cached per device).
int device_sm_count();

// The forward lists an item's key tiles under a block mask in shared memory,
// at most this many per row (its list capacity); a call with a block mask
// over more key tiles returns FA_ERR_UNSUPPORTED before enqueuing anything.
constexpr int kFwdMaxMaskedKeyTiles = 2048;

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous kernel in the stream drains, and waits for it on the
// device (grid_dep_wait() in fa_ptx.cuh, the first statement of every kernel
// launched this way).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dep(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                              cudaStream_t st, const Args &...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Forward: a persistent grid of at most one CTA per SM over (query-tile pair,
// b*h) work items; the workspace's words 2 and 3 hold its item counter.
cudaError_t launch_fwd(int d, const FwdParams &p, cudaStream_t st);
int fwd_smem_bytes(int d);
// Forward with a chosen key-tile width (64 or 128); p.qpc sets the query
// tiles per CTA.
cudaError_t launch_fwd_tiles(int d, int block_k, const FwdParams &p, cudaStream_t st);
// Ragged batches: packed [total][H][d] sequences (cu_q, cu_k offsets).
cudaError_t launch_fwd_varlen(int d, const FwdParams &p, cudaStream_t st);
// FP8 forward (d = 128): e4m3 Q, K, V^T with per-block scales.
cudaError_t launch_fwd_fp8(const FwdParams &p, cudaStream_t st);
// The forward's split of the last wave: at most this many parts, one slot of
// kFwdSplitSlotBytes each (two query tiles x 128 rows: 128 fp32 of O, m, l).
constexpr int kFwdSplitMaxParts = 512;
constexpr size_t kFwdSplitSlotBytes = 2 * 128 * (128 + 2) * 4;
// FP8 block quantisation of one bf16 tensor [BH][N][d] (V: transposed);
// with signs (Q, K only), of the incoherently rotated rows (x * signs) H.
cudaError_t launch_quant_fp8(int d, const void *X, void *Y, float *scales, int BH, int N, int transpose,
                             const int8_t *signs, cudaStream_t st);

// Backward: D = rowsum(dO * O) and dQacc = 0; the main kernel; dQ = bf16(scale * dQacc).
cudaError_t launch_bwd_pre(int d, const void *O, const void *dO, float *Dvec, float *dQacc,
                           int64_t rows, cudaStream_t st);
cudaError_t launch_bwd_main(int d, const BwdParams &p, cudaStream_t st);
// Ragged batches: packed [total][H][d] sequences (cu_q, cu_k offsets).
cudaError_t launch_bwd_main_varlen(int d, const BwdParams &p, cudaStream_t st);
cudaError_t launch_bwd_convert(int d, const float *dQacc, void *dQ, int64_t elems, float scale,
                               cudaStream_t st);
int bwd_query_block(int d);
// Workspace of the backward without the d = 128 split area: the status block,
// D and the dQ accumulator (what fa_bwd requires).
size_t bwd_base_workspace_bytes(int B, int H, int N, int d);
// The d = 128 split: at most this many split items (byte counters in the
// status block's words 8..63) and parts (fp32 slots of 128 x 256).
constexpr int kSplitMaxItems = 224;
constexpr int kSplitMaxParts = 256;
// d = 64: the persistent kernel (fa_bwd64.cu); the workspace's words 2 and 3
// hold its item counter.
cudaError_t launch_bwd64_main(const BwdParams &p, cudaStream_t st);
cudaError_t launch_bwd64_main_varlen(const BwdParams &p, cudaStream_t st);
int bwd64_smem_bytes();
// d = 128: the 128-row query block kernel (fa_bwd128.cu).
cudaError_t launch_bwd128_main(const BwdParams &p, cudaStream_t st);
cudaError_t launch_bwd128_main_varlen(const BwdParams &p, cudaStream_t st);
int bwd128_smem_bytes();
int bwd_dq_box_rows(int d);
int bwd_smem_bytes(int d);

// Decode: split-KV partials, then the merge.
cudaError_t launch_decode(int d, const DecParams &p, cudaStream_t st);
cudaError_t launch_decode_merge(int d, const float *Opart, const float *Lpart, void *O, float *LSE,
                                int64_t rows, int splits, cudaStream_t st);

// Failure-path self-test: a bounded wait on a barrier nothing completes.
cudaError_t launch_selftest_wait(unsigned *status, unsigned *result, cudaStream_t st);

// Plan export.
cudaError_t launch_plan(int B, int N, int causal, const int32_t *key_len,
                        const uint8_t *block_mask, uint8_t *plan, unsigned *status,
                        cudaStream_t st);

}  // namespace fa
