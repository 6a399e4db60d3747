// fa_api.cu -- the C ABI declared in include/fa.h: argument checks, TMA
// descriptor encoding, kernel launches, the host-buffer convenience path and
// the device status word.  Host code only; the kernels live in fa_fwd.cu and
// fa_bwd.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

using fa::BwdParams;
using fa::DecParams;
using fa::FwdParams;

constexpr size_t kStatusBytes = 256;

inline size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 3-D bf16 view [BH][N][d] of a contiguous [B, H, N, d] tensor; box of
// 64 columns x box_rows rows x 1 head, 128-byte swizzle, zero fill outside.
bool encode_bf16_3d(CUtensorMap *m, const void *ptr, int d, int N, int BH, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view [total][H][d] of packed (ragged-batch) bf16 rows: box of 64
// columns of one head x box_rows rows, 128-byte swizzle.
bool encode_bf16_thd(CUtensorMap *m, const void *ptr, int d, int H, int total, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)total};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D byte view [outer][rows][inner] of e4m3 codes; box of 128 bytes x
// box_rows rows, 128-byte swizzle (FP8 Q, K: inner = d = 128; V^T: inner =
// Np, rows = d).
bool encode_u8_3d(CUtensorMap *m, const void *ptr, int inner, int rows, int outer, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)outer};
    cuuint64_t strides[2] = {(cuuint64_t)inner, (cuuint64_t)rows * inner};
    cuuint32_t box[3] = {128, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp32 view [BH][N][d] of the dQ accumulator; box of 32 columns (128
// bytes) x box_rows rows, 128-byte swizzle (target of the TMA reduce-add).
bool encode_f32_3d(CUtensorMap *m, const void *ptr, int d, int N, int BH, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
    cuuint32_t box[3] = {32, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp32 view [total][H][d] of a ragged batch's dQ accumulator; box of
// 32 columns of one head x box_rows rows, 128-byte swizzle.
bool encode_f32_thd(CUtensorMap *m, const void *ptr, int d, int H, int total, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)total};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)H * d * 4};
    cuuint32_t box[3] = {32, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Checks shared by fa_fwd / fa_bwd / fa_tile_plan.  Returns FA_OK, or the
// error to report; *empty is set when there is nothing to compute.
fa_status check_sizes(int B, int H, int N, int d, bool *empty) {
    *empty = false;
    if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARGUMENT;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if ((int64_t)B * H * N == 0) {
        *empty = true;
        return FA_OK;
    }
    const int64_t BH = (int64_t)B * H;
    const int64_t T = ((int64_t)N + 127) / 128;
    if (BH > INT_MAX || T * BH > INT_MAX) return FA_ERR_UNSUPPORTED;
    // TMA: global byte strides below 2^40
    if ((int64_t)N * d * 2 >= (int64_t(1) << 40)) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }

using fa::kFwdMaxMaskedKeyTiles;

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace

namespace fa {
size_t bwd_base_workspace_bytes(int B, int H, int N, int d) {
    if (B < 0 || H < 0 || N < 0 || d <= 0) return 0;
    const size_t rows = (size_t)B * H * N;
    return kStatusBytes + round256(rows * 4) + round256(rows * (size_t)d * 4);
}
}  // namespace fa

namespace {
// d = 128: slots for the split of the last wave's items (fa_bwd128.cu), one
// fp32 [128 keys][dK 128 | dV 128] slot per part; at most four parts per
// item, one per query block, kSplitMaxParts in all.  Their counters live in
// the status block, so this area needs no zero fill.
constexpr size_t kSplitSlotBytes = 128 * 256 * 4;
size_t bwd_split_parts(int B, int H, int N, int d) {
    if (d != 128 || B <= 0 || H <= 0 || N <= 128) return 0;
    const int64_t T = (N + 127) / 128;
    const int64_t bh = (int64_t)B * H;
    const int64_t per = T * std::min<int64_t>(4, T);
    if (bh >= fa::kSplitMaxParts || per >= fa::kSplitMaxParts) return fa::kSplitMaxParts;
    return (size_t)std::min<int64_t>(fa::kSplitMaxParts, bh * per);
}
// d = 128, at least 32 key tiles: slots for the forward's split of its last
// wave (fa_fwd_fp8.cu), at most four parts per item of two query tiles, 16
// key tiles per part at least, kFwdSplitMaxParts in all.
size_t fwd_split_parts(int B, int H, int N, int d) {
    if (d != 128 || B <= 0 || H <= 0 || N < 32 * 128) return 0;
    const int64_t T = (N + 127) / 128;
    const int64_t bh = (int64_t)B * H;
    const int64_t per = (T + 1) / 2 * std::min<int64_t>(4, T / 16);
    if (bh >= fa::kFwdSplitMaxParts || per >= fa::kFwdSplitMaxParts) return fa::kFwdSplitMaxParts;
    return (size_t)std::min<int64_t>(fa::kFwdSplitMaxParts, bh * per);
}
}  // namespace

extern "C" {

int fa_tile_size(void) { return fa::kTile; }

size_t fa_fwd_workspace_size(int B, int H, int N, int d) {
    return kStatusBytes + fwd_split_parts(B, H, N, d) * fa::kFwdSplitSlotBytes;
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
    const size_t base = fa::bwd_base_workspace_bytes(B, H, N, d);
    if (base == 0) return 0;
    return base + bwd_split_parts(B, H, N, d) * kSplitSlotBytes;
}

const char *fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "ok";
        case FA_ERR_INVALID_ARGUMENT: return "invalid argument";
        case FA_ERR_UNSUPPORTED: return "unsupported configuration";
        case FA_ERR_WORKSPACE: return "workspace missing or too small";
        case FA_ERR_CUDA: return "CUDA error";
        case FA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case FA_ERR_DEVICE_BAD_KEY_LEN: return "key_len value outside [0, N] (clamped)";
    }
    return "unknown status";
}

// Persistent grids hand out work items head-major (the heaviest items of a
// head first) unless the items differ in length and spreading them across
// heads keeps L2 useful.  Spread order (the heaviest items of every head
// first) gives the shortest tail: head-major would start the last head's
// heaviest item near the end of the launch, where it runs alone.  But the
// CTAs at work at one time then touch as many heads as there are CTAs, so it
// is taken only when the data of all heads is within about 1.5 L2 capacities
// (the forward's K and V; the backward's Q, dO, K, V and fp32 dQ accumulator)
// or when there are few enough heads that each one still has several CTAs at
// work on it.  Measured on one GPU: causal B8 H16 N1024 d64 step 0.184 ->
// 0.155 ms; causal d128 forwards B1 H16 N16384 0.905 -> 0.814 ms, B4 H16
// N4096 0.283 -> 0.267 ms, B16 H16 N1024 0.128 -> 0.117 ms (134 MB of K and
// V); block-sparse B2 H16 N8192 d64 backward 0.315 -> 0.242 ms; a ragged
// batch of 16 x 16 sequence-heads (329 MB of K and V) was slower spread,
// 0.501 -> 0.549 ms.
// When neither holds (non-ragged problems only) the heads go in groups of 8,
// the items spread across a group's heads and the groups in order, so that
// the last items handed out are the last group's lightest while the CTAs at
// work touch about 8 heads.  The value is the group size the kernels map
// item indices with: every head (spread), 8, or 0 (head-major).
constexpr double kSpreadL2Bytes = 192.0 * (1 << 20);
static int spread_items(bool lengths_vary, double bytes, int64_t heads, bool ragged = false) {
    if (!lengths_vary) return 0;
    if (bytes <= kSpreadL2Bytes || heads * 4 <= fa::device_sm_count()) return (int)heads;
    return (ragged || heads <= 8) ? 0 : 8;
}

fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int N,
                 int d, float softmax_scale, int causal, const int32_t *key_len,
                 const uint8_t *block_mask, void *workspace, size_t workspace_bytes, void *stream) {
    bool empty = false;
    fa_status st = check_sizes(B, H, N, d, &empty);
    if (st != FA_OK) return st;
    if (!scale_ok(softmax_scale)) return FA_ERR_INVALID_ARGUMENT;
    if (empty) return FA_OK;
    if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARGUMENT;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
        return FA_ERR_INVALID_ARGUMENT;
    if (!workspace || !aligned16(workspace) || workspace_bytes < kStatusBytes) return FA_ERR_WORKSPACE;
    if (block_mask && (N + 127) / 128 > kFwdMaxMaskedKeyTiles) return FA_ERR_UNSUPPORTED;

    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    const int BH = B * H;
    if (!encode_bf16_3d(&p.tmQ, Q, d, N, BH, 128) || !encode_bf16_3d(&p.tmK, K, d, N, BH, 128) ||
        !encode_bf16_3d(&p.tmV, V, d, N, BH, 128))
        return FA_ERR_CUDA;
    p.O = O;
    p.LSE = LSE;
    p.key_len = key_len;
    p.block_mask = block_mask;
    p.status = static_cast<unsigned *>(workspace);
    p.H = H;
    p.N = N;
    p.BH = BH;
    p.Tq = (N + 127) / 128;
    p.Tk = p.Tq;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = softmax_scale * kLog2e;
    p.spread = spread_items(causal || key_len || block_mask, 4.0 * BH * N * d, BH);
    return fa::launch_fwd(d, p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_tiles(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int N, int d,
                       float softmax_scale, int causal, const int32_t *key_len, const uint8_t *block_mask, int block_q,
                       int block_k, void *workspace, size_t workspace_bytes, void *stream) {
    if (block_q != 128 && block_q != 256) return FA_ERR_UNSUPPORTED;
    if (block_k != 64 && block_k != 128) return FA_ERR_UNSUPPORTED;
    bool empty = false;
    fa_status st = check_sizes(B, H, N, d, &empty);
    if (st != FA_OK) return st;
    if (!scale_ok(softmax_scale)) return FA_ERR_INVALID_ARGUMENT;
    if (empty) return FA_OK;
    if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARGUMENT;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
        return FA_ERR_INVALID_ARGUMENT;
    if (!workspace || !aligned16(workspace) || workspace_bytes < kStatusBytes) return FA_ERR_WORKSPACE;
    if (block_mask && (N + block_k - 1) / block_k > kFwdMaxMaskedKeyTiles) return FA_ERR_UNSUPPORTED;
    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    const int BH = B * H;
    if (!encode_bf16_3d(&p.tmQ, Q, d, N, BH, 128) || !encode_bf16_3d(&p.tmK, K, d, N, BH, block_k) ||
        !encode_bf16_3d(&p.tmV, V, d, N, BH, block_k))
        return FA_ERR_CUDA;
    p.O = O;
    p.LSE = LSE;
    p.key_len = key_len;
    p.block_mask = block_mask;
    p.status = static_cast<unsigned *>(workspace);
    p.H = H;
    p.N = N;
    p.BH = BH;
    p.Tq = (N + 127) / 128;
    p.Tk = (N + block_k - 1) / block_k;
    p.qpc = block_q / 128;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = softmax_scale * kLog2e;
    return fa::launch_fwd_tiles(d, block_k, p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                                  : FA_ERR_CUDA;
}

fa_status fa_fwd_varlen(const void *Q, const void *K, const void *V, void *O, float *LSE, const int32_t *cu_seqlens_q,
                        const int32_t *cu_seqlens_k, int B, int H, int total_q, int total_k, int max_seqlen_q, int d,
                        float softmax_scale, int causal, void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 0 || H <= 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0) return FA_ERR_INVALID_ARGUMENT;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!scale_ok(softmax_scale)) return FA_ERR_INVALID_ARGUMENT;
    if (B == 0 || total_q == 0 || max_seqlen_q == 0) return FA_OK;
    const int64_t Tq = ((int64_t)max_seqlen_q + 127) / 128;
    if ((int64_t)B * H > INT_MAX || (Tq + 1) / 2 * (int64_t)B * H > INT_MAX) return FA_ERR_UNSUPPORTED;
    if ((int64_t)total_q * H * d * 2 >= (int64_t(1) << 40) || (int64_t)total_k * H * d * 2 >= (int64_t(1) << 40))
        return FA_ERR_UNSUPPORTED;
    if (!Q || !O || !LSE || !cu_seqlens_q || !cu_seqlens_k || !aligned16(Q) || !aligned16(O) || !aligned16(LSE))
        return FA_ERR_INVALID_ARGUMENT;
    if (total_k > 0 && (!K || !V || !aligned16(K) || !aligned16(V))) return FA_ERR_INVALID_ARGUMENT;
    if (!workspace || !aligned16(workspace) || workspace_bytes < fa_fwd_workspace_size(1, 1, 1, d))
        return FA_ERR_WORKSPACE;
    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    // a sequence without keys still needs valid maps: point K, V at Q then
    // (no key tile is ever loaded for it)
    const void *Km = total_k > 0 ? K : Q, *Vm = total_k > 0 ? V : Q;
    const int tk = total_k > 0 ? total_k : total_q;
    if (!encode_bf16_thd(&p.tmQ, Q, d, H, total_q, 128) || !encode_bf16_thd(&p.tmK, Km, d, H, tk, 128) ||
        !encode_bf16_thd(&p.tmV, Vm, d, H, tk, 128))
        return FA_ERR_CUDA;
    p.O = O;
    p.LSE = LSE;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.total_q = total_q;
    p.total_k = total_k;
    p.status = static_cast<unsigned *>(workspace);
    p.H = H;
    p.N = 0;
    p.BH = B * H;
    p.Tq = (int)Tq;
    p.Tk = 0;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = softmax_scale * kLog2e;
    p.spread = spread_items(true, 4.0 * total_k * H * d, (int64_t)B * H, true);
    return fa::launch_fwd_varlen(d, p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_quantize_fp8(const void *X, void *X8, float *scales, int B, int H, int N, int d, int transpose,
                          void *stream) {
    bool empty = false;
    fa_status st = check_sizes(B, H, N, d, &empty);
    if (st != FA_OK) return st;
    if (empty) return FA_OK;
    if (!X || !X8 || !scales || !aligned16(X) || !aligned16(X8) || !aligned16(scales))
        return FA_ERR_INVALID_ARGUMENT;
    return fa::launch_quant_fp8(d, X, X8, scales, B * H, N, transpose ? 1 : 0, nullptr,
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
}

fa_status fa_quantize_fp8_rotated(const void *X, void *X8, float *scales, const int8_t *signs, int B, int H, int N,
                                  int d, void *stream) {
    bool empty = false;
    fa_status st = check_sizes(B, H, N, d, &empty);
    if (st != FA_OK) return st;
    if (empty) return FA_OK;
    if (!X || !X8 || !scales || !signs || !aligned16(X) || !aligned16(X8) || !aligned16(scales) || !aligned16(signs))
        return FA_ERR_INVALID_ARGUMENT;
    return fa::launch_quant_fp8(d, X, X8, scales, B * H, N, 0, signs, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
}

fa_status fa_fwd_fp8(const void *Q8, const void *K8, const void *Vt8, const float *sQ, const float *sK,
                     const float *sV, void *O, float *LSE, int B, int H, int N, int d, float softmax_scale,
                     int causal, const int32_t *key_len, const uint8_t *block_mask, void *workspace,
                     size_t workspace_bytes, void *stream) {
    bool empty = false;
    fa_status st = check_sizes(B, H, N, d, &empty);
    if (st != FA_OK) return st;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if (!scale_ok(softmax_scale)) return FA_ERR_INVALID_ARGUMENT;
    if (empty) return FA_OK;
    if (!Q8 || !K8 || !Vt8 || !sQ || !sK || !sV || !O || !LSE) return FA_ERR_INVALID_ARGUMENT;
    if (!aligned16(Q8) || !aligned16(K8) || !aligned16(Vt8) || !aligned16(O) || !aligned16(LSE))
        return FA_ERR_INVALID_ARGUMENT;
    if (!workspace || !aligned16(workspace) || workspace_bytes < kStatusBytes) return FA_ERR_WORKSPACE;
    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    const int BH = B * H;
    const int Np = (N + 15) / 16 * 16;
    if (!encode_u8_3d(&p.tmQ, Q8, d, N, BH, 128) || !encode_u8_3d(&p.tmK, K8, d, N, BH, 128) ||
        !encode_u8_3d(&p.tmV, Vt8, Np, d, BH, d))
        return FA_ERR_CUDA;
    p.sQ = sQ;
    p.sK = sK;
    p.sV = sV;
    p.O = O;
    p.LSE = LSE;
    p.key_len = key_len;
    p.block_mask = block_mask;
    p.status = static_cast<unsigned *>(workspace);
    p.H = H;
    p.N = N;
    p.BH = BH;
    p.Tq = (N + 127) / 128;
    p.Tk = p.Tq;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = softmax_scale * kLog2e;
    // the split area, when the workspace holds it (the launcher decides whether to split)
    const size_t parts = fwd_split_parts(B, H, N, d);
    if (parts >= 2 && workspace_bytes >= kStatusBytes + parts * fa::kFwdSplitSlotBytes) {
        p.split_cnt = p.status + 8;
        p.split_buf = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + kStatusBytes);
        p.split_cap = (int)parts;
    }
    return fa::launch_fwd_fp8(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_fp8_rotated(const void *Q8, const void *K8, const void *Vt8, const float *sQ, const float *sK,
                             const float *sV, void *O, float *LSE, int B, int H, int N, int d, float softmax_scale,
                             int causal, const int32_t *key_len, const uint8_t *block_mask, void *workspace,
                             size_t workspace_bytes, void *stream) {
    if (!scale_ok(softmax_scale)) return FA_ERR_INVALID_ARGUMENT;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    // the rotated scores are d times the unrotated ones: (Q s H)(K s H)^T = d Q K^T
    return fa_fwd_fp8(Q8, K8, Vt8, sQ, sK, sV, O, LSE, B, H, N, d, softmax_scale / (float)d, causal, key_len,
                      block_mask, workspace, workspace_bytes, stream);
}

namespace {
struct BwdWs {
    unsigned *status;
    float *Dvec, *dQacc;
};
BwdWs bwd_ws(void *workspace, int B, int H, int N) {
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t rows = (size_t)B * H * N;
    return BwdWs{reinterpret_cast<unsigned *>(ws), reinterpret_cast<float *>(ws + kStatusBytes),
                 reinterpret_cast<float *>(ws + kStatusBytes + round256(rows * 4))};
}
fa_status bwd_common_checks(int B, int H, int N, int d, float scale, void *workspace, size_t workspace_bytes,
                            bool *empty) {
    fa_status st = check_sizes(B, H, N, d, empty);
    if (st != FA_OK) return st;
    if (!scale_ok(scale)) return FA_ERR_INVALID_ARGUMENT;
    if (*empty) return FA_OK;
    if (!workspace || !aligned16(workspace) || workspace_bytes < fa::bwd_base_workspace_bytes(B, H, N, d))
        return FA_ERR_WORKSPACE;
    return FA_OK;
}
}  // namespace

fa_status fa_bwd_preprocess(const void *O, const void *dO, int B, int H, int N, int d, void *workspace,
                            size_t workspace_bytes, void *stream) {
    bool empty = false;
    fa_status st = bwd_common_checks(B, H, N, d, 1.f, workspace, workspace_bytes, &empty);
    if (st != FA_OK || empty) return st;
    if (!O || !dO || !aligned16(O) || !aligned16(dO)) return FA_ERR_INVALID_ARGUMENT;
    const BwdWs w = bwd_ws(workspace, B, H, N);
    return fa::launch_bwd_pre(d, O, dO, w.Dvec, w.dQacc, (int64_t)B * H * N, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
}

fa_status fa_bwd_main(const void *Q, const void *K, const void *V, const float *LSE, const void *dO, void *dK,
                      void *dV, int B, int H, int N, int d, float softmax_scale, int causal,
                      const int32_t *key_len, const uint8_t *block_mask, void *workspace,
                      size_t workspace_bytes, void *stream) {
    bool empty = false;
    fa_status st = bwd_common_checks(B, H, N, d, softmax_scale, workspace, workspace_bytes, &empty);
    if (st != FA_OK || empty) return st;
    const void *ptrs[] = {Q, K, V, LSE, dO, dK, dV};
    for (const void *x : ptrs)
        if (!x || !aligned16(x)) return FA_ERR_INVALID_ARGUMENT;
    if (block_mask && (N + 127) / 128 > kFwdMaxMaskedKeyTiles) return FA_ERR_UNSUPPORTED;
    const BwdWs w = bwd_ws(workspace, B, H, N);
    const int BH = B * H;
    BwdParams p;
    std::memset(&p, 0, sizeof(p));
    const int BQ = fa::bwd_query_block(d);
    if (!encode_bf16_3d(&p.tmQ, Q, d, N, BH, BQ) || !encode_bf16_3d(&p.tmdO, dO, d, N, BH, BQ) ||
        !encode_bf16_3d(&p.tmK, K, d, N, BH, 128) || !encode_bf16_3d(&p.tmV, V, d, N, BH, 128) ||
        !encode_f32_3d(&p.tmdQ, w.dQacc, d, N, BH, fa::bwd_dq_box_rows(d)))
        return FA_ERR_CUDA;
    p.LSE = LSE;
    p.Dvec = w.Dvec;
    p.dQacc = w.dQacc;
    p.dK = dK;
    p.dV = dV;
    p.key_len = key_len;
    p.block_mask = block_mask;
    p.status = w.status;
    p.H = H;
    p.N = N;
    p.BH = BH;
    p.Tk = (N + 127) / 128;
    p.Tqb = (N + BQ - 1) / BQ;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = softmax_scale * kLog2e;
    p.scale = softmax_scale;
    p.spread = spread_items(causal || key_len || block_mask, 12.0 * BH * N * d, BH);
    // the split area, when the workspace holds it (the launcher decides whether to split)
    const size_t base = fa::bwd_base_workspace_bytes(B, H, N, d);
    const size_t parts = bwd_split_parts(B, H, N, d);
    if (parts >= 2 && workspace_bytes >= base + parts * kSplitSlotBytes) {
        p.split_cnt = w.status + 8;
        p.split_buf = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + base);
        p.split_cap = (int)parts;
    }
    return fa::launch_bwd_main(d, p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bwd_postprocess(void *dQ, int B, int H, int N, int d, float softmax_scale, const void *workspace,
                             size_t workspace_bytes, void *stream) {
    bool empty = false;
    fa_status st =
        bwd_common_checks(B, H, N, d, softmax_scale, const_cast<void *>(workspace), workspace_bytes, &empty);
    if (st != FA_OK || empty) return st;
    if (!dQ || !aligned16(dQ)) return FA_ERR_INVALID_ARGUMENT;
    const BwdWs w = bwd_ws(const_cast<void *>(workspace), B, H, N);
    return fa::launch_bwd_convert(d, w.dQacc, dQ, (int64_t)B * H * N * d, softmax_scale,
                                  static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
}

fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const float *LSE, const void *dO,
                 void *dQ, void *dK, void *dV, int B, int H, int N, int d, float softmax_scale, int causal,
                 const int32_t *key_len, const uint8_t *block_mask, void *workspace, size_t workspace_bytes,
                 void *stream) {
    bool empty = false;
    fa_status st = bwd_common_checks(B, H, N, d, softmax_scale, workspace, workspace_bytes, &empty);
    if (st != FA_OK || empty) return st;
    const void *ptrs[] = {Q, K, V, O, LSE, dO, dQ, dK, dV};
    for (const void *x : ptrs)
        if (!x || !aligned16(x)) return FA_ERR_INVALID_ARGUMENT;
    // the main stage's own check, made here so that a rejected call enqueues nothing
    if (block_mask && (N + 127) / 128 > kFwdMaxMaskedKeyTiles) return FA_ERR_UNSUPPORTED;
    st = fa_bwd_preprocess(O, dO, B, H, N, d, workspace, workspace_bytes, stream);
    if (st != FA_OK) return st;
    st = fa_bwd_main(Q, K, V, LSE, dO, dK, dV, B, H, N, d, softmax_scale, causal, key_len, block_mask, workspace,
                     workspace_bytes, stream);
    if (st != FA_OK) return st;
    return fa_bwd_postprocess(dQ, B, H, N, d, softmax_scale, workspace, workspace_bytes, stream);
}

size_t fa_bwd_varlen_workspace_size(int H, int total_q, int d) {
    if (H < 0 || total_q < 0 || d <= 0) return 0;
    return fa::bwd_base_workspace_bytes(1, H, total_q, d);
}

fa_status fa_bwd_varlen(const void *Q, const void *K, const void *V, const void *O, const float *LSE, const void *dO,
                        void *dQ, void *dK, void *dV, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int B,
                        int H, int total_q, int total_k, int max_seqlen_k, int d, float softmax_scale, int causal,
                        void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 0 || H <= 0 || total_q < 0 || total_k < 0 || max_seqlen_k < 0) return FA_ERR_INVALID_ARGUMENT;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!scale_ok(softmax_scale)) return FA_ERR_INVALID_ARGUMENT;
    if (B == 0 || (total_q == 0 && total_k == 0)) return FA_OK;
    const int64_t Tk = ((int64_t)max_seqlen_k + 127) / 128;
    if ((int64_t)B * H > INT_MAX || Tk * B * H > INT_MAX) return FA_ERR_UNSUPPORTED;
    if ((int64_t)total_q * H * d * 4 >= (int64_t(1) << 40) || (int64_t)total_k * H * d * 2 >= (int64_t(1) << 40))
        return FA_ERR_UNSUPPORTED;
    if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID_ARGUMENT;
    if (total_q > 0) {
        const void *ptrs[] = {Q, O, LSE, dO, dQ};
        for (const void *x : ptrs)
            if (!x || !aligned16(x)) return FA_ERR_INVALID_ARGUMENT;
    }
    if (total_k > 0) {
        const void *ptrs[] = {K, V, dK, dV};
        for (const void *x : ptrs)
            if (!x || !aligned16(x)) return FA_ERR_INVALID_ARGUMENT;
    }
    if (!workspace || !aligned16(workspace) || workspace_bytes < fa_bwd_varlen_workspace_size(H, total_q, d))
        return FA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const BwdWs w = bwd_ws(workspace, 1, H, total_q);
    // D = rowsum(dO * O) and the accumulator zeroed, over the [total_q][H] rows
    if (total_q > 0 &&
        fa::launch_bwd_pre(d, O, dO, w.Dvec, w.dQacc, (int64_t)total_q * H, s) != cudaSuccess)
        return FA_ERR_CUDA;
    if (total_k > 0 && Tk > 0) {
        BwdParams p;
        std::memset(&p, 0, sizeof(p));
        // without queries the maps still need a valid base: point them at K
        // (no query block is ever loaded then)
        const void *Qm = total_q > 0 ? Q : K, *dOm = total_q > 0 ? dO : K;
        const int tq = total_q > 0 ? total_q : total_k;
        if (!encode_bf16_thd(&p.tmQ, Qm, d, H, tq, 128) || !encode_bf16_thd(&p.tmdO, dOm, d, H, tq, 128) ||
            !encode_bf16_thd(&p.tmK, K, d, H, total_k, 128) || !encode_bf16_thd(&p.tmV, V, d, H, total_k, 128) ||
            !encode_f32_thd(&p.tmdQ, total_q > 0 ? (const void *)w.dQacc : K, d, H, tq, fa::bwd_dq_box_rows(d)))
            return FA_ERR_CUDA;
        p.LSE = LSE;
        p.Dvec = w.Dvec;
        p.dQacc = w.dQacc;
        p.dK = dK;
        p.dV = dV;
        p.cu_q = cu_seqlens_q;
        p.cu_k = cu_seqlens_k;
        p.total_q = total_q;
        p.total_k = total_k;
        p.status = w.status;
        p.H = H;
        p.N = 0;
        p.BH = B * H;
        p.Tk = (int)Tk;
        p.Tqb = 0;
        p.causal = causal ? 1 : 0;
        p.scale_log2 = softmax_scale * kLog2e;
        p.scale = softmax_scale;
        p.spread = spread_items(true, 4.0 * total_k * H * d + 8.0 * total_q * H * d, (int64_t)B * H, true);
        if (fa::launch_bwd_main_varlen(d, p, s) != cudaSuccess) return FA_ERR_CUDA;
    }
    if (total_q > 0 &&
        fa::launch_bwd_convert(d, w.dQacc, dQ, (int64_t)total_q * H * d, softmax_scale, s) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

// ------------------------------------------------------------------ decode (split KV)
namespace {
constexpr int kDecodeMaxSplits = 64;

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n <= 0)
        return 148;
    return n;
}

// splits actually used for a problem: the request (<= 0: enough CTAs for
// two waves), at most one per key tile and at most kDecodeMaxSplits, then
// tightened so that no split is empty.
void decode_splits(int Tq, int BH, int Tk, bool ragged, int requested, int *splits, int *tiles_per_split) {
    int sp = requested;
    if (sp <= 0) {
        // one CTA fits on an SM (the K/V ring takes most of shared memory) and
        // the kernel streams K/V from HBM: with equal cache lengths fill the
        // SMs in one wave and never start a second, partly empty one; with
        // per-batch lengths the longest cache would set the time of a single
        // wave, so cut the work into about three waves of shorter pieces
        // (pieces past a batch's length end at once) and let the block
        // scheduler balance them
        const int64_t items = (int64_t)Tq * BH;
        sp = (int)std::max<int64_t>(1, (ragged ? 3 : 1) * (int64_t)sm_count() / items);
    }
    sp = std::max(1, std::min(sp, std::min(std::max(Tk, 1), kDecodeMaxSplits)));
    const int tps = (std::max(Tk, 1) + sp - 1) / sp;
    *tiles_per_split = tps;
    *splits = (std::max(Tk, 1) + tps - 1) / tps;
}
}  // namespace

size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits) {
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0) return 0;
    const int Tk = (Nk + 127) / 128;
    const int sp = std::max(1, std::min(num_splits > 0 ? num_splits : kDecodeMaxSplits,
                                        std::min(std::max(Tk, 1), kDecodeMaxSplits)));
    const size_t rows = (size_t)B * H * Nq;
    return kStatusBytes + round256((size_t)sp * rows * (size_t)d * 4) + round256((size_t)sp * rows * 4);
}

fa_status fa_decode(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int Nq, int Nk,
                    int d, float softmax_scale, int causal, const int32_t *kv_len, int num_splits, void *workspace,
                    size_t workspace_bytes, void *stream) {
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return FA_ERR_INVALID_ARGUMENT;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!scale_ok(softmax_scale)) return FA_ERR_INVALID_ARGUMENT;
    if ((int64_t)B * H * Nq == 0) return FA_OK;
    const int64_t BH = (int64_t)B * H;
    const int Tq = (Nq + 127) / 128, Tk = (Nk + 127) / 128;
    if (BH > INT_MAX || BH * Tq * kDecodeMaxSplits > INT_MAX) return FA_ERR_UNSUPPORTED;
    if ((int64_t)std::max(Nq, Nk) * d * 2 >= (int64_t(1) << 40)) return FA_ERR_UNSUPPORTED;
    if (!Q || !O || !LSE || !aligned16(Q) || !aligned16(O) || !aligned16(LSE)) return FA_ERR_INVALID_ARGUMENT;
    if (Nk > 0 && (!K || !V || !aligned16(K) || !aligned16(V))) return FA_ERR_INVALID_ARGUMENT;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < fa_decode_workspace_size(B, H, Nq, Nk, d, num_splits))
        return FA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int splits = 0, tps = 0;
    decode_splits(Tq, (int)BH, Tk, kv_len != nullptr, num_splits, &splits, &tps);
    const int64_t rows = BH * Nq;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *Opart = reinterpret_cast<float *>(ws + kStatusBytes);
    float *Lpart = reinterpret_cast<float *>(ws + kStatusBytes + round256((size_t)splits * rows * (size_t)d * 4));
    if (Nk == 0)   // nothing visible anywhere: the merge of zero splits writes O = 0, LSE = -inf
        return fa::launch_decode_merge(d, Opart, Lpart, O, LSE, rows, 0, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    DecParams p;
    std::memset(&p, 0, sizeof(p));
    if (!encode_bf16_3d(&p.tmQ, Q, d, Nq, (int)BH, 128) || !encode_bf16_3d(&p.tmK, K, d, Nk, (int)BH, 128) ||
        !encode_bf16_3d(&p.tmV, V, d, Nk, (int)BH, 128) ||
        (Nq <= 32 && !encode_bf16_3d(&p.tmQs, Q, d, Nq, (int)BH, 32)))
        return FA_ERR_CUDA;
    p.Opart = Opart;
    p.Lpart = Lpart;
    if (splits == 1) {   // the single split is the whole answer: written directly, no merge launch
        p.O = O;
        p.LSE = LSE;
    }
    p.kv_len = kv_len;
    p.status = reinterpret_cast<unsigned *>(ws);
    p.H = H;
    p.Nq = Nq;
    p.Nk = Nk;
    p.BH = (int)BH;
    p.Tq = Tq;
    p.Tk = Tk;
    p.splits = splits;
    p.tiles_per_split = tps;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = softmax_scale * kLog2e;
    if (fa::launch_decode(d, p, s) != cudaSuccess) return FA_ERR_CUDA;
    if (splits == 1) return FA_OK;
    return fa::launch_decode_merge(d, Opart, Lpart, O, LSE, rows, splits, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_tile_plan(int B, int N, int causal, const int32_t *key_len, const uint8_t *block_mask,
                       uint8_t *plan, void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 0 || N < 0) return FA_ERR_INVALID_ARGUMENT;
    if ((int64_t)B * N == 0) return FA_OK;
    const int64_t T = ((int64_t)N + 127) / 128;
    if (T * T * B > ((int64_t)1 << 40)) return FA_ERR_UNSUPPORTED;
    if (!plan) return FA_ERR_INVALID_ARGUMENT;
    if (!workspace || !aligned16(workspace) || workspace_bytes < kStatusBytes) return FA_ERR_WORKSPACE;
    return fa::launch_plan(B, N, causal ? 1 : 0, key_len, block_mask, plan, static_cast<unsigned *>(workspace),
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
}

fa_status fa_get_device_status(const void *workspace, void *stream) {
    if (!workspace) return FA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned w[2] = {0, 0};
    if (cudaMemcpyAsync(w, workspace, sizeof(w), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
    return static_cast<fa_status>(w[0]);
}

fa_status fa_selftest_wait_timeout(void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace || !aligned16(workspace) || workspace_bytes < 32) return FA_ERR_WORKSPACE;
    unsigned *w = static_cast<unsigned *>(workspace);
    // words 0 and 1: status and wait site (as for every kernel); 4..6: the test's own results
    return fa::launch_selftest_wait(w, w + 4, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                                : FA_ERR_CUDA;
}

fa_status fa_reset_device_status(void *workspace, void *stream) {
    if (!workspace) return FA_ERR_WORKSPACE;
    return cudaMemsetAsync(workspace, 0, 8, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                                 : FA_ERR_CUDA;
}

// ------------------------------------------------------------------ host-buffer path
namespace {
// The host path runs in chunks of (b, h) pairs, so that a chunk's kernels
// start as soon as its own inputs are on the device and its outputs go back
// while later chunks still compute: only the first chunk's upload and the
// last chunk's download stay exposed.  A chunk is either whole batches
// (b0 .. b0+nb-1, every head) or a head range of one batch, so that key_len
// applies to it through an offset pointer; its rows are contiguous in every
// [B,H,N,...] array.
constexpr int kMaxHostChunks = 8;
constexpr int kHostChunkTarget = 4;
// Below this many elements per bf16 tensor the step is bound by the copies
// (host <-> device runs at ~200 GB/s per direction; a 2^23-element problem
// moves ~150 MB for ~0.2 ms of kernels) and one chunk is as fast; four
// chunks measured better than eight on the long-context shape (more
// launches, smaller grids).
constexpr size_t kHostChunkMinElems = (size_t)1 << 24;

struct HostChunk {
    int b0, nb, h0, nh;
    size_t row0;        // first (b, h, n) row: (b0 * H + h0) * N
    size_t ws_off;      // this chunk's kernel workspace inside the attention region
};

struct HostLayout {
    size_t attn_ws, q, k, v, o, dO, dQ, dK, dV, lse, klen, bmask, total;
    int nchunks;
    HostChunk chunk[kMaxHostChunks];
};

int host_chunks(int B, int H, int N, int d, HostChunk *c) {
    const size_t elems = (size_t)B * H * N * d;
    // LSE rows are fp32 and the kernels want 16-byte aligned bases: N % 4 == 0
    // keeps every chunk boundary aligned
    if (elems < kHostChunkMinElems || N % 4 != 0 || (size_t)B * H < 2) {
        c[0] = {0, B, 0, H, 0, 0};
        return 1;
    }
    int n = 0;
    if (B >= kHostChunkTarget) {
        for (int i = 0; i < kHostChunkTarget; ++i) {
            const int b0 = (int)((long long)B * i / kHostChunkTarget);
            const int b1 = (int)((long long)B * (i + 1) / kHostChunkTarget);
            c[n++] = {b0, b1 - b0, 0, H, 0, 0};
        }
    } else {
        const int g = std::min(H, (kHostChunkTarget + B - 1) / B);
        for (int b = 0; b < B; ++b)
            for (int i = 0; i < g; ++i) {
                const int h0 = (int)((long long)H * i / g), h1 = (int)((long long)H * (i + 1) / g);
                c[n++] = {b, 1, h0, h1 - h0, 0, 0};
            }
    }
    for (int i = 0; i < n; ++i) c[i].row0 = ((size_t)c[i].b0 * H + c[i].h0) * N;
    return n;
}

HostLayout host_layout(int B, int H, int N, int d, int with_bwd) {
    HostLayout L;
    const size_t rows = (size_t)B * H * N, t = round256(rows * (size_t)d * 2);
    const size_t nb = ((size_t)N + 127) / 128;
    L.nchunks = host_chunks(B, H, N, d, L.chunk);
    size_t off = 0;
    L.attn_ws = off;
    for (int i = 0; i < L.nchunks; ++i) {
        const HostChunk &c = L.chunk[i];
        L.chunk[i].ws_off = off;
        off += round256(with_bwd ? fa_bwd_workspace_size(c.nb, c.nh, N, d) : fa_fwd_workspace_size(c.nb, c.nh, N, d));
    }
    L.q = off; off += t;
    L.k = off; off += t;
    L.v = off; off += t;
    L.o = off; off += t;
    L.dO = off; off += with_bwd ? t : 0;
    L.dQ = off; off += with_bwd ? t : 0;
    L.dK = off; off += with_bwd ? t : 0;
    L.dV = off; off += with_bwd ? t : 0;
    L.lse = off; off += round256(rows * 4);
    L.klen = off; off += round256((size_t)B * 4);
    L.bmask = off; off += round256(nb * nb);
    L.total = off;
    return L;
}
}  // namespace

size_t fa_host_workspace_size(int B, int H, int N, int d, int with_backward) {
    if (B < 0 || H < 0 || N < 0 || d <= 0) return 0;
    return host_layout(B, H, N, d, with_backward ? 1 : 0).total;
}

namespace {
// Streams and events of one host-path call: an upload stream, a download
// stream and one compute stream per chunk (so that the chunks' kernels can
// share the SMs).  They are made for the call and released when it returns;
// CUDA frees a stream or event whose queued work is still pending once that
// work has completed, so nothing outlives the call's own work.
struct HostStreams {
    bool ok = false;
    int n = 0;
    cudaStream_t up = nullptr, down = nullptr, comp[kMaxHostChunks] = {};
    cudaEvent_t start = nullptr, down_done = nullptr, in[kMaxHostChunks] = {}, dO_in[kMaxHostChunks] = {},
                fwd_done[kMaxHostChunks] = {}, bwd_done[kMaxHostChunks] = {};
    explicit HostStreams(int nchunks) : n(nchunks) {
        auto mk_s = [](cudaStream_t *s) { return cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) == cudaSuccess; };
        auto mk_e = [](cudaEvent_t *e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
        ok = mk_s(&up) && mk_s(&down) && mk_e(&start) && mk_e(&down_done);
        for (int i = 0; ok && i < n; ++i)
            ok = mk_s(&comp[i]) && mk_e(&in[i]) && mk_e(&dO_in[i]) && mk_e(&fwd_done[i]) && mk_e(&bwd_done[i]);
    }
    ~HostStreams() {
        for (cudaEvent_t e : {start, down_done})
            if (e) cudaEventDestroy(e);
        for (int i = 0; i < kMaxHostChunks; ++i) {
            for (cudaEvent_t e : {in[i], dO_in[i], fwd_done[i], bwd_done[i]})
                if (e) cudaEventDestroy(e);
            if (comp[i]) cudaStreamDestroy(comp[i]);
        }
        if (up) cudaStreamDestroy(up);
        if (down) cudaStreamDestroy(down);
    }
    HostStreams(const HostStreams &) = delete;
    HostStreams &operator=(const HostStreams &) = delete;
};
}  // namespace

fa_status fa_attention_host(const void *Q, const void *K, const void *V, const void *dO, void *O, float *LSE,
                            void *dQ, void *dK, void *dV, int B, int H, int N, int d, float softmax_scale,
                            int causal, const int32_t *key_len, const uint8_t *block_mask, void *dev_workspace,
                            size_t dev_workspace_bytes, void *stream) {
    bool empty = false;
    fa_status st = check_sizes(B, H, N, d, &empty);
    if (st != FA_OK) return st;
    if (!scale_ok(softmax_scale)) return FA_ERR_INVALID_ARGUMENT;
    if (empty) return FA_OK;
    const int bwd = dO != nullptr;
    if (!Q || !K || !V || !O || !LSE || (bwd && (!dQ || !dK || !dV))) return FA_ERR_INVALID_ARGUMENT;
    const HostLayout L = host_layout(B, H, N, d, bwd);
    if (!dev_workspace || !aligned16(dev_workspace) || dev_workspace_bytes < L.total) return FA_ERR_WORKSPACE;
    if (block_mask && (N + 127) / 128 > kFwdMaxMaskedKeyTiles) return FA_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *w = static_cast<uint8_t *>(dev_workspace);
    const size_t nb = ((size_t)N + 127) / 128;
    HostStreams streams(L.nchunks);
    HostStreams *hs = &streams;
    if (!hs->ok) return FA_ERR_CUDA;
    // An error in the middle of queueing must not return while copies or
    // kernels already queued still use the caller's buffers: wait for every
    // side stream first, so that work the caller puts on `stream` afterwards
    // is ordered after all of this call's work, as on success.
    auto fail = [hs](fa_status e) -> fa_status {
        cudaStreamSynchronize(hs->up);
        cudaStreamSynchronize(hs->down);
        for (int i = 0; i < hs->n; ++i) cudaStreamSynchronize(hs->comp[i]);
        return e;
    };
    {
        auto after = [](cudaEvent_t e, cudaStream_t from, cudaStream_t to) {
            return cudaEventRecord(e, from) == cudaSuccess && cudaStreamWaitEvent(to, e, 0) == cudaSuccess;
        };
        auto h2d = [&](size_t off, const void *src, size_t n) {
            return cudaMemcpyAsync(w + off, src, n, cudaMemcpyHostToDevice, hs->up) == cudaSuccess;
        };
        auto d2h = [&](void *dst, size_t off, size_t n) {
            return cudaMemcpyAsync(dst, w + off, n, cudaMemcpyDeviceToHost, hs->down) == cudaSuccess;
        };
        // everything starts after the work already on `stream`
        if (cudaEventRecord(hs->start, s) != cudaSuccess || cudaStreamWaitEvent(hs->up, hs->start, 0) != cudaSuccess ||
            cudaStreamWaitEvent(hs->down, hs->start, 0) != cudaSuccess)
            return fail(FA_ERR_CUDA);
        for (int i = 0; i < L.nchunks; ++i)
            if (cudaStreamWaitEvent(hs->comp[i], hs->start, 0) != cudaSuccess) return fail(FA_ERR_CUDA);
        // uploads: masks, then each chunk's Q, K, V, then each chunk's dO
        if (key_len && !h2d(L.klen, key_len, (size_t)B * 4)) return fail(FA_ERR_CUDA);
        if (block_mask && !h2d(L.bmask, block_mask, nb * nb)) return fail(FA_ERR_CUDA);
        const size_t row_bytes = (size_t)d * 2;
        auto cbytes = [&](const HostChunk &c) { return (size_t)c.nb * c.nh * N * row_bytes; };
        auto at = [](const void *p, size_t off) { return static_cast<const uint8_t *>(p) + off; };
        for (int i = 0; i < L.nchunks; ++i) {
            const HostChunk &c = L.chunk[i];
            const size_t o = c.row0 * row_bytes, n = cbytes(c);
            if (!h2d(L.q + o, at(Q, o), n) || !h2d(L.k + o, at(K, o), n) || !h2d(L.v + o, at(V, o), n) ||
                !after(hs->in[i], hs->up, hs->comp[i]))
                return fail(FA_ERR_CUDA);
        }
        if (bwd)
            for (int i = 0; i < L.nchunks; ++i) {
                const HostChunk &c = L.chunk[i];
                const size_t o = c.row0 * row_bytes;
                if (!h2d(L.dO + o, at(dO, o), cbytes(c)) || !after(hs->dO_in[i], hs->up, hs->comp[i]))
                    return fail(FA_ERR_CUDA);
            }
        // kernels: chunk i on compute stream i
        for (int i = 0; i < L.nchunks; ++i) {
            const HostChunk &c = L.chunk[i];
            const size_t o = c.row0 * row_bytes;
            const int32_t *kl = key_len ? reinterpret_cast<const int32_t *>(w + L.klen) + c.b0 : nullptr;
            const uint8_t *bm = block_mask ? w + L.bmask : nullptr;
            float *lse = reinterpret_cast<float *>(w + L.lse) + c.row0;
            uint8_t *ws = w + L.attn_ws + c.ws_off;
            const size_t ws_bytes = bwd ? fa_bwd_workspace_size(c.nb, c.nh, N, d) : fa_fwd_workspace_size(c.nb, c.nh, N, d);
            st = fa_fwd(w + L.q + o, w + L.k + o, w + L.v + o, w + L.o + o, lse, c.nb, c.nh, N, d, softmax_scale, causal,
                        kl, bm, ws, ws_bytes, hs->comp[i]);
            if (st != FA_OK) return fail(st);
            if (!after(hs->fwd_done[i], hs->comp[i], hs->down)) return fail(FA_ERR_CUDA);
            if (!d2h(static_cast<uint8_t *>(O) + o, L.o + o, cbytes(c)) ||
                !d2h(LSE + c.row0, L.lse + c.row0 * 4, (size_t)c.nb * c.nh * N * 4))
                return fail(FA_ERR_CUDA);
            if (bwd) {
                st = fa_bwd(w + L.q + o, w + L.k + o, w + L.v + o, w + L.o + o, lse, w + L.dO + o, w + L.dQ + o,
                            w + L.dK + o, w + L.dV + o, c.nb, c.nh, N, d, softmax_scale, causal, kl, bm, ws, ws_bytes,
                            hs->comp[i]);
                if (st != FA_OK) return fail(st);
                if (!after(hs->bwd_done[i], hs->comp[i], hs->down)) return fail(FA_ERR_CUDA);
                if (!d2h(static_cast<uint8_t *>(dQ) + o, L.dQ + o, cbytes(c)) ||
                    !d2h(static_cast<uint8_t *>(dK) + o, L.dK + o, cbytes(c)) ||
                    !d2h(static_cast<uint8_t *>(dV) + o, L.dV + o, cbytes(c)))
                    return fail(FA_ERR_CUDA);
            }
        }
        // the download stream has waited for every chunk's kernels, which waited
        // for every upload: `stream` resumes after the last download
        if (!after(hs->down_done, hs->down, s)) return fail(FA_ERR_CUDA);
    }
    for (int i = 0; i < L.nchunks; ++i) {
        st = fa_get_device_status(w + L.attn_ws + L.chunk[i].ws_off, stream);
        if (st != FA_OK) return st;
    }
    return FA_OK;
}

}  // extern "C"
