// fa_tiles.cuh -- the tile-skipping rule shared by the forward, backward and
// plan-export kernels, and the kernel parameter blocks.
//
// Block-sparse skipping follows the "Attention" chapter (learn-kernels.com,
// block-sparse paragraph): a block the mask zeroes is never loaded.  Causal
// and key-padding masks skip the same way whenever a whole tile is masked.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace fa {

constexpr int kTile = 128;           // query/key tile edge = block_mask block edge
constexpr unsigned kTileSkip = 0, kTileFull = 1, kTilePartial = 2;
// plan value for a tile whose class disagrees with a kernel's visit rule
constexpr unsigned kTileRuleMismatch = 3;

// Class of the tile of query rows [q0, q0 + qn) (all < N) and key columns
// [k0, k0 + kw) (columns >= N count as masked): skip if every element is
// masked, full if none is, partial otherwise.
//   kvis     keys < kvis are visible by length: min(N, key_len[b])
//   mask_on  the tile's block_mask entry (1 when there is no block mask)
__host__ __device__ __forceinline__ unsigned tile_class(int q0, int qn, int k0, int kw, int kvis,
                                                        int causal, int mask_on) {
    const int q_last = q0 + qn - 1, k_last = k0 + kw - 1;
    if (!mask_on || qn <= 0) return kTileSkip;
    if (k0 >= kvis) return kTileSkip;
    if (causal && k0 > q_last) return kTileSkip;
    const bool full = (k_last < kvis) && (!causal || k_last <= q0);
    return full ? kTileFull : kTilePartial;
}

// tile_class for decode shapes: the queries are the last rows of the
// sequence, so with the causal mask query i sees key j iff j <= i + shift
// (shift = kv_len - Nq; 0 gives tile_class).
__host__ __device__ __forceinline__ unsigned tile_class_shift(int q0, int qn, int k0, int kw, int kvis,
                                                              int causal, int shift) {
    const int q_last = q0 + qn - 1, k_last = k0 + kw - 1;
    if (qn <= 0 || k0 >= kvis) return kTileSkip;
    if (causal && k0 > q_last + shift) return kTileSkip;
    const bool full = (k_last < kvis) && (!causal || k_last <= q0 + shift);
    return full ? kTileFull : kTilePartial;
}

// The kernels' own O(1) visit rules when there is no block mask (with a
// block mask they test tile_class tile by tile).  fa_plan_kernel checks both
// against tile_class on every tile, so the exported plan shows a wrong rule.
//
// Forward: the key tiles of width bc that the query tile [q0, q0 + qn) visits
// are exactly [0, fwd_key_tile_end): keys below kvis and, under the causal
// mask, at most the tile's last row + shift.
__host__ __device__ __forceinline__ int fwd_key_tile_end(int q0, int qn, int kvis, int causal, int shift,
                                                         int bc) {
    int lim = kvis;
    if (causal && q0 + qn + shift < lim) lim = q0 + qn + shift;
    return (qn > 0 && lim > 0) ? (lim + bc - 1) / bc : 0;
}

// Backward: the query blocks of bq rows that see the key tile starting at k0
// are exactly [bwd_query_block_begin, Tqb): none when the tile lies past
// kvis; under the causal mask, from the first block whose last row reaches
// k0 (+ shift for a bottom-right diagonal: row i sees key j iff j <= i + shift).
__host__ __device__ __forceinline__ int bwd_query_block_begin(int k0, int kvis, int causal, int shift, int bq,
                                                              int Tqb) {
    if (k0 >= kvis) return Tqb;
    if (!causal) return 0;
    const int first_row = k0 - shift;          // the first query row that sees key k0
    if (first_row <= 0) return 0;
    const int qb = first_row / bq;
    return qb < Tqb ? qb : Tqb;
}

// Visible-key bound for batch b: min(N, key_len[b]) with key_len clamped to
// [0, N]; out-of-range values are reported through *bad.
__device__ __forceinline__ int key_visible_bound(const int32_t *key_len, int b, int N, bool *bad) {
    if (!key_len) return N;
    int v = key_len[b];
    if (v < 0 || v > N) {
        *bad = true;
        v = v < 0 ? 0 : N;
    }
    return v;
}

struct FwdParams {
    CUtensorMap tmQ, tmK, tmV;       // [BH][N][d] bf16, box {64, 128, 1}, 128B swizzle; FP8: Q, K e4m3
                                     // [BH][N][d] box {128, 128, 1}, V^T e4m3 [BH][d][Np] box {128, d, 1}
    const float *sQ, *sK, *sV;       // FP8 only: per-(bh, 128-row block) scales [BH][T]
    // ragged batches only: sequence b owns query rows cu_q[b]..cu_q[b+1]-1 of
    // Q, O [total_q][H][d] and key rows cu_k[b]..cu_k[b+1]-1 of K, V
    // [total_k][H][d]; LSE is [H][total_q]; the maps view [total][H][d]
    const int32_t *cu_q, *cu_k;
    int total_q, total_k;
    int qpc;                         // fa_fwd_tiles only: query tiles per CTA (1 or 2)
    void *O;                         // bf16 [BH][N][d]
    float *LSE;                      // fp32 [BH][N]
    const int32_t *key_len;          // device [B] or null
    const uint8_t *block_mask;       // device [nb][nb] or null
    unsigned *status;                // workspace words 0 (status) and 1 (detail)
    int H, N, BH, Tq, Tk;
    int causal;
    float scale_log2;                // softmax_scale * log2(e)
    int spread;                      // persistent grid: 0 head-major, else the items handed out in
                                     // groups of `spread` heads (every head: the heaviest pairs of
                                     // every head first), pair-major inside a group
    // FP8 forward, every tile full: the items (query-tile pair, b*h) from
    // split_from on are each run as split_f CTAs over consecutive ranges of key
    // tiles (split_f < 2: none).  Part j of item split_from + t writes its
    // unnormalised fp32 O rows and (m, l) to split_buf slot t * split_f + j
    // (kFwdSplitSlotBytes: O as [query tile 2][column group 32][row 128] float4,
    // then (m, l) as [query tile 2][row 128] float2) and counts itself in byte
    // t % 4 of split_cnt[t / 4] (workspace words 8..63); the part that counts
    // last merges the slots, writes O and LSE and sets its byte back to zero.
    // The host supplies split_buf, split_cnt and split_cap (slots the buffer
    // holds; 0: no split); the launcher sets split_from and split_f.
    float *split_buf;
    unsigned *split_cnt;
    int split_cap;
    int split_from, split_f;
};

struct DecParams {
    CUtensorMap tmQ;                 // [BH][Nq][d] bf16, box {64, 128, 1}
    CUtensorMap tmQs;                // the same, box {64, 32, 1} (Nq <= 32: the query rows in each quarter)
    CUtensorMap tmK, tmV;            // [BH][Nk][d] bf16, box {64, 128, 1}
    float *Opart;                    // [splits][BH][Nq][d] fp32, each split's normalised output
    float *Lpart;                    // [splits][BH][Nq] fp32, each split's log-sum-exp (-inf: none visible)
    void *O;                         // with one split: bf16 [BH][Nq][d] written directly (no merge), else null
    float *LSE;                      // with one split: fp32 [BH][Nq] natural-log LSE, else null
    const int32_t *kv_len;           // device [B] or null
    unsigned *status;
    int H, Nq, Nk, BH, Tq, Tk, splits, tiles_per_split;
    int causal;
    float scale_log2;
};

struct BwdParams {
    CUtensorMap tmQ, tmdO;           // box {64, BQ, 1}
    CUtensorMap tmK, tmV;            // box {64, 128, 1}
    CUtensorMap tmdQ;                // fp32 [BH][N][d], box {32, 32 or BQ, 1}, 128B swizzle
    const float *LSE;                // fp32 [BH][N]
    const float *Dvec;               // fp32 [BH][N]: rowsum(dO * O)
    float *dQacc;                    // fp32 [BH][N][d]
    void *dK, *dV;                   // bf16 [BH][N][d]
    const int32_t *key_len;
    const uint8_t *block_mask;
    // ragged batches only: sequence b owns query rows cu_q[b]..cu_q[b+1]-1 of
    // Q, dO, dQ [total_q][H][d] and key rows cu_k[b]..cu_k[b+1]-1 of K, V, dK,
    // dV [total_k][H][d]; LSE is [H][total_q], D and the dQ accumulator follow
    // the [total_q][H] row order; the maps view [total][H][d] (box {64, 1, rows},
    // the accumulator {32, 1, 32})
    const int32_t *cu_q, *cu_k;
    int total_q, total_k;
    unsigned *status;
    int H, N, BH, Tk, Tqb;           // Tqb = ceil(N / BQ); ragged: Tk covers the longest key sequence
    int causal;
    float scale_log2;                // softmax_scale * log2(e)
    float scale;                     // softmax_scale
    int spread;                      // d = 64 persistent grid: 0 head-major, else items (key tile,
                                     // b*h) taken in groups of `spread` heads, key-tile-major inside a
                                     // group (every head: key tile 0 of every head first)
    // d = 128, every tile full: the items (key tile, b*h) from split_from on
    // are each run as split_f CTAs over consecutive ranges of query blocks
    // (split_f < 2: none).  Part j of item split_from + t writes its fp32 dK
    // (unscaled) and dV to split_buf slot t * split_f + j (128 KiB: 64 column
    // groups of 4, dK's then dV's, each 128 key rows of float4) and counts
    // itself in byte t % 4 of
    // split_cnt[t / 4] (workspace words 8..63: at most 224 split items); the
    // part that counts last adds the others' slots to its own, writes dK, dV
    // and sets its byte back to zero.  The host supplies split_buf, split_cnt
    // and split_cap (slots the buffer holds; 0: no split); the launcher sets
    // split_from and split_f.
    float *split_buf;
    unsigned *split_cnt;
    int split_cap;
    int split_from, split_f;
};

// The sequence a CTA of a ragged batch works on: query rows [q_start,
// q_start + Lq), key rows [k_start, k_start + Lk).  Offsets outside [0, total]
// or negative lengths, or a key length past the grid's key tiles (max_k_rows),
// make it invalid: *bad is set and both lengths become 0 (the sequence is
// skipped).
__device__ __forceinline__ void varlen_sequence(const int32_t *cu_q, const int32_t *cu_k, int b, int total_q,
                                                int total_k, int max_q_rows, int max_k_rows, int *q_start,
                                                int *Lq, int *k_start, int *Lk, bool *bad) {
    *q_start = cu_q[b];
    *Lq = cu_q[b + 1] - *q_start;
    *k_start = cu_k[b];
    *Lk = cu_k[b + 1] - *k_start;
    if (*q_start < 0 || *Lq < 0 || *q_start + *Lq > total_q || *k_start < 0 || *Lk < 0 ||
        *k_start + *Lk > total_k || *Lq > max_q_rows || *Lk > max_k_rows) {
        *bad = true;
        *Lq = *Lk = 0;
    }
}

}  // namespace fa
