/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact IO-aware attention library.
 *
 * The operation ("FlashAttention: Mathematical Foundations, IO-Aware Tiling,
 * Online Softmax, and Recomputation Dynamics", section "The GPU Memory
 * Hierarchy and the Attention Memory Wall"):
 *
 *     O = softmax(softmax_scale * Q K^T [+ mask]) V,   Q, K, V of shape (N, d),
 *
 * per (batch b, head h).  The forward pass writes only O and one fp32 number
 * per query row, LSE = m + ln(l) (the row maximum m and normaliser l of the
 * online softmax folded together; "The Attention Matrix You Never Write
 * Down", section "Tiling forward, recomputing backward": only the output and
 * a small per-row normalisation statistic go back to HBM).  The backward
 * pass rebuilds the score and probability tiles on chip from Q, K and LSE
 * (same page and section; "Backward Pass and Activation Recomputation" on
 * the mathematical-foundations page) and produces dQ, dK, dV for the loss
 * sum(O * dO).  The N x N score matrix is never written to memory.
 *
 * Conventions shared by every entry point
 *   - Tensors are contiguous [B, H, N, d] row-major (d fastest), bf16
 *     (Q, K, V, O, dO, dQ, dK, dV); LSE is fp32 [B, H, N].
 *   - Device pointers are owned by the caller and must be 16-byte aligned.
 *     The library allocates no device memory and keeps no state between
 *     calls apart from cached kernel attributes.
 *   - d must be 64 or 128 (else FA_ERR_UNSUPPORTED).  B, H, N >= 0; when
 *     B*H*N == 0 the call does nothing and returns FA_OK.  Q and K share N
 *     (self-attention).  softmax_scale must be finite and > 0 (the usual
 *     value is 1/sqrt(d)).
 *   - causal != 0 keeps key j for query i iff j <= i (top-left aligned).
 *   - key_len: NULL, or a DEVICE int32 [B]: key j of batch b is kept iff
 *     j < key_len[b] (queries are never masked).  Values are read on the
 *     device; a value outside [0, N] is clamped and flagged in the
 *     workspace status word (FA_ERR_DEVICE_BAD_KEY_LEN).
 *   - block_mask: NULL, or a DEVICE uint8 [nb][nb], nb = ceil(N / 128),
 *     shared by every (b, h): the 128 x 128 block (query block r, key block
 *     c) is kept iff block_mask[r * nb + c] != 0 ("Attention" chapter of
 *     learn-kernels.com, block-sparse paragraph: blocks the mask zeroes are
 *     skipped, never loaded).  With a block_mask nb may be at most 2048
 *     (the forward lists a row's key tiles in shared memory; fa_fwd_tiles:
 *     2048 key tiles of its width), else the call returns
 *     FA_ERR_UNSUPPORTED, like every argument error before anything is
 *     enqueued.
 *   - A query row with no visible key gets O = 0, LSE = -inf and contributes
 *     nothing to the gradients.
 *   - stream is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous: they validate, enqueue and return.  Argument errors are
 *     returned before anything is enqueued.  Errors found on the device (a
 *     wait that timed out, a bad key_len) are written to the first word of
 *     the workspace and read back with fa_get_device_status().
 *   - The workspace must be zero-filled once before its first use.  Word 0
 *     is the status word, which the library only ever sets, never clears
 *     (fa_reset_device_status() clears it).  The persistent kernels (the
 *     forward, the d = 64 backward) hand out their work items from a counter
 *     in words 2 and 3, which every launch leaves at zero again; the d = 128 backward and the FP8 forward keep
 *     the counters of their last-wave splits (fa_bwd_workspace_size,
 *     fa_fwd_workspace_size) in words 8..63, also left at zero.  After a
 *     call that recorded a device-side timeout, zero-fill the workspace
 *     again before reusing it.  A workspace therefore serves one call at a
 *     time: calls that may run concurrently (different streams) need
 *     workspaces of their own.
 *   - No entry point throws or exits; there is no CPU fallback.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARGUMENT = 1,   /* null/misaligned pointer, negative size, bad scale */
    FA_ERR_UNSUPPORTED = 2,        /* d not in {64, 128}, sizes beyond the 32-bit grid limits,
                                      a block_mask over more than 2048 key tiles */
    FA_ERR_WORKSPACE = 3,          /* workspace NULL or smaller than the call needs (*_workspace_size) */
    FA_ERR_CUDA = 4,               /* a CUDA runtime call or kernel launch failed */
    FA_ERR_DEVICE_TIMEOUT = 5,     /* a device-side wait gave up (kernel returned early) */
    FA_ERR_DEVICE_BAD_KEY_LEN = 6  /* a key_len value was outside [0, N] and was clamped */
} fa_status;

/* Size of the 128 x 128 tile (and of a block_mask block). */
int fa_tile_size(void);

/* Bytes of device workspace for fa_fwd and fa_fwd_fp8: the 256-byte status
 * block (status word, the persistent forward grid's work-item counter), and
 * for d = 128 with at least 32 key tiles (N >= 4096) the FP8 forward's split
 * area: 130 KiB per CTA of a split item, for min(512, B * H * ceil(T / 2) *
 * min(4, T / 16)) of them (T = ceil(N / 128)).  With no mask and N a multiple
 * of 128 every FP8 forward item (two query tiles) takes the same time; the
 * items past the last full wave of one CTA per SM run as 2-4 CTAs each over
 * parts of the key range, whose unnormalised O and running (max, sum) meet in
 * that area, the last to finish merging them.  The calls accept the 256-byte
 * status block alone and then do not split. */
size_t fa_fwd_workspace_size(int B, int H, int N, int d);

/* Bytes of device workspace fa_bwd uses: the 256-byte status block, the
 * fp32 row dot-products D = rowsum(dO * O) [B, H, N] and the fp32 dQ
 * accumulator [B, H, N, d], each 256-byte aligned; for d = 128 and N > 128
 * then the split area: 128 KiB per CTA of a split key tile, for
 * min(256, B * H * ceil(N / 128) * min(4, ceil(N / 128))) of them.  With no
 * mask and N a multiple of 128 every key tile takes the same time; the main
 * kernel runs one CTA per SM at a time, and the key tiles past its last full
 * wave run as 2-4 CTAs each over parts of the query range, whose fp32 dK and
 * dV meet in that area.  The calls accept a workspace without the split area
 * (status block, D and accumulator only) and then do not split. */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Forward.  Q, K, V: device bf16 [B, H, N, d] (read).  O: device bf16
 * [B, H, N, d] (written).  LSE: device fp32 [B, H, N] (written, natural log:
 * P_ij = exp(softmax_scale * q_i.k_j - LSE_i) for visible keys).
 * One kernel launch: a persistent grid of at most one CTA per SM taking
 * (pair of 128-row query tiles, b, h) work items from the workspace
 * counter.  With a block_mask, N may be at most 2048 * 128 (the key tiles of
 * a row are listed in shared memory), else FA_ERR_UNSUPPORTED.
 */
fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                 int N, int d, float softmax_scale, int causal, const int32_t *key_len,
                 const uint8_t *block_mask, void *workspace, size_t workspace_bytes,
                 void *stream);

/*
 * The forward with a chosen tile shape, for the block-size sweep
 * ("Attention" chapter, FlashAttention paragraph: widening the block
 * shrinks HBM traffic and runtime up to a point).  block_q: query rows per
 * CTA, 128 or 256 (fa_fwd uses 256: two 128-row tiles); block_k: key rows per
 * tile, 64 or 128 (fa_fwd: 128).  Other values: FA_ERR_UNSUPPORTED (a 256-key
 * tile does not fit: its S rows need 256 of the 512 TMEM columns per query
 * tile, and at d = 128 one K plus one V tile take 128 KB of shared memory).
 * Arguments, results and masks otherwise as fa_fwd; the block_mask keeps its
 * 128 x 128 granularity.  One kernel launch.
 */
fa_status fa_fwd_tiles(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                       int N, int d, float softmax_scale, int causal, const int32_t *key_len,
                       const uint8_t *block_mask, int block_q, int block_k, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * Forward of a ragged batch ("Attention" chapter, serving paragraph: the
 * ragged layouts inference engines keep their sequences in): B sequences of
 * different lengths packed one after another.  Q, O: device bf16
 * [total_q, H, d]; K, V: device bf16 [total_k, H, d]; LSE: device fp32
 * [H, total_q] (natural log).  cu_seqlens_q, cu_seqlens_k: device int32
 * [B + 1], non-decreasing offsets from 0 to total_q / total_k: sequence b
 * owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows
 * cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1.  max_seqlen_q (host): at least the
 * longest query length (it sizes the grid).  Lq queries of a sequence are its
 * last Lq positions among its Lk keys (a cached prefix when Lk > Lq): with
 * causal != 0 query i sees key j iff j <= i + Lk - Lq.  A row that sees no
 * key gets O = 0, LSE = -inf.  Offsets outside [0, total], a negative length
 * or a query length beyond the grid max_seqlen_q sizes (rounded up to whole
 * 128-row tiles): that sequence is skipped and FA_ERR_DEVICE_BAD_KEY_LEN is
 * recorded in the workspace status word.
 * Workspace: fa_fwd_workspace_size(1, 1, 1, d) bytes.  One kernel launch.
 */
fa_status fa_fwd_varlen(const void *Q, const void *K, const void *V, void *O, float *LSE,
                        const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int B, int H,
                        int total_q, int total_k, int max_seqlen_q, int d, float softmax_scale,
                        int causal, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward of a ragged batch (the layout of fa_fwd_varlen) for the loss
 * sum(O * dO): the gradients of each packed sequence on its own, with the
 * same bottom-right causal alignment (query i of a sequence sees key j iff
 * j <= i + Lk - Lq).  Q, O, dO: device bf16 [total_q, H, d] (read); K, V:
 * device bf16 [total_k, H, d] (read); LSE: device fp32 [H, total_q] from
 * fa_fwd_varlen with the same arguments (read).  dQ: device bf16
 * [total_q, H, d]; dK, dV: device bf16 [total_k, H, d] (written; the keys of
 * a sequence without queries get zero gradients).  cu_seqlens_q,
 * cu_seqlens_k: device int32 [B + 1] offsets as for fa_fwd_varlen.
 * max_seqlen_k (host): at least the longest key length (it sizes the grid).
 * An invalid sequence (offsets outside [0, total], a negative length, a key
 * length beyond max_seqlen_k rounded up to whole 128-row tiles) is skipped
 * and FA_ERR_DEVICE_BAD_KEY_LEN recorded in the workspace status word.
 * Workspace: fa_bwd_varlen_workspace_size(H, total_q, d) bytes (status
 * word, D = rowsum(dO * O) and the fp32 dQ accumulator, [total_q, H] rows).
 * Three kernel launches, as fa_bwd.
 */
size_t fa_bwd_varlen_workspace_size(int H, int total_q, int d);
fa_status fa_bwd_varlen(const void *Q, const void *K, const void *V, const void *O, const float *LSE,
                        const void *dO, void *dQ, void *dK, void *dV, const int32_t *cu_seqlens_q,
                        const int32_t *cu_seqlens_k, int B, int H, int total_q, int total_k,
                        int max_seqlen_k, int d, float softmax_scale, int causal, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * FP8 block quantisation ("FlashAttention: Mathematical Foundations ...",
 * section "Architectural Evolution", FlashAttention-3 paragraph:
 * block-quantised FP8 matmuls with dynamic scaling).  X: device bf16
 * [B, H, N, d] (read).  A block is 128 consecutive rows of one (b, h); its
 * scale, written to scales (device fp32 [B, H, ceil(N / 128)]), is
 * amax / 448 (0 for an all-zero block), and each element becomes the e4m3
 * code of x / scale (fp32 division, nearest-even, saturating to +-448).
 * X8 (device, written): e4m3 codes [B, H, N, d], or with transpose != 0
 * [B, H, d, Np], Np = ceil(N / 16) * 16, columns N..Np-1 zero (the layout
 * fa_fwd_fp8 wants for V).  One kernel launch, no workspace.
 */
fa_status fa_quantize_fp8(const void *X, void *X8, float *scales, int B, int H, int N, int d,
                          int transpose, void *stream);

/*
 * FP8 block quantisation with incoherent processing (the "Attention" chapter
 * of learn-kernels.com, FlashAttention-3 paragraph: "block quantization with
 * incoherent processing"), for Q and K.  Each row x of X (device bf16
 * [B, H, N, d], read) is first rotated to (x * signs) H: signs is a device
 * int8 [d] vector of +1 / -1 (16-byte aligned; the caller draws it at
 * random and uses the same one for Q and K), H the unnormalised d x d
 * Sylvester-Hadamard matrix, applied as the fast Walsh-Hadamard transform
 * in fp32 (stages h = 1, 2, ..., d/2, each pair (i, i + h) becoming
 * (x_i + x_{i+h}, x_i - x_{i+h})).  Then as fa_quantize_fp8 without
 * transpose: codes X8 [B, H, N, d] and scales [B, H, ceil(N / 128)] of the
 * rotated values.  Since (Q s H)(K s H)^T = d Q K^T, the forward on
 * rotated Q and K is fa_fwd_fp8_rotated, which takes the softmax scale of
 * the unrotated problem and removes the factor d itself.  V is quantised
 * unrotated.  One kernel launch, no workspace.
 */
fa_status fa_quantize_fp8_rotated(const void *X, void *X8, float *scales, const int8_t *signs, int B,
                                  int H, int N, int d, void *stream);

/*
 * FP8 forward (d = 128 only; other d: FA_ERR_UNSUPPORTED).  Q8, K8: e4m3
 * [B, H, N, d]; Vt8: e4m3 [B, H, d, Np] (fa_quantize_fp8 with transpose);
 * sQ, sK, sV: their block scales [B, H, ceil(N / 128)]; all device, read.
 * Computes exact attention of the values the codes stand for (code * block
 * scale) with both products on the FP8 tensor cores; the probabilities are
 * rounded to e4m3 for the P.V product (this, not the inputs, sets the
 * accuracy: about 2^-5 relative per probability).  O (bf16), LSE (fp32,
 * natural log), masks and workspace as fa_fwd (the split of the last wave,
 * fa_fwd_workspace_size, is this call's; each part rounds its probabilities
 * against its own running maximum).  One kernel launch.
 */
fa_status fa_fwd_fp8(const void *Q8, const void *K8, const void *Vt8, const float *sQ,
                     const float *sK, const float *sV, void *O, float *LSE, int B, int H, int N,
                     int d, float softmax_scale, int causal, const int32_t *key_len,
                     const uint8_t *block_mask, void *workspace, size_t workspace_bytes,
                     void *stream);

/*
 * FP8 forward after incoherent processing ("Attention" chapter of
 * learn-kernels.com, FlashAttention-3 paragraph).  Q8, K8 and sQ, sK come
 * from fa_quantize_fp8_rotated (the rows of Q and K rotated by diag(signs) H,
 * with the same signs for both); Vt8, sV from fa_quantize_fp8 with
 * transpose (V is not rotated).  softmax_scale is the scale of the
 * unrotated attention (usually 1/sqrt(d)): the rotated scores carry a
 * factor d ((Q s H)(K s H)^T = d Q K^T), which this call removes by running
 * fa_fwd_fp8 with softmax_scale / d.  Everything else as fa_fwd_fp8.
 */
fa_status fa_fwd_fp8_rotated(const void *Q8, const void *K8, const void *Vt8, const float *sQ,
                             const float *sK, const float *sV, void *O, float *LSE, int B, int H,
                             int N, int d, float softmax_scale, int causal, const int32_t *key_len,
                             const uint8_t *block_mask, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * Backward for the loss sum(O * dO).  Q, K, V, O, dO: device bf16 [B, H, N, d]
 * (read); LSE: device fp32 [B, H, N] from fa_fwd with the same arguments
 * (read).  dQ, dK, dV: device bf16 [B, H, N, d] (written).  Three kernel
 * launches: D = rowsum(dO * O) with the dQ accumulator zeroed; the main
 * kernel (one CTA per 128-key tile, recomputing S and P tile by tile; the
 * last wave's tiles split over several CTAs, see fa_bwd_workspace_size);
 * the fp32 -> bf16 conversion of dQ.
 */
fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const float *LSE,
                 const void *dO, void *dQ, void *dK, void *dV, int B, int H, int N, int d,
                 float softmax_scale, int causal, const int32_t *key_len,
                 const uint8_t *block_mask, void *workspace, size_t workspace_bytes,
                 void *stream);

/*
 * fa_bwd in its three stages, for callers that want to schedule or time them
 * separately.  Same arguments and preconditions as fa_bwd; the stages must be
 * enqueued in this order on one stream with the same workspace.
 *   fa_bwd_preprocess:  D = rowsum(dO * O) (fp32) and dQ accumulator = 0
 *                       (reads O, dO; writes the workspace).
 *   fa_bwd_main:        one CTA per 128-key tile: recompute S^T and P^T,
 *                       dP^T, dS^T; write dK, dV; add dQ contributions into
 *                       the workspace accumulator.
 *   fa_bwd_postprocess: dQ = bf16(softmax_scale * accumulator).
 */
fa_status fa_bwd_preprocess(const void *O, const void *dO, int B, int H, int N, int d,
                            void *workspace, size_t workspace_bytes, void *stream);
fa_status fa_bwd_main(const void *Q, const void *K, const void *V, const float *LSE, const void *dO,
                      void *dK, void *dV, int B, int H, int N, int d, float softmax_scale,
                      int causal, const int32_t *key_len, const uint8_t *block_mask,
                      void *workspace, size_t workspace_bytes, void *stream);
fa_status fa_bwd_postprocess(void *dQ, int B, int H, int N, int d, float softmax_scale,
                             const void *workspace, size_t workspace_bytes, void *stream);

/*
 * Decode-time attention ("Attention" chapter of learn-kernels.com, decoding
 * paragraph: the same IO-aware framing applied to the small, frequent
 * product of a few new tokens against a growing key/value cache).
 *   Q: device bf16 [B, H, Nq, d], the newest Nq tokens; K, V: device bf16
 *   [B, H, Nk, d], the cache; O: device bf16 [B, H, Nq, d]; LSE: device fp32
 *   [B, H, Nq] (natural log).  kv_len: NULL or device int32 [B], the valid
 *   cache length of each batch (key j visible iff j < kv_len[b]; values
 *   outside [0, Nk] are clamped and flagged).  causal != 0: the queries are
 *   the last Nq positions, query i sees key j iff j <= kv_len[b] - Nq + i
 *   (bottom-right alignment).  num_splits: how many CTAs share the key tiles
 *   of one (query tile, b, h); <= 0 picks the most that still fit the GPU's
 *   SMs in one wave, or about three waves when kv_len is given (at least
 *   1, at most 64).  Each split writes a normalised fp32 partial output and its
 *   log-sum-exp into the workspace; a second kernel merges them with the
 *   block-merge identity ("FlashAttention: Mathematical Foundations ...",
 *   section "Incremental Online Updates").  Two kernel launches; with a
 *   single split, one (it writes O and LSE itself).
 * fa_decode_workspace_size: bytes for the status word and the partials,
 * for the same num_splits argument.
 */
size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits);
fa_status fa_decode(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                    int Nq, int Nk, int d, float softmax_scale, int causal, const int32_t *kv_len,
                    int num_splits, void *workspace, size_t workspace_bytes, void *stream);

/*
 * The tile-skipping decisions the kernels take, exported so that they can be
 * checked exactly.  plan: device uint8 [B][T][T], T = ceil(N / 128), written
 * with 0 = skip (every element of the 128 x 128 tile masked; the tile is
 * never loaded), 1 = full (no element masked), 2 = partial (element masks
 * applied).  Element set of tile (r, c): query rows i in [128r, 128r+128)
 * with i < N, key columns j in [128c, 128c+128); j >= N counts as masked.
 * Computed by the same device function the kernels take their full /
 * partial decisions with, and checked on every tile against the rules the
 * kernels skip with (without a block mask the forward visits a contiguous
 * range of key tiles and the backward a contiguous range of query blocks,
 * each found in O(1)): a tile where either rule disagrees with its class is
 * written as 3, a value no correct plan contains.
 */
fa_status fa_tile_plan(int B, int N, int causal, const int32_t *key_len,
                       const uint8_t *block_mask, uint8_t *plan, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * Host-buffer convenience: Q, K, V (and dO unless NULL) are HOST bf16 arrays;
 * O, LSE (and dQ, dK, dV when dO != NULL) are HOST outputs.  key_len and
 * block_mask, when given, are HOST arrays too.  The call copies the inputs
 * into dev_workspace, runs fa_fwd (and fa_bwd), copies the outputs back and
 * synchronises the stream before returning.  Pinned host memory makes the
 * copies asynchronous.  Large problems (at least 2^24 elements per tensor,
 * N a multiple of 4, B*H >= 2) run in up to 8 chunks of whole batches or of
 * a head range of one batch: each chunk's kernels start once its own inputs
 * are on the device, on a compute stream of their own so that chunks share
 * the SMs, and its outputs are copied back while later chunks compute.
 * Uploads and downloads each have a stream.  These streams and their events
 * are made for the call and released when it returns (nothing persists);
 * they are ordered after the work already queued on `stream`, which in turn
 * waits for all of them.  Results are
 * bit-identical to fa_fwd / fa_bwd on device buffers except dQ (summed by
 * reduce-adds in a varying order).
 * dev_workspace: device memory of at least fa_host_workspace_size() bytes,
 * zero-filled once before first use.
 */
size_t fa_host_workspace_size(int B, int H, int N, int d, int with_backward);
fa_status fa_attention_host(const void *Q, const void *K, const void *V, const void *dO, void *O,
                            float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int d,
                            float softmax_scale, int causal, const int32_t *key_len,
                            const uint8_t *block_mask, void *dev_workspace,
                            size_t dev_workspace_bytes, void *stream);

/*
 * fa_bwd without a workspace, for callers that cannot allocate device memory
 * (code that must not call cudaMalloc where it runs, or that is handed only
 * its input and output buffers).  The pages have no counterpart: this is a
 * packaging of fa_bwd, not part of the method.
 *
 * Same arguments, meaning and results as fa_bwd, minus the workspace.  The
 * scratch (status word, D, dQ accumulator, and the d = 128 split area when
 * it fits) is a 64 MiB array built into the library and held by every GPU
 * that loads it until the process exits.
 *   - Problems needing more, i.e. B*H*N*(4 + 4*d) + 256 bytes > 64 MiB (for
 *     example B*H*N > 130,000 rows at d = 128), return FA_ERR_WORKSPACE
 *     before anything is enqueued.
 *   - Allocates nothing.  The first call on a device looks up the array's
 *     device address, with that device current, and keeps it for the
 *     device's CUDA context (a context made after cudaDeviceReset gets a
 *     new lookup); make that first call before any stream capture.
 *   - Arguments are checked as fa_bwd checks them before the GPU is
 *     touched: a rejected call enqueues nothing and leaves the array as it
 *     was.
 *   - All calls share the array and see the previous call's contents; each
 *     call clears the status word and zeroes the accumulator first.  Calls
 *     that overlap on the GPU race on the array: serialise them.
 *   - Device-side status is not reported here (use fa_bwd for that).
 */
fa_status fa_bwd_noalloc(const void *Q, const void *K, const void *V, const void *O,
                         const float *LSE, const void *dO, void *dQ, void *dK, void *dV, int B,
                         int H, int N, int d, float softmax_scale, int causal,
                         const int32_t *key_len, const uint8_t *block_mask, void *stream);

/* Synchronise stream and return the workspace status word (FA_OK if no
 * device-side error was recorded). */
fa_status fa_get_device_status(const void *workspace, void *stream);

/* Enqueue a clear of the workspace status word on stream. */
fa_status fa_reset_device_status(void *workspace, void *stream);

/*
 * Failure-path self-test.  Launches one warp that waits, with the same
 * bounded wait every kernel here uses for its barriers, on a barrier phase
 * that nothing completes.  The wait gives up after the kernels' wait limit
 * (2 s), records FA_ERR_DEVICE_TIMEOUT in the workspace status word (word 1:
 * the wait site, 0x5e1f) and raises the CTA's abort flag; a second wait
 * returns at once through that flag; the kernel then exits normally.
 * workspace: zero-filled device memory of at least 32 bytes; besides the
 * status words it receives in words 4..6 the outcome of the two waits
 * (0 = gave up) and 1 if the second wait returned well before the limit.
 * No GPU fault, trap or hang is involved: the context stays usable.
 */
fa_status fa_selftest_wait_timeout(void *workspace, size_t workspace_bytes, void *stream);

/* Static string for a status code. */
const char *fa_status_string(fa_status s);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
