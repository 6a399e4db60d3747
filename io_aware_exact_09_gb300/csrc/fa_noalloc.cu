// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass for callers that cannot
// allocate device memory.
//
// fa_bwd needs a caller-provided workspace (a status word, the fp32 row
// dot-products D = rowsum(dO * O) and the fp32 dQ accumulator).  Some callers
// cannot provide one: code running where cudaMalloc is not allowed or would
// stall the whole device (a latency-critical loop, a region under a memory
// manager that owns every byte), a plug-in that is handed only its input and
// output buffers, or a host program with no allocator of its own.  For them
// this entry point takes only the inputs and outputs and uses a scratch array
// that is part of the library: a file-scope __device__ array of
// kScratchBytes, which every GPU that loads the library holds until the
// process exits.
//
// Limits and behaviour:
//   - B*H*N*(4 + 4*d) + 256 bytes must fit in kScratchBytes (64 MiB); larger
//     problems are rejected with FA_ERR_WORKSPACE before anything is
//     enqueued.  Use fa_bwd with a workspace for those.
//   - No cudaMalloc, cudaFree or other allocating call is made.  The first
//     call on each device (more exactly, in each CUDA context: after
//     cudaDeviceReset the device has a new one) looks up the array's device
//     address with cudaGetSymbolAddress, with that device current, and
//     caches it for that context; make that first call before any stream
//     capture.
//   - Arguments are checked (sizes, the softmax scale, null or misaligned
//     pointers) before anything touches the GPU: a rejected call enqueues
//     nothing and leaves the array as it was.
//   - Every call shares the one array and finds the previous call's contents
//     in it.  The status word is cleared and the dQ accumulator is zeroed at
//     the start of every call; D is fully overwritten.  Calls whose work
//     overlaps on the GPU (different streams, or several host threads) race
//     on the array: serialise them.
//   - Device-side status (a timed-out wait, a clamped key_len) lands in the
//     array's status word, which this entry point does not report; callers
//     that need it use fa_bwd and fa_get_device_status.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_dev[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// cuCtxGetCurrent through the runtime's driver entry point (the library does
// not link the driver library itself); null if it cannot be found.
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// Device address of g_bwd_scratch on the current device (in host code the
// array's name is only a stand-in, not an address).  Looked up with
// cudaGetSymbolAddress once per device and context: a context made after a
// cudaDeviceReset gets a fresh lookup instead of a stale address.
void *scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    CtxGetCurrentFn get_ctx = ctx_get_current();
    CUcontext ctx = nullptr;
    if (g_scratch_dev[dev] && get_ctx && get_ctx(&ctx) == CUDA_SUCCESS && ctx == g_scratch_ctx[dev])
        return g_scratch_dev[dev];
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return nullptr;
    ctx = nullptr;
    if (get_ctx && get_ctx(&ctx) == CUDA_SUCCESS && ctx) {
        g_scratch_dev[dev] = p;
        g_scratch_ctx[dev] = ctx;
    } else {
        g_scratch_dev[dev] = nullptr;   // no context handle to key on: look up on every call
    }
    return p;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void *Q, const void *K, const void *V, const void *O,
                                    const float *LSE, const void *dO, void *dQ, void *dK, void *dV,
                                    int B, int H, int N, int d, float softmax_scale, int causal,
                                    const int32_t *key_len, const uint8_t *block_mask, void *stream) {
    // every argument check fa_bwd makes, before the GPU is touched, so that a
    // rejected call writes nothing into the shared array
    if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARGUMENT;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return FA_ERR_INVALID_ARGUMENT;
    if ((int64_t)B * H * N == 0) return FA_OK;
    const void *ptrs[] = {Q, K, V, O, LSE, dO, dQ, dK, dV};
    for (const void *x : ptrs)
        if (!x || !aligned16(x)) return FA_ERR_INVALID_ARGUMENT;
    if (block_mask && (N + 127) / 128 > fa::kFwdMaxMaskedKeyTiles) return FA_ERR_UNSUPPORTED;
    // what fa_bwd requires (status block, D, accumulator); the d = 128 split
    // area after it is used when the array holds that too
    const size_t need = fa::bwd_base_workspace_bytes(B, H, N, d);
    if (need == 0 || need > kScratchBytes) return FA_ERR_WORKSPACE;
    void *ws = scratch_address();
    if (!ws) return FA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // clear the status word the previous call left (D and the dQ accumulator
    // are rewritten by the preprocessing kernel inside fa_bwd)
    if (cudaMemsetAsync(ws, 0, 8, s) != cudaSuccess) return FA_ERR_CUDA;
    return fa_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, N, d, softmax_scale, causal, key_len, block_mask, ws,
                  kScratchBytes, stream);
}
