"""GB300 (sm_103a) exact IO-aware attention: Python binding of the C ABI.

Every entry point of ``include/fa.h`` is exposed here under the same name,
taking torch tensors (device memory) or numpy arrays (host memory) and
passing their raw pointers and sizes through ctypes.  This module does
argument marshalling only; all computation runs in the CUDA kernels of
``libfa_gb300.so``.  If the library has not been built, every call raises:
there is no fallback path.

Convenience wrappers ``attention_forward`` / ``attention_backward`` allocate
outputs and the workspace with torch (PyTorch supplies device memory and
streams) and call ``fa_fwd`` / ``fa_bwd``.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfa_gb300.so")

FA_OK = 0
STATUS_NAMES = {
    0: "FA_OK", 1: "FA_ERR_INVALID_ARGUMENT", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_WORKSPACE",
    4: "FA_ERR_CUDA", 5: "FA_ERR_DEVICE_TIMEOUT", 6: "FA_ERR_DEVICE_BAD_KEY_LEN",
}

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__("%s: %s (%d)" % (where, STATUS_NAMES.get(self.status, "?"), self.status))


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    from . import _builder as _b
    return _b.build(force=force)


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libfa_gb300.so is not built; call io_aware_exact_09_gb300.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.fa_tile_size.argtypes = []
            L.fa_tile_size.restype = i
            L.fa_fwd_workspace_size.argtypes = [i, i, i, i]
            L.fa_fwd_workspace_size.restype = sz
            L.fa_bwd_workspace_size.argtypes = [i, i, i, i]
            L.fa_bwd_workspace_size.restype = sz
            L.fa_host_workspace_size.argtypes = [i, i, i, i, i]
            L.fa_host_workspace_size.restype = sz
            L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, vp, sz, vp]
            L.fa_fwd.restype = i
            L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, vp, sz, vp]
            L.fa_bwd.restype = i
            L.fa_bwd_preprocess.argtypes = [vp, vp, i, i, i, i, vp, sz, vp]
            L.fa_bwd_preprocess.restype = i
            L.fa_bwd_main.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, vp, sz, vp]
            L.fa_bwd_main.restype = i
            L.fa_bwd_postprocess.argtypes = [vp, i, i, i, i, f, vp, sz, vp]
            L.fa_bwd_postprocess.restype = i
            L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, vp]
            L.fa_bwd_noalloc.restype = i
            L.fa_decode_workspace_size.argtypes = [i, i, i, i, i, i]
            L.fa_decode_workspace_size.restype = sz
            L.fa_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp, sz, vp]
            L.fa_decode.restype = i
            L.fa_fwd_tiles.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, i, i, vp, sz, vp]
            L.fa_fwd_tiles.restype = i
            L.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp]
            L.fa_fwd_varlen.restype = i
            L.fa_bwd_varlen_workspace_size.argtypes = [i, i, i]
            L.fa_bwd_varlen_workspace_size.restype = sz
            L.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp]
            L.fa_bwd_varlen.restype = i
            L.fa_quantize_fp8.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
            L.fa_quantize_fp8.restype = i
            L.fa_quantize_fp8_rotated.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
            L.fa_quantize_fp8_rotated.restype = i
            L.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, vp, sz, vp]
            L.fa_fwd_fp8.restype = i
            L.fa_fwd_fp8_rotated.argtypes = L.fa_fwd_fp8.argtypes
            L.fa_fwd_fp8_rotated.restype = i
            L.fa_tile_plan.argtypes = [i, i, i, vp, vp, vp, vp, sz, vp]
            L.fa_tile_plan.restype = i
            L.fa_attention_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp,
                                            vp, sz, vp]
            L.fa_attention_host.restype = i
            L.fa_get_device_status.argtypes = [vp, vp]
            L.fa_get_device_status.restype = i
            L.fa_selftest_wait_timeout.argtypes = [vp, sz, vp]
            L.fa_selftest_wait_timeout.restype = i
            L.fa_reset_device_status.argtypes = [vp, vp]
            L.fa_reset_device_status.restype = i
            L.fa_status_string.argtypes = [i]
            L.fa_status_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


EXPORTED = ("fa_tile_size", "fa_fwd_workspace_size", "fa_bwd_workspace_size", "fa_fwd", "fa_bwd",
            "fa_bwd_preprocess", "fa_bwd_main", "fa_bwd_postprocess", "fa_bwd_noalloc",
            "fa_decode_workspace_size", "fa_decode", "fa_fwd_tiles", "fa_fwd_varlen", "fa_bwd_varlen_workspace_size",
            "fa_bwd_varlen", "fa_quantize_fp8", "fa_quantize_fp8_rotated", "fa_fwd_fp8", "fa_fwd_fp8_rotated",
            "fa_tile_plan",
            "fa_host_workspace_size", "fa_attention_host", "fa_get_device_status", "fa_reset_device_status",
            "fa_selftest_wait_timeout", "fa_status_string")


# ---------------------------------------------------------------- marshalling helpers
def _p(t):
    """Raw pointer of a torch tensor / numpy array, or None."""
    if t is None:
        return None
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _check(status, where):
    if status != FA_OK:
        raise FAError(status, where)


# ---------------------------------------------------------------- ABI, same names
def fa_tile_size() -> int:
    return lib().fa_tile_size()


def fa_fwd_workspace_size(B, H, N, d) -> int:
    return lib().fa_fwd_workspace_size(B, H, N, d)


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return lib().fa_bwd_workspace_size(B, H, N, d)


def fa_host_workspace_size(B, H, N, d, with_backward) -> int:
    return lib().fa_host_workspace_size(B, H, N, d, int(bool(with_backward)))


def fa_fwd(Q, K, V, O, LSE, B, H, N, d, softmax_scale, causal, key_len, block_mask, workspace,
           workspace_bytes, stream=None) -> int:
    return lib().fa_fwd(_p(Q), _p(K), _p(V), _p(O), _p(LSE), B, H, N, d, float(softmax_scale),
                        int(bool(causal)), _p(key_len), _p(block_mask), _p(workspace),
                        int(workspace_bytes), _stream(stream))


def fa_fwd_tiles(Q, K, V, O, LSE, B, H, N, d, softmax_scale, causal, key_len, block_mask, block_q, block_k,
                 workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_fwd_tiles(_p(Q), _p(K), _p(V), _p(O), _p(LSE), B, H, N, d, float(softmax_scale),
                              int(bool(causal)), _p(key_len), _p(block_mask), int(block_q), int(block_k),
                              _p(workspace), int(workspace_bytes), _stream(stream))


def fa_fwd_varlen(Q, K, V, O, LSE, cu_seqlens_q, cu_seqlens_k, B, H, total_q, total_k, max_seqlen_q, d,
                  softmax_scale, causal, workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_fwd_varlen(_p(Q), _p(K), _p(V), _p(O), _p(LSE), _p(cu_seqlens_q), _p(cu_seqlens_k), B, H,
                               total_q, total_k, max_seqlen_q, d, float(softmax_scale), int(bool(causal)),
                               _p(workspace), int(workspace_bytes), _stream(stream))


def attention_varlen(Q, K, V, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, softmax_scale=None, causal=False,
                     ws=None, stream=None, check_status=False):
    """O [total_q, H, d], LSE [H, total_q] = fa_fwd_varlen(...) on bf16 CUDA tensors."""
    import torch
    total_q, H, d = (int(x) for x in Q.shape)
    total_k = int(K.shape[0])
    B = int(cu_seqlens_q.numel()) - 1
    scale = (1.0 / d ** 0.5) if softmax_scale is None else softmax_scale
    O = torch.empty_like(Q)
    LSE = torch.empty((H, total_q), dtype=torch.float32, device=Q.device)
    if ws is None:
        ws = workspace(fa_fwd_workspace_size(1, 1, 1, d), Q.device)
    _check(fa_fwd_varlen(Q, K, V, O, LSE, cu_seqlens_q, cu_seqlens_k, B, H, total_q, total_k, max_seqlen_q, d,
                         scale, causal, ws, ws.numel(), stream), "fa_fwd_varlen")
    if check_status:
        _check(fa_get_device_status(ws, stream), "fa_fwd_varlen (device)")
    return O, LSE


def fa_bwd_varlen_workspace_size(H, total_q, d) -> int:
    return lib().fa_bwd_varlen_workspace_size(H, total_q, d)


def fa_bwd_varlen(Q, K, V, O, LSE, dO, dQ, dK, dV, cu_seqlens_q, cu_seqlens_k, B, H, total_q, total_k, max_seqlen_k,
                  d, softmax_scale, causal, workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_bwd_varlen(_p(Q), _p(K), _p(V), _p(O), _p(LSE), _p(dO), _p(dQ), _p(dK), _p(dV),
                               _p(cu_seqlens_q), _p(cu_seqlens_k), B, H, total_q, total_k, max_seqlen_k, d,
                               float(softmax_scale), int(bool(causal)), _p(workspace), int(workspace_bytes),
                               _stream(stream))


def attention_varlen_backward(Q, K, V, O, LSE, dO, cu_seqlens_q, cu_seqlens_k, max_seqlen_k, softmax_scale=None,
                              causal=False, ws=None, stream=None, check_status=False):
    """dQ [total_q, H, d], dK, dV [total_k, H, d] = fa_bwd_varlen(...) on bf16 CUDA tensors."""
    import torch
    total_q, H, d = (int(x) for x in Q.shape)
    total_k = int(K.shape[0])
    B = int(cu_seqlens_q.numel()) - 1
    scale = (1.0 / d ** 0.5) if softmax_scale is None else softmax_scale
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    if ws is None:
        ws = workspace(fa_bwd_varlen_workspace_size(H, total_q, d), Q.device)
    _check(fa_bwd_varlen(Q, K, V, O, LSE, dO, dQ, dK, dV, cu_seqlens_q, cu_seqlens_k, B, H, total_q, total_k,
                         max_seqlen_k, d, scale, causal, ws, ws.numel(), stream), "fa_bwd_varlen")
    if check_status:
        _check(fa_get_device_status(ws, stream), "fa_bwd_varlen (device)")
    return dQ, dK, dV


def fa_quantize_fp8(X, X8, scales, B, H, N, d, transpose, stream=None) -> int:
    return lib().fa_quantize_fp8(_p(X), _p(X8), _p(scales), B, H, N, d, int(bool(transpose)), _stream(stream))


def fa_quantize_fp8_rotated(X, X8, scales, signs, B, H, N, d, stream=None) -> int:
    return lib().fa_quantize_fp8_rotated(_p(X), _p(X8), _p(scales), _p(signs), B, H, N, d, _stream(stream))


def fa_fwd_fp8(Q8, K8, Vt8, sQ, sK, sV, O, LSE, B, H, N, d, softmax_scale, causal, key_len, block_mask,
               workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_fwd_fp8(_p(Q8), _p(K8), _p(Vt8), _p(sQ), _p(sK), _p(sV), _p(O), _p(LSE), B, H, N, d,
                            float(softmax_scale), int(bool(causal)), _p(key_len), _p(block_mask), _p(workspace),
                            int(workspace_bytes), _stream(stream))


def fa_fwd_fp8_rotated(Q8, K8, Vt8, sQ, sK, sV, O, LSE, B, H, N, d, softmax_scale, causal, key_len, block_mask,
                       workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_fwd_fp8_rotated(_p(Q8), _p(K8), _p(Vt8), _p(sQ), _p(sK), _p(sV), _p(O), _p(LSE), B, H, N, d,
                                    float(softmax_scale), int(bool(causal)), _p(key_len), _p(block_mask),
                                    _p(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, N, d, softmax_scale, causal, key_len, block_mask,
           workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_bwd(_p(Q), _p(K), _p(V), _p(O), _p(LSE), _p(dO), _p(dQ), _p(dK), _p(dV), B, H, N,
                        d, float(softmax_scale), int(bool(causal)), _p(key_len), _p(block_mask),
                        _p(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_preprocess(O, dO, B, H, N, d, workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_bwd_preprocess(_p(O), _p(dO), B, H, N, d, _p(workspace), int(workspace_bytes),
                                   _stream(stream))


def fa_bwd_main(Q, K, V, LSE, dO, dK, dV, B, H, N, d, softmax_scale, causal, key_len, block_mask,
                workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_bwd_main(_p(Q), _p(K), _p(V), _p(LSE), _p(dO), _p(dK), _p(dV), B, H, N, d,
                             float(softmax_scale), int(bool(causal)), _p(key_len), _p(block_mask),
                             _p(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_postprocess(dQ, B, H, N, d, softmax_scale, workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_bwd_postprocess(_p(dQ), B, H, N, d, float(softmax_scale), _p(workspace),
                                    int(workspace_bytes), _stream(stream))


def fa_bwd_noalloc(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, N, d, softmax_scale, causal, key_len,
                   block_mask, stream=None) -> int:
    """fa_bwd using the library's built-in scratch instead of a workspace, for
    callers that cannot allocate device memory (limits in include/fa.h)."""
    return lib().fa_bwd_noalloc(_p(Q), _p(K), _p(V), _p(O), _p(LSE), _p(dO), _p(dQ), _p(dK), _p(dV), B,
                                H, N, d, float(softmax_scale), int(bool(causal)), _p(key_len),
                                _p(block_mask), _stream(stream))


def fa_decode_workspace_size(B, H, Nq, Nk, d, num_splits=0) -> int:
    return lib().fa_decode_workspace_size(B, H, Nq, Nk, d, int(num_splits))


def fa_decode(Q, K, V, O, LSE, B, H, Nq, Nk, d, softmax_scale, causal, kv_len, num_splits, workspace,
              workspace_bytes, stream=None) -> int:
    return lib().fa_decode(_p(Q), _p(K), _p(V), _p(O), _p(LSE), B, H, Nq, Nk, d, float(softmax_scale),
                           int(bool(causal)), _p(kv_len), int(num_splits), _p(workspace),
                           int(workspace_bytes), _stream(stream))


def fa_tile_plan(B, N, causal, key_len, block_mask, plan, workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_tile_plan(B, N, int(bool(causal)), _p(key_len), _p(block_mask), _p(plan),
                              _p(workspace), int(workspace_bytes), _stream(stream))


def fa_attention_host(Q, K, V, dO, O, LSE, dQ, dK, dV, B, H, N, d, softmax_scale, causal, key_len,
                      block_mask, dev_workspace, dev_workspace_bytes, stream=None) -> int:
    return lib().fa_attention_host(_p(Q), _p(K), _p(V), _p(dO), _p(O), _p(LSE), _p(dQ), _p(dK),
                                   _p(dV), B, H, N, d, float(softmax_scale), int(bool(causal)),
                                   _p(key_len), _p(block_mask), _p(dev_workspace),
                                   int(dev_workspace_bytes), _stream(stream))


def fa_get_device_status(workspace, stream=None) -> int:
    return lib().fa_get_device_status(_p(workspace), _stream(stream))


def fa_selftest_wait_timeout(workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_selftest_wait_timeout(_p(workspace), int(workspace_bytes), _stream(stream))


def fa_reset_device_status(workspace, stream=None) -> int:
    return lib().fa_reset_device_status(_p(workspace), _stream(stream))


def fa_status_string(status) -> str:
    return lib().fa_status_string(int(status)).decode()


# ---------------------------------------------------------------- torch conveniences
def _dims(Q):
    if Q.dim() != 4:
        raise ValueError("expected [B, H, N, d]")
    return tuple(int(x) for x in Q.shape)


def workspace(nbytes, device):
    import torch
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def attention_forward(Q, K, V, softmax_scale=None, causal=False, key_len=None, block_mask=None,
                      ws=None, out=None, stream=None, check_status=False):
    """O, LSE = fa_fwd(Q, K, V, ...) on bf16 CUDA tensors [B, H, N, d]."""
    import torch
    B, H, N, d = _dims(Q)
    scale = (1.0 / d ** 0.5) if softmax_scale is None else softmax_scale
    if out is None:
        O = torch.empty_like(Q)
        LSE = torch.empty((B, H, N), dtype=torch.float32, device=Q.device)
    else:
        O, LSE = out
    need = fa_fwd_workspace_size(B, H, N, d)
    if ws is None:
        ws = workspace(need, Q.device)
    _check(fa_fwd(Q, K, V, O, LSE, B, H, N, d, scale, causal, key_len, block_mask, ws, ws.numel(),
                  stream), "fa_fwd")
    if check_status:
        _check(fa_get_device_status(ws, stream), "fa_fwd (device)")
    return O, LSE


def quantize_fp8(X, transpose=False, stream=None, signs=None):
    """(codes, scales) = fa_quantize_fp8(X): codes uint8 [B, H, N, d] (transpose:
    [B, H, d, Np], Np = ceil(N / 16) * 16), scales fp32 [B, H, ceil(N / 128)].
    With signs (device int8 [d] of +-1), the codes of the incoherently
    rotated rows (fa_quantize_fp8_rotated; not with transpose)."""
    import torch
    B, H, N, d = _dims(X)
    Np = (N + 15) // 16 * 16
    X8 = torch.empty((B, H, d, Np) if transpose else (B, H, N, d), dtype=torch.uint8, device=X.device)
    sc = torch.empty((B, H, (N + 127) // 128), dtype=torch.float32, device=X.device)
    if signs is not None:
        if transpose:
            raise ValueError("the rotation applies to Q and K, not to the transposed V")
        _check(fa_quantize_fp8_rotated(X, X8, sc, signs, B, H, N, d, stream), "fa_quantize_fp8_rotated")
    else:
        _check(fa_quantize_fp8(X, X8, sc, B, H, N, d, transpose, stream), "fa_quantize_fp8")
    return X8, sc


def attention_forward_fp8(Q, K, V, softmax_scale=None, causal=False, key_len=None, block_mask=None, ws=None,
                          stream=None, check_status=False, signs=None):
    """O, LSE of the FP8 forward on bf16 CUDA tensors [B, H, N, 128]: Q, K and V
    are block-quantised (fa_quantize_fp8), then fa_fwd_fp8 runs.  With signs
    (device int8 [d] of random +-1), Q and K are quantised with incoherent
    processing (fa_quantize_fp8_rotated) and fa_fwd_fp8_rotated runs (it takes
    the scores' extra factor d out of the softmax scale)."""
    import torch
    B, H, N, d = _dims(Q)
    scale = (1.0 / d ** 0.5) if softmax_scale is None else softmax_scale
    Q8, sQ = quantize_fp8(Q, False, stream, signs)
    K8, sK = quantize_fp8(K, False, stream, signs)
    Vt8, sV = quantize_fp8(V, True, stream)
    O = torch.empty_like(Q)
    LSE = torch.empty((B, H, N), dtype=torch.float32, device=Q.device)
    need = fa_fwd_workspace_size(B, H, N, d)
    if ws is None:
        ws = workspace(need, Q.device)
    call, name = (fa_fwd_fp8, "fa_fwd_fp8") if signs is None else (fa_fwd_fp8_rotated, "fa_fwd_fp8_rotated")
    _check(call(Q8, K8, Vt8, sQ, sK, sV, O, LSE, B, H, N, d, scale, causal, key_len, block_mask, ws,
                ws.numel(), stream), name)
    if check_status:
        _check(fa_get_device_status(ws, stream), "fa_fwd_fp8 (device)")
    return O, LSE


def attention_backward(Q, K, V, O, LSE, dO, softmax_scale=None, causal=False, key_len=None,
                       block_mask=None, ws=None, out=None, stream=None, check_status=False):
    """dQ, dK, dV = fa_bwd(...) on bf16 CUDA tensors [B, H, N, d]."""
    import torch
    B, H, N, d = _dims(Q)
    scale = (1.0 / d ** 0.5) if softmax_scale is None else softmax_scale
    if out is None:
        dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    else:
        dQ, dK, dV = out
    need = fa_bwd_workspace_size(B, H, N, d)
    if ws is None:
        ws = workspace(need, Q.device)
    _check(fa_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, N, d, scale, causal, key_len, block_mask,
                  ws, ws.numel(), stream), "fa_bwd")
    if check_status:
        _check(fa_get_device_status(ws, stream), "fa_bwd (device)")
    return dQ, dK, dV


def tile_plan(B, N, causal=False, key_len=None, block_mask=None, device="cuda", stream=None):
    """uint8 [B, T, T] tile classes (0 skip, 1 full, 2 partial) from the device."""
    import torch
    T = (N + 127) // 128
    plan = torch.full((B, T, T), 255, dtype=torch.uint8, device=device)
    ws = workspace(256, device)
    _check(fa_tile_plan(B, N, causal, key_len, block_mask, plan, ws, ws.numel(), stream), "fa_tile_plan")
    _check(fa_get_device_status(ws, stream), "fa_tile_plan (device)")
    return plan


def attention_decode(Q, K, V, softmax_scale=None, causal=False, kv_len=None, num_splits=0, ws=None,
                     stream=None, check_status=False):
    """O, LSE = fa_decode(...): Q [B, H, Nq, d] against the cache K, V [B, H, Nk, d]."""
    import torch
    B, H, Nq, d = _dims(Q)
    Nk = int(K.shape[2])
    scale = (1.0 / d ** 0.5) if softmax_scale is None else softmax_scale
    O = torch.empty_like(Q)
    LSE = torch.empty((B, H, Nq), dtype=torch.float32, device=Q.device)
    need = fa_decode_workspace_size(B, H, Nq, Nk, d, num_splits)
    if ws is None:
        ws = workspace(need, Q.device)
    _check(fa_decode(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, causal, kv_len, num_splits, ws, ws.numel(),
                     stream), "fa_decode")
    if check_status:
        _check(fa_get_device_status(ws, stream), "fa_decode (device)")
    return O, LSE
