"""fp64 CPU oracle for exact scaled dot-product attention (test infrastructure).

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library (the CUDA path in
``io_aware_exact_09_gb300``) never imports it, and this package never imports
the product library: the two share no code.

The arithmetic lives in ``fa_oracle.c`` (plain C, fp64, OpenMP over rows);
this module only builds it with gcc and marshals numpy arrays through ctypes.
``online.py`` holds the pages' two-block merge identity, ``io_model.py``
the page-2 traffic/time model and ``incoherent.py`` the Hadamard rotation
of the FP8 forward's incoherent processing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into liboracle.so beside it (gcc, -O3, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O3", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB points the tests' mutation check at a deliberately
            # broken copy of the oracle; normally the library is built here.
            path = os.environ.get("ORACLE_LIB") or build()
            lib = ctypes.CDLL(path)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            bp = ctypes.POINTER(ctypes.c_uint8)
            lp = ctypes.POINTER(ctypes.c_int64)
            i, dbl = ctypes.c_int, ctypes.c_double
            common = [i, i, i, i, dbl, i, ip, bp, i]
            lib.oracle_fwd.argtypes = [dp, dp, dp] + common + [dp, dp, dp]
            lib.oracle_bwd.argtypes = [dp, dp, dp, dp] + common + [dp, dp, dp, dp, dp]
            lib.oracle_query_rows.argtypes = [dp, dp, dp, dp] + common + [i, lp, dp, dp, dp]
            lib.oracle_key_rows.argtypes = [dp, dp, dp, dp] + common + [i, lp, dp, dp]
            lib.oracle_tile_plan.argtypes = [i, i, i, ip, bp, i, i, i, bp]
            lib.oracle_decode.argtypes = [dp, dp, dp, i, i, i, i, i, dbl, i, ip, dp, dp]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_bwd_rect.argtypes = [dp, dp, dp, dp, i, i, i, i, dbl, i, dp, dp, dp, dp, dp]
            lib.oracle_bwd_rect.restype = ctypes.c_int
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_ubyte
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_ubyte]
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            fp = ctypes.POINTER(ctypes.c_float)
            lib.oracle_quantize_fp8.argtypes = [fp, i, i, i, i, bp, fp]
            lib.oracle_quantize_fp8.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            for f in (lib.oracle_fwd, lib.oracle_bwd, lib.oracle_query_rows,
                      lib.oracle_key_rows, lib.oracle_tile_plan, lib.oracle_num_threads):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    return a


def _shapes(*arrays):
    """Self-attention: every operand is [B, H, N, d] with the same shape."""
    shp = arrays[0].shape
    if len(shp) != 4:
        raise ValueError("expected [B, H, N, d], got %r" % (shp,))
    for a in arrays[1:]:
        if a is not None and a.shape != shp:
            raise ValueError("operand shapes differ: %r vs %r" % (a.shape, shp))
    return shp


def _check_masks(B, N, kl, bm, mask_block):
    if kl is not None and kl.shape != (B,):
        raise ValueError("key_len must have shape [B]")
    if bm is not None:
        nb = (N + mask_block - 1) // mask_block
        if bm.shape != (nb, nb):
            raise ValueError("block_mask must have shape [%d, %d]" % (nb, nb))


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _masks(key_len, block_mask):
    kl = None if key_len is None else np.ascontiguousarray(np.asarray(key_len, dtype=np.int32))
    bm = None if block_mask is None else np.ascontiguousarray(np.asarray(block_mask, dtype=np.uint8))
    return kl, bm


def num_threads() -> int:
    """OpenMP threads the oracle runs with (its `cores`)."""
    return int(_load().oracle_num_threads())


def attention_fwd(Q, K, V, scale, causal=False, key_len=None, block_mask=None,
                  mask_block=128, return_P=False):
    """O, LSE (and optionally P) of softmax(scale*QK^T [+mask]) V, fp64.

    Q, K, V: arrays [B, H, N, d].  key_len: int [B] or None.  block_mask:
    uint8 [ceil(N/mask_block)]^2 or None.
    """
    lib = _load()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, d = _shapes(Q, K, V)
    kl, bm = _masks(key_len, block_mask)
    _check_masks(B, N, kl, bm, mask_block)
    O = np.zeros((B, H, N, d), np.float64)
    LSE = np.zeros((B, H, N), np.float64)
    P = np.zeros((B, H, N, N), np.float64) if return_P else None
    rc = lib.oracle_fwd(_ptr(Q, ctypes.c_double), _ptr(K, ctypes.c_double), _ptr(V, ctypes.c_double),
                        B, H, N, d, float(scale), int(bool(causal)), _ptr(kl, ctypes.c_int32),
                        _ptr(bm, ctypes.c_uint8), int(mask_block), _ptr(O, ctypes.c_double),
                        _ptr(LSE, ctypes.c_double), _ptr(P, ctypes.c_double))
    if rc != 0:
        raise RuntimeError("oracle_fwd failed: %d" % rc)
    return (O, LSE, P) if return_P else (O, LSE)


def attention_bwd(Q, K, V, dO, scale, causal=False, key_len=None, block_mask=None, mask_block=128):
    """O, LSE, dQ, dK, dV for the loss sum(O * dO), fp64 (full materialisation)."""
    lib = _load()
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, N, d = _shapes(Q, K, V, dO)
    kl, bm = _masks(key_len, block_mask)
    _check_masks(B, N, kl, bm, mask_block)
    O = np.zeros((B, H, N, d), np.float64)
    LSE = np.zeros((B, H, N), np.float64)
    dQ, dK, dV = (np.zeros((B, H, N, d), np.float64) for _ in range(3))
    c = ctypes.c_double
    rc = lib.oracle_bwd(_ptr(Q, c), _ptr(K, c), _ptr(V, c), _ptr(dO, c), B, H, N, d, float(scale),
                        int(bool(causal)), _ptr(kl, ctypes.c_int32), _ptr(bm, ctypes.c_uint8),
                        int(mask_block), _ptr(O, c), _ptr(LSE, c), _ptr(dQ, c), _ptr(dK, c),
                        _ptr(dV, c))
    if rc != 0:
        raise RuntimeError("oracle_bwd failed: %d" % rc)
    return O, LSE, dQ, dK, dV


def query_rows(Q, K, V, dO, scale, rows, causal=False, key_len=None, block_mask=None,
               mask_block=128):
    """O, LSE and dQ for chosen query rows; rows are flat (b*H+h)*N+i indices.

    dO may be None (then dQ is not computed and None is returned for it).
    """
    lib = _load()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    dOa = None if dO is None else _f64(dO)
    B, H, N, d = _shapes(Q, K, V, dOa)
    kl, bm = _masks(key_len, block_mask)
    _check_masks(B, N, kl, bm, mask_block)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.size
    O = np.zeros((n, d), np.float64)
    LSE = np.zeros((n,), np.float64)
    dQ = np.zeros((n, d), np.float64) if dOa is not None else None
    c = ctypes.c_double
    rc = lib.oracle_query_rows(_ptr(Q, c), _ptr(K, c), _ptr(V, c), _ptr(dOa, c), B, H, N, d,
                               float(scale), int(bool(causal)), _ptr(kl, ctypes.c_int32),
                               _ptr(bm, ctypes.c_uint8), int(mask_block), n,
                               _ptr(rows, ctypes.c_int64), _ptr(O, c), _ptr(LSE, c), _ptr(dQ, c))
    if rc != 0:
        raise RuntimeError("oracle_query_rows failed: %d" % rc)
    return O, LSE, dQ


def key_rows(Q, K, V, dO, scale, keys, causal=False, key_len=None, block_mask=None,
             mask_block=128):
    """dK and dV for chosen key rows; keys are flat (b*H+h)*N+j indices."""
    lib = _load()
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, N, d = _shapes(Q, K, V, dO)
    kl, bm = _masks(key_len, block_mask)
    _check_masks(B, N, kl, bm, mask_block)
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.int64))
    n = keys.size
    dK = np.zeros((n, d), np.float64)
    dV = np.zeros((n, d), np.float64)
    c = ctypes.c_double
    rc = lib.oracle_key_rows(_ptr(Q, c), _ptr(K, c), _ptr(V, c), _ptr(dO, c), B, H, N, d,
                             float(scale), int(bool(causal)), _ptr(kl, ctypes.c_int32),
                             _ptr(bm, ctypes.c_uint8), int(mask_block), n,
                             _ptr(keys, ctypes.c_int64), _ptr(dK, c), _ptr(dV, c))
    if rc != 0:
        raise RuntimeError("oracle_key_rows failed: %d" % rc)
    return dK, dV


def tile_plan(B, N, causal=False, key_len=None, block_mask=None, mask_block=128,
              tile_q=128, tile_k=128):
    """uint8 [B, Tq, Tk]: 0 skip, 1 full, 2 partial, by brute force over elements."""
    lib = _load()
    kl, bm = _masks(key_len, block_mask)
    _check_masks(B, N, kl, bm, mask_block)
    Tq = (N + tile_q - 1) // tile_q
    Tk = (N + tile_k - 1) // tile_k
    plan = np.zeros((B, Tq, Tk), np.uint8)
    rc = lib.oracle_tile_plan(B, N, int(bool(causal)), _ptr(kl, ctypes.c_int32),
                              _ptr(bm, ctypes.c_uint8), int(mask_block), tile_q, tile_k,
                              _ptr(plan, ctypes.c_uint8))
    if rc != 0:
        raise RuntimeError("oracle_tile_plan failed: %d" % rc)
    return plan


def attention_decode(Q, K, V, scale, causal=False, kv_len=None):
    """O, LSE of Nq query rows against Nk cached keys (fp64).

    Q: [B, H, Nq, d]; K, V: [B, H, Nk, d]; kv_len: int [B] or None.  With
    causal, query i sees keys j <= kv_len[b] - Nq + i (the queries are the
    last Nq positions)."""
    lib = _load()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    if Q.ndim != 4 or K.shape != V.shape or K.ndim != 4 or Q.shape[:2] != K.shape[:2] or Q.shape[3] != K.shape[3]:
        raise ValueError("expected Q [B, H, Nq, d] and K, V [B, H, Nk, d]")
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    kl = None if kv_len is None else np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32))
    if kl is not None and kl.shape != (B,):
        raise ValueError("kv_len must have shape [B]")
    O = np.zeros((B, H, Nq, d), np.float64)
    LSE = np.zeros((B, H, Nq), np.float64)
    c = ctypes.c_double
    rc = lib.oracle_decode(_ptr(Q, c), _ptr(K, c), _ptr(V, c), B, H, Nq, Nk, d, float(scale),
                           int(bool(causal)), _ptr(kl, ctypes.c_int32), _ptr(O, c), _ptr(LSE, c))
    if rc != 0:
        raise RuntimeError("oracle_decode failed: %d" % rc)
    return O, LSE


def attention_varlen(Q, K, V, cu_q, cu_k, scale, causal=False):
    """Ragged batch (packed sequences), fp64.

    Q: [total_q, H, d], K, V: [total_k, H, d]; sequence b owns query rows
    cu_q[b]..cu_q[b+1]-1 and key rows cu_k[b]..cu_k[b+1]-1.  Each sequence is
    attended on its own; its Lq queries are the last Lq positions of its Lk
    keys, so with causal query i sees key j iff j <= i + Lk - Lq (the decode
    reading, bottom-right; Lq = Lk gives the square causal mask).  Returns
    O [total_q, H, d] and LSE [H, total_q].  Each sequence goes through
    attention_decode on its own slice."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    cu_q = np.asarray(cu_q, np.int64)
    cu_k = np.asarray(cu_k, np.int64)
    if Q.ndim != 3 or K.ndim != 3 or K.shape != V.shape or Q.shape[1:] != K.shape[1:]:
        raise ValueError("expected Q [total_q, H, d] and K, V [total_k, H, d]")
    if cu_q.shape != cu_k.shape or cu_q.ndim != 1 or cu_q[0] != 0 or cu_k[0] != 0 or \
            cu_q[-1] != Q.shape[0] or cu_k[-1] != K.shape[0] or np.any(np.diff(cu_q) < 0) or np.any(np.diff(cu_k) < 0):
        raise ValueError("cu_q / cu_k must be [B + 1] offsets from 0 to total, non-decreasing")
    H, d = Q.shape[1], Q.shape[2]
    O = np.zeros(Q.shape, np.float64)
    LSE = np.full((H, Q.shape[0]), -np.inf, np.float64)
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        if q1 == q0:
            continue
        qb = np.ascontiguousarray(Q[q0:q1].transpose(1, 0, 2))[None]
        kb = np.ascontiguousarray(K[k0:k1].transpose(1, 0, 2))[None]
        vb = np.ascontiguousarray(V[k0:k1].transpose(1, 0, 2))[None]
        ob, lb = attention_decode(qb, kb, vb, scale, causal=causal)
        O[q0:q1] = ob[0].transpose(1, 0, 2)
        LSE[:, q0:q1] = lb[0]
    return O, LSE


def attention_bwd_rect(Q, K, V, dO, scale, causal=False):
    """O, LSE, dQ, dK, dV of Nq query rows against Nk keys (fp64), the queries
    being the last Nq positions (with causal, query i sees key j iff
    j <= i + Nk - Nq).  Q, dO: [B, H, Nq, d]; K, V: [B, H, Nk, d]."""
    lib = _load()
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    if Q.ndim != 4 or K.shape != V.shape or K.ndim != 4 or Q.shape != dO.shape or Q.shape[:2] != K.shape[:2] \
            or Q.shape[3] != K.shape[3]:
        raise ValueError("expected Q, dO [B, H, Nq, d] and K, V [B, H, Nk, d]")
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    O = np.zeros((B, H, Nq, d), np.float64)
    LSE = np.zeros((B, H, Nq), np.float64)
    dQ = np.zeros((B, H, Nq, d), np.float64)
    dK, dV = np.zeros((B, H, Nk, d), np.float64), np.zeros((B, H, Nk, d), np.float64)
    c = ctypes.c_double
    rc = lib.oracle_bwd_rect(_ptr(Q, c), _ptr(K, c), _ptr(V, c), _ptr(dO, c), B * H, Nq, Nk, d, float(scale),
                             int(bool(causal)), _ptr(O, c), _ptr(LSE, c), _ptr(dQ, c), _ptr(dK, c), _ptr(dV, c))
    if rc != 0:
        raise RuntimeError("oracle_bwd_rect failed: %d" % rc)
    return O, LSE, dQ, dK, dV


def attention_varlen_bwd(Q, K, V, dO, cu_q, cu_k, scale, causal=False):
    """Forward and backward of a ragged batch (packed sequences), fp64.

    Layouts as attention_varlen: Q, dO [total_q, H, d], K, V [total_k, H, d],
    offsets cu_q, cu_k [B + 1].  Each sequence is attended on its own, its Lq
    queries being the last Lq of its Lk positions (bottom-right causal).
    Returns O, dQ [total_q, H, d], LSE [H, total_q] and dK, dV [total_k, H, d];
    a sequence without queries gets dK = dV = 0 for its keys, one without keys
    O = dQ = 0 and LSE = -inf.  Each sequence goes through attention_bwd_rect
    on its own slice."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    cu_q = np.asarray(cu_q, np.int64)
    cu_k = np.asarray(cu_k, np.int64)
    if Q.ndim != 3 or K.ndim != 3 or K.shape != V.shape or Q.shape != dO.shape or Q.shape[1:] != K.shape[1:]:
        raise ValueError("expected Q, dO [total_q, H, d] and K, V [total_k, H, d]")
    if cu_q.shape != cu_k.shape or cu_q.ndim != 1 or cu_q[0] != 0 or cu_k[0] != 0 or \
            cu_q[-1] != Q.shape[0] or cu_k[-1] != K.shape[0] or np.any(np.diff(cu_q) < 0) or np.any(np.diff(cu_k) < 0):
        raise ValueError("cu_q / cu_k must be [B + 1] offsets from 0 to total, non-decreasing")
    H = Q.shape[1]
    O, dQ = np.zeros(Q.shape, np.float64), np.zeros(Q.shape, np.float64)
    dK, dV = np.zeros(K.shape, np.float64), np.zeros(K.shape, np.float64)
    LSE = np.full((H, Q.shape[0]), -np.inf, np.float64)
    tr = lambda X, a, b: np.ascontiguousarray(X[a:b].transpose(1, 0, 2))[None]
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        ob, lb, dqb, dkb, dvb = attention_bwd_rect(tr(Q, q0, q1), tr(K, k0, k1), tr(V, k0, k1), tr(dO, q0, q1),
                                                   scale, causal=causal)
        O[q0:q1] = ob[0].transpose(1, 0, 2)
        dQ[q0:q1] = dqb[0].transpose(1, 0, 2)
        LSE[:, q0:q1] = lb[0]
        dK[k0:k1] = dkb[0].transpose(1, 0, 2)
        dV[k0:k1] = dvb[0].transpose(1, 0, 2)
    return O, LSE, dQ, dK, dV


E4M3_MAX = 448.0
FP8_BLOCK = 128


def e4m3_encode(x):
    """e4m3 codes (uint8) of fp32 values: nearest, ties to even, saturating."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    flat, of = x.reshape(-1), out.reshape(-1)
    for k in range(flat.size):
        of[k] = lib.oracle_e4m3_encode(float(flat[k]))
    return out


def e4m3_table():
    """fp64 value of each of the 256 e4m3 codes (NaN for the two NaN codes)."""
    lib = _load()
    return np.array([lib.oracle_e4m3_decode(c) for c in range(256)], np.float64)


def quantize_fp8(X, transpose=False):
    """Block quantisation of X [B, H, N, d] (bf16 values as fp32/fp64):
    codes uint8 [B, H, N, d] (with transpose: [B, H, d, Np], Np = ceil(N/16)*16)
    and scales fp32 [B, H, ceil(N/128)] (amax / 448; 0 for an all-zero block)."""
    lib = _load()
    X = np.ascontiguousarray(np.asarray(X, dtype=np.float32))
    if X.ndim != 4:
        raise ValueError("expected X [B, H, N, d]")
    B, H, N, d = X.shape
    T = (N + FP8_BLOCK - 1) // FP8_BLOCK
    Np = (N + 15) // 16 * 16
    codes = np.zeros((B, H, d, Np) if transpose else (B, H, N, d), np.uint8)
    scales = np.zeros((B, H, T), np.float32)
    fp = ctypes.POINTER(ctypes.c_float)
    rc = lib.oracle_quantize_fp8(X.ctypes.data_as(fp), B * H, N, d, int(bool(transpose)),
                                 codes.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), scales.ctypes.data_as(fp))
    if rc != 0:
        raise RuntimeError("oracle_quantize_fp8 failed: %d" % rc)
    return codes, scales


def dequantize_fp8(codes, scales, N, transpose=False):
    """fp64 [B, H, N, d] values the codes stand for: e4m3(code) * scale of the
    code's 128-row block."""
    codes = np.asarray(codes)
    vals = e4m3_table()[codes]
    if transpose:
        vals = np.swapaxes(vals, 2, 3)[:, :, :N, :]
    rows = np.arange(N) // FP8_BLOCK
    return vals * np.asarray(scales, np.float64)[:, :, rows][..., None]


def quantize_fp8_rotated(X, signs):
    """Block quantisation of the incoherently rotated X [B, H, N, d]:
    quantize_fp8(rotate(X, signs)) (codes [B, H, N, d], scales [B, H, T])."""
    from .incoherent import rotate
    return quantize_fp8(rotate(X, signs), False)


from .online import merge_blocks, online_fold  # noqa: E402,F401
from .io_model import io_model  # noqa: E402,F401
