"""Seeded synthetic inputs for the attention workloads.

This module holds input generation only -- no attention arithmetic.  It is
the one module both the oracle-side checks and the CUDA path's tests/bench
draw their inputs from.

Recipe (every workload): a CPU ``torch.Generator`` seeded with the
workload's seed draws, in this order, Q, K, V, dO as fp32 N(0, 1) tensors of
shape [B, H, N, d] (times ``input_scale``), each rounded to bf16 with
round-to-nearest-even; then the per-sequence key lengths (if any); then the
block-sparsity mask (if any).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

MASK_BLOCK = 128


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    seed: int
    causal: bool = False
    input_scale: float = 1.0
    key_len_range: Optional[tuple] = None      # inclusive (lo, hi) or None
    sparse_density: Optional[float] = None     # target fraction of nonzero blocks, or None
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads the method is evaluated on: a small exact check, a
# GPT-2-medium-shaped causal layer, a BERT-large-shaped encoder layer with key
# padding, a long-context layer (run non-causal and causal) and a
# block-sparse layer.
WORKLOADS = {
    "small_b1h2n128d64": Workload("small_b1h2n128d64", 1, 2, 128, 64, 1000,
                                  description="B1 H2 N128 d64, no mask"),
    "gpt2m_causal_b8h16n1024d64": Workload("gpt2m_causal_b8h16n1024d64", 8, 16, 1024, 64, 1001,
                                           causal=True,
                                           description="GPT-2-medium shape, causal"),
    "bertl_keypad_b16h16n512d64": Workload("bertl_keypad_b16h16n512d64", 16, 16, 512, 64, 1002,
                                           key_len_range=(128, 512),
                                           description="BERT-large shape, key padding U[128,512]"),
    "longctx_b1h16n16384d128": Workload("longctx_b1h16n16384d128", 1, 16, 16384, 128, 1003,
                                        input_scale=0.5,
                                        description="long context, N=16384, d=128, inputs x0.5"),
    "longctx_causal_b1h16n16384d128": Workload("longctx_causal_b1h16n16384d128", 1, 16, 16384, 128,
                                               1003, causal=True, input_scale=0.5,
                                               description="long context, causal"),
    "blocksparse_b2h16n8192d64": Workload("blocksparse_b2h16n8192d64", 2, 16, 8192, 64, 1004,
                                          sparse_density=0.15,
                                          description="block-sparse, band 3 + 4 global + random, s~0.15"),
}


@dataclass(frozen=True)
class DecodeWorkload:
    """Nq new query rows per (b, h) against a key/value cache of Nk rows."""
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    seed: int
    causal: bool = False
    kv_len_range: Optional[tuple] = None       # inclusive (lo, hi) or None (full caches)
    description: str = ""

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# Decode shapes (the pages give none): one new token per sequence against a
# 32K cache with 32 heads of d=128, and a speculative-decoding-like step
# (4 new tokens, causal) over ragged caches of up to 16K with d=64.
DECODE_WORKLOADS = {
    "decode_b4h32q1k32768d128": DecodeWorkload("decode_b4h32q1k32768d128", 4, 32, 1, 32768, 128, 1005,
                                               description="B4 H32, 1 new token, full 32K caches, d=128"),
    "decode_ragged_b16h8q4k16384d64": DecodeWorkload("decode_ragged_b16h8q4k16384d64", 16, 8, 4, 16384, 64,
                                                     1006, causal=True, kv_len_range=(1024, 16384),
                                                     description="B16 H8, 4 new tokens (causal), "
                                                                 "cache lengths U[1024, 16384], d=64"),
}


def make_decode_inputs(w: DecodeWorkload, B=None, H=None):
    """Q [B, H, Nq, d], K, V [B, H, Nk, d] (bf16 from fp32 N(0, 1), drawn in
    that order) and kv_len (int32 [B] or None) from the workload's seed.
    B and H may be lowered to draw a smaller case with the same recipe and
    seed (a bounded CPU sample); its values are not a slice of the full draw."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    gen = torch.Generator().manual_seed(w.seed)
    Q = to_bf16(torch.randn((B, H, w.Nq, w.d), generator=gen, dtype=torch.float32))
    K = to_bf16(torch.randn((B, H, w.Nk, w.d), generator=gen, dtype=torch.float32))
    V = to_bf16(torch.randn((B, H, w.Nk, w.d), generator=gen, dtype=torch.float32))
    kv_len = None
    if w.kv_len_range is not None:
        kv_len = draw_key_len(B, w.kv_len_range[0], w.kv_len_range[1], gen)
    return {"Q": Q, "K": K, "V": V, "kv_len": kv_len, "causal": w.causal, "scale": w.softmax_scale}


def decode_visible_keys(w: DecodeWorkload, kv_len=None) -> int:
    """Number of (b, h, key) cache rows a decode step must read: every row
    below the batch's cache length (all Nk when there are no lengths)."""
    if kv_len is None:
        return w.B * w.H * w.Nk
    return w.H * sum(min(max(int(x), 0), w.Nk) for x in kv_len)


@dataclass(frozen=True)
class VarlenWorkload:
    """A ragged batch of B packed sequences of H heads: query lengths drawn
    U{lo..hi}; each sequence's keys are its queries (Lk = Lq) unless
    k_extra_range adds a cached prefix (Lk = Lq + U{lo..hi})."""
    name: str
    B: int
    H: int
    d: int
    seed: int
    q_len_range: tuple
    k_extra_range: Optional[tuple] = None
    causal: bool = True
    description: str = ""

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# Ragged batches (the pages name the layout, not sizes): a prefill batch of
# 16 sequences of 256..4096 tokens, and a chunked-prefill batch whose new
# chunks of 128..1024 tokens attend to cached prefixes of up to 8192 tokens.
VARLEN_WORKLOADS = {
    "varlen_prefill_b16h16d128": VarlenWorkload("varlen_prefill_b16h16d128", 16, 16, 128, 1007, (256, 4096),
                                                description="16 sequences, lengths U{256..4096}, causal, d=128"),
    "varlen_chunked_b16h16d128": VarlenWorkload("varlen_chunked_b16h16d128", 16, 16, 128, 1008, (128, 1024),
                                                k_extra_range=(0, 8192),
                                                description="16 chunks of U{128..1024} new tokens after cached "
                                                            "prefixes of U{0..8192}, causal, d=128"),
}


def make_varlen_inputs(w: VarlenWorkload):
    """Lengths first (query lengths, then prefix lengths), then Q [total_q, H, d]
    and K, V [total_k, H, d] (bf16 from fp32 N(0, 1)); cu_q, cu_k int32 [B + 1]."""
    gen = torch.Generator().manual_seed(w.seed)
    lq = torch.randint(w.q_len_range[0], w.q_len_range[1] + 1, (w.B,), generator=gen, dtype=torch.int64)
    lk = lq.clone()
    if w.k_extra_range is not None:
        lk = lk + torch.randint(w.k_extra_range[0], w.k_extra_range[1] + 1, (w.B,), generator=gen,
                                dtype=torch.int64)
    cu_q = torch.zeros(w.B + 1, dtype=torch.int32)
    cu_k = torch.zeros(w.B + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(lq, 0).to(torch.int32)
    cu_k[1:] = torch.cumsum(lk, 0).to(torch.int32)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    Q = to_bf16(torch.randn((tq, w.H, w.d), generator=gen, dtype=torch.float32))
    K = to_bf16(torch.randn((tk, w.H, w.d), generator=gen, dtype=torch.float32))
    V = to_bf16(torch.randn((tk, w.H, w.d), generator=gen, dtype=torch.float32))
    return {"Q": Q, "K": K, "V": V, "cu_q": cu_q, "cu_k": cu_k, "max_q": int(lq.max()), "causal": w.causal,
            "scale": w.softmax_scale}


def varlen_fwd_flops(cu_q, cu_k, H, d, causal) -> float:
    """4 * d * H * (number of visible (query, key) pairs), causal bottom-right."""
    pairs = 0
    for b in range(len(cu_q) - 1):
        lq = int(cu_q[b + 1]) - int(cu_q[b])
        lk = int(cu_k[b + 1]) - int(cu_k[b])
        if not causal:
            pairs += lq * lk
        else:
            sh = lk - lq
            # query i sees min(lk, max(0, i + sh + 1)) keys
            pairs += sum(min(lk, max(0, i + sh + 1)) for i in range(lq))
    return 4.0 * d * H * pairs


def to_bf16(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> bf16 with round-to-nearest-even (torch's conversion)."""
    return x.to(torch.bfloat16)


def draw_qkvdo(B, H, N, d, gen: torch.Generator, input_scale: float = 1.0):
    out = []
    for _ in range(4):
        x = torch.randn((B, H, N, d), generator=gen, dtype=torch.float32)
        if input_scale != 1.0:
            x = x * input_scale
        out.append(to_bf16(x))
    return out


def draw_key_len(B: int, lo: int, hi: int, gen: torch.Generator) -> torch.Tensor:
    """int32 [B], uniform integers in [lo, hi]."""
    return torch.randint(lo, hi + 1, (B,), generator=gen, dtype=torch.int64).to(torch.int32)


def draw_block_mask(N: int, density: float, gen: torch.Generator, block: int = MASK_BLOCK,
                    band: int = 1, n_global: int = 4) -> torch.Tensor:
    """uint8 [nb, nb]: blocks with |r - c| <= band, plus key-block columns
    0..n_global-1, plus blocks drawn uniformly without replacement from the
    rest until round(density * nb^2) blocks are nonzero."""
    nb = (N + block - 1) // block
    m = torch.zeros((nb, nb), dtype=torch.uint8)
    r = torch.arange(nb)
    m[(r[:, None] - r[None, :]).abs() <= band] = 1
    m[:, :min(n_global, nb)] = 1
    target = int(round(density * nb * nb))
    free = (m.flatten() == 0).nonzero().flatten()
    need = max(0, target - int(m.sum()))
    if need > 0 and free.numel() > 0:
        perm = torch.randperm(free.numel(), generator=gen)
        m.view(-1)[free[perm[:need]]] = 1
    return m


def make_inputs(w: Workload, with_dO: bool = True):
    """All inputs of a workload on the CPU: dict with Q, K, V, dO (bf16),
    key_len (int32 [B] or None), block_mask (uint8 [nb, nb] or None), causal,
    scale."""
    gen = torch.Generator().manual_seed(w.seed)
    Q, K, V, dO = draw_qkvdo(w.B, w.H, w.N, w.d, gen, w.input_scale)
    key_len = None
    if w.key_len_range is not None:
        key_len = draw_key_len(w.B, w.key_len_range[0], w.key_len_range[1], gen)
    block_mask = None
    if w.sparse_density is not None:
        block_mask = draw_block_mask(w.N, w.sparse_density, gen)
    return {"Q": Q, "K": K, "V": V, "dO": dO if with_dO else None, "key_len": key_len,
            "block_mask": block_mask, "causal": w.causal, "scale": w.softmax_scale}


def make_case(B, H, N, d, seed, causal=False, key_len=None, block_mask=None, input_scale=1.0,
              key_len_range=None, sparse_density=None):
    """Ad-hoc case with the same recipe (for tests: ragged N, odd shapes)."""
    w = Workload("case", B, H, N, d, seed, causal=causal, input_scale=input_scale,
                 key_len_range=key_len_range, sparse_density=sparse_density)
    c = make_inputs(w)
    if key_len is not None:
        c["key_len"] = torch.as_tensor(key_len, dtype=torch.int32)
    if block_mask is not None:
        c["block_mask"] = torch.as_tensor(block_mask, dtype=torch.uint8)
    return c


def algorithmic_fwd_flops(B, H, N, d, causal=False, key_len=None, block_mask=None,
                          block=MASK_BLOCK) -> float:
    """Forward FLOPs counted the way the workloads are reported: 4*B*H*N^2*d,
    halved for causal; with key padding or a block mask only the unmasked
    (q, k) pairs count (4*d per pair)."""
    if key_len is None and block_mask is None:
        f = 4.0 * B * H * N * N * d
        return f / 2 if causal else f
    pairs_per_b = []
    for b in range(B):
        kl = N if key_len is None else int(min(max(int(key_len[b]), 0), N))
        if block_mask is None:
            pairs = float(N) * kl if not causal else float(sum(min(i + 1, kl) for i in range(N)))
        else:
            bm = torch.as_tensor(block_mask)
            nb = bm.shape[0]
            pairs = 0.0
            for r in range(nb):
                for c in range(nb):
                    if not bm[r, c]:
                        continue
                    rows = min(block, N - r * block)
                    k0, k1 = c * block, min((c + 1) * block, N, kl)
                    if k1 <= k0:
                        continue
                    if not causal:
                        pairs += rows * (k1 - k0)
                    else:
                        for i in range(r * block, r * block + rows):
                            pairs += max(0, min(k1, i + 1) - k0)
        pairs_per_b.append(pairs)
    return 4.0 * H * d * sum(pairs_per_b)
