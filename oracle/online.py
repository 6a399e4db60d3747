"""The online-softmax identities the pages state, in their notation (fp64, numpy).

Test infrastructure: used only to pin the oracle (and, through it, the
kernels) to the pages' own statement of why tiling is exact.

- ``merge_blocks``: "FlashAttention: Mathematical Foundations, IO-Aware
  Tiling, Online Softmax, and Recomputation Dynamics", section "Incremental
  Online Updates": two blocks of a score row with local statistics
  (m1, l1) and (m2, l2) combine as m_new = max(m1, m2),
  l_new = l1 exp(m1 - m_new) + l2 exp(m2 - m_new), and the normalised block
  outputs combine with weights l1 exp(m1 - m_new) / l_new and
  l2 exp(m2 - m_new) / l_new.  The page writes the second weight as
  exp(-m_new) / l_new applied to sum_j exp(x_j) V_j; that is the same number
  but overflows when evaluated literally, so it is evaluated as
  exp(x_j - m2) relative to the block's own maximum (reading of a
  numerically unsafe form, not a change of value).
- ``online_fold``: "The Attention Matrix You Never Write Down", section "The
  running-statistics trick", steps 1-4: carry (m, l, o) per query; for each
  new block take m' = max(m, local max), multiply l and o by exp(m - m'),
  add the block's exp(x - m') and exp(x - m') V; after the last block divide
  o by l.  The tiling page's update rule ("IO-Aware Tiling Algorithm") prints
  the correction factor with an inverse, diag(exp(m_i - m_i_new))^-1, which
  contradicts the running-statistics page and its own final
  diag(l_i)^-1 normalisation; the fold follows the multiply-by-exp(m - m')
  reading.
"""
from __future__ import annotations

import numpy as np


def block_stats(x, v):
    """Local statistics of one block: m = max x, l = sum exp(x - m), O = softmax(x) v.

    x: [..., n] scores (may hold -inf), v: [n, d].  A block with every score
    -inf has m = -inf, l = 0 and O = 0.
    """
    x = np.asarray(x, np.float64)
    v = np.asarray(v, np.float64)
    m = np.max(x, axis=-1)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    e = np.exp(x - m_safe[..., None])
    e = np.where(np.isneginf(x), 0.0, e)
    l = e.sum(axis=-1)
    with np.errstate(invalid="ignore", divide="ignore"):
        O = np.where(l[..., None] > 0, (e @ v) / np.where(l > 0, l, 1.0)[..., None], 0.0)
    return m, l, O


def merge_blocks(m1, l1, O1, m2, l2, O2):
    """Combine two blocks' (m, l, normalised O) into the statistics of their union."""
    m1, l1, O1 = np.asarray(m1, np.float64), np.asarray(l1, np.float64), np.asarray(O1, np.float64)
    m2, l2, O2 = np.asarray(m2, np.float64), np.asarray(l2, np.float64), np.asarray(O2, np.float64)
    m_new = np.maximum(m1, m2)
    ref = np.where(np.isfinite(m_new), m_new, 0.0)
    w1 = np.where(np.isneginf(m1), 0.0, l1 * np.exp(np.where(np.isneginf(m1), 0.0, m1) - ref))
    w2 = np.where(np.isneginf(m2), 0.0, l2 * np.exp(np.where(np.isneginf(m2), 0.0, m2) - ref))
    l_new = w1 + w2
    safe = np.where(l_new > 0, l_new, 1.0)
    O_new = np.where((l_new > 0)[..., None],
                     (w1 / safe)[..., None] * O1 + (w2 / safe)[..., None] * O2, 0.0)
    return m_new, l_new, O_new


def online_fold(x, v, block):
    """Single sweep over key blocks with running (m, l, o); returns (O, LSE).

    x: [q, n] scores (may hold -inf), v: [n, d], block: keys per step.
    """
    x = np.asarray(x, np.float64)
    v = np.asarray(v, np.float64)
    q, n = x.shape
    d = v.shape[1]
    m = np.full(q, -np.inf)
    l = np.zeros(q)
    o = np.zeros((q, d))
    for s in range(0, n, block):
        xb = x[:, s:s + block]
        vb = v[s:s + block]
        m_new = np.maximum(m, xb.max(axis=1))
        ref = np.where(np.isfinite(m_new), m_new, 0.0)
        corr = np.where(np.isneginf(m), 0.0, np.exp(np.where(np.isneginf(m), 0.0, m) - ref))
        p = np.where(np.isneginf(xb), 0.0, np.exp(xb - ref[:, None]))
        l = l * corr + p.sum(axis=1)
        o = o * corr[:, None] + p @ vb
        m = m_new
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    O = np.where((l > 0)[:, None], o / np.where(l > 0, l, 1.0)[:, None], 0.0)
    return O, lse
