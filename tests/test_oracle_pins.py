"""Pins for the fp64 oracle: each check comes from the pages or from mathematics,
never from the oracle's own formula retyped.  A dropped term, a wrong sign,
a transposed operand or a wrong mask index in the oracle fails at least one
of these.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.online import block_stats, merge_blocks, online_fold


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def element_mask(B, N, causal, key_len, block_mask, mb=128):
    """[B, N, N] bool of visible (query, key) pairs, written from the mask
    readings directly (independent of the oracle's C predicate)."""
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    out = np.ones((B, N, N), bool)
    if causal:
        out &= (j <= i)[None]
    if key_len is not None:
        out &= (j[None] < np.asarray(key_len)[:, None, None])
    if block_mask is not None:
        bm = np.asarray(block_mask).astype(bool)
        out &= bm[i // mb, j // mb][None]
    return out


MASK_KINDS = [
    dict(),
    dict(causal=True),
    dict(key_len=[5, 16]),
    dict(block_mask=np.array([[1, 0], [1, 1]], np.uint8), mask_block=8),
    dict(causal=True, key_len=[9, 13], block_mask=np.array([[1, 0], [1, 1]], np.uint8),
         mask_block=8),
]


# ---------------------------------------------------------------- forward pins

@pytest.mark.parametrize("kw", MASK_KINDS)
def test_rows_of_P_sum_to_one_and_masked_entries_are_zero(kw):
    # step 2 of the attention lab: softmax turns each score row into weights
    # that add up to exactly 1.
    B, H, N, d = 2, 2, 16, 8
    Q, K, V = rnd((B, H, N, d), 1), rnd((B, H, N, d), 2), rnd((B, H, N, d), 3)
    O, LSE, P = oracle.attention_fwd(Q, K, V, 0.3, return_P=True, **kw)
    vis = element_mask(B, N, kw.get("causal", False), kw.get("key_len"), kw.get("block_mask"),
                       kw.get("mask_block", 128))
    for b in range(B):
        has = vis[b].any(axis=1)
        np.testing.assert_allclose(P[b].sum(-1)[:, has], 1.0, rtol=0, atol=1e-12)
        assert np.all(P[b][:, ~vis[b]] == 0.0)
        assert np.all(P[b] >= 0)


@pytest.mark.parametrize("kw", MASK_KINDS)
def test_zero_query_gives_column_mean_of_visible_V(kw):
    B, H, N, d = 2, 3, 16, 8
    Q = np.zeros((B, H, N, d))
    K, V = rnd((B, H, N, d), 4), rnd((B, H, N, d), 5)
    O, LSE = oracle.attention_fwd(Q, K, V, 0.7, **kw)
    vis = element_mask(B, N, kw.get("causal", False), kw.get("key_len"), kw.get("block_mask"),
                       kw.get("mask_block", 128))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                keys = np.nonzero(vis[b, i])[0]
                if keys.size == 0:
                    assert np.all(O[b, h, i] == 0) and LSE[b, h, i] == -np.inf
                    continue
                np.testing.assert_allclose(O[b, h, i], V[b, h, keys].mean(0), atol=1e-12, rtol=0)
                # all scores 0 -> LSE = ln(#visible keys)
                assert abs(LSE[b, h, i] - math.log(keys.size)) < 1e-12


def test_one_hot_dominant_score_selects_value_row():
    # orthonormal keys; query i points along key pi(i) with length 50, so
    # its score there is 50 and 0 elsewhere: softmax is one-hot to 1e-21.
    B, H, N, d = 1, 2, 16, 16
    K = np.zeros((B, H, N, d))
    basis = np.linalg.qr(rnd((d, d), 6))[0]
    K[0, :] = basis[:N]
    V = rnd((B, H, N, d), 7)
    perm = np.random.default_rng(8).permutation(N)
    Q = np.zeros((B, H, N, d))
    for i in range(N):
        Q[0, :, i] = 50.0 * K[0, :, perm[i]]
    O, LSE = oracle.attention_fwd(Q, K, V, 1.0)
    np.testing.assert_allclose(O[0], V[0][:, perm], atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, 50.0, atol=1e-12)


def test_lse_equals_log_of_plain_exp_sum():
    # small scores: LSE_i = ln sum_j exp(s_ij) with no max shift, summed with fsum
    B, H, N, d = 1, 2, 12, 4
    Q, K, V = rnd((B, H, N, d), 9, 0.3), rnd((B, H, N, d), 10, 0.3), rnd((B, H, N, d), 11)
    scale = 0.5
    O, LSE = oracle.attention_fwd(Q, K, V, scale)
    for h in range(H):
        for i in range(N):
            s = [scale * sum(Q[0, h, i, t] * K[0, h, j, t] for t in range(d)) for j in range(N)]
            ref = math.log(math.fsum(math.exp(x) for x in s))
            assert abs(LSE[0, h, i] - ref) < 1e-12
            w = [math.exp(x - ref) for x in s]
            o = [math.fsum(w[j] * V[0, h, j, t] for j in range(N)) for t in range(d)]
            np.testing.assert_allclose(O[0, h, i], o, atol=1e-12, rtol=0)


@pytest.mark.parametrize("kw", MASK_KINDS)
def test_forward_matches_torch_library_sdpa(kw):
    # an independent library routine: torch's scaled_dot_product_attention in
    # fp64 with an explicit boolean mask (rows that keep at least one key).
    B, H, N, d = 2, 2, 16, 8
    Q, K, V = rnd((B, H, N, d), 12), rnd((B, H, N, d), 13), rnd((B, H, N, d), 14)
    scale = 0.37
    O, LSE = oracle.attention_fwd(Q, K, V, scale, **kw)
    vis = element_mask(B, N, kw.get("causal", False), kw.get("key_len"), kw.get("block_mask"),
                       kw.get("mask_block", 128))
    m = torch.from_numpy(vis)[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q), torch.from_numpy(K), torch.from_numpy(V), attn_mask=m, scale=scale)
    s = scale * torch.from_numpy(Q) @ torch.from_numpy(K).transpose(-1, -2)
    s = s.masked_fill(~m, -math.inf)
    lse_ref = torch.logsumexp(s, dim=-1)
    rows = vis.any(-1)  # [B, N]
    for b in range(B):
        np.testing.assert_allclose(O[b][:, rows[b]], ref[b][:, rows[b]].numpy(), atol=1e-12, rtol=0)
        np.testing.assert_allclose(LSE[b][:, rows[b]], lse_ref[b][:, rows[b]].numpy(), atol=1e-12,
                                   rtol=0)


def torch_attn(Q, K, V, scale):
    """A library routine on an explicitly given key set (fp64): O and LSE."""
    q, k, v = (torch.from_numpy(np.ascontiguousarray(x)) for x in (Q, K, V))
    O = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)
    L = torch.logsumexp(scale * q @ k.transpose(-1, -2), dim=-1)
    return O.numpy(), L.numpy()


def test_two_block_merge_equals_full_softmax():
    # "Incremental Online Updates": splitting the keys in two, computing each
    # half alone and merging with the page's rule gives the full result.
    B, H, N, d = 1, 3, 40, 8
    Q, K, V = rnd((B, H, N, d), 15), rnd((B, H, N, d), 16, 2.0), rnd((B, H, N, d), 17)
    scale = 0.9
    O, LSE = oracle.attention_fwd(Q, K, V, scale)
    for n1 in (1, 13, 20, 39):
        # each half through the oracle: the first n1 keys via key_len = n1, the
        # rest by rotating them to the front and key_len = N - n1
        O1, L1 = oracle.attention_fwd(Q, K, V, scale, key_len=[n1])
        Kr, Vr = np.roll(K, -n1, axis=2), np.roll(V, -n1, axis=2)
        O2, L2 = oracle.attention_fwd(Q, Kr, Vr, scale, key_len=[N - n1])
        # the same halves from a library routine on the explicit key subsets
        T1 = torch_attn(Q, K[:, :, :n1], V[:, :, :n1], scale)
        T2 = torch_attn(Q, K[:, :, n1:], V[:, :, n1:], scale)
        np.testing.assert_allclose(O1, T1[0], atol=1e-12, rtol=0)
        np.testing.assert_allclose(O2, T2[0], atol=1e-12, rtol=0)
        np.testing.assert_allclose(L2, T2[1], atol=1e-12, rtol=0)
        # (m, l) = (LSE, 1) is an exact representation of a block's statistics
        m, l, Om = merge_blocks(L1, np.ones_like(L1), O1, L2, np.ones_like(L2), O2)
        np.testing.assert_allclose(Om, O, atol=1e-12, rtol=0)
        np.testing.assert_allclose(m + np.log(l), LSE, atol=1e-12, rtol=0)


def test_k_way_merge_in_random_order_and_online_fold():
    rng = np.random.default_rng(18)
    q, n, d = 7, 64, 5
    x = rng.standard_normal((q, n)) * 3
    x[2, :] = -np.inf            # a row with nothing visible
    x[3, 10:] = -np.inf          # a row visible only in the first block
    v = rng.standard_normal((n, d))
    # reference: the oracle's three-pass softmax on the same scores.  Build
    # Q, K so that scale * Q K^T = x exactly: K = identity rows, Q = x.
    Qx = np.zeros((1, 1, n, n)); Qx[0, 0, :q] = np.where(np.isfinite(x), x, 0.0)
    Kx = np.zeros((1, 1, n, n)); Kx[0, 0] = np.eye(n)
    Vx = np.zeros((1, 1, n, n)); Vx[0, 0, :, :d] = v     # zero-padded to the same d
    O_ref, L_ref = oracle.attention_fwd(Qx, Kx, Vx, 1.0)
    O_ref = O_ref[..., :d]
    finite_rows = [r for r in range(q) if np.isfinite(x[r]).all()]
    # k-way merge of 8 blocks in random order
    order = rng.permutation(8)
    acc = None
    for blk in order:
        sl = slice(8 * blk, 8 * blk + 8)
        st = block_stats(x[:, sl], v[sl])
        acc = st if acc is None else merge_blocks(*acc, *st)
    m, l, Om = acc
    for r in finite_rows:
        np.testing.assert_allclose(Om[r], O_ref[0, 0, r], atol=1e-12, rtol=0)
        assert abs(m[r] + math.log(l[r]) - L_ref[0, 0, r]) < 1e-12
    assert np.all(Om[2] == 0) and l[2] == 0
    # row 3 against a direct softmax over its first 10 scores
    w = np.exp(x[3, :10] - x[3, :10].max()); w /= w.sum()
    np.testing.assert_allclose(Om[3], w @ v[:10], atol=1e-12, rtol=0)
    # the single-sweep running-statistics fold, several block sizes
    for blk in (1, 5, 16, 64):
        Of, Lf = online_fold(x, v, blk)
        for r in finite_rows:
            np.testing.assert_allclose(Of[r], O_ref[0, 0, r], atol=1e-12, rtol=0)
            assert abs(Lf[r] - L_ref[0, 0, r]) < 1e-12
        assert np.all(Of[2] == 0) and Lf[2] == -np.inf


# ---------------------------------------------------------------- mask pins

def test_key_padding_equals_truncated_key_set():
    B, H, N, d = 3, 2, 20, 8
    Q, K, V = rnd((B, H, N, d), 19), rnd((B, H, N, d), 20), rnd((B, H, N, d), 21)
    kl = [7, 20, 1]
    O, LSE = oracle.attention_fwd(Q, K, V, 0.4, key_len=kl)
    for b in range(B):
        Ot, Lt = torch_attn(Q[b:b + 1], K[b:b + 1, :, :kl[b]], V[b:b + 1, :, :kl[b]], 0.4)
        np.testing.assert_allclose(O[b:b + 1], Ot, atol=1e-12, rtol=0)
        np.testing.assert_allclose(LSE[b:b + 1], Lt, atol=1e-12, rtol=0)


def test_causal_equals_prefix_key_set():
    B, H, N, d = 1, 2, 17, 8
    Q, K, V = rnd((B, H, N, d), 22), rnd((B, H, N, d), 23), rnd((B, H, N, d), 24)
    O, LSE = oracle.attention_fwd(Q, K, V, 0.4, causal=True)
    for i in range(N):
        Ot, Lt = torch_attn(Q[:, :, i:i + 1], K[:, :, :i + 1], V[:, :, :i + 1], 0.4)
        np.testing.assert_allclose(O[:, :, i:i + 1], Ot, atol=1e-12, rtol=0)
        np.testing.assert_allclose(LSE[:, :, i:i + 1], Lt, atol=1e-12, rtol=0)
        # and the oracle itself with key_len = i + 1 instead of the causal flag
        Ok, Lk = oracle.attention_fwd(Q, K, V, 0.4, key_len=[i + 1])
        np.testing.assert_allclose(O[:, :, i], Ok[:, :, i], atol=1e-12, rtol=0)


def test_block_mask_equals_gathered_key_blocks():
    B, H, N, d, mb = 1, 2, 30, 8, 8            # 4 blocks, last one ragged (6 keys)
    Q, K, V = rnd((B, H, N, d), 25), rnd((B, H, N, d), 26), rnd((B, H, N, d), 27)
    bm = np.array([[1, 0, 0, 1], [0, 1, 1, 0], [1, 1, 1, 1], [0, 0, 0, 1]], np.uint8)
    O, LSE = oracle.attention_fwd(Q, K, V, 0.4, block_mask=bm, mask_block=mb)
    for r in range(4):
        keys = np.concatenate([np.arange(c * mb, min((c + 1) * mb, N)) for c in range(4) if bm[r, c]])
        rows = slice(r * mb, min((r + 1) * mb, N))
        Ot, Lt = torch_attn(Q[:, :, rows], K[:, :, keys], V[:, :, keys], 0.4)
        np.testing.assert_allclose(O[:, :, rows], Ot, atol=1e-12, rtol=0)
        np.testing.assert_allclose(LSE[:, :, rows], Lt, atol=1e-12, rtol=0)


def test_oracle_rejects_mismatched_shapes():
    Q = rnd((1, 1, 8, 4), 1)
    with pytest.raises(ValueError):
        oracle.attention_fwd(Q, Q[:, :, :4], Q, 1.0)
    with pytest.raises(ValueError):
        oracle.attention_fwd(Q, Q, Q, 1.0, key_len=[1, 2])


def test_fully_masked_rows_convention():
    B, H, N, d = 2, 1, 8, 4
    Q, K, V, dO = (rnd((B, H, N, d), s) for s in (28, 29, 30, 31))
    O, LSE, dQ, dK, dV = oracle.attention_bwd(Q, K, V, dO, 0.5, key_len=[0, 3])
    assert np.all(O[0] == 0) and np.all(LSE[0] == -np.inf)
    assert np.all(dQ[0] == 0) and np.all(dK[0] == 0) and np.all(dV[0] == 0)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(dQ))
    assert np.all(dK[1, :, 3:] == 0) and np.all(dV[1, :, 3:] == 0)


# ---------------------------------------------------------------- backward pins

def loss(Q, K, V, dO, scale, kw):
    O, _ = oracle.attention_fwd(Q, K, V, scale, **kw)
    return float(np.sum(O * dO))


@pytest.mark.parametrize("kw", MASK_KINDS)
def test_gradients_match_central_finite_differences(kw):
    B, H, N, d = 2, 1, 16, 8
    Q, K, V, dO = (rnd((B, H, N, d), s) for s in (32, 33, 34, 35))
    scale = 0.45
    _, _, dQ, dK, dV = oracle.attention_bwd(Q, K, V, dO, scale, **kw)
    h = 1e-5
    for name, X, G in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        fd = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = X[idx]
            X[idx] = old + h
            lp = loss(Q, K, V, dO, scale, kw)
            X[idx] = old - h
            lm = loss(Q, K, V, dO, scale, kw)
            X[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(fd - G) / max(np.linalg.norm(G), 1e-30)
        assert err <= 1e-6, (name, err)


@pytest.mark.parametrize("kw", MASK_KINDS)
def test_gradients_match_torch_autograd(kw):
    B, H, N, d = 2, 2, 16, 8
    Q, K, V, dO = (rnd((B, H, N, d), s) for s in (36, 37, 38, 39))
    scale = 0.6
    O, LSE, dQ, dK, dV = oracle.attention_bwd(Q, K, V, dO, scale, **kw)
    vis = element_mask(B, N, kw.get("causal", False), kw.get("key_len"), kw.get("block_mask"),
                       kw.get("mask_block", 128))
    tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (Q, K, V))
    s = scale * tq @ tk.transpose(-1, -2)
    m = torch.from_numpy(vis)[:, None]
    s = s.masked_fill(~m, -math.inf)
    p = torch.softmax(s, dim=-1)
    p = torch.nan_to_num(p, nan=0.0)     # rows with no visible key -> zero weights
    o = p @ tv
    (o * torch.from_numpy(dO)).sum().backward()
    np.testing.assert_allclose(O, o.detach().numpy(), atol=1e-10, rtol=0)
    np.testing.assert_allclose(dQ, tq.grad.numpy(), atol=1e-10, rtol=0)
    np.testing.assert_allclose(dK, tk.grad.numpy(), atol=1e-10, rtol=0)
    np.testing.assert_allclose(dV, tv.grad.numpy(), atol=1e-10, rtol=0)


@pytest.mark.parametrize("kw", MASK_KINDS)
def test_row_sampled_functions_match_full_materialisation(kw):
    B, H, N, d = 2, 2, 16, 8
    Q, K, V, dO = (rnd((B, H, N, d), s) for s in (40, 41, 42, 43))
    scale = 0.3
    O, LSE, dQ, dK, dV = oracle.attention_bwd(Q, K, V, dO, scale, **kw)
    rows = np.array([0, 5, 15, 16, 31, 40, 63])
    Or, Lr, dQr = oracle.query_rows(Q, K, V, dO, scale, rows, **kw)
    flat = lambda X: X.reshape(B * H * N, -1)
    np.testing.assert_allclose(Or, flat(O)[rows], atol=1e-12, rtol=0)
    np.testing.assert_allclose(Lr, LSE.reshape(-1)[rows], atol=1e-12, rtol=0)
    np.testing.assert_allclose(dQr, flat(dQ)[rows], atol=1e-12, rtol=0)
    dKr, dVr = oracle.key_rows(Q, K, V, dO, scale, rows, **kw)
    np.testing.assert_allclose(dKr, flat(dK)[rows], atol=1e-12, rtol=0)
    np.testing.assert_allclose(dVr, flat(dV)[rows], atol=1e-12, rtol=0)


def test_dV_is_column_sum_of_dO_when_Q_is_zero_and_single_key_gets_all_weight():
    # Q = 0: every P row is uniform, 1/N, so dV_j = sum_i dO_i / N; dK is a
    # sum of multiples of the (zero) query rows; dQ_i = (1/N) sum_j
    # (dO_i.V_j - dO_i.Vbar) K_j since D_i = dO_i.O_i = dO_i.Vbar.
    B, H, N, d = 1, 1, 10, 4
    Q = np.zeros((B, H, N, d))
    K, V, dO = rnd((B, H, N, d), 44), rnd((B, H, N, d), 45), rnd((B, H, N, d), 46)
    _, _, dQ, dK, dV = oracle.attention_bwd(Q, K, V, dO, 1.0)
    np.testing.assert_allclose(dV[0, 0], np.tile(dO[0, 0].sum(0) / N, (N, 1)), atol=1e-12)
    np.testing.assert_allclose(dK, 0.0, atol=1e-12)
    # dQ_i = sum_j (1/N)(dO_i.V_j - dO_i.Vbar) K_j
    Vbar = V[0, 0].mean(0)
    ref = np.stack([sum((dO[0, 0, i] @ (V[0, 0, j] - Vbar)) * K[0, 0, j] for j in range(N)) / N
                    for i in range(N)])
    np.testing.assert_allclose(dQ[0, 0], ref, atol=1e-12)


# ---------------------------------------------------------------- tile plan pins

def test_tile_plan_causal_closed_form():
    for N in (512, 300, 128, 1):
        plan = oracle.tile_plan(2, N, causal=True)
        T = (N + 127) // 128
        for i in range(T):
            for j in range(T):
                # below the diagonal: full; on it: partial (keys above the
                # diagonal, and keys >= N in a ragged last tile, are masked)
                want = 0 if j > i else (1 if j < i else 2)
                assert plan[0, i, j] == want and plan[1, i, j] == want


def test_tile_plan_key_padding_and_tail_closed_form():
    N = 300                                          # tiles 0..2, last one 44 keys wide
    plan = oracle.tile_plan(4, N, key_len=[300, 128, 129, 0])
    assert plan.shape == (4, 3, 3)
    assert (plan[0, :, 0] == 1).all() and (plan[0, :, 1] == 1).all() and (plan[0, :, 2] == 2).all()
    assert (plan[1, :, 0] == 1).all() and (plan[1, :, 1:] == 0).all()
    assert (plan[2, :, 0] == 1).all() and (plan[2, :, 1] == 2).all() and (plan[2, :, 2] == 0).all()
    assert (plan[3] == 0).all()


def test_tile_plan_block_mask_counts():
    from synthetic import draw_block_mask
    bm = draw_block_mask(8192, 0.15, torch.Generator().manual_seed(1004)).numpy()
    plan = oracle.tile_plan(1, 8192, block_mask=bm)
    assert int((plan[0] != 0).sum()) == 614
    assert int((plan[0] == 2).sum()) == 0               # N divisible by 128: no partial tiles
    assert np.array_equal(plan[0] != 0, bm.astype(bool))


# ---------------------------------------------------------------- decode shapes

def test_decode_equals_square_oracle_when_shapes_agree():
    # Nq = Nk: key padding by kv_len is the square key_len mask, and the
    # bottom-right causal alignment coincides with the top-left one
    B, H, N, d = 2, 2, 24, 8
    Q, K, V = rnd((B, H, N, d), 50), rnd((B, H, N, d), 51), rnd((B, H, N, d), 52)
    O, L = oracle.attention_fwd(Q, K, V, 0.3, key_len=[24, 10])
    Od, Ld = oracle.attention_decode(Q, K, V, 0.3, kv_len=[24, 10])
    np.testing.assert_allclose(Od, O, atol=1e-12, rtol=0)
    np.testing.assert_allclose(Ld, L, atol=1e-12, rtol=0)
    O, L = oracle.attention_fwd(Q, K, V, 0.3, causal=True)
    Od, Ld = oracle.attention_decode(Q, K, V, 0.3, causal=True)
    np.testing.assert_allclose(Od, O, atol=1e-12, rtol=0)
    np.testing.assert_allclose(Ld, L, atol=1e-12, rtol=0)


def test_decode_matches_library_sdpa_with_explicit_mask():
    B, H, Nq, Nk, d = 2, 3, 5, 37, 8
    Q, K, V = rnd((B, H, Nq, d), 53), rnd((B, H, Nk, d), 54), rnd((B, H, Nk, d), 55)
    kl = [37, 20]
    for causal in (False, True):
        O, L = oracle.attention_decode(Q, K, V, 0.4, causal=causal, kv_len=kl)
        for b in range(B):
            i = np.arange(Nq)[:, None]
            j = np.arange(Nk)[None, :]
            vis = j < kl[b]
            if causal:
                vis = vis & (j <= kl[b] - Nq + i)
            m = torch.from_numpy(vis)
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(Q[b]), torch.from_numpy(K[b]), torch.from_numpy(V[b]), attn_mask=m, scale=0.4)
            s = 0.4 * torch.from_numpy(Q[b]) @ torch.from_numpy(K[b]).transpose(-1, -2)
            lref = torch.logsumexp(s.masked_fill(~m, -math.inf), dim=-1)
            np.testing.assert_allclose(O[b], ref.numpy(), atol=1e-12, rtol=0)
            np.testing.assert_allclose(L[b], lref.numpy(), atol=1e-12, rtol=0)


def test_decode_split_keys_merge_to_the_whole():
    # the split-KV decode reading: partial (O, LSE) over key ranges merge by
    # the "Incremental Online Updates" rule into the full result
    B, H, Nq, Nk, d = 1, 2, 3, 50, 8
    Q, K, V = rnd((B, H, Nq, d), 56), rnd((B, H, Nk, d), 57, 2.0), rnd((B, H, Nk, d), 58)
    O, L = oracle.attention_decode(Q, K, V, 0.5)
    acc = None
    for a, b in ((0, 7), (7, 30), (30, 50)):
        Op, Lp = oracle.attention_decode(Q, K[:, :, a:b], V[:, :, a:b], 0.5)
        st = (Lp, np.ones_like(Lp), Op)
        acc = st if acc is None else merge_blocks(*acc, *st)
    np.testing.assert_allclose(acc[2], O, atol=1e-12, rtol=0)
    np.testing.assert_allclose(acc[0] + np.log(acc[1]), L, atol=1e-12, rtol=0)


def _packed(lens_q, lens_k, H, d, seed):
    g = torch.Generator().manual_seed(seed)
    tq, tk = sum(lens_q), sum(lens_k)
    Q = torch.randn((tq, H, d), generator=g, dtype=torch.float64).numpy()
    K = torch.randn((tk, H, d), generator=g, dtype=torch.float64).numpy()
    V = torch.randn((tk, H, d), generator=g, dtype=torch.float64).numpy()
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    return Q, K, V, cu_q, cu_k


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_square_oracle_per_sequence(causal):
    """Lq = Lk: each packed sequence equals the square oracle on that sequence alone."""
    lens = [5, 1, 17, 0, 9]
    H, d = 2, 8
    Q, K, V, cu_q, cu_k = _packed(lens, lens, H, d, seed=31)
    O, L = oracle.attention_varlen(Q, K, V, cu_q, cu_k, 0.3, causal=causal)
    for b, n in enumerate(lens):
        if n == 0:
            continue
        sl = slice(cu_q[b], cu_q[b + 1])
        tr = lambda X: X[sl].transpose(1, 0, 2)[None]
        rO, rL = oracle.attention_fwd(tr(Q), tr(K), tr(V), 0.3, causal=causal)
        assert np.max(np.abs(O[sl].transpose(1, 0, 2) - rO[0])) < 1e-12
        assert np.max(np.abs(L[:, sl] - rL[0])) < 1e-12


def test_varlen_matches_library_sdpa_with_bottom_right_mask():
    """Lq < Lk (queries are the last positions): torch fp64 SDPA with the
    bottom-right causal mask written out, sequence by sequence."""
    lens_q, lens_k = [3, 7, 1], [10, 7, 4]
    H, d = 3, 16
    Q, K, V, cu_q, cu_k = _packed(lens_q, lens_k, H, d, seed=32)
    O, L = oracle.attention_varlen(Q, K, V, cu_q, cu_k, 0.25, causal=True)
    for b, (lq, lk) in enumerate(zip(lens_q, lens_k)):
        q = torch.from_numpy(Q[cu_q[b]:cu_q[b + 1]].transpose(1, 0, 2).copy())
        k = torch.from_numpy(K[cu_k[b]:cu_k[b + 1]].transpose(1, 0, 2).copy())
        v = torch.from_numpy(V[cu_k[b]:cu_k[b + 1]].transpose(1, 0, 2).copy())
        i = torch.arange(lq)[:, None]
        j = torch.arange(lk)[None, :]
        mask = j <= i + (lk - lq)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=0.25)
        got = O[cu_q[b]:cu_q[b + 1]].transpose(1, 0, 2)
        assert np.max(np.abs(got - ref.numpy())) < 1e-12


def test_varlen_rejects_bad_offsets():
    Q, K, V, cu_q, cu_k = _packed([2, 3], [2, 3], 1, 4, seed=33)
    with pytest.raises(ValueError):
        oracle.attention_varlen(Q, K, V, cu_q[::-1], cu_k, 0.5)
    with pytest.raises(ValueError):
        oracle.attention_varlen(Q, K, V, cu_q, cu_k[:-1], 0.5)


# ---------------------------------------------------------------- ragged-batch backward

@pytest.mark.parametrize("causal", [False, True])
def test_varlen_bwd_equals_square_oracle_per_sequence(causal):
    """Lq = Lk: each packed sequence's O, LSE, dQ, dK, dV equal the square
    oracle (pinned by finite differences and autograd) on that sequence alone."""
    lens = [5, 1, 17, 0, 9]
    H, d = 2, 8
    Q, K, V, cu_q, cu_k = _packed(lens, lens, H, d, seed=41)
    dO = np.random.default_rng(42).standard_normal(Q.shape)
    O, L, dQ, dK, dV = oracle.attention_varlen_bwd(Q, K, V, dO, cu_q, cu_k, 0.35, causal=causal)
    for b, n in enumerate(lens):
        if n == 0:
            continue
        sl = slice(cu_q[b], cu_q[b + 1])
        tr = lambda X: X[sl].transpose(1, 0, 2)[None]
        rO, rL, rdQ, rdK, rdV = oracle.attention_bwd(tr(Q), tr(K), tr(V), tr(dO), 0.35, causal=causal)
        back = lambda X: X[0].transpose(1, 0, 2)
        for got, ref in ((O[sl], back(rO)), (dQ[sl], back(rdQ)), (dK[sl], back(rdK)), (dV[sl], back(rdV))):
            assert np.max(np.abs(got - ref)) < 1e-12
        assert np.max(np.abs(L[:, sl] - rL[0])) < 1e-12


def test_varlen_bwd_matches_torch_autograd_bottom_right():
    """Lq != Lk, causal, bottom-right (queries are the last positions): torch
    fp64 autograd of softmax with the mask written out, sequence by sequence.
    Includes a sequence with no queries, one with no keys, and one with
    Lk < Lq whose first queries see no key (zero output, zero gradient)."""
    lens_q, lens_k = [3, 7, 1, 0, 4, 5], [10, 7, 4, 3, 0, 2]
    H, d, scale = 3, 16, 0.3
    Q, K, V, cu_q, cu_k = _packed(lens_q, lens_k, H, d, seed=43)
    dO = np.random.default_rng(44).standard_normal(Q.shape)
    O, L, dQ, dK, dV = oracle.attention_varlen_bwd(Q, K, V, dO, cu_q, cu_k, scale, causal=True)
    for b, (lq, lk) in enumerate(zip(lens_q, lens_k)):
        sq, sk = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        t = lambda X, s: torch.from_numpy(X[s].transpose(1, 0, 2).copy()).requires_grad_(True)
        q, k, v = t(Q, sq), t(K, sk), t(V, sk)
        g = torch.from_numpy(dO[sq].transpose(1, 0, 2).copy())
        i = torch.arange(lq)[:, None]
        j = torch.arange(lk)[None, :]
        s = (scale * q @ k.transpose(-1, -2)).masked_fill(~(j <= i + (lk - lq)), -math.inf)
        p = torch.nan_to_num(torch.softmax(s, dim=-1), nan=0.0)
        o = p @ v
        if lq and lk:
            (o * g).sum().backward()
        grads = [x.grad if x.grad is not None else torch.zeros_like(x) for x in (q, k, v)]
        back = lambda X: X.detach().numpy().transpose(1, 0, 2)
        np.testing.assert_allclose(O[sq], back(o), atol=1e-10, rtol=0)
        np.testing.assert_allclose(dQ[sq], back(grads[0]), atol=1e-10, rtol=0)
        np.testing.assert_allclose(dK[sk], back(grads[1]), atol=1e-10, rtol=0)
        np.testing.assert_allclose(dV[sk], back(grads[2]), atol=1e-10, rtol=0)
        if lq > lk:
            assert np.all(dQ[sq][: lq - lk] == 0) and np.all(np.isneginf(L[:, sq][:, : lq - lk]))


def test_varlen_bwd_matches_central_finite_differences():
    """Gradients of sum(O * dO) by central differences of the ragged forward
    (itself pinned against torch's SDPA with the bottom-right mask)."""
    lens_q, lens_k = [3, 2, 4], [5, 2, 3]
    H, d, scale = 1, 4, 0.55
    Q, K, V, cu_q, cu_k = _packed(lens_q, lens_k, H, d, seed=45)
    dO = np.random.default_rng(46).standard_normal(Q.shape)
    _, _, dQ, dK, dV = oracle.attention_varlen_bwd(Q, K, V, dO, cu_q, cu_k, scale, causal=True)

    def loss():
        O, _ = oracle.attention_varlen(Q, K, V, cu_q, cu_k, scale, causal=True)
        return float(np.sum(O * dO))

    h = 1e-5
    for name, X, G in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        fd = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = X[idx]
            X[idx] = old + h
            lp = loss()
            X[idx] = old - h
            lm = loss()
            X[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(fd - G) / max(np.linalg.norm(G), 1e-30)
        assert err <= 1e-6, (name, err)
