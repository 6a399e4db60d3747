"""Ragged batches (fa_fwd_varlen, fa_bwd_varlen) against the fp64 oracle: packed sequences
of uneven lengths, cached prefixes (Lk > Lq, bottom-right causal), queries
without a visible key (Lk < Lq under the causal mask), empty sequences, bad
offsets, and both ragged workloads at full size on sampled sequences."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import LSE_MAX_ABS, O_MAX_ABS, O_REL_FRO, rel_fro
from synthetic import VARLEN_WORKLOADS, make_varlen_inputs

pytestmark = pytest.mark.gpu


def packed(lens_q, lens_k, H, d, seed):
    g = torch.Generator().manual_seed(seed)
    tq, tk = sum(lens_q), sum(lens_k)
    Q = torch.randn((tq, H, d), generator=g).to(torch.bfloat16)
    K = torch.randn((tk, H, d), generator=g).to(torch.bfloat16)
    V = torch.randn((tk, H, d), generator=g).to(torch.bfloat16)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32)
    return Q, K, V, cu_q, cu_k


def run(Q, K, V, cu_q, cu_k, max_q, causal, scale=None):
    import io_aware_exact_09_gb300 as fa
    O, L = fa.attention_varlen(Q.cuda(), K.cuda(), V.cuda(), cu_q.cuda(), cu_k.cuda(), max_q, scale, causal,
                               check_status=True)
    torch.cuda.synchronize()
    return O.double().cpu().numpy(), L.double().cpu().numpy()


def check(O, L, rO, rL, label):
    fin = np.isfinite(rL)                          # [H, total_q]
    assert np.all(L[~fin] == -np.inf), label
    rows_empty = ~fin.T                            # [total_q, H]
    assert np.all(O[rows_empty] == 0), label
    assert np.all(np.isfinite(O)), label
    assert rel_fro(O, rO) <= O_REL_FRO, (label, rel_fro(O, rO))
    assert np.max(np.abs(O - rO)) <= O_MAX_ABS, label
    if fin.any():
        assert np.max(np.abs(L[fin] - rL[fin])) <= LSE_MAX_ABS, label


CASES = [
    # lens_q, lens_k
    ([1, 127, 128, 129, 300, 0, 5], None),               # prefill: Lk = Lq
    ([64, 200, 1], [1000, 333, 129]),                    # cached prefixes: Lk > Lq
    ([300, 50], [100, 50]),                              # Lk < Lq: early queries see nothing (causal)
    ([513, 1024], [513, 1024]),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_oracle(case, d, causal):
    lq, lk = CASES[case]
    lk = lq if lk is None else lk
    Q, K, V, cu_q, cu_k = packed(lq, lk, 3, d, seed=100 * case + d + causal)
    O, L = run(Q, K, V, cu_q, cu_k, max(lq), causal)
    rO, rL = oracle.attention_varlen(Q.double().numpy(), K.double().numpy(), V.double().numpy(), cu_q.numpy(),
                                     cu_k.numpy(), 1.0 / d ** 0.5, causal=causal)
    check(O, L, rO, rL, (case, d, causal))


def test_varlen_bad_offsets_are_flagged_and_skipped():
    import io_aware_exact_09_gb300 as fa
    Q, K, V, cu_q, cu_k = packed([100, 100], [100, 100], 2, 64, seed=7)
    bad_q = torch.tensor([0, 150, 100], dtype=torch.int32)         # second length negative
    with pytest.raises(fa.FAError) as e:
        run(Q, K, V, bad_q, cu_k, 150, False)
    assert e.value.status == 6
    # a query length beyond the grid max_seqlen_q sizes (whole 128-row
    # tiles) is flagged too
    Q, K, V, cu_q, cu_k = packed([300, 100], [300, 100], 2, 64, seed=8)
    with pytest.raises(fa.FAError) as e:
        run(Q, K, V, cu_q, cu_k, 100, False)
    assert e.value.status == 6


def test_varlen_rejects_bad_arguments():
    import io_aware_exact_09_gb300 as fa
    ws = fa.workspace(fa.fa_fwd_workspace_size(1, 1, 1, 64), "cuda")
    x = torch.zeros((10, 2, 80), dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 10], dtype=torch.int32, device="cuda")
    L = torch.zeros((2, 10), device="cuda")
    assert fa.fa_fwd_varlen(x, x, x, x, L, cu, cu, 1, 2, 10, 10, 10, 80, 0.1, 0, ws, ws.numel()) == 2
    assert fa.fa_fwd_varlen(x, x, x, x, L, None, cu, 1, 2, 10, 10, 10, 64, 0.1, 0, ws, ws.numel()) == 1


@pytest.mark.parametrize("name", sorted(VARLEN_WORKLOADS))
def test_varlen_full_size_sampled(name):
    """Both ragged workloads at full size (the launch bench.py times): the
    shortest and the longest sequence and one more, on two heads each."""
    w = VARLEN_WORKLOADS[name]
    c = make_varlen_inputs(w)
    O, L = run(c["Q"], c["K"], c["V"], c["cu_q"], c["cu_k"], c["max_q"], w.causal)
    cu_q, cu_k = c["cu_q"].numpy(), c["cu_k"].numpy()
    lens = np.diff(cu_q)
    picks = sorted({int(np.argmin(lens)), int(np.argmax(lens)), w.B // 2})
    for b in picks:
        for h in (0, w.H - 1):
            sq = slice(cu_q[b], cu_q[b + 1])
            sk = slice(cu_k[b], cu_k[b + 1])
            f = lambda X, s: X[s, h:h + 1].double().numpy().transpose(1, 0, 2)[None]
            rO, rL = oracle.attention_decode(f(c["Q"], sq), f(c["K"], sk), f(c["V"], sk), w.softmax_scale,
                                             causal=w.causal)
            got = O[sq, h]
            assert rel_fro(got, rO[0, 0]) <= O_REL_FRO, (name, b, h, rel_fro(got, rO[0, 0]))
            assert np.max(np.abs(got - rO[0, 0])) <= O_MAX_ABS, (name, b, h)
            assert np.max(np.abs(L[h, sq] - rL[0, 0])) <= LSE_MAX_ABS, (name, b, h)


# ---------------------------------------------------------------- backward (fa_bwd_varlen)

def run_bwd(Q, K, V, dO, cu_q, cu_k, max_q, max_k, causal, scale=None, prefill_nan=True):
    """Forward then backward of a ragged batch through the C ABI; the gradient
    buffers start as NaN so that an element the kernels never write shows."""
    import io_aware_exact_09_gb300 as fa
    Qd, Kd, Vd, dOd = (x.cuda().contiguous() for x in (Q, K, V, dO))
    cq, ck = cu_q.cuda(), cu_k.cuda()
    O, L = fa.attention_varlen(Qd, Kd, Vd, cq, ck, max_q, scale, causal, check_status=True)
    d = Q.shape[2]
    sc = (1.0 / d ** 0.5) if scale is None else scale
    H, tq, tk = Q.shape[1], Q.shape[0], K.shape[0]
    B = cu_q.numel() - 1
    dQ, dK, dV = (torch.full_like(x, float("nan")) for x in (Qd, Kd, Vd))
    ws = fa.workspace(fa.fa_bwd_varlen_workspace_size(H, tq, d), "cuda")
    st = fa.fa_bwd_varlen(Qd, Kd, Vd, O, L, dOd, dQ, dK, dV, cq, ck, B, H, tq, tk, max_k, d, sc, causal, ws,
                          ws.numel())
    assert st == 0, fa.fa_status_string(st)
    assert fa.fa_get_device_status(ws) == 0
    torch.cuda.synchronize()
    f = lambda t: t.double().cpu().numpy()
    return f(O), f(L), f(dQ), f(dK), f(dV)


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_matches_oracle(case, d, causal):
    from gpu_common import GRAD_REL_FRO
    lq, lk = CASES[case]
    lk = lq if lk is None else lk
    Q, K, V, cu_q, cu_k = packed(lq, lk, 3, d, seed=300 + 100 * case + d + causal)
    dO = torch.randn(Q.shape, generator=torch.Generator().manual_seed(7 + case)).to(torch.bfloat16)
    O, L, dQ, dK, dV = run_bwd(Q, K, V, dO, cu_q, cu_k, max(lq), max(lk), causal)
    f64 = lambda t: t.double().numpy()
    rO, rL, rdQ, rdK, rdV = oracle.attention_varlen_bwd(f64(Q), f64(K), f64(V), f64(dO), cu_q.numpy(), cu_k.numpy(),
                                                        1.0 / d ** 0.5, causal=causal)
    check(O, L, rO, rL, (case, d, causal))
    for got, ref, name in ((dQ, rdQ, "dQ"), (dK, rdK, "dK"), (dV, rdV, "dV")):
        assert np.all(np.isfinite(got)), (case, d, causal, name)
        assert rel_fro(got, ref) <= GRAD_REL_FRO, (case, d, causal, name, rel_fro(got, ref))
    # exact zeros where the definition gives zero: query rows that see no key,
    # keys of sequences without queries
    fin = np.isfinite(rL).T                       # [total_q, H]
    assert np.all(dQ[~fin] == 0), (case, d, causal)
    for b in range(len(lq)):
        if lq[b] == 0:
            assert np.all(dK[cu_k[b]:cu_k[b + 1]] == 0) and np.all(dV[cu_k[b]:cu_k[b + 1]] == 0)


def test_varlen_backward_bad_offsets_are_flagged():
    import io_aware_exact_09_gb300 as fa
    Q, K, V, cu_q, cu_k = packed([100, 100], [100, 100], 2, 64, seed=9)
    g = lambda x: x.cuda().contiguous()
    O, L = fa.attention_varlen(g(Q), g(K), g(V), cu_q.cuda(), cu_k.cuda(), 100, None, False, check_status=True)
    bad_k = torch.tensor([0, 150, 100], dtype=torch.int32, device="cuda")     # second key length negative
    dQ, dK, dV = (torch.empty_like(g(x)) for x in (Q, K, V))
    ws = fa.workspace(fa.fa_bwd_varlen_workspace_size(2, 200, 64), "cuda")
    assert fa.fa_bwd_varlen(g(Q), g(K), g(V), O, L, g(Q), dQ, dK, dV, cu_q.cuda(), bad_k, 2, 2, 200, 200, 150, 64,
                            0.125, 0, ws, ws.numel()) == 0
    assert fa.fa_get_device_status(ws) == 6
    # a key length past the grid's max_seqlen_k (whole 128-row tiles) is flagged too
    ws.zero_()
    Q, K, V, cu_q, cu_k = packed([50, 50], [300, 100], 2, 64, seed=10)
    O, L = fa.attention_varlen(g(Q), g(K), g(V), cu_q.cuda(), cu_k.cuda(), 50, None, False, check_status=True)
    dQ, dK, dV = (torch.empty_like(g(x)) for x in (Q, K, V))
    assert fa.fa_bwd_varlen(g(Q), g(K), g(V), O, L, g(Q), dQ, dK, dV, cu_q.cuda(), cu_k.cuda(), 2, 2, 100, 400, 100,
                            64, 0.125, 0, ws, ws.numel()) == 0
    assert fa.fa_get_device_status(ws) == 6


def test_varlen_backward_rejects_bad_arguments():
    import io_aware_exact_09_gb300 as fa
    ws = fa.workspace(fa.fa_bwd_varlen_workspace_size(2, 10, 64), "cuda")
    x = torch.zeros((10, 2, 64), dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 10], dtype=torch.int32, device="cuda")
    L = torch.zeros((2, 10), device="cuda")
    args = lambda d, scale, cu_q: (x, x, x, x, L, x, x, x, x, cu_q, cu, 1, 2, 10, 10, 10, d, scale, 0, ws, ws.numel())
    assert fa.fa_bwd_varlen(*args(80, 0.1, cu)) == 2
    assert fa.fa_bwd_varlen(*args(64, float("nan"), cu)) == 1
    assert fa.fa_bwd_varlen(*args(64, 0.1, None)) == 1
    assert fa.fa_bwd_varlen(x, x, x, x, L, x, x, x, x, cu, cu, 1, 2, 10, 10, 10, 64, 0.1, 0, ws, 16) == 3


@pytest.mark.parametrize("name", sorted(VARLEN_WORKLOADS))
def test_varlen_backward_full_size_sampled(name):
    """Both ragged workloads at full size, forward and backward in the launch
    configuration bench.py times; the oracle checks the shortest, the longest
    and a middle sequence on the first and last head (each sequence's
    gradients depend on that sequence alone)."""
    from gpu_common import GRAD_REL_FRO
    w = VARLEN_WORKLOADS[name]
    c = make_varlen_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 1)
    dO = torch.randn(c["Q"].shape, generator=g).to(torch.bfloat16)
    cu_q, cu_k = c["cu_q"].numpy(), c["cu_k"].numpy()
    max_k = int(np.max(np.diff(cu_k)))
    O, L, dQ, dK, dV = run_bwd(c["Q"], c["K"], c["V"], dO, c["cu_q"], c["cu_k"], c["max_q"], max_k, w.causal)
    for t in (dQ, dK, dV):
        assert np.all(np.isfinite(t)), name
    lens = np.diff(cu_q)
    picks = sorted({int(np.argmin(lens)), int(np.argmax(lens)), w.B // 2})
    for b in picks:
        sq, sk = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        for h in (0, w.H - 1):
            f = lambda X, s: X[s, h:h + 1].double().numpy().transpose(1, 0, 2)[None]
            rO, rL, rdQ, rdK, rdV = oracle.attention_bwd_rect(f(c["Q"], sq), f(c["K"], sk), f(c["V"], sk), f(dO, sq),
                                                              w.softmax_scale, causal=w.causal)
            assert rel_fro(O[sq, h], rO[0, 0]) <= O_REL_FRO, (name, b, h)
            for got, ref, nm in ((dQ[sq, h], rdQ[0, 0], "dQ"), (dK[sk, h], rdK[0, 0], "dK"), (dV[sk, h], rdV[0, 0], "dV")):
                assert rel_fro(got, ref) <= GRAD_REL_FRO, (name, b, h, nm, rel_fro(got, ref))
