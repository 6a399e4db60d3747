"""Ragged batches (fa_fwd_varlen) against the fp64 oracle: packed sequences
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
