"""Split-KV decode (fa_decode) vs the fp64 decode oracle: a few query rows
against a long key/value cache, every split count, causal (bottom-right) and
per-batch cache lengths, ragged tails, empty caches."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import LSE_MAX_ABS, O_MAX_ABS, O_REL_FRO, rel_fro

pytestmark = pytest.mark.gpu


def draw(B, H, Nq, Nk, d, seed):
    g = torch.Generator().manual_seed(seed)
    Q = torch.randn((B, H, Nq, d), generator=g).to(torch.bfloat16)
    K = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16)
    V = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16)
    return Q, K, V


def run(Q, K, V, causal, kv_len, splits):
    import io_aware_exact_09_gb300 as fa
    kl = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32).cuda()
    O, L = fa.attention_decode(Q.cuda(), K.cuda(), V.cuda(), None, causal, kl, splits, check_status=True)
    torch.cuda.synchronize()
    return O.double().cpu().numpy(), L.double().cpu().numpy()


def check(O, L, rO, rL, label):
    fin = np.isfinite(rL)
    assert np.all(L[~fin] == -np.inf) and np.all(O[~fin] == 0), label
    if fin.any():
        assert rel_fro(O[fin], rO[fin]) <= O_REL_FRO, (label, rel_fro(O[fin], rO[fin]))
        assert np.max(np.abs(O - rO)) <= O_MAX_ABS, label
        assert np.max(np.abs(L[fin] - rL[fin])) <= LSE_MAX_ABS, label


CASES = [
    # B, H, Nq, Nk, d
    (2, 3, 1, 1000, 128),
    (1, 2, 4, 4133, 64),
    (2, 2, 16, 300, 128),
    (1, 2, 130, 777, 64),
    (1, 1, 1, 1, 128),
    (2, 4, 8, 2048, 128),
    (1, 2, 32, 1500, 64),       # the most query rows of the quartered softmax
    (1, 1, 33, 600, 128),       # one past it: whole-row softmax, two warps with rows
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_decode_matches_oracle(case, splits):
    B, H, Nq, Nk, d = case
    Q, K, V = draw(B, H, Nq, Nk, d, seed=sum(case) + splits)
    f = lambda t: t.double().numpy()
    for causal in (False, True):
        kv = [Nk] if B == 1 else [Nk, max(1, Nk // 3)]
        O, L = run(Q, K, V, causal, kv, splits)
        rO, rL = oracle.attention_decode(f(Q), f(K), f(V), 1.0 / d ** 0.5, causal=causal, kv_len=kv)
        check(O, L, rO, rL, (case, splits, causal))


def test_decode_splits_agree_and_edge_lengths():
    B, H, Nq, Nk, d = 3, 2, 4, 1500, 128
    Q, K, V = draw(B, H, Nq, Nk, d, seed=5)
    f = lambda t: t.double().numpy()
    # kv_len 0 (nothing visible), 2 < Nq with causal (the first queries see
    # nothing), and the full cache
    kv = [0, 2, Nk]
    for causal in (False, True):
        rO, rL = oracle.attention_decode(f(Q), f(K), f(V), 1.0 / d ** 0.5, causal=causal, kv_len=kv)
        outs = [run(Q, K, V, causal, kv, sp) for sp in (1, 2, 7, 64)]
        for O, L in outs:
            check(O, L, rO, rL, ("edge", causal))
        for O, L in outs[1:]:
            assert np.max(np.abs(O - outs[0][0])) <= 2e-2


def test_decode_empty_cache():
    Q, K, V = draw(2, 2, 3, 0, 64, seed=9)
    O, L = run(Q, K.reshape(2, 2, 0, 64), V.reshape(2, 2, 0, 64), False, None, 0)
    assert np.all(O == 0) and np.all(L == -np.inf)
