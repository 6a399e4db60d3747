"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (a plug-in handed only its input and output buffers, code that must
not call cudaMalloc where it runs).  It takes no workspace and uses the
library's built-in scratch array instead.  It must give the same gradients
as fa_bwd with a workspace, and agree with the fp64 oracle, on two calls in a row (the second call finds the
first call's scratch contents and must clear what has to start at zero), and
reject problems larger than the scratch before launching anything.

Kept in a file of its own that pytest collects last, so that a run that
stops at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import io_aware_exact_09_gb300 as fa
import oracle
from synthetic import make_case

GRAD_REL_FRO = 1e-2   # the gradient bound the other parity tests use


def rel_fro(a, b):
    a = a.double().cpu()
    b = b.double().cpu()
    return float(torch.linalg.norm(a - b) / torch.linalg.norm(b))


def test_noalloc_rejects_oversize_before_any_gpu_work():
    fa.build()
    L = fa.lib()
    # 16 heads x 16384 rows at d = 128 need ~135 MB of scratch: more than the built-in 64 MiB
    assert L.fa_bwd_noalloc(256, 256, 256, 256, 256, 256, 256, 256, 256, 1, 16, 16384, 128, 0.1, 0,
                            None, None, None) == 3
    assert L.fa_bwd_noalloc(256, 256, 256, 256, 256, 256, 256, 256, 256, 1, 1, 128, 96, 0.1, 0,
                            None, None, None) == 2
    assert L.fa_bwd_noalloc(None, None, None, None, None, None, None, None, None, 0, 1, 128, 64, 0.1, 0,
                            None, None, None) == 0


def test_noalloc_rejects_bad_arguments_before_touching_the_gpu():
    """A NaN or non-positive scale, a null or misaligned pointer: FA_ERR_INVALID_ARGUMENT
    (1), returned before any CUDA call (here, on a machine without a GPU, a call
    that reached the CUDA runtime would fail with FA_ERR_CUDA instead), so a
    rejected call cannot clear the status word of a call still running."""
    fa.build()
    L = fa.lib()
    ok = [256] * 9
    for scale in (float("nan"), 0.0, -1.0, float("inf")):
        assert L.fa_bwd_noalloc(*ok, 1, 2, 128, 64, scale, 0, None, None, None) == 1, scale
    for k in range(9):
        for bad in (None, 264):
            args = list(ok)
            args[k] = bad
            assert L.fa_bwd_noalloc(*args, 1, 2, 128, 64, 0.125, 0, None, None, None) == 1, (k, bad)


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_matches_workspace_backward_twice(d):
    fa.build()
    c = make_case(2, 3, 300, d, seed=77 + d, causal=True, key_len=[300, 170])
    scale = 1.0 / d ** 0.5
    Q, K, V, dO = (c[k].cuda() for k in ("Q", "K", "V", "dO"))
    kl = c["key_len"].cuda()
    O, LSE = fa.attention_forward(Q, K, V, scale, True, kl, None, check_status=True)
    rQ, rK, rV = fa.attention_backward(Q, K, V, O, LSE, dO, scale, True, kl, None, check_status=True)
    B, H, N, _ = Q.shape
    f64 = lambda t: t.to(torch.float64).numpy()
    _, _, odQ, odK, odV = oracle.attention_bwd(f64(c["Q"]), f64(c["K"]), f64(c["V"]), f64(c["dO"]), scale,
                                                causal=True, key_len=c["key_len"].numpy())
    orel = lambda got, ref: float(np.linalg.norm(got.double().cpu().numpy() - ref) / np.linalg.norm(ref))
    for call in range(2):
        dQ, dK, dV = (torch.full_like(Q, float("nan")) for _ in range(3))
        st = fa.fa_bwd_noalloc(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, N, d, scale, True, kl, None)
        assert st == 0, fa.fa_status_string(st)
        torch.cuda.synchronize()
        for got, ref, name in ((dQ, rQ, "dQ"), (dK, rK, "dK"), (dV, rV, "dV")):
            assert bool(torch.isfinite(got).all()), (call, name)
            assert rel_fro(got, ref) <= GRAD_REL_FRO, (call, name, rel_fro(got, ref))
        # and against the fp64 oracle directly, with the same bound
        for got, ref, name in ((dQ, odQ, "dQ"), (dK, odK, "dK"), (dV, odV, "dV")):
            assert orel(got, ref) <= GRAD_REL_FRO, (call, name, "oracle", orel(got, ref))
        # dK and dV are not accumulated across CTAs: identical to the workspace path
        assert torch.equal(dK, rK) and torch.equal(dV, rV), call


@pytest.mark.gpu
def test_noalloc_plain_d128_uses_the_split_and_matches():
    """d = 128 with every tile full: the built-in array holds the split area
    for this size (the last wave's key tiles run in parts), so fa_bwd_noalloc
    takes the same plan as fa_bwd with a full workspace: dK and dV bit for
    bit, dQ within the parity bound, every output against the oracle too;
    twice, since the split's counters must be back at zero for the next
    call."""
    fa.build()
    B, H, N, d = 1, 2, 1024, 128
    c = make_case(B, H, N, d, seed=91)
    scale = 1.0 / d ** 0.5
    Q, K, V, dO = (c[k].cuda() for k in ("Q", "K", "V", "dO"))
    O, LSE = fa.attention_forward(Q, K, V, scale, False, check_status=True)
    rQ, rK, rV = fa.attention_backward(Q, K, V, O, LSE, dO, scale, False, check_status=True)
    f64 = lambda t: t.to(torch.float64).numpy()
    _, _, odQ, odK, odV = oracle.attention_bwd(f64(c["Q"]), f64(c["K"]), f64(c["V"]), f64(c["dO"]), scale)
    orel = lambda got, ref: float(np.linalg.norm(got.double().cpu().numpy() - ref) / np.linalg.norm(ref))
    for call in range(2):
        dQ, dK, dV = (torch.full_like(Q, float("nan")) for _ in range(3))
        st = fa.fa_bwd_noalloc(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, N, d, scale, False, None, None)
        assert st == 0, fa.fa_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(dK, rK) and torch.equal(dV, rV), call
        assert rel_fro(dQ, rQ) <= GRAD_REL_FRO, call
        for got, ref, name in ((dQ, odQ, "dQ"), (dK, odK, "dK"), (dV, odV, "dV")):
            assert orel(got, ref) <= GRAD_REL_FRO, (call, name, orel(got, ref))
