"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare with the fp64 oracle on the same seeded inputs."""
import numpy as np
import torch

import io_aware_exact_09_gb300 as fa

# Acceptance bounds (bf16 inputs, fp32 accumulation) against the fp64 oracle.
O_REL_FRO = 5e-3
O_MAX_ABS = 2e-2
LSE_MAX_ABS = 1e-3
GRAD_REL_FRO = 1e-2


def rel_fro(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    num = np.linalg.norm(a - b)
    return num / den if den > 0 else num


def to_dev(case, device="cuda"):
    out = {}
    for k in ("Q", "K", "V", "dO"):
        out[k] = None if case.get(k) is None else case[k].to(device).contiguous()
    out["key_len"] = None if case.get("key_len") is None else case["key_len"].to(device)
    out["block_mask"] = None if case.get("block_mask") is None else case["block_mask"].contiguous().to(device)
    return out


def run_cuda(case, backward=True, device="cuda"):
    """O, LSE (and dQ, dK, dV) from fa_fwd / fa_bwd, as fp64 numpy arrays."""
    g = to_dev(case, device)
    O, LSE = fa.attention_forward(g["Q"], g["K"], g["V"], case["scale"], case["causal"], g["key_len"],
                                  g["block_mask"], check_status=True)
    res = {"O": O, "LSE": LSE}
    if backward:
        dQ, dK, dV = fa.attention_backward(g["Q"], g["K"], g["V"], O, LSE, g["dO"], case["scale"],
                                           case["causal"], g["key_len"], g["block_mask"], check_status=True)
        res.update(dQ=dQ, dK=dK, dV=dV)
    torch.cuda.synchronize()
    return {k: v.detach().to("cpu", torch.float64).numpy() for k, v in res.items()}


def oracle_args(case):
    kl = None if case.get("key_len") is None else case["key_len"].numpy()
    bm = None if case.get("block_mask") is None else case["block_mask"].numpy()
    return dict(causal=case["causal"], key_len=kl, block_mask=bm)


def f64(t):
    return t.to(torch.float64).numpy()


def check_forward(got_O, got_LSE, ref_O, ref_LSE, label=""):
    fin = np.isfinite(ref_LSE)
    # rows with no visible key: O = 0, LSE = -inf
    assert np.all(got_LSE[~fin] == -np.inf), label
    assert np.all(got_O[~fin] == 0), label
    assert np.all(np.isfinite(got_O)), label
    e_rel = rel_fro(got_O, ref_O)
    e_abs = float(np.max(np.abs(got_O - ref_O))) if got_O.size else 0.0
    e_lse = float(np.max(np.abs(got_LSE[fin] - ref_LSE[fin]))) if fin.any() else 0.0
    assert e_rel <= O_REL_FRO, (label, "O rel", e_rel)
    assert e_abs <= O_MAX_ABS, (label, "O abs", e_abs)
    assert e_lse <= LSE_MAX_ABS, (label, "LSE", e_lse)
    return e_rel, e_abs, e_lse


def check_grads(got, ref, label=""):
    errs = {}
    for k in ("dQ", "dK", "dV"):
        assert np.all(np.isfinite(got[k])), (label, k)
        errs[k] = rel_fro(got[k], ref[k])
        assert errs[k] <= GRAD_REL_FRO, (label, k, errs[k])
    return errs
