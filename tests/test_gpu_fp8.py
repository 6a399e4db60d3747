"""FP8 forward: the block quantiser (fa_quantize_fp8) is compared byte for
byte with the oracle's; the FP8 attention (fa_fwd_fp8) against the fp64
oracle's exact attention of the values the codes stand for.

Tolerance of the FP8 attention.  Its inputs are exact (the oracle reads the
same codes and scales); what differs is that the kernel rounds every
probability to e4m3 for the P.V product.  One e4m3 rounding has relative
error at most 2^-4, and for values spread over a binade its RMS is
2^-4 * sqrt(E[(2^e/x)^2] / 3) ~= 0.027.  With value rows that are not
correlated with the rounding errors, the RMS relative error of O is the
same 0.027, so the O relative-Frobenius bound is twice that, 0.05; the
worst case of one row (every rounding in the same direction) is
2^-4 * max|V| plus the bf16 rounding of O, the max-abs bound.  (Probabilities
below e4m3's normal range, p * sV_j / max sV < 2^-6, round to a 2^-9 grid
instead; on these inputs the scores of a row lie within a few units and the
block-scale ratios near 1, so few fall there.)  LSE uses the unrounded
probabilities: the bf16 bound 1e-3 applies."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import LSE_MAX_ABS, f64, rel_fro
from synthetic import WORKLOADS, make_case, make_inputs

pytestmark = pytest.mark.gpu

FP8_O_REL_FRO = 0.05


def fp8_max_abs(Vh):
    # e4m3 rounding of P (2^-4 relative in the normal range) plus the bf16
    # rounding of O (2^-9 relative), both against max |V|
    return (2.0 ** -4 + 2.0 ** -9) * float(np.max(np.abs(Vh)))


def quant_gpu(X, transpose):
    import io_aware_exact_09_gb300 as fa
    X8, sc = fa.quantize_fp8(X.cuda().contiguous(), transpose)
    torch.cuda.synchronize()
    return X8.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("shape", [(1, 2, 300, 128), (2, 1, 128, 64), (1, 1, 17, 128), (1, 2, 1000, 128),
                                   (2, 2, 129, 64)])
@pytest.mark.parametrize("transpose", [False, True])
def test_quantize_bit_exact(shape, transpose):
    B, H, N, d = shape
    g = torch.Generator().manual_seed(sum(shape) + transpose)
    X = torch.randn(shape, generator=g)
    X[0, 0, :min(N, 128)] *= 1e3                      # a block with a wide range
    if N > 128:
        X[-1, -1, 128:256] = 0.0                      # an all-zero block
    X[0, -1, 0, :5] = torch.tensor([-0.0, 1e-30, -1e-30, 3.0, -3.0])
    X = X.to(torch.bfloat16)
    codes, sc = quant_gpu(X, transpose)
    rc, rs = oracle.quantize_fp8(X.float().numpy(), transpose)
    assert np.array_equal(sc.view(np.uint32), rs.view(np.uint32))
    assert codes.shape == rc.shape
    assert np.array_equal(codes, rc), int(np.sum(codes != rc))


def run_fp8(case):
    import io_aware_exact_09_gb300 as fa
    dev = lambda t: None if t is None else t.cuda().contiguous()
    O, L = fa.attention_forward_fp8(dev(case["Q"]), dev(case["K"]), dev(case["V"]), case["scale"], case["causal"],
                                    dev(case["key_len"]), dev(case["block_mask"]), check_status=True)
    torch.cuda.synchronize()
    return O.double().cpu().numpy(), L.double().cpu().numpy()


def dequantized(case):
    N = case["Q"].shape[2]
    out = []
    for k, tr in (("Q", False), ("K", False), ("V", True)):
        codes, sc = oracle.quantize_fp8(case[k].float().numpy(), tr)
        out.append(oracle.dequantize_fp8(codes, sc, N, tr))
    return out


def check_fp8(O, L, rO, rL, Vh, label):
    fin = np.isfinite(rL)
    assert np.all(L[~fin] == -np.inf) and np.all(O[~fin] == 0), label
    assert np.all(np.isfinite(O)), label
    e = rel_fro(O, rO)
    assert e <= FP8_O_REL_FRO, (label, "O rel", e)
    assert np.max(np.abs(O - rO)) <= fp8_max_abs(Vh), (label, "O abs", np.max(np.abs(O - rO)))
    assert np.max(np.abs(L[fin] - rL[fin])) <= LSE_MAX_ABS, (label, "LSE")
    return e


@pytest.mark.parametrize("N", [128, 200, 512, 1000])
@pytest.mark.parametrize("mask", ["none", "causal", "key_len", "block"])
def test_fwd_fp8_matches_oracle(N, mask):
    kw = {}
    if mask == "causal":
        kw["causal"] = True
    elif mask == "key_len":
        kw["key_len"] = [max(1, N // 3), N]
    elif mask == "block":
        nb = (N + 127) // 128
        bm = (np.random.default_rng(N).random((nb, nb)) < 0.5).astype(np.uint8)
        np.fill_diagonal(bm, 1)
        kw["block_mask"] = bm
    case = make_case(2, 2, N, 128, seed=N + len(mask), **kw)
    O, L = run_fp8(case)
    Qh, Kh, Vh = dequantized(case)
    kl = None if case["key_len"] is None else case["key_len"].numpy()
    bm = None if case["block_mask"] is None else case["block_mask"].numpy()
    rO, rL = oracle.attention_fwd(Qh, Kh, Vh, case["scale"], causal=case["causal"], key_len=kl, block_mask=bm)
    check_fp8(O, L, rO, rL, Vh, (N, mask))


def test_fwd_fp8_rejects_d64_and_bad_args():
    import io_aware_exact_09_gb300 as fa
    x = torch.zeros((1, 1, 128, 64), dtype=torch.uint8, device="cuda")
    s = torch.zeros((1, 1, 1), device="cuda")
    O = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    L = torch.zeros((1, 1, 128), device="cuda")
    ws = fa.workspace(fa.fa_fwd_workspace_size(1, 1, 128, 64), "cuda")
    assert fa.fa_fwd_fp8(x, x, x, s, s, s, O, L, 1, 1, 128, 64, 0.125, 0, None, None, ws, ws.numel()) == 2
    assert fa.fa_fwd_fp8(None, x, x, s, s, s, O, L, 1, 1, 128, 128, 0.125, 0, None, None, ws, ws.numel()) == 1


def test_fwd_fp8_full_size_sampled_rows():
    """The long-context shape (B=1, H=16, N=16384, d=128) in the launch
    configuration bench.py times: sampled query rows of two heads."""
    w = WORKLOADS["longctx_b1h16n16384d128"]
    case = make_inputs(w, with_dO=False)
    O, L = run_fp8(case)
    Qh, Kh, Vh = dequantized(case)
    B, H, N, d = w.B, w.H, w.N, w.d
    rng = np.random.default_rng(5)
    rows = []
    for h in (0, H - 1):
        rows += [h * N + r for r in sorted(rng.choice(N, 24, replace=False))]
    rows = np.array(rows, np.int64)
    rO, rL, _ = oracle.query_rows(Qh, Kh, Vh, np.zeros_like(Qh), case["scale"], rows)
    flat = lambda X: X.reshape(B * H * N, -1)
    check_fp8(flat(O)[rows], L.reshape(-1)[rows], rO, rL, Vh, "full size")


@pytest.mark.parametrize("causal", [True, False])
def test_fwd_fp8_is_deterministic(causal):
    """Repeated runs give the same bits.  (The softmax warps run ahead of the
    P.V products here; an epilogue that waited on the per-tile barrier's
    parity could pass two phases early and read O before the last products
    landed, which showed up as run-to-run differences under the causal mask.)"""
    case = make_case(2, 2, 512, 128, seed=518, causal=causal)
    outs = [run_fp8(case) for _ in range(12)]
    for O, L in outs[1:]:
        assert np.array_equal(O, outs[0][0]) and np.array_equal(L, outs[0][1])


# ---------------------------------------------------------------- incoherent processing
def random_signs(d, seed):
    return torch.where(torch.rand(d, generator=torch.Generator().manual_seed(seed)) < 0.5, -1, 1).to(torch.int8)


@pytest.mark.parametrize("shape", [(1, 2, 300, 128), (2, 1, 128, 64), (1, 1, 17, 128), (2, 2, 129, 64)])
def test_quantize_rotated_bit_exact(shape):
    import io_aware_exact_09_gb300 as fa
    B, H, N, d = shape
    g = torch.Generator().manual_seed(sum(shape) + 7)
    X = torch.randn(shape, generator=g)
    X[..., 3] *= 50.0                                 # an outlier channel
    if N > 128:
        X[-1, -1, 128:256] = 0.0                      # an all-zero block stays zero after the rotation
    X = X.to(torch.bfloat16)
    s = random_signs(d, d + N)
    X8, sc = fa.quantize_fp8(X.cuda().contiguous(), False, signs=s.cuda())
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_fp8_rotated(X.float().numpy(), s.numpy())
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    codes = X8.cpu().numpy()
    assert np.array_equal(codes, rc), int(np.sum(codes != rc))


def rotated_reference(case, s):
    N, d = case["Q"].shape[2], case["Q"].shape[3]
    q = oracle.dequantize_fp8(*oracle.quantize_fp8_rotated(case["Q"].float().numpy(), s), N)
    k = oracle.dequantize_fp8(*oracle.quantize_fp8_rotated(case["K"].float().numpy(), s), N)
    v = oracle.dequantize_fp8(*oracle.quantize_fp8(case["V"].float().numpy(), True), N, True)
    return q, k, v, case["scale"] / d


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_fwd_fp8_incoherent_matches_oracle(mask):
    import io_aware_exact_09_gb300 as fa
    case = make_case(2, 2, 512, 128, seed=71, causal=(mask == "causal"))
    s = random_signs(128, 72)
    O, L = fa.attention_forward_fp8(case["Q"].cuda().contiguous(), case["K"].cuda().contiguous(),
                                    case["V"].cuda().contiguous(), case["scale"], case["causal"],
                                    check_status=True, signs=s.cuda())
    torch.cuda.synchronize()
    q, k, v, sc = rotated_reference(case, s.numpy())
    rO, rL = oracle.attention_fwd(q, k, v, sc, causal=case["causal"])
    check_fp8(O.double().cpu().numpy(), L.double().cpu().numpy(), rO, rL, v, mask)


def test_incoherent_processing_lowers_fp8_error_with_outliers():
    """The effect the rotation exists for, through the kernels: with a few
    large channels in Q and K, the FP8 output is closer to the exact
    attention of the bf16 inputs with the rotation than without."""
    import io_aware_exact_09_gb300 as fa
    g = torch.Generator().manual_seed(73)
    B, H, N, d = 1, 4, 1024, 128
    Q, K, V = (torch.randn((B, H, N, d), generator=g) for _ in range(3))
    ch = torch.randperm(d, generator=g)[:4]
    Q[..., ch] *= 40.0
    K[..., ch] *= 40.0
    Q, K, V = (t.to(torch.bfloat16) for t in (Q, K, V))
    scale = 1.0 / (d ** 0.5 * 40.0)
    rO, _ = oracle.attention_fwd(f64(Q), f64(K), f64(V), scale)
    dev = lambda t: t.cuda().contiguous()
    err = {}
    for name, s in (("plain", None), ("rotated", random_signs(d, 74).cuda())):
        O, _ = fa.attention_forward_fp8(dev(Q), dev(K), dev(V), scale, False, check_status=True, signs=s)
        err[name] = float(np.linalg.norm(O.double().cpu().numpy() - rO) / np.linalg.norm(rO))
    assert err["plain"] / err["rotated"] > 1.5, err


def fp8_split_factor(B, H, N, sms):
    """The launcher's plan for the plain FP8 forward: items (query-tile pairs
    x B x H) past the last full wave, parts per item (2..4, 16 key tiles per
    part at least), the f whose parts' waves end soonest."""
    T = N // 128
    items = B * H * ((T + 1) // 2)
    rem = items % sms
    if rem == 0 or rem > 224 or T < 32:
        return 0
    cap = min(512, B * H * ((T + 1) // 2) * min(4, T // 16))
    best, best_len = 1, 1.0
    for f in range(2, 5):
        if f > T // 16 or rem * f > cap:
            break
        ln = -(-rem * f // sms) / f
        if ln < best_len - 1e-12:
            best, best_len = f, ln
    return best if best >= 2 else 0


# (B, H, N) on 152 SMs: f = 2 (64 items of 32 key tiles), f = 3 (96 items of
# 64), f = 4 (32 items of 64), f = 2 with an odd tile count (68 items of 33 key
# tiles; every head's last pair holds one query tile, and is split too), f = 2
# on a two-batch input (64 items of 32)
FP8_SPLIT_SHAPES = [(1, 4, 4096), (1, 3, 8192), (1, 1, 8192), (1, 4, 4224), (2, 2, 4096)]


@pytest.mark.parametrize("B,H,N", FP8_SPLIT_SHAPES)
def test_fwd_fp8_split_matches_oracle_and_unsplit(B, H, N):
    """The plain FP8 forward's last wave split over 2-4 CTAs per item (each
    over its own key tiles, the last to finish merging the parts' O and
    (m, l)): parity with the oracle, agreement with the unsplit kernel (a
    256-byte workspace, which has no room for the parts), bit-identical
    repeats (the merge's order does not depend on which part ends last), and
    the status block's counters back at zero."""
    import io_aware_exact_09_gb300 as fa
    d = 128
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    f = fp8_split_factor(B, H, N, sms)
    case = make_case(B, H, N, d, seed=H * 7 + N)
    dev = lambda t: t.cuda().contiguous()
    Q, K, V = dev(case["Q"]), dev(case["K"]), dev(case["V"])
    need = fa.fa_fwd_workspace_size(B, H, N, d)
    assert need > 256
    ws = fa.workspace(need, "cuda")
    O, L = fa.attention_forward_fp8(Q, K, V, case["scale"], False, ws=ws, check_status=True)
    torch.cuda.synchronize()
    assert int(ws[32:256].view(torch.int32).abs().sum()) == 0, f
    if f >= 2:
        assert int((ws[256:] != 0).sum()) > 0, f              # the parts' slots were written: the split ran
    for _ in range(3):
        O2, L2 = fa.attention_forward_fp8(Q, K, V, case["scale"], False, ws=ws)
        assert torch.equal(O, O2) and torch.equal(L, L2), f
    assert fa.fa_get_device_status(ws) == 0
    assert int(ws[32:256].view(torch.int32).abs().sum()) == 0
    ws0 = fa.workspace(256, "cuda")
    O0, L0 = fa.attention_forward_fp8(Q, K, V, case["scale"], False, ws=ws0, check_status=True)
    On, Ln, O0n, L0n = (t.double().cpu().numpy() for t in (O, L, O0, L0))
    # each part rounds its probabilities to e4m3 against its own running
    # maximum, so O agrees with the unsplit kernel's within the FP8 bound (not
    # bit for bit); LSE sums unrounded probabilities: fp32 rounding only
    assert rel_fro(On, O0n) <= FP8_O_REL_FRO, ("split vs unsplit", f, rel_fro(On, O0n))
    assert np.max(np.abs(Ln - L0n)) <= 1e-4, ("split vs unsplit LSE", f, np.max(np.abs(Ln - L0n)))
    Qh, Kh, Vh = dequantized(case)
    rO, rL = oracle.attention_fwd(Qh, Kh, Vh, case["scale"], causal=False)
    check_fp8(On, Ln, rO, rL, Vh, ("split", f))


def test_fwd_fp8_split_plan_covers_the_intended_factors():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    fs = [fp8_split_factor(B, H, N, sms) for B, H, N in FP8_SPLIT_SHAPES]
    if sms == 152:
        assert fs == [2, 3, 4, 2, 2], fs
    # 8 key tiles per part would be too short: B4 H16 N4096 does not split
    assert fp8_split_factor(4, 16, 4096, 152) == 0
    # the long-context shape: 1,024 items, 112 past six waves of 152 -> 4 parts each
    assert fp8_split_factor(1, 16, 16384, 152) == 4


def test_fwd_fp8_full_size_sampled():
    """The long-context workload at full size, as the benchmark runs it (its
    last wave split four ways): sampled query rows of the first and last
    head and of random heads against the oracle's rows of the dequantised
    inputs."""
    import io_aware_exact_09_gb300 as fa
    from test_gpu_fullsize import sample_rows
    w = WORKLOADS["longctx_b1h16n16384d128"]
    case = make_inputs(w)
    B, H, N, d = w.B, w.H, w.N, w.d
    dev = lambda t: t.cuda().contiguous()
    O, L = fa.attention_forward_fp8(dev(case["Q"]), dev(case["K"]), dev(case["V"]), case["scale"], False,
                                    check_status=True)
    torch.cuda.synchronize()
    rows, _ = sample_rows(B, H, N, np.random.default_rng(99))
    Qh, Kh, Vh = dequantized(case)
    O_r, L_r, _ = oracle.query_rows(Qh, Kh, Vh, None, case["scale"], rows)
    gO = O.double().cpu().numpy().reshape(B * H * N, d)[rows]
    gL = L.double().cpu().numpy().reshape(-1)[rows]
    assert np.all(np.isfinite(gO))
    e = rel_fro(gO, O_r)
    assert e <= FP8_O_REL_FRO, e
    assert np.max(np.abs(gO - O_r)) <= fp8_max_abs(Vh), np.max(np.abs(gO - O_r))
    assert np.max(np.abs(gL - L_r)) <= LSE_MAX_ABS, np.max(np.abs(gL - L_r))
