"""NaN canaries: every output buffer is filled with NaN before the call, so an
element a kernel forgets to write stays NaN.  Each entry point runs on shapes
with ragged tails, masked and fully masked rows, and the result must hold no
NaN and equal, bit for bit, the same call into freshly allocated buffers
(whose values the parity tests compare with the oracle).  Rows with no
visible key must come out as O = 0 and LSE = -inf."""
import numpy as np
import pytest
import torch

from synthetic import make_case

pytestmark = pytest.mark.gpu

NAN = float("nan")


def nan_like(t, dtype=None):
    return torch.full(t.shape if hasattr(t, "shape") else t, NAN, dtype=dtype or t.dtype, device="cuda")


def assert_written(label, *ts):
    for i, t in enumerate(ts):
        assert not torch.isnan(t).any().item(), (label, i, int(torch.isnan(t).sum()))


def dev(c, k):
    return None if c[k] is None else c[k].cuda().contiguous()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kind", ["plain", "masked"])
def test_forward_and_backward_write_every_element(d, kind):
    import io_aware_exact_09_gb300 as fa
    B, H, N = 2, 2, 333
    kw = dict(causal=True, key_len=[333, 150], block_mask=[[0, 0, 0], [0, 1, 0], [1, 1, 1]]) if kind == "masked" \
        else {}
    c = make_case(B, H, N, d, seed=41 + d, **kw)
    Q, K, V, dO = (dev(c, k) for k in ("Q", "K", "V", "dO"))
    kl, bm = dev(c, "key_len"), dev(c, "block_mask")
    causal = c["causal"]

    def run(fill):
        O = nan_like(Q) if fill else torch.empty_like(Q)
        L = torch.full((B, H, N), NAN if fill else 0.0, dtype=torch.float32, device="cuda")
        ws = fa.workspace(fa.fa_fwd_workspace_size(B, H, N, d), "cuda")
        assert fa.fa_fwd(Q, K, V, O, L, B, H, N, d, c["scale"], causal, kl, bm, ws, ws.numel()) == 0
        assert fa.fa_get_device_status(ws) == 0
        dQ, dK, dV = ((nan_like(Q) if fill else torch.empty_like(Q)) for _ in range(3))
        wb = fa.workspace(fa.fa_bwd_workspace_size(B, H, N, d), "cuda")
        assert fa.fa_bwd(Q, K, V, O, L, dO, dQ, dK, dV, B, H, N, d, c["scale"], causal, kl, bm, wb, wb.numel()) == 0
        assert fa.fa_get_device_status(wb) == 0
        torch.cuda.synchronize()
        return O, L, dQ, dK, dV

    O, L, dQ, dK, dV = run(True)
    # LSE is -inf (not NaN) exactly on rows with no visible key
    assert_written((d, kind), O, dQ, dK, dV)
    assert not torch.isnan(L).any().item()
    empty = torch.isinf(L)
    assert torch.all(O[empty] == 0)
    if kind == "masked":
        assert empty.any()                          # the mask leaves some rows without a key
    O2, L2, dQ2, dK2, dV2 = run(False)
    assert torch.equal(O, O2) and torch.equal(L, L2) and torch.equal(dK, dK2) and torch.equal(dV, dV2)
    # dQ is summed by reduce-adds in varying order
    assert torch.allclose(dQ.float(), dQ2.float(), rtol=1e-2, atol=1e-3)


@pytest.mark.parametrize("block_q,block_k", [(256, 64), (128, 128), (128, 64)])
def test_other_tile_shapes_write_every_element(block_q, block_k):
    import io_aware_exact_09_gb300 as fa
    B, H, N, d = 1, 2, 300, 128
    c = make_case(B, H, N, d, seed=43, causal=True, key_len=[200])
    Q, K, V = (dev(c, k) for k in ("Q", "K", "V"))
    kl = dev(c, "key_len")
    O, L = nan_like(Q), torch.full((B, H, N), NAN, device="cuda")
    ws = fa.workspace(fa.fa_fwd_workspace_size(B, H, N, d), "cuda")
    assert fa.fa_fwd_tiles(Q, K, V, O, L, B, H, N, d, c["scale"], True, kl, None, block_q, block_k, ws,
                           ws.numel()) == 0
    assert fa.fa_get_device_status(ws) == 0
    assert_written((block_q, block_k), O)
    assert not torch.isnan(L).any().item()


@pytest.mark.parametrize("splits", [1, 3, 0])
def test_decode_writes_every_element(splits):
    import io_aware_exact_09_gb300 as fa
    B, H, Nq, Nk, d = 3, 2, 5, 1000, 64
    g = torch.Generator().manual_seed(47)
    Q, K, V = (torch.randn(s, generator=g).to(torch.bfloat16).cuda()
               for s in ((B, H, Nq, d), (B, H, Nk, d), (B, H, Nk, d)))
    kv = torch.tensor([1000, 3, 0], dtype=torch.int32, device="cuda")   # the last batch sees nothing
    O, L = nan_like(Q), torch.full((B, H, Nq), NAN, device="cuda")
    ws = fa.workspace(fa.fa_decode_workspace_size(B, H, Nq, Nk, d, splits), "cuda")
    assert fa.fa_decode(Q, K, V, O, L, B, H, Nq, Nk, d, 0.125, True, kv, splits, ws, ws.numel()) == 0
    assert fa.fa_get_device_status(ws) == 0
    assert_written(splits, O)
    assert not torch.isnan(L).any().item()
    assert torch.all(O[2] == 0) and torch.all(torch.isinf(L[2]))


def test_varlen_writes_every_element():
    import io_aware_exact_09_gb300 as fa
    lens_q, lens_k, H, d = [1, 129, 0, 300], [1, 129, 5, 100], 2, 128
    g = torch.Generator().manual_seed(53)
    tq, tk = sum(lens_q), sum(lens_k)
    Q, K, V = (torch.randn(s, generator=g).to(torch.bfloat16).cuda() for s in ((tq, H, d), (tk, H, d), (tk, H, d)))
    cu = lambda ls: torch.tensor(np.concatenate([[0], np.cumsum(ls)]), dtype=torch.int32, device="cuda")
    O, L = nan_like(Q), torch.full((H, tq), NAN, device="cuda")
    ws = fa.workspace(fa.fa_fwd_workspace_size(1, 1, 1, d), "cuda")
    assert fa.fa_fwd_varlen(Q, K, V, O, L, cu(lens_q), cu(lens_k), len(lens_q), H, tq, tk, max(lens_q), d,
                            d ** -0.5, True, ws, ws.numel()) == 0
    assert fa.fa_get_device_status(ws) == 0
    assert_written("varlen", O)
    assert not torch.isnan(L).any().item()


def test_fp8_forward_writes_every_element():
    import io_aware_exact_09_gb300 as fa
    B, H, N, d = 1, 2, 300, 128
    c = make_case(B, H, N, d, seed=59, causal=True, key_len=[200])
    Q, K, V = (dev(c, k) for k in ("Q", "K", "V"))
    kl = dev(c, "key_len")
    Q8, sQ = fa.quantize_fp8(Q, False)
    K8, sK = fa.quantize_fp8(K, False)
    Vt8, sV = fa.quantize_fp8(V, True)
    O, L = nan_like(Q), torch.full((B, H, N), NAN, device="cuda")
    ws = fa.workspace(fa.fa_fwd_workspace_size(B, H, N, d), "cuda")
    assert fa.fa_fwd_fp8(Q8, K8, Vt8, sQ, sK, sV, O, L, B, H, N, d, c["scale"], True, kl, None, ws,
                         ws.numel()) == 0
    assert fa.fa_get_device_status(ws) == 0
    assert_written("fp8", O)
    assert not torch.isnan(L).any().item()
