"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times: the CUDA path runs on the whole workload; the oracle checks
sampled query rows (O, LSE, dQ) and sampled key rows (dK, dV), which it
computes one by one from the plain definition."""
import numpy as np
import pytest
import torch

import oracle
from synthetic import DECODE_WORKLOADS, WORKLOADS, make_case, make_decode_inputs, make_inputs
from gpu_common import GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, O_REL_FRO, f64, oracle_args, rel_fro, run_cuda

pytestmark = pytest.mark.gpu

FULL = ["gpt2m_causal_b8h16n1024d64", "bertl_keypad_b16h16n512d64", "longctx_b1h16n16384d128",
        "longctx_causal_b1h16n16384d128", "blocksparse_b2h16n8192d64"]


def sample_rows(B, H, N, rng, n_heads=2, per_head=24):
    """Flat (b*H+h)*N+i indices: first and last head plus random ones; in
    each, the first and last row, the rows around tile edges, random rows."""
    BH = B * H
    heads = sorted(set([0, BH - 1] + list(rng.choice(BH, size=min(BH, n_heads), replace=False))))
    rows = []
    for bh in heads:
        pick = {0, N - 1, min(127, N - 1), min(128, N - 1)}
        pick |= set(int(x) for x in rng.choice(N, size=min(N, per_head), replace=False))
        rows += [bh * N + i for i in sorted(pick)]
    return np.array(rows, np.int64), heads


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    w = WORKLOADS[name]
    case = make_inputs(w)
    got = run_cuda(case)
    B, H, N, d = w.B, w.H, w.N, w.d
    rng = np.random.default_rng(2024)
    qrows, _ = sample_rows(B, H, N, rng)
    Q, K, V, dO = (f64(case[k]) for k in ("Q", "K", "V", "dO"))
    oa = oracle_args(case)
    O_r, L_r, dQ_r = oracle.query_rows(Q, K, V, dO, case["scale"], qrows, **oa)
    flat = lambda X: X.reshape(B * H * N, -1)
    gO, gL, gdQ = flat(got["O"])[qrows], got["LSE"].reshape(-1)[qrows], flat(got["dQ"])[qrows]
    assert np.all(np.isfinite(gO)) and np.all(np.isfinite(gdQ))
    assert rel_fro(gO, O_r) <= O_REL_FRO, rel_fro(gO, O_r)
    assert np.max(np.abs(gO - O_r)) <= O_MAX_ABS
    fin = np.isfinite(L_r)
    assert np.max(np.abs(gL[fin] - L_r[fin])) <= LSE_MAX_ABS
    assert rel_fro(gdQ, dQ_r) <= GRAD_REL_FRO, rel_fro(gdQ, dQ_r)
    # key rows: dK, dV need every query row of the head, so fewer heads
    krows, _ = sample_rows(B, H, N, np.random.default_rng(7), n_heads=0, per_head=12)
    if N * N * d > 2 ** 34:
        krows = krows[krows < N]          # one head only at the longest lengths
    dK_r, dV_r = oracle.key_rows(Q, K, V, dO, case["scale"], krows, **oa)
    gdK, gdV = flat(got["dK"])[krows], flat(got["dV"])[krows]
    assert rel_fro(gdK, dK_r) <= GRAD_REL_FRO, rel_fro(gdK, dK_r)
    assert rel_fro(gdV, dV_r) <= GRAD_REL_FRO, rel_fro(gdV, dV_r)
    # properties that hold at any size, on every row
    for k in ("O", "dQ", "dK", "dV"):
        assert np.all(np.isfinite(got[k])), k


def test_tile_plan_bit_exact_on_workloads():
    import io_aware_exact_09_gb300 as fa
    for name in ("gpt2m_causal_b8h16n1024d64", "bertl_keypad_b16h16n512d64", "blocksparse_b2h16n8192d64",
                 "longctx_causal_b1h16n16384d128"):
        w = WORKLOADS[name]
        case = make_inputs(w, with_dO=False)
        kl = case["key_len"]
        bm = case["block_mask"]
        got = fa.tile_plan(w.B, w.N, w.causal, None if kl is None else kl.cuda(),
                           None if bm is None else bm.cuda()).cpu().numpy()
        ref = oracle.tile_plan(w.B, w.N, w.causal, None if kl is None else kl.numpy(),
                               None if bm is None else bm.numpy())
        assert np.array_equal(got, ref), name


@pytest.mark.parametrize("N", [1, 100, 300, 1000])
def test_tile_plan_bit_exact_ragged(N):
    import io_aware_exact_09_gb300 as fa
    rng = np.random.default_rng(N)
    T = (N + 127) // 128
    kl = rng.integers(0, N + 1, size=3).astype(np.int32)
    bm = (rng.random((T, T)) < 0.6).astype(np.uint8)
    for causal in (False, True):
        for use_kl in (False, True):
            for use_bm in (False, True):
                got = fa.tile_plan(3, N, causal, torch.from_numpy(kl).cuda() if use_kl else None,
                                   torch.from_numpy(bm).cuda() if use_bm else None)
                ref = oracle.tile_plan(3, N, causal, kl if use_kl else None, bm if use_bm else None)
                assert np.array_equal(got.cpu().numpy(), ref), (N, causal, use_kl, use_bm)


@pytest.mark.parametrize("N", [1, 127, 128, 129, 255, 256, 257, 640, 1000])
def test_visit_rules_match_tile_classes_at_tile_edges(N):
    """Without a block mask the forward visits a contiguous range of key tiles
    and the backward a contiguous range of query blocks, each found in O(1);
    the exported plan writes 3 wherever either range disagrees with the tile's
    class.  Key lengths at, just below and just above every tile edge (and 0,
    1, N), with and without the causal mask: the plan must equal the oracle's
    brute-force enumeration, so a range one tile too long or too short fails."""
    import io_aware_exact_09_gb300 as fa
    edges = {0, 1, N} | {e + o for e in range(0, N + 1, 128) for o in (-1, 0, 1) if 0 <= e + o <= N}
    kl = np.array(sorted(edges), np.int32)
    for causal in (False, True):
        for use_kl in (False, True):
            B = len(kl) if use_kl else 2
            got = fa.tile_plan(B, N, causal, torch.from_numpy(kl).cuda() if use_kl else None, None).cpu().numpy()
            ref = oracle.tile_plan(B, N, causal, kl if use_kl else None, None)
            assert not np.any(got == 3), (N, causal, use_kl)
            assert np.array_equal(got, ref), (N, causal, use_kl)


def test_host_buffer_path_matches_device_path():
    import io_aware_exact_09_gb300 as fa
    w = WORKLOADS["bertl_keypad_b16h16n512d64"]
    case = make_inputs(w)
    B, H, N, d = w.B, w.H, w.N, w.d
    pin = lambda t: t.contiguous().pin_memory()
    Qh, Kh, Vh, dOh = (pin(case[k]) for k in ("Q", "K", "V", "dO"))
    O = torch.empty_like(Qh).pin_memory()
    LSE = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    dQ, dK, dV = (torch.empty_like(Qh).pin_memory() for _ in range(3))
    kl = case["key_len"].contiguous()
    need = fa.fa_host_workspace_size(B, H, N, d, 1)
    ws = fa.workspace(need, "cuda")
    st = fa.fa_attention_host(Qh, Kh, Vh, dOh, O, LSE, dQ, dK, dV, B, H, N, d, case["scale"], False, kl,
                              None, ws, ws.numel())
    assert st == 0, fa.fa_status_string(st)
    dev = run_cuda(case)
    assert np.array_equal(O.double().numpy(), dev["O"])
    assert np.array_equal(LSE.double().numpy(), dev["LSE"])
    assert np.array_equal(dK.double().numpy(), dev["dK"])
    assert np.array_equal(dV.double().numpy(), dev["dV"])
    # dQ goes through fp32 atomics whose order varies: compare within tolerance
    assert rel_fro(dQ.double().numpy(), dev["dQ"]) < 1e-3


@pytest.mark.parametrize("B,H,N,d,key_len", [(2, 8, 8192, 128, [8192, 2500]),
                                              (4, 8, 8192, 64, [8192, 300, 5000, 8191])])
def test_host_buffer_path_in_chunks_with_key_len(B, H, N, d, key_len):
    """Large enough to run in chunks: with B = 2 each chunk is a head range of
    one batch, with B = 4 one whole batch; either way the kernels see the
    chunk's key_len through an offset pointer.  The forward and dK, dV are
    per-head deterministic, so the chunked host path gives the device path's
    bits; the forward-only call too."""
    import io_aware_exact_09_gb300 as fa
    case = make_case(B, H, N, d, seed=37, causal=True, key_len=key_len)
    pin = lambda t: t.contiguous().pin_memory()
    Qh, Kh, Vh, dOh = (pin(case[k]) for k in ("Q", "K", "V", "dO"))
    kl = case["key_len"].contiguous()
    dev = run_cuda(case)
    for with_bwd in (1, 0):
        O = torch.empty_like(Qh).pin_memory()
        LSE = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        dQ, dK, dV = (torch.empty_like(Qh).pin_memory() for _ in range(3))
        ws = fa.workspace(fa.fa_host_workspace_size(B, H, N, d, with_bwd), "cuda")
        st = fa.fa_attention_host(Qh, Kh, Vh, dOh if with_bwd else None, O, LSE, dQ if with_bwd else None,
                                  dK if with_bwd else None, dV if with_bwd else None, B, H, N, d, case["scale"],
                                  True, kl, None, ws, ws.numel())
        assert st == 0, fa.fa_status_string(st)
        assert np.array_equal(O.double().numpy(), dev["O"])
        assert np.array_equal(LSE.double().numpy(), dev["LSE"])
        if with_bwd:
            assert np.array_equal(dK.double().numpy(), dev["dK"])
            assert np.array_equal(dV.double().numpy(), dev["dV"])
            assert rel_fro(dQ.double().numpy(), dev["dQ"]) < 1e-3


def test_host_buffer_path_orders_its_streams():
    """fa_attention_host runs on its own upload, download and per-chunk compute
    streams.  Work already queued on the caller's stream must finish first:
    here it zeroes the whole device workspace (slowly, many times), which
    would wipe the uploaded inputs if a copy ran ahead of it.  Repeated calls
    on a non-default stream give the device path's bits each time (the shape
    runs in four chunks)."""
    import io_aware_exact_09_gb300 as fa
    B, H, N, d = 1, 16, 8192, 128
    case = make_case(B, H, N, d, seed=31)
    pin = lambda t: t.contiguous().pin_memory()
    Qh, Kh, Vh, dOh = (pin(case[k]) for k in ("Q", "K", "V", "dO"))
    dev = run_cuda(case)
    need = fa.fa_host_workspace_size(B, H, N, d, 1)
    ws = fa.workspace(need, "cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(3):
            O = torch.empty_like(Qh).pin_memory()
            LSE = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
            dQ, dK, dV = (torch.empty_like(Qh).pin_memory() for _ in range(3))
            for _ in range(50):
                ws.zero_()
            st = fa.fa_attention_host(Qh, Kh, Vh, dOh, O, LSE, dQ, dK, dV, B, H, N, d, case["scale"], False, None,
                                      None, ws, ws.numel(), stream)
            assert st == 0, fa.fa_status_string(st)
            assert np.array_equal(O.double().numpy(), dev["O"])
            assert np.array_equal(LSE.double().numpy(), dev["LSE"])
            assert np.array_equal(dK.double().numpy(), dev["dK"])
            assert np.array_equal(dV.double().numpy(), dev["dV"])
            assert rel_fro(dQ.double().numpy(), dev["dQ"]) < 1e-3


@pytest.mark.parametrize("name", sorted(DECODE_WORKLOADS))
def test_decode_full_size_sampled(name):
    """Decode workloads at full size with the split count bench.py uses
    (automatic): sampled (b, h) pairs against the fp64 decode oracle."""
    import io_aware_exact_09_gb300 as fa
    w = DECODE_WORKLOADS[name]
    c = make_decode_inputs(w)
    kl = None if c["kv_len"] is None else c["kv_len"].cuda()
    O, L = fa.attention_decode(c["Q"].cuda(), c["K"].cuda(), c["V"].cuda(), w.softmax_scale, w.causal, kl, 0,
                               check_status=True)
    torch.cuda.synchronize()
    O, L = O.double().cpu().numpy(), L.double().cpu().numpy()
    rng = np.random.default_rng(w.seed)
    picks = [(0, 0), (w.B - 1, w.H - 1)] + [(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(4)]
    for b, h in picks:
        sl = lambda t: t[b:b + 1, h:h + 1].double().numpy()
        kvb = None if c["kv_len"] is None else [int(c["kv_len"][b])]
        rO, rL = oracle.attention_decode(sl(c["Q"]), sl(c["K"]), sl(c["V"]), w.softmax_scale, causal=w.causal,
                                         kv_len=kvb)
        o, l = O[b:b + 1, h:h + 1], L[b:b + 1, h:h + 1]
        assert rel_fro(o, rO) <= O_REL_FRO, (name, b, h, rel_fro(o, rO))
        assert np.max(np.abs(o - rO)) <= O_MAX_ABS, (name, b, h)
        assert np.max(np.abs(l - rL)) <= LSE_MAX_ABS, (name, b, h)


@pytest.mark.parametrize("B,H,N,d", [(8, 16, 4096, 128), (16, 16, 2048, 64), (5, 20, 4096, 128),
                                     (7, 13, 4096, 64)])
def test_grouped_item_order_sampled(B, H, N, d):
    """Masked shapes past the spread rule (working set beyond L2, many heads):
    the persistent forward (8 x 16 x 4096 x 128, 5 x 20 x 4096 x 128) and the
    d = 64 backward (16 x 16 x 2048 x 64, 7 x 13 x 4096 x 64) hand out their
    items in groups of 8 heads, and the d = 128 backward numbers its blocks the
    same way; with 100 and 91 heads the last group holds 4 and 3.  Sampled
    query rows (O, LSE, dQ) and key rows (dK, dV) of the first, the last and
    random heads against the oracle."""
    case = make_case(B, H, N, d, seed=B * H + N + d, causal=True)
    case["scale"] = 1.0 / d ** 0.5
    got = run_cuda(case)
    rng = np.random.default_rng(11)
    qrows, _ = sample_rows(B, H, N, rng, n_heads=3, per_head=16)
    Q, K, V, dO = (f64(case[k]) for k in ("Q", "K", "V", "dO"))
    oa = oracle_args(case)
    O_r, L_r, dQ_r = oracle.query_rows(Q, K, V, dO, case["scale"], qrows, **oa)
    flat = lambda X: X.reshape(B * H * N, -1)
    gO, gL, gdQ = flat(got["O"])[qrows], got["LSE"].reshape(-1)[qrows], flat(got["dQ"])[qrows]
    assert rel_fro(gO, O_r) <= O_REL_FRO, rel_fro(gO, O_r)
    assert np.max(np.abs(gO - O_r)) <= O_MAX_ABS
    assert np.max(np.abs(gL - L_r)) <= LSE_MAX_ABS
    assert rel_fro(gdQ, dQ_r) <= GRAD_REL_FRO, rel_fro(gdQ, dQ_r)
    krows, _ = sample_rows(B, H, N, np.random.default_rng(13), n_heads=3, per_head=8)
    dK_r, dV_r = oracle.key_rows(Q, K, V, dO, case["scale"], krows, **oa)
    gdK, gdV = flat(got["dK"])[krows], flat(got["dV"])[krows]
    assert rel_fro(gdK, dK_r) <= GRAD_REL_FRO, rel_fro(gdK, dK_r)
    assert rel_fro(gdV, dV_r) <= GRAD_REL_FRO, rel_fro(gdV, dV_r)
    for k in ("O", "dQ", "dK", "dV"):
        assert np.all(np.isfinite(got[k])), k
