"""The seeded input recipe: deterministic, right shapes, right mask statistics."""
import torch

from synthetic import WORKLOADS, draw_block_mask, draw_key_len, make_case, algorithmic_fwd_flops


def test_inputs_are_deterministic_bf16():
    a = make_case(2, 3, 77, 64, seed=5)
    b = make_case(2, 3, 77, 64, seed=5)
    for k in ("Q", "K", "V", "dO"):
        assert a[k].dtype == torch.bfloat16 and a[k].shape == (2, 3, 77, 64)
        assert torch.equal(a[k], b[k])
    c = make_case(2, 3, 77, 64, seed=6)
    assert not torch.equal(a["Q"], c["Q"])


def test_block_mask_recipe_statistics():
    bm = draw_block_mask(8192, 0.15, torch.Generator().manual_seed(1004))
    assert bm.shape == (64, 64) and bm.dtype == torch.uint8
    assert int(bm.sum()) == 614                       # round(0.15 * 4096)
    r = torch.arange(64)
    assert bool((bm[(r[:, None] - r[None, :]).abs() <= 1] == 1).all())   # band of width 3
    assert bool((bm[:, :4] == 1).all())                                   # 4 global key columns


def test_key_len_range():
    kl = draw_key_len(1000, 128, 512, torch.Generator().manual_seed(3))
    assert kl.dtype == torch.int32 and int(kl.min()) >= 128 and int(kl.max()) <= 512


def test_workload_table_shapes_and_flops():
    w = WORKLOADS["longctx_b1h16n16384d128"]
    assert (w.B, w.H, w.N, w.d) == (1, 16, 16384, 128) and w.input_scale == 0.5
    assert abs(algorithmic_fwd_flops(1, 16, 16384, 128) - 2.199e12) / 2.199e12 < 1e-3
    assert abs(algorithmic_fwd_flops(1, 16, 16384, 128, causal=True) - 1.0995e12) / 1.1e12 < 1e-3
    assert abs(algorithmic_fwd_flops(8, 16, 1024, 64, causal=True) - 17.18e9) / 17.18e9 < 1e-3
    # key padding counts only unmasked pairs
    f = algorithmic_fwd_flops(2, 1, 256, 64, key_len=[128, 256])
    assert f == 4.0 * 64 * (256 * 128 + 256 * 256)
