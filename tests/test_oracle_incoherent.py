"""Pins of the incoherent-processing rotation (oracle/incoherent.py) and of
the rotated block quantiser, against mathematics that does not depend on the
transform's implementation: the Sylvester matrix's defining properties, the
explicit matrix product, the dot-product identity that makes the rotation
harmless, and the effect it exists for (a smaller FP8 error when a few
channels carry outliers)."""
import numpy as np
import pytest

import oracle
from oracle.incoherent import hadamard, rotate


def signs(d, seed):
    return np.where(np.random.default_rng(seed).random(d) < 0.5, -1, 1).astype(np.int8)


@pytest.mark.parametrize("d", [1, 2, 4, 64, 128, 256])
def test_sylvester_matrix(d):
    H = hadamard(d)
    assert set(np.unique(H)) <= {-1.0, 1.0}
    assert np.array_equal(H, H.T)
    assert np.array_equal(H @ H.T, d * np.eye(d))
    if d >= 2:       # the recursive structure: H_2n = [[H, H], [H, -H]]
        h = hadamard(d // 2)
        assert np.array_equal(H, np.block([[h, h], [h, -h]]))


@pytest.mark.parametrize("d", [64, 128])
def test_transform_is_the_matrix_product_on_exact_inputs(d):
    # small integers: every partial sum is exact in fp32, so the transform
    # must give (x * s) H bit for bit
    x = np.random.default_rng(d).integers(-64, 64, (5, 7, d)).astype(np.float32)
    s = signs(d, d + 1)
    assert np.array_equal(rotate(x, s), ((x * s) @ hadamard(d)).astype(np.float32))


def test_transform_rounding_bound_on_bf16_values():
    import torch
    d = 128
    x = torch.randn(64, d).mul(torch.logspace(-3, 3, d)).to(torch.bfloat16).float().numpy()
    s = signs(d, 9)
    exact = (x.astype(np.float64) * s) @ hadamard(d)
    err = np.abs(rotate(x, s).astype(np.float64) - exact)
    # each of the log2(d) stages rounds once, by at most half an ulp of a
    # partial sum bounded by sum |x|
    bound = np.log2(d) * 2.0 ** -24 * np.abs(x).sum(axis=1, keepdims=True)
    assert np.all(err <= bound)


def test_rotation_keeps_scores_up_to_d():
    rng = np.random.default_rng(3)
    Q, K = rng.standard_normal((2, 50, 128))
    M = np.diag(signs(128, 4).astype(np.float64)) @ hadamard(128)
    assert np.allclose((Q @ M) @ (K @ M).T, 128 * Q @ K.T, rtol=1e-12, atol=1e-9)


def test_rotated_quantiser_is_quantiser_of_rotated_values():
    rng = np.random.default_rng(5)
    X = rng.standard_normal((1, 2, 300, 128)).astype(np.float32)
    s = signs(128, 6)
    c1, s1 = oracle.quantize_fp8_rotated(X, s)
    c2, s2 = oracle.quantize_fp8(rotate(X, s), False)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def outlier_case(seed, N=256, d=128, n_out=4, mag=40.0):
    import torch
    g = torch.Generator().manual_seed(seed)
    Q, K, V = (torch.randn((1, 1, N, d), generator=g) for _ in range(3))
    ch = torch.randperm(d, generator=g)[:n_out]
    Q[..., ch] *= mag             # a few channels carry most of the magnitude
    K[..., ch] *= mag
    f = lambda t: t.to(torch.bfloat16).double().numpy()
    return f(Q), f(K), f(V)


def fp8_error(Q, K, V, scale, s=None):
    N = Q.shape[2]
    d = Q.shape[3]
    rO, _ = oracle.attention_fwd(Q, K, V, scale)
    if s is None:
        q = oracle.dequantize_fp8(*oracle.quantize_fp8(Q), N)
        k = oracle.dequantize_fp8(*oracle.quantize_fp8(K), N)
        sc = scale
    else:
        q = oracle.dequantize_fp8(*oracle.quantize_fp8_rotated(Q, s), N)
        k = oracle.dequantize_fp8(*oracle.quantize_fp8_rotated(K, s), N)
        sc = scale / d
    v = oracle.dequantize_fp8(*oracle.quantize_fp8(V, True), N, True)
    O, _ = oracle.attention_fwd(q, k, v, sc)
    return np.linalg.norm(O - rO) / np.linalg.norm(rO)


def test_rotation_lowers_fp8_error_with_outlier_channels():
    ratios = []
    for seed in (11, 12, 13):
        Q, K, V = outlier_case(seed)
        scale = 1.0 / (128 ** 0.5 * 40.0)      # keep the softmax in a moderate range
        plain = fp8_error(Q, K, V, scale)
        rot = fp8_error(Q, K, V, scale, signs(128, seed))
        ratios.append(plain / rot)
    assert min(ratios) > 1.5, ratios
