"""Pins of the oracle's FP8 block quantiser (e4m3 codes, per-block scales):
the format's closed forms, a library conversion (torch.float8_e4m3fn) on
every bf16 value in range and every tie, and the properties the block
scaling guarantees."""
import numpy as np
import pytest
import torch

import oracle


def test_e4m3_table_closed_forms():
    t = oracle.e4m3_table()
    assert t[0x00] == 0.0 and t[0x38] == 1.0 and t[0x7E] == 448.0
    assert t[0x01] == 2.0 ** -9 and t[0x07] == 7 * 2.0 ** -9 and t[0x08] == 2.0 ** -6
    assert t[0x40] == 2.0 and t[0x3C] == 1.5
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)                 # strictly increasing magnitudes
    assert np.array_equal(t[0x80:0xFF], -pos)       # sign bit
    # spacing: 2^(e-3) inside binade e, subnormal spacing 2^-9
    for c in range(0x08, 0x7E):
        e = (c >> 3) - 7
        assert t[c + 1] - t[c] == 2.0 ** (e - 3)


def test_e4m3_decode_encode_round_trip():
    t = oracle.e4m3_table()
    codes = np.array([c for c in range(256) if not np.isnan(t[c])], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(t[codes].astype(np.float32)), codes)


def _torch_e4m3(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_library_on_every_bf16_value():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) <= 448.0)]
    assert np.array_equal(oracle.e4m3_encode(x), _torch_e4m3(x))


def test_e4m3_ties_to_even_and_neighbours_match_library():
    t = oracle.e4m3_table()[:0x7F]
    mids = (t[:-1] + t[1:]) / 2
    x = np.concatenate([mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                        np.nextafter(mids.astype(np.float32), np.float32(1e9))]).astype(np.float32)
    x = np.concatenate([x, -x])
    got = oracle.e4m3_encode(x)
    assert np.array_equal(got, _torch_e4m3(x))
    # at an exact tie the even mantissa wins
    tie = oracle.e4m3_encode(mids.astype(np.float32))
    assert np.all(tie % 2 == 0)


def test_e4m3_saturates_and_keeps_sign():
    x = np.array([448.0, 449.0, 464.0, 480.0, 1e30, np.inf, -500.0, -np.inf, -0.0, -1e-30], np.float32)
    assert list(oracle.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x80, 0x80]


def _bf16_values(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("N,d", [(300, 64), (128, 128), (17, 128), (129, 64)])
def test_block_quantisation_properties(N, d):
    X = _bf16_values((2, 3, N, d), seed=N + d)
    X[1, 2, :min(N, 128)] *= 40.0                      # one block with a much larger range
    codes, scales = oracle.quantize_fp8(X)
    T = (N + 127) // 128
    assert scales.shape == (2, 3, T) and scales.dtype == np.float32
    Xh = oracle.dequantize_fp8(codes, scales, N)
    tab = oracle.e4m3_table()
    for b in range(2):
        for h in range(3):
            for t in range(T):
                blk = X[b, h, 128 * t:128 * t + 128]
                amax = np.float32(np.abs(blk).max())
                sc = scales[b, h, t]
                assert sc == np.float32(amax / np.float32(448.0))
                cb = codes[b, h, 128 * t:128 * t + 128]
                # the largest element lands on +-448
                assert np.all(np.abs(tab[cb[np.abs(blk) == amax]]) == 448.0)
                err = np.abs(Xh[b, h, 128 * t:128 * t + 128] - blk)
                normal = np.abs(blk) >= 2.0 ** -6 * sc
                assert np.all(err[normal] <= 2.0 ** -4 * np.abs(blk[normal]) * (1 + 1e-6))
                assert np.all(err[~normal] <= 2.0 ** -10 * sc * (1 + 1e-6))


def test_transposed_layout_and_zero_block():
    N, d = 200, 64
    X = _bf16_values((1, 2, N, d), seed=3)
    X[0, 1, 128:] = 0.0                                # an all-zero block
    codes, scales = oracle.quantize_fp8(X)
    ct, st = oracle.quantize_fp8(X, transpose=True)
    Np = (N + 15) // 16 * 16
    assert ct.shape == (1, 2, d, Np)
    assert np.array_equal(st, scales)
    assert np.array_equal(ct[:, :, :, :N], np.swapaxes(codes, 2, 3))
    assert np.all(ct[:, :, :, N:] == 0)
    assert scales[0, 1, 1] == 0.0 and np.all(codes[0, 1, 128:] == 0)
    assert np.all(oracle.dequantize_fp8(codes, scales, N)[0, 1, 128:] == 0.0)
    assert np.array_equal(oracle.dequantize_fp8(ct, st, N, transpose=True), oracle.dequantize_fp8(codes, scales, N))


def test_fp8_attention_definition_is_close_to_bf16_attention():
    """The FP8 forward's definition (exact attention of the values the codes
    stand for) stays within the quantisation error of the bf16 attention."""
    N, d = 256, 128
    Q, K, V = (_bf16_values((1, 2, N, d), seed=s) for s in (11, 12, 13))
    deq = lambda X: oracle.dequantize_fp8(*oracle.quantize_fp8(X), N)
    O8, L8 = oracle.attention_fwd(deq(Q), deq(K), deq(V), d ** -0.5)
    O, L = oracle.attention_fwd(Q.astype(np.float64), K.astype(np.float64), V.astype(np.float64), d ** -0.5)
    rel = np.linalg.norm(O8 - O) / np.linalg.norm(O)
    assert 1e-4 < rel < 0.08
    assert np.max(np.abs(L8 - L)) < 0.05
