"""Incoherent processing for the FP8 forward (test infrastructure, part of
the oracle).

The "Attention" chapter of learn-kernels.com (its paragraph on the Hopper
generation and FlashAttention-3) names block quantization with incoherent
processing as the FP8 method and credits it with a lower numerical error
than a baseline FP8 attention; no page gives a formula.
The reading taken here (the usual meaning of incoherent processing): before
block quantisation, Q and K are multiplied along the head dimension by a
random orthogonal matrix, M = diag(s) H, with s a vector of random signs (an
input: the caller draws it) and H the Walsh-Hadamard matrix.  Because
M M^T = d I, (Q M)(K M)^T = d Q K^T, so the attention of the rotated,
quantised Q and K with softmax scale `scale / d` approximates the original
one; the rotation spreads a few large channels over all d channels, so a
block's amax (its quantisation step) shrinks relative to its typical values.
V is not rotated.

H is the unnormalised Sylvester matrix (H_1 = [1], H_2n = [[H, H], [H, -H]]),
applied as the fast Walsh-Hadamard transform in fp32, stage h = 1, 2, 4, ...,
d/2 mapping each pair (i, i + h) inside a block of 2h to (x_i + x_{i+h},
x_i - x_{i+h}).  Each stage is one fp32 addition per element, so the result
is a definite fp32 value that the device computes identically."""
import numpy as np


def hadamard(d: int) -> np.ndarray:
    """The d x d Sylvester-Hadamard matrix (entries +-1, H H^T = d I), fp64."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


def rotate(X, signs) -> np.ndarray:
    """(X * signs) H along the last axis, by the fast Walsh-Hadamard transform
    in fp32 (X: values of bf16 tensors, any leading shape; signs: +-1 [d])."""
    y = np.asarray(X, np.float32) * np.asarray(signs, np.float32)
    y = y.astype(np.float32)
    d = y.shape[-1]
    lead = y.shape[:-1]
    h = 1
    while h < d:
        y = y.reshape(lead + (d // (2 * h), 2, h))
        a, b = y[..., 0, :], y[..., 1, :]
        y = np.stack([(a + b).astype(np.float32), (a - b).astype(np.float32)], axis=-2).reshape(lead + (d,))
        h *= 2
    return y
