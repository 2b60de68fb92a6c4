"""Orthogonal rotation of q and k before FP8 quantisation (test
infrastructure only).

ZYFA README, "Using FP8 attention in a model": a Hadamard rotation of q and k
before quantisation roughly halves the input error; the rotation is
R = diag(s) H / sqrt(d) with H the d x d Hadamard matrix of Sylvester's
construction (H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]) and s a vector of
random signs, applied to each head row as x @ R (after RoPE; v is left
unrotated).  R is orthogonal, so (qR)(kR)^T = qk^T and only the rounding of
the quantised inputs changes.  A 192-channel head has no Hadamard matrix of
its own size, so there the README mixes a DCT of length 3 with a Hadamard
matrix of order 64; the reading taken here is the Kronecker product
R = diag(s) (C3^T kron H_64) / 8, with C3 the orthonormal DCT-II matrix
C3[k, n] = a_k cos(pi (2n + 1) k / 6), a_0 = sqrt(1/3), a_k = sqrt(2/3):
row block n of x (columns 64n .. 64n+63) is transformed by H_64 / 8 and the
three blocks are mixed by the DCT.

The signs are an input (the README draws them from a seeded generator); the
quantisation of the rotated values is ``quantize.fp8_quantize_f64``.
Pinned by ``tests/test_oracle.py::test_rotation_*``.
"""

from __future__ import annotations

import math

import numpy as np

from .quantize import fp8_quantize_f64


def hadamard_f64(n: int) -> np.ndarray:
    """Sylvester's n x n Hadamard matrix (n a power of two), entries +-1."""
    if n < 1 or n & (n - 1):
        raise ValueError("n must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def dct3_f64() -> np.ndarray:
    """Orthonormal 3-point DCT-II matrix, rows = frequencies k, columns = samples n."""
    c = np.empty((3, 3))
    for k in range(3):
        a = math.sqrt(1.0 / 3.0) if k == 0 else math.sqrt(2.0 / 3.0)
        for n in range(3):
            c[k, n] = a * math.cos(math.pi * (2 * n + 1) * k / 6.0)
    return c


def rotation_f64(d: int, signs) -> np.ndarray:
    """The d x d rotation applied as x @ R (d = 128, or 192 in DCT x Hadamard form)."""
    s = np.asarray(signs, dtype=np.float64).reshape(d)
    if d == 192:
        core = np.kron(dct3_f64().T, hadamard_f64(64)) / 8.0
    else:
        core = hadamard_f64(d) / math.sqrt(d)
    return s[:, None] * core


def rotate_f64(x: np.ndarray, signs) -> np.ndarray:
    """x (..., d) @ R in float64."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    return x @ rotation_f64(d, signs)


def fp8_quantize_rotated_f64(x: np.ndarray, signs):
    """(codes, descale) of x @ R: rotation then per-tensor e4m3 quantisation."""
    return fp8_quantize_f64(rotate_f64(x, signs))
