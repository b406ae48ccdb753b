"""Independent numpy restatements used only to pin the oracle (dense matmul forms).

The E2M1 table comes from the golden grid fixture, not from the oracle.
"""
import numpy as np

from conftest import read_golden

E2M1 = np.array([float(v) for _, v in read_golden("e2m1_grid.txt")], dtype=np.float64)


def dequant(fp4, e8m0):
    """packed [..., R, K/2] + scales [..., R, K/32] -> fp64 [..., R, K]."""
    lo = fp4 & 0xF
    hi = fp4 >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(fp4.shape[:-1] + (fp4.shape[-1] * 2,))
    vals = E2M1[codes]
    sc = np.ldexp(1.0, e8m0.astype(np.int64) - 127)
    return vals * np.repeat(sc, 32, axis=-1)


def bf16_to_f64(x16):
    return (x16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def silu(z):
    return z / (1.0 + np.exp(-z))


def dense_moe(x, W1, W3, W2, G):
    """y = sum_e G[:, e] * (silu(x W1_e^T) * (x W3_e^T)) W2_e^T, all fp64 matmuls."""
    y = np.zeros((x.shape[0], W2.shape[1]))
    for e in range(W1.shape[0]):
        h = silu(x @ W1[e].T) * (x @ W3[e].T)
        y += G[:, e:e + 1] * (h @ W2[e].T)
    return y
