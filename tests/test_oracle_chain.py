"""Pins of the oracle's chain of layers: x_{l+1} = bf16_RNE(y_l + r * x_l).

One layer without the residual is the layer itself; zero weights make every layer's output 0,
so the residual chain returns x and the plain chain returns zeros; and a two-layer chain of
single-expert layers (k = 1: each layer is a dense SwiGLU FFN) is recomputed here from the
format definitions with numpy and a pure-Python round-to-nearest-even, independent of the C
code.
"""
import math
import struct

import numpy as np
import pytest

from oracle import oracle as O
from synth import layers as LY

# E2M1 magnitudes of codes 0..7 (sign in bit 3): the format definition
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _decode(fp4, e8m0):
    """packed [R, K/2] + scales [R, K/32] -> fp64 [R, K]"""
    R, half = fp4.shape
    K = 2 * half
    out = np.empty((R, K))
    for r in range(R):
        for i in range(K):
            b = int(fp4[r, i // 2])
            c = (b >> 4) if i % 2 else (b & 0xF)
            v = E2M1[c & 7] * (-1.0 if c & 8 else 1.0)
            out[r, i] = v * 2.0 ** (int(e8m0[r, i // 32]) - 127)
    return out


def _bf16_rne(v: float) -> int:
    """bits of the bf16 nearest to v (ties to even), for normal magnitudes"""
    if v == 0.0:
        return 0x8000 if math.copysign(1.0, v) < 0 else 0
    m, e = math.frexp(v)                       # v = m * 2^e, 0.5 <= |m| < 1
    r = round(m * 256.0)                       # 8 significant bits; Python rounds ties to even
    val = math.ldexp(r, e - 8)                 # exact, representable in binary32
    return struct.unpack("<I", struct.pack("<f", val))[0] >> 16


def _bf16_val(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def _layer(seed, T, H, I, E, k):
    L = LY.Layer("chain", H, I, E, k, T, seed)
    return L, LY.host_logits(L), LY.host_packed_weights(L, O.mxfp4_quantize)


@pytest.mark.parametrize("mode", [O.ACT_EXACT, O.ACT_MXFP8])
def test_one_layer_without_residual_is_the_layer(mode):
    L, lg, w = _layer(3, 12, 128, 64, 6, 2)
    x = LY.host_x(L)
    y16, _, _ = O.moe_forward(x, lg, *w, L.k, mode)
    assert (O.moe_chain(x, [lg], [w], L.k, mode) == y16).all()


def test_zero_weights_return_x_with_residual_and_zero_without():
    L, lg, w = _layer(4, 7, 64, 32, 4, 2)
    x = LY.host_x(L)
    zero = tuple(np.zeros_like(a) for a in w)
    out = O.moe_chain(x, [lg, lg, lg], [zero, zero, zero], L.k, O.ACT_EXACT, residual=True)
    assert (out == x).all()
    out = O.moe_chain(x, [lg, lg], [zero, zero], L.k, O.ACT_EXACT, residual=False)
    assert (out == 0).all()


def test_two_dense_layers_with_residual_by_hand():
    T, H, I = 4, 64, 32
    layers = [_layer(10 + l, T, H, I, 1, 1) for l in range(2)]
    x = LY.host_x(layers[0][0])
    cur = [[_bf16_val(b) for b in row] for row in x]
    for _, _, (w13, s13, w2, s2) in layers:
        W13 = _decode(w13[0], s13[0])           # [2I, H]
        W2 = _decode(w2[0], s2[0])              # [H, I]
        nxt = []
        for row in cur:
            a = np.array(row)
            z = W13 @ a
            g, u = z[:I], z[I:]
            h = g / (1.0 + np.exp(-g)) * u      # silu(gate) * up
            y = W2 @ h
            nxt.append([_bf16_val(_bf16_rne(float(y[o]) + row[o])) for o in range(H)])
        cur = nxt
    want = np.array([[_bf16_rne(v) for v in row] for row in cur], dtype=np.uint16)
    got = O.moe_chain(x, [lg for _, lg, _ in layers], [w for _, _, w in layers], 1,
                      O.ACT_EXACT, residual=True)
    assert (got == want).all()


def test_chain_rejects_bad_arguments():
    L, lg, w = _layer(5, 4, 64, 32, 4, 2)
    with pytest.raises((AssertionError, ValueError)):
        O.moe_chain(LY.host_x(L), [], [], L.k)
