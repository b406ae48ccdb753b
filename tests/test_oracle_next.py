"""Pins of the oracle's router logits, MXFP8 weight packing and dense FP8 projection.

Each function is checked against something other than itself: numpy's fp64 matmul of
independently decoded operands (torch's bf16 / float8_e4m3fn decoders), closed forms
(one-hot rows, identity weights), exact power-of-two scaling and torch's bf16 rounding.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from synth import synth as S


def _bf16_to_f64(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()


def _e4m3_to_f64(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def _decode_mxfp8(codes, scales):
    K = codes.shape[-1]
    return _e4m3_to_f64(codes) * np.repeat(2.0 ** (scales.astype(np.float64) - 127), 32,
                                          axis=-1).reshape(codes.shape[:-1] + (K,))


# ------------------------------------------------------------------ router logits

@pytest.mark.parametrize("T,H,E", [(5, 256, 8), (16, 384, 40), (3, 2048, 64)])
def test_router_logits_equal_numpy_matmul(T, H, E):
    x, w = S.x_bf16(T + H, T, H), S.router_bf16(E + H, E, H)
    got = O.router_logits(x, w)
    ref = _bf16_to_f64(x) @ _bf16_to_f64(w).T          # [T, E]: catches a transposed W
    assert got.shape == (T, E)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_router_logits_one_hot_rows_pick_weight_columns():
    T, H, E = 6, 256, 12
    w = S.router_bf16(7, E, H)
    x = np.zeros((T, H), dtype=np.uint16)
    cols = [0, 1, 77, 128, 200, 255]
    for t, c in enumerate(cols):
        x[t, c] = 0x3F80                                  # bf16 1.0
    got = O.router_logits(x, w)
    for t, c in enumerate(cols):
        assert np.array_equal(got[t], _bf16_to_f64(w[:, c]))


# ------------------------------------------------------------------ MXFP8 weight packing

def test_mxfp8_quantize_matrix_scale_rule_and_codes():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((9, 96)) * 0.02).astype(np.float32)
    w[1] = 0.0                                            # amax 0 -> scale code 0, codes +0
    w[2, :32] = 2.0 ** -5                                 # amax an exact power of two
    w[3, :32] = np.linspace(-3e4, 3e4, 32, dtype=np.float32)  # large values
    codes, sc = O.mxfp8_quantize(w)
    for r in range(w.shape[0]):
        for b in range(3):
            blk = w[r, 32 * b:32 * b + 32].astype(np.float64)
            amax = np.abs(blk).max()
            exp = 0 if amax == 0 else int(np.floor(np.log2(amax))) - 8 + 127
            assert sc[r, b] == max(0, min(254, exp))
            q = torch.from_numpy(blk / 2.0 ** (int(sc[r, b]) - 127)).clamp(-448, 448).to(
                torch.float8_e4m3fn)
            assert np.array_equal(codes[r, 32 * b:32 * b + 32], q.view(torch.uint8).numpy())
    assert (codes[1] == 0).all() and (sc[1] == 0).all()


# ------------------------------------------------------------------ dense FP8 projection

def _dense_case(T, K, N, seed):
    x = S.x_bf16(seed, T, K)
    codes, sc = O.mxfp8_quantize(S.dense_w_f32(seed, N, K))
    return x, codes, sc


@pytest.mark.parametrize("T,K,N", [(4, 64, 48), (7, 256, 96)])
def test_dense_exact_equals_numpy_matmul(T, K, N):
    x, codes, sc = _dense_case(T, K, N, 11)
    y16, y64 = O.dense_forward(x, codes, sc, O.ACT_EXACT)
    ref = _bf16_to_f64(x) @ _decode_mxfp8(codes, sc).T    # [T, N]
    np.testing.assert_allclose(y64, ref, rtol=1e-12, atol=1e-15)
    rounded = torch.from_numpy(y64).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y16, rounded)


def test_dense_mxfp8_mode_quantizes_x_per_block():
    T, K, N = 5, 128, 40
    x, codes, sc = _dense_case(T, K, N, 12)
    _, y64 = O.dense_forward(x, codes, sc, O.ACT_MXFP8)
    xq = np.stack([_decode_mxfp8(*O.mxfp8_quantize_row(_bf16_to_f64(x[t]))) for t in range(T)])
    np.testing.assert_allclose(y64, xq @ _decode_mxfp8(codes, sc).T, rtol=1e-12, atol=1e-15)


def test_dense_identity_weights_return_x():
    T, K = 6, 64
    x = S.x_bf16(13, T, K)
    codes = np.zeros((K, K), dtype=np.uint8)
    np.fill_diagonal(codes, 0x38)                          # E4M3 1.0
    sc = np.full((K, K // 32), 127, dtype=np.uint8)
    y16, _ = O.dense_forward(x, codes, sc, O.ACT_EXACT)
    assert np.array_equal(y16, x)


def test_dense_scale_plumbing_doubles_output():
    x, codes, sc = _dense_case(3, 96, 24, 14)
    _, y = O.dense_forward(x, codes, sc, O.ACT_MXFP8)
    _, y2 = O.dense_forward(x, codes, (sc + 1).astype(np.uint8), O.ACT_MXFP8)
    assert np.array_equal(y2, 2.0 * y)


def test_dense_rejects_bad_shapes():
    with pytest.raises(ValueError):
        O.dense_forward(np.zeros((2, 40), np.uint16), np.zeros((3, 40), np.uint8),
                        np.zeros((3, 1), np.uint8))
