"""Pins of the oracle's layer forward (CPU only).

- k = 1, E = 1 reduces to a dense SwiGLU FFN: numpy fp64 matmuls on independently decoded
  weights.
- Tiny layers against a dense numpy form that runs every expert and gates with a one-hot
  (top-k) weight matrix built by Python's sort.
- k = E: the output is the softmax-weighted sum of every expert.
- Token permutation equivariance (exact), power-of-two scale invariance (exact doubling).
- MXFP8 emulation: act1 equals the separately quantized x; bf16 mode is close to exact.
"""
import numpy as np
import pytest
from scipy.special import softmax

import _np_ref as R


def make_layer(S, O, T, H, I, E, seed):
    x = S.x_bf16(seed, T, H)
    lg = S.logits(seed, T, E)
    w13, s13 = O.mxfp4_quantize(S.w13_f32(seed, E, I, H))
    w2, s2 = O.mxfp4_quantize(S.w2_f32(seed, E, H, I))
    return x, lg, w13, s13, w2, s2


def test_single_expert_is_dense_swiglu(synth_mod, oracle_mod):
    T, H, I = 6, 96, 64
    x, lg, w13, s13, w2, s2 = make_layer(synth_mod, oracle_mod, T, H, I, 1, 21)
    y16, y64, h = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, 1, want_h=True)
    W13 = R.dequant(w13, s13)[0]
    W2 = R.dequant(w2, s2)[0]
    xf = R.bf16_to_f64(x)
    hr = R.silu(xf @ W13[:I].T) * (xf @ W13[I:].T)
    yr = hr @ W2.T
    np.testing.assert_allclose(h[:, 0, :], hr, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(y64, yr, rtol=1e-11, atol=1e-15)


@pytest.mark.parametrize("T,H,I,E,k", [(16, 256, 128, 8, 2), (5, 64, 32, 6, 3)])
def test_tiny_layer_matches_dense_form(synth_mod, oracle_mod, T, H, I, E, k):
    x, lg, w13, s13, w2, s2 = make_layer(synth_mod, oracle_mod, T, H, I, E, T + E)
    _, y64, _ = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, k)
    G = np.zeros((T, E))
    for t in range(T):
        sel = sorted(range(E), key=lambda e: (-float(lg[t, e]), e))[:k]
        G[t, sel] = softmax(lg[t, sel].astype(np.float64))
    W13 = R.dequant(w13, s13)
    yr = R.dense_moe(R.bf16_to_f64(x), W13[:, :I], W13[:, I:], R.dequant(w2, s2), G)
    np.testing.assert_allclose(y64, yr, rtol=1e-10, atol=1e-14)


def test_k_equals_E_is_softmax_mixture(synth_mod, oracle_mod):
    T, H, I, E = 4, 64, 32, 5
    x, lg, w13, s13, w2, s2 = make_layer(synth_mod, oracle_mod, T, H, I, E, 3)
    _, y64, _ = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, E)
    G = softmax(lg.astype(np.float64), axis=1)
    W13 = R.dequant(w13, s13)
    yr = R.dense_moe(R.bf16_to_f64(x), W13[:, :I], W13[:, I:], R.dequant(w2, s2), G)
    np.testing.assert_allclose(y64, yr, rtol=1e-10, atol=1e-14)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_token_permutation_equivariance(synth_mod, oracle_mod, mode):
    T, H, I, E, k = 12, 128, 64, 8, 2
    x, lg, w13, s13, w2, s2 = make_layer(synth_mod, oracle_mod, T, H, I, E, 9)
    y16, y64, _ = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, k, mode)
    p = np.random.default_rng(0).permutation(T)
    y16p, y64p, _ = oracle_mod.moe_forward(x[p], lg[p], w13, s13, w2, s2, k, mode)
    assert (y64p == y64[p]).all() and (y16p == y16[p]).all()


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_power_of_two_scale_plumbing(synth_mod, oracle_mod, mode):
    """+1 on every w2 scale code, or on every up-half w13 scale code, doubles y exactly."""
    T, H, I, E, k = 8, 128, 64, 4, 2
    x, lg, w13, s13, w2, s2 = make_layer(synth_mod, oracle_mod, T, H, I, E, 4)
    _, y64, _ = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, k, mode)
    _, y64b, _ = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2 + 1, k, mode)
    assert (y64b == 2 * y64).all()
    s13u = s13.copy()
    s13u[:, I:] += 1
    _, y64c, _ = oracle_mod.moe_forward(x, lg, w13, s13u, w2, s2, k, mode)
    assert (y64c == 2 * y64).all()
    # the gate half is not linear (silu): its scales change y
    s13g = s13.copy()
    s13g[:, :I] += 1
    _, y64d, _ = oracle_mod.moe_forward(x, lg, w13, s13g, w2, s2, k, mode)
    assert not (y64d == 2 * y64).all()


def test_mxfp8_mode_uses_quantized_x(synth_mod, oracle_mod):
    """In MXFP8 mode with k = E = 1 and an identity-like check: the gate/up input equals the
    separately quantized x (via h for a single expert vs numpy on the dequantized x)."""
    T, H, I = 3, 64, 32
    x, lg, w13, s13, w2, s2 = make_layer(synth_mod, oracle_mod, T, H, I, 1, 8)
    _, _, h = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, 1, 1, want_h=True)
    xf = R.bf16_to_f64(x)
    xq = np.empty_like(xf)
    for t in range(T):
        codes, sc = oracle_mod.mxfp8_quantize_row(xf[t])
        xq[t] = [oracle_mod.e4m3_value(c) * 2.0 ** (int(sc[i // 32]) - 127)
                 for i, c in enumerate(codes)]
    W13 = R.dequant(w13, s13)[0]
    hr = R.silu(xq @ W13[:I].T) * (xq @ W13[I:].T)
    for t in range(T):
        codes, sc = oracle_mod.mxfp8_quantize_row(hr[t])
        hq = np.array([oracle_mod.e4m3_value(c) * 2.0 ** (int(sc[i // 32]) - 127)
                       for i, c in enumerate(codes)])
        # tiny summation-order differences may flip a rounding; compare closely
        np.testing.assert_allclose(h[t, 0], hq, rtol=0.07, atol=1e-12)
        assert np.mean(h[t, 0] == hq) > 0.95


def test_modes_are_close(synth_mod, oracle_mod):
    T, H, I, E, k = 16, 256, 128, 8, 2
    x, lg, w13, s13, w2, s2 = make_layer(synth_mod, oracle_mod, T, H, I, E, 0)
    _, ye, _ = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, k, 0)
    _, ym, _ = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, k, 1)
    _, yb, _ = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, k, 2)
    rel = lambda a: np.linalg.norm(a - ye) / np.linalg.norm(ye)
    assert rel(yb) < 5e-3
    assert 5e-3 < rel(ym) < 0.1     # two E4M3 roundings: a few percent


def test_rejects_bad_arguments(synth_mod, oracle_mod):
    x, lg, w13, s13, w2, s2 = make_layer(synth_mod, oracle_mod, 2, 64, 32, 2, 1)
    with pytest.raises(ValueError):
        oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, 3)


def test_literal_nested_loops_equal_the_oracle_bit_for_bit(synth_mod, oracle_mod):
    """The layer written out as plain Python loops over tokens, slots, rows and the reduction
    index — weights decoded from the E2M1 grid and 2^(s - 127), top-k by a linear scan (the
    first of equal logits kept), softmax of the selected logits, sums in the same index order
    — gives the oracle's fp64 output exactly (no fused multiply-adds on either side)."""
    import math
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    T, H, I, E, k = 3, 64, 32, 4, 2
    x, lg, w13, s13, w2, s2 = make_layer(synth_mod, oracle_mod, T, H, I, E, 77)
    _, y64, _ = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, k)

    def wv(fp4, sc, e, r, c):
        byte = int(fp4[e, r, c // 2])
        nib = (byte >> 4) if c % 2 else (byte & 0xF)
        mag = grid[nib & 7] * (-1.0 if nib & 8 else 1.0)
        return mag * 2.0 ** (int(sc[e, r, c // 32]) - 127)

    want = np.zeros((T, H))
    for t in range(T):
        a = [float(R.bf16_to_f64(x[t:t + 1, h:h + 1])[0, 0]) for h in range(H)]
        taken, sel = set(), []
        for _ in range(k):
            best = -1
            for e in range(E):
                if e not in taken and (best < 0 or float(lg[t, e]) > float(lg[t, best])):
                    best = e
            taken.add(best)
            sel.append(best)
        m = float(lg[t, sel[0]])
        s = 0.0
        for e in sel:
            s += math.exp(float(lg[t, e]) - m)
        g = [math.exp(float(lg[t, e]) - m) / s for e in sel]
        d = []
        for e in sel:
            hv = []
            for i in range(I):
                gate = up = 0.0
                for h in range(H):
                    gate += wv(w13, s13, e, i, h) * a[h]
                    up += wv(w13, s13, e, I + i, h) * a[h]
                hv.append(gate / (1.0 + math.exp(-gate)) * up)
            row = []
            for o in range(H):
                acc = 0.0
                for i in range(I):
                    acc += wv(w2, s2, e, o, i) * hv[i]
                row.append(acc)
            d.append(row)
        for o in range(H):
            acc = 0.0
            for j in range(k):
                acc += g[j] * d[j][o]
            want[t, o] = acc
    assert (y64 == want).all()


def test_bf16_mode_rounds_h_to_the_nearest_bf16(synth_mod, oracle_mod):
    """bf16-emulation mode (act1 the identity on the bf16 x, act2 = round h to bf16), pinned
    against numpy and torch: with one expert, the oracle's h must be bf16 values (torch's own
    bf16 cast leaves them unchanged), each within half a bf16 step of the exact fp64 h that
    numpy computes from independently decoded weights, equal to torch's rounding of that h
    almost everywhere (torch may round fp64 -> fp32 -> bf16 twice), and y must be that
    rounded h times W2 — not the exact layer's y, so a skipped act2 fails."""
    import torch
    T, H, I = 6, 96, 64
    x, lg, w13, s13, w2, s2 = make_layer(synth_mod, oracle_mod, T, H, I, 1, 31)
    _, y64, h = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, 1, 2, want_h=True)
    _, yex, _ = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, 1, 0)
    W13 = R.dequant(w13, s13)[0]
    W2 = R.dequant(w2, s2)[0]
    xf = R.bf16_to_f64(x)
    hr = R.silu(xf @ W13[:I].T) * (xf @ W13[I:].T)
    hg = h[:, 0, :]
    as_bf16 = torch.from_numpy(hg).to(torch.bfloat16).to(torch.float64).numpy()
    assert (as_bf16 == hg).all()
    step = np.ldexp(1.0, np.floor(np.log2(np.abs(hr))).astype(np.int64) - 7)
    assert (np.abs(hg - hr) <= 0.5 * step * (1 + 1e-9)).all()
    tb = torch.from_numpy(hr).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.mean(tb == hg) > 0.99
    np.testing.assert_allclose(y64, hg @ W2.T, rtol=1e-11, atol=1e-15)
    assert not np.allclose(y64, yex, rtol=1e-5, atol=0)
    # act1 is the identity: the exact layer's h equals numpy's unrounded h
    _, _, hx = oracle_mod.moe_forward(x, lg, w13, s13, w2, s2, 1, 0, want_h=True)
    np.testing.assert_allclose(hx[:, 0, :], hr, rtol=1e-12, atol=1e-15)
