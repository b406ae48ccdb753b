"""Pins of the oracle's format codecs and MXFP4/MXFP8 quantizers (CPU only).

Each check compares the oracle with something other than itself: the E2M1 grid and rounding
table of the layer's MXFP4 rule (golden fixtures), exact closed forms (2^(c-127), frexp),
torch's own float8_e4m3fn and bfloat16 conversions, a hand-worked block, round trips and the
quantizer's error bound.
"""
import math
import struct

import numpy as np
import pytest
import torch

from conftest import read_golden

GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def f32(v):
    return struct.unpack("<f", struct.pack("<f", v))[0]


def test_e2m1_decode_matches_grid(oracle_mod):
    for code, val in read_golden("e2m1_grid.txt"):
        got = oracle_mod.e2m1_value(int(code))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e2m1_rounding_table(oracle_mod):
    for q, code in read_golden("e2m1_rounding.txt"):
        assert oracle_mod.e2m1_encode(float(q)) == int(code), q


def test_e2m1_encode_roundtrip_all_codes(oracle_mod):
    for c in range(16):
        assert oracle_mod.e2m1_encode(oracle_mod.e2m1_value(c)) == c


def test_e8m0_closed_form(oracle_mod):
    for c in range(255):
        assert oracle_mod.e8m0_value(c) == math.ldexp(1.0, c - 127) == 2.0 ** (c - 127)
    assert math.isnan(oracle_mod.e8m0_value(255))


def test_e4m3_decode_matches_torch(oracle_mod):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle_mod.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(got)
        else:
            assert got == ref[c], c


def test_e4m3_encode_matches_torch_in_range(oracle_mod):
    rng = np.random.default_rng(7)
    vals = list(rng.standard_normal(3000) * rng.choice([1e-3, 0.05, 1, 30, 200], 3000))
    # every midpoint between adjacent finite magnitudes (exact in fp32: 5 significant bits)
    mags = sorted({oracle_mod.e4m3_value(c) for c in range(0x7F)})
    vals += [(a + b) / 2 for a, b in zip(mags, mags[1:])]
    vals += [-(a + b) / 2 for a, b in zip(mags, mags[1:])]
    vals = [f32(v) for v in vals if abs(v) <= 448]
    ref = torch.tensor(vals, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)
    for v, r in zip(vals, ref.tolist()):
        assert oracle_mod.e4m3_encode(v) == r, v


def test_e4m3_saturates(oracle_mod):
    assert oracle_mod.e4m3_encode(449.0) == 0x7E
    assert oracle_mod.e4m3_encode(511.9) == 0x7E
    assert oracle_mod.e4m3_encode(-1e9) == 0xFE


def test_bf16_rne_matches_torch(oracle_mod):
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2**32, 4000, dtype=np.uint64).astype(np.uint32)
    bits = bits[((bits >> 23) & 0xFF) != 0xFF]          # finite only
    ties = (bits & 0xFFFF0000) | 0x8000                   # exact halfway cases
    allb = np.concatenate([bits, ties]).astype(np.uint32)
    f = allb.view(np.float32)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for v, r in zip(f.tolist(), ref.tolist()):
        assert oracle_mod.bf16_from_double(v) == r, v


def test_floor_log2_f32(oracle_mod):
    rng = np.random.default_rng(5)
    vals = np.abs(rng.standard_normal(2000).astype(np.float32)) * np.float32(1e-3)
    vals = list(vals) + [np.float32(2.0) ** -149, np.float32(3e-45), np.float32(1e-40),
                         np.float32(1.1754942e-38), np.float32(3.4e38), np.float32(1.0)]
    for v in vals:
        v = float(v)
        if v == 0:
            continue
        m, e = math.frexp(v)
        assert oracle_mod.floor_log2_f32(v) == e - 1, v


def test_mxfp4_hand_worked_block(oracle_mod):
    rows = read_golden("mxfp4_block.txt")
    scale = int(rows[0][1])
    vals = [float(r[0]) for r in rows[1:]]
    codes = [int(r[1]) for r in rows[1:]]
    w = np.zeros((1, 64), dtype=np.float32)
    w[0, :len(vals)] = vals
    fp4, sc = oracle_mod.mxfp4_quantize(w)
    assert sc[0, 0] == scale and sc[0, 1] == 0
    got = [(fp4[0, i // 2] >> (4 * (i % 2))) & 0xF for i in range(len(vals))]
    assert got == codes


@pytest.mark.parametrize("s", list(range(0, 253, 3)) + [252, 1, 2])
def test_mxfp4_roundtrip_every_code_and_scale(oracle_mod, s):
    """Blocks made of exact grid points x 2^(s-127), with amax = 6 * 2^(s-127), come back
    with scale code s and the same 16 element codes."""
    X = math.ldexp(1.0, s - 127)
    codes = np.array(list(range(16)) * 2, dtype=np.int64)
    codes[7] = 7                                        # amax = 6 X
    vals = np.array([oracle_mod.e2m1_value(c) * X for c in codes], dtype=np.float32)
    assert all(float(v) == oracle_mod.e2m1_value(c) * X for v, c in zip(vals, codes))
    fp4, sc = oracle_mod.mxfp4_quantize(vals.reshape(1, 32))
    assert sc[0, 0] == s
    got = [(fp4[0, i // 2] >> (4 * (i % 2))) & 0xF for i in range(32)]
    assert got == list(codes)


def test_mxfp4_saturation_and_clamp(oracle_mod):
    # 7X and 7.99X share the scale of 4X..8X and saturate to +-6
    X = 2.0 ** -7
    w = np.zeros((1, 32), dtype=np.float32)
    w[0, :4] = [7 * X, -7.99 * X, 4 * X, 6 * X]
    fp4, sc = oracle_mod.mxfp4_quantize(w)
    assert sc[0, 0] == 120
    assert [(fp4[0, i // 2] >> (4 * (i % 2))) & 0xF for i in range(4)] == [7, 15, 6, 7]
    # amax below 2^-125: exponent clamps at code 0 and elements use 2^-127
    w = np.zeros((1, 32), dtype=np.float32)
    w[0, 0] = np.float32(2.0 ** -130)
    w[0, 1] = np.float32(-(2.0 ** -127))
    fp4, sc = oracle_mod.mxfp4_quantize(w)
    assert sc[0, 0] == 0
    assert fp4[0, 0] == (0 | (10 << 4))          # 2^-3 -> 0 ; -1.0 -> code 10
    # all-zero block: scale code 0, codes 0
    fp4, sc = oracle_mod.mxfp4_quantize(np.zeros((2, 64), dtype=np.float32))
    assert not sc.any() and not fp4.any()


def test_mxfp4_error_bound_random(oracle_mod):
    """|dequant(q(w)) - w| <= half the grid step at |w|/X (unsaturated), and the scale puts
    amax in [4X, 8X)."""
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    w[3, 5] = 0.0
    fp4, sc = oracle_mod.mxfp4_quantize(w)
    for r in range(w.shape[0]):
        for c in range(w.shape[1]):
            X = oracle_mod.e8m0_value(int(sc[r, c // 32]))
            code = (int(fp4[r, c // 2]) >> (4 * (c % 2))) & 0xF
            q = abs(float(w[r, c])) / X
            step = 0.5 if q < 2 else (1.0 if q < 4 else 2.0)
            err = abs(oracle_mod.e2m1_value(code) - float(w[r, c]) / X)
            assert err <= step / 2 + 1e-12 or q >= 6
        for b in range(w.shape[1] // 32):
            amax = float(np.abs(w[r, b * 32:(b + 1) * 32]).max())
            X = oracle_mod.e8m0_value(int(sc[r, b]))
            assert 4 * X <= amax < 8 * X


def test_mxfp8_row_quantizer(oracle_mod):
    """Scale = 2^(floor(log2 amax) - 8); element codes equal torch's own E4M3 rounding of
    v / scale; amax == 0 gives scale code 0."""
    rng = np.random.default_rng(2)
    v = rng.standard_normal(256) * np.repeat([1.0, 1e-3, 50.0, 1e-30, 3.0, 0.0, 1.0, 7.0], 32)
    v = v.astype(np.float32).astype(np.float64)
    codes, sc = oracle_mod.mxfp8_quantize_row(v)
    for b in range(8):
        blk = v[b * 32:(b + 1) * 32]
        amax = np.abs(blk).max()
        if amax == 0:
            assert sc[b] == 0 and not (codes[b * 32:(b + 1) * 32] & 0x7F).any()
            assert ((codes[b * 32:(b + 1) * 32] >> 7) == np.signbit(blk)).all()
            continue
        e = math.frexp(amax)[1] - 1 - 8
        assert sc[b] == e + 127
        q = torch.tensor(blk / 2.0 ** e, dtype=torch.float32)   # exact: power-of-two scaling
        assert (q.abs() < 512).all()
        ref = q.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert (codes[b * 32:(b + 1) * 32] == ref).all()
