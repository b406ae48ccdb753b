"""GPU parity of layers whose widths the GEMMs do not take directly: H or I a multiple of 32
but not of 128, and FP4 weights that are 16- but not 32-byte aligned.  Such layers run on
zero-padded copies (H and I rounded up to 128) made in the scratch.

Bars: the same as the other layer tests (MXFP8 mode within rel-Frobenius 1e-2 and max|err| <=
4e-2 * rms of the oracle's MXFP8 emulation; bf16 mode within 5e-3 of the exact oracle), and
bit-identity with the explicitly zero-padded layer, which is what the copies claim to be.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import mxfp4_expert_layer_dflash_b300 as moe  # noqa: E402
from gpu_util import bf16_to_f64, dev, host_bf16, max_err_over_rms, rel_fro  # noqa: E402
from synth import layers as LY  # noqa: E402
from synth import synth as S  # noqa: E402

MXFP8_FRO, MXFP8_MAX, BF16_FRO = 1e-2, 4e-2, 5e-3


@pytest.fixture(scope="module")
def O():
    from oracle import oracle
    return oracle


def _r128(v):
    return (v + 127) // 128 * 128


def _case(O, T, H, I, E, k, seed):
    L = LY.Layer("padded", H, I, E, k, T, seed)
    return L, LY.host_x(L), LY.host_logits(L), LY.host_packed_weights(L, O.mxfp4_quantize)


def _forward(x, lg, w, T, H, I, E, k, **kw):
    y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_ex(x, lg, *w, T, H, I, E, k, y, **kw)
    assert moe.moe_mxfp4_get_status() == 0
    return y


def _zero_padded(x, w, H, I):
    """The layer padded by hand: H and I rounded up to 128, gate rows at [0, I) and up rows at
    [Ip, Ip + I) of each expert's w13, every added element and scale code zero."""
    Hp, Ip = _r128(H), _r128(I)
    w13, s13, w2, s2 = w
    E = w13.shape[0]
    pw13 = np.zeros((E, 2 * Ip, Hp // 2), np.uint8)
    ps13 = np.zeros((E, 2 * Ip, Hp // 32), np.uint8)
    for dst, src, c in ((pw13, w13, H // 2), (ps13, s13, H // 32)):
        dst[:, :I, :c] = src[:, :I]
        dst[:, Ip:Ip + I, :c] = src[:, I:]
    pw2 = np.zeros((E, Hp, Ip // 2), np.uint8)
    ps2 = np.zeros((E, Hp, Ip // 32), np.uint8)
    pw2[:, :H, :I // 2] = w2
    ps2[:, :H, :I // 32] = s2
    px = np.zeros((x.shape[0], Hp), np.uint16)
    px[:, :H] = x
    return px, (pw13, ps13, pw2, ps2), Hp, Ip


SHAPES = [(16, 160, 96, 8, 2), (5, 32, 32, 3, 2), (40, 288, 160, 16, 4), (8, 2080, 1056, 16, 8),
          (1, 6176, 2080, 4, 2)]


@pytest.mark.parametrize("T,H,I,E,k", SHAPES)
@pytest.mark.parametrize("act,path", [(moe.MOE_ACT_MXFP8, moe.MOE_PATH_AUTO),
                                      (moe.MOE_ACT_MXFP8, moe.MOE_PATH_MULTI),
                                      (moe.MOE_ACT_MXFP8, moe.MOE_PATH_PERSISTENT),
                                      (moe.MOE_ACT_BF16, moe.MOE_PATH_AUTO)])
def test_widths_multiple_of_32_match_oracle(O, T, H, I, E, k, act, path):
    L, x, lg, w = _case(O, T, H, I, E, k, T + H + I)
    y = _forward(dev(x), dev(lg), [dev(a) for a in w], T, H, I, E, k, act_mode=act, path=path)
    yg = bf16_to_f64(host_bf16(y))
    if act == moe.MOE_ACT_MXFP8:
        _, yref, _ = O.moe_forward(x, lg, *w, k, O.ACT_MXFP8)
        f, m = rel_fro(yg, yref), max_err_over_rms(yg, yref)
        print(f"T={T} H={H} I={I}: mxfp8 fro={f:.3e} max/rms={m:.3e}")
        assert f <= MXFP8_FRO and m <= MXFP8_MAX
    else:
        _, yref, _ = O.moe_forward(x, lg, *w, k, O.ACT_EXACT)
        f = rel_fro(yg, yref)
        print(f"T={T} H={H} I={I}: bf16 fro={f:.3e}")
        assert f <= BF16_FRO


@pytest.mark.parametrize("T,H,I,E,k", SHAPES[:4])
@pytest.mark.parametrize("act", [moe.MOE_ACT_MXFP8, moe.MOE_ACT_BF16])
def test_padded_copies_equal_the_zero_padded_layer(O, T, H, I, E, k, act):
    """The copies the library makes are the layer padded with zeros: the same bits as running
    the hand-padded layer at the padded widths."""
    L, x, lg, w = _case(O, T, H, I, E, k, 7 * T + H)
    y = _forward(dev(x), dev(lg), [dev(a) for a in w], T, H, I, E, k, act_mode=act)
    px, pw, Hp, Ip = _zero_padded(x, w, H, I)
    yp = _forward(dev(px), dev(lg), [dev(a) for a in pw], T, Hp, Ip, E, k, act_mode=act)
    assert torch.equal(y.view(torch.int16), yp[:, :H].view(torch.int16))


def _misaligned(t, offset=16):
    """a copy of t whose data starts `offset` bytes past a 256-byte boundary"""
    buf = torch.empty(t.numel() * t.element_size() + 256, dtype=torch.uint8, device=t.device)
    out = buf[offset:offset + t.numel() * t.element_size()]
    out.copy_(t.reshape(-1).view(torch.uint8))
    return out


@pytest.mark.parametrize("name", ["tiny", "mid_t8"])
def test_fp4_weights_16_byte_aligned(O, name):
    """FP4 weights only 16-byte aligned give the same bits as aligned ones, with the library's
    scratch and with a caller workspace of moe_mxfp4_workspace_size_padded bytes."""
    L = LY.LAYERS[name]
    w = [dev(a) for a in LY.host_packed_weights(L, O.mxfp4_quantize)]
    x, lg = dev(LY.host_x(L)), dev(LY.host_logits(L))
    args = (L.T, L.H, L.I, L.E, L.k)
    ya = _forward(x, lg, w, *args)
    wm = [_misaligned(w[0]), w[1], _misaligned(w[2]), w[3]]
    assert wm[0].data_ptr() % 32 == 16 and wm[2].data_ptr() % 32 == 16
    yb = _forward(x, lg, wm, *args)
    assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))
    n = moe.moe_mxfp4_workspace_size_padded(*args)
    assert n > moe.moe_mxfp4_workspace_size(*args)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    yc = _forward(x, lg, wm, *args, workspace=ws, workspace_bytes=n)
    assert torch.equal(ya.view(torch.int16), yc.view(torch.int16))
    with pytest.raises(moe.MoeError) as e:
        _forward(x, lg, wm, *args, workspace=ws, workspace_bytes=moe.moe_mxfp4_workspace_size(*args))
    assert e.value.status == moe.MOE_ERR_NO_MEMORY


def test_padded_layer_with_caller_workspace_allocates_nothing(O):
    T, H, I, E, k = 16, 160, 96, 8, 2
    L, x, lg, w = _case(O, T, H, I, E, k, 3)
    xd, lgd, wd = dev(x), dev(lg), [dev(a) for a in w]
    n = moe.moe_mxfp4_workspace_size(T, H, I, E, k)
    assert n == moe.moe_mxfp4_workspace_size_padded(T, H, I, E, k)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    before = moe.moe_mxfp4_alloc_count()
    y1 = _forward(xd, lgd, wd, T, H, I, E, k, workspace=ws, workspace_bytes=n)
    assert moe.moe_mxfp4_alloc_count() == before
    y2 = _forward(xd, lgd, wd, T, H, I, E, k)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_padded_routed_layer_matches_oracle(O):
    """The router in front of a padded layer: its weights are padded with the activations."""
    T, H, I, E, k = 8, 160, 96, 8, 2
    L, x, _, w = _case(O, T, H, I, E, k, 11)
    w_r = S.router_bf16(L.seed, E, H)
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_routed(dev(x), dev(w_r), *(dev(a) for a in w), T, H, I, E, k, y)
    assert moe.moe_mxfp4_get_status() == 0
    ref_logits = O.router_logits(x, w_r)
    tol = 64 * 2.0 ** -24 * (np.abs(bf16_to_f64(x)) @ np.abs(bf16_to_f64(w_r)).T)
    top = -np.sort(-ref_logits, axis=1)[:, :k + 1]
    sep = np.all(np.diff(-top, axis=1) > 2 * tol.max(axis=1)[:, None], axis=1)
    assert sep.sum() >= T // 2
    _, yref, _ = O.moe_forward(x, ref_logits.astype(np.float32), *w, k, O.ACT_MXFP8)
    yg = bf16_to_f64(host_bf16(y))
    assert rel_fro(yg[sep], yref[sep]) <= MXFP8_FRO
    assert max_err_over_rms(yg[sep], yref[sep]) <= MXFP8_MAX


def test_padded_noalloc_equals_forward(O):
    T, H, I, E, k = 16, 160, 96, 8, 2
    L, x, lg, w = _case(O, T, H, I, E, k, 5)
    xd, lgd, wd = dev(x), dev(lg), [dev(a) for a in w]
    y1 = _forward(xd, lgd, wd, T, H, I, E, k)
    y2 = torch.empty_like(y1)
    moe.moe_mxfp4_forward_noalloc(xd, lgd, *wd, T, H, I, E, k, y2)
    assert moe.moe_mxfp4_get_status() == 0
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
