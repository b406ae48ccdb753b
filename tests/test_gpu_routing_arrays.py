"""The routing arrays and activation codes of the kernels the forward actually runs, read back
and compared with the oracle bit for bit.

The forward leaves its intermediate arrays in a caller workspace at the offsets
moe_mxfp4_workspace_layout names.  So these tests run the real forward (and the real chain) on
a workspace of their own and then check, against the fp64 oracle:
- step (1): topk_idx bit-exact, topk_w within 1e-6 relative (fp32 expf against fp64 exp);
- steps (2)-(4): cnt, off, perm, pos bit-exact (the oracle's stable counting sort);
- act1: xq/xs in slot order equal the oracle's MXFP8 rule applied to x[perm[slot]] (E4M3
  codes and E8M0 scales, bit-exact), or x itself in the bf16 mode;
- act2 (GEMM1's epilogue): hq/hs against the oracle's MXFP8-emulation h, where fp32 against
  fp64 accumulation may flip a rounding: codes equal on >= 98 % of the entries, values within
  rel-Frobenius 1e-2.
That covers the one-launch routing kernel of small token blocks (T <= 32), the general kernels
(T > 32, or MOE_DEBUG_SPLIT_ROUTING), the chain's routing kernels for every layer, and the
chain's fused combine + next-layer activation step.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import mxfp4_expert_layer_dflash_b300 as moe  # noqa: E402
from gpu_util import bf16_to_f64, dev, host_bf16  # noqa: E402
from synth import layers as LY  # noqa: E402


@pytest.fixture(scope="module")
def O():
    from oracle import oracle
    return oracle


def _region(ws, off, n, dtype):
    size = np.dtype(dtype).itemsize
    return ws[off:off + n * size].cpu().numpy().view(dtype)


def _ws_arrays(ws, lay, T, H, I, E, k, act):
    """the forward's arrays from workspace `ws` (a uint8 CUDA tensor) at layout `lay`"""
    TK = T * k
    a = {"idx": _region(ws, lay.topk_idx, TK, np.int32).reshape(T, k),
         "w": _region(ws, lay.topk_w, TK, np.float32).reshape(T, k),
         "cnt": _region(ws, lay.cnt, E, np.int32), "off": _region(ws, lay.off, E + 1, np.int32),
         "perm": _region(ws, lay.perm, TK, np.int32), "pos": _region(ws, lay.pos, TK, np.int32)}
    if act == moe.MOE_ACT_MXFP8:
        a["xq"] = _region(ws, lay.xq, TK * H, np.uint8).reshape(TK, H)
        a["xs"] = _region(ws, lay.xs, TK * H // 32, np.uint8).reshape(TK, H // 32)
        a["hq"] = _region(ws, lay.hq, TK * I, np.uint8).reshape(TK, I)
        a["hs"] = _region(ws, lay.hs, TK * I // 32, np.uint8).reshape(TK, I // 32)
    else:
        a["xq"] = _region(ws, lay.xq, TK * H, np.uint16).reshape(TK, H)
    return a


def _check_routing(O, a, lg, k):
    ridx, rw = O.route(lg, k)
    assert (a["idx"] == ridx).all()
    np.testing.assert_allclose(a["w"], rw, rtol=1e-6, atol=1e-7)
    rcnt, roff, rperm, rpos = O.route_arrays(ridx, lg.shape[1])
    assert (a["cnt"] == rcnt).all() and (a["off"] == roff).all()
    assert (a["perm"] == rperm).all() and (a["pos"] == rpos).all()
    return rpos.reshape(lg.shape[0], k)


def _quant_rows(O, x_bits):
    """the oracle's MXFP8 codes and scales of each bf16 row"""
    codes, scales = [], []
    for r in range(x_bits.shape[0]):
        c, s = O.mxfp8_quantize_row(bf16_to_f64(x_bits[r]))
        codes.append(c)
        scales.append(s)
    return np.stack(codes), np.stack(scales)


def _check_act1(O, a, x_bits, pos, act):
    if act == moe.MOE_ACT_MXFP8:
        codes, scales = _quant_rows(O, x_bits)
        for j in range(pos.shape[1]):
            assert (a["xq"][pos[:, j]] == codes).all()
            assert (a["xs"][pos[:, j]] == scales).all()
    else:
        for j in range(pos.shape[1]):
            assert (a["xq"][pos[:, j]] == x_bits).all()


def _e4m3_values(O, codes, scales):
    tab = np.array([O.e4m3_value(c) for c in range(256)])
    v = tab[codes.astype(np.int64)]
    s = np.repeat(2.0 ** (scales.astype(np.float64) - 127), 32, axis=1)
    return v * s


def _forward_ws(inp, L, act, flags=0, path=moe.MOE_PATH_AUTO):
    lay = moe.moe_mxfp4_workspace_layout(L.T, L.H, L.I, L.E, L.k, act)
    ws = torch.zeros(lay.total, dtype=torch.uint8, device="cuda")
    y = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_ex(*inp, L.T, L.H, L.I, L.E, L.k, y, act_mode=act, path=path,
                             workspace=ws, workspace_bytes=lay.total, debug_flags=flags)
    assert moe.moe_mxfp4_get_status() == 0
    return _ws_arrays(ws, lay, L.T, L.H, L.I, L.E, L.k, act), y


CASES = [("tiny", 0), ("tiny", moe.MOE_DEBUG_SPLIT_ROUTING), ("mid_t8", 0),
         ("mid_t8", moe.MOE_DEBUG_SPLIT_ROUTING), ("full_t8", 0), ("full_t256", 0)]


@pytest.mark.parametrize("act", [moe.MOE_ACT_MXFP8, moe.MOE_ACT_BF16])
@pytest.mark.parametrize("name,flags", CASES)
def test_forward_routing_arrays_and_act1_codes(O, name, flags, act):
    """The forward's own routing arrays and activation codes (the one-launch small-block kernel
    at T <= 32 unless MOE_DEBUG_SPLIT_ROUTING; the top-k, permutation and activation kernels
    otherwise), bit for bit against the oracle."""
    L = LY.LAYERS[name]
    x, lg = LY.host_x(L), LY.host_logits(L)
    inp = (dev(x), dev(lg)) + tuple(LY.device_packed_weights(L, moe.mxfp4_quantize))
    a, _ = _forward_ws(inp, L, act, flags)
    pos = _check_routing(O, a, lg, L.k)
    _check_act1(O, a, x, pos, act)
    del inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("path", [moe.MOE_PATH_MULTI, moe.MOE_PATH_PERSISTENT,
                                  moe.MOE_PATH_GEMMS])
@pytest.mark.parametrize("name", ["tiny", "mid_t8"])
def test_forward_act2_codes_against_emulation(O, name, path):
    """GEMM1's SwiGLU + MXFP8 epilogue output (hq/hs) against the oracle's act2(h): the same
    rule applied to an fp64 h, so codes agree except where fp32 accumulation moves a value
    across a rounding boundary."""
    L = LY.LAYERS[name]
    x, lg = LY.host_x(L), LY.host_logits(L)
    w = LY.host_packed_weights(L, O.mxfp4_quantize)
    inp = (dev(x), dev(lg)) + tuple(dev(t) for t in w)
    a, _ = _forward_ws(inp, L, moe.MOE_ACT_MXFP8, path=path)
    pos = _check_routing(O, a, lg, L.k)
    _, _, h = O.moe_forward(x, lg, *w, L.k, O.ACT_MXFP8, want_h=True)   # [T, k, I]
    got = _e4m3_values(O, a["hq"], a["hs"])
    want = h.reshape(L.T * L.k, L.I)
    g = got[pos.reshape(-1)]
    agree = float(np.mean(g == want))
    rel = float(np.linalg.norm(g - want) / np.linalg.norm(want))
    print(f"{name}: act2 codes agree on {agree:.4f}, rel-Frobenius {rel:.2e}")
    assert agree >= 0.98 and rel <= 1e-2


SMALL_T = [1, 2, 5, 8, 16, 31, 32]


@pytest.mark.parametrize("E", [1, 8, 64, 384, 1000])
def test_small_block_routing_kernel_bit_exact(O, E):
    """moe_mxfp4_route runs the forward's kernels for its T: at T <= 32 the one-launch
    small-block routing kernel.  Every T of a small block x k in {1, 2, 8, 16} (k <= E), on
    random logits and on tie-heavy ones (values on a 0.5 grid, one row all equal)."""
    rng = np.random.default_rng(E)
    for T in SMALL_T:
        for k in (1, 2, 8, 16):
            if k > E:
                continue
            for ties in (False, True):
                lg = rng.standard_normal((T, E)).astype(np.float32)
                if ties:
                    lg = (np.round(lg * 2) / 2).astype(np.float32)
                    lg[T // 2] = 0.5
                out = [torch.empty(n, dtype=dt, device="cuda") for n, dt in
                       [(T * k, torch.int32), (T * k, torch.float32), (E, torch.int32),
                        (E + 1, torch.int32), (T * k, torch.int32), (T * k, torch.int32)]]
                moe.moe_mxfp4_route(dev(lg), T, E, k, *out)
                assert moe.moe_mxfp4_get_status() == 0
                o = [t.cpu().numpy() for t in out]
                a = {"idx": o[0].reshape(T, k), "w": o[1].reshape(T, k), "cnt": o[2],
                     "off": o[3], "perm": o[4], "pos": o[5]}
                _check_routing(O, a, lg, k)


@pytest.mark.parametrize("act,path", [(moe.MOE_ACT_MXFP8, moe.MOE_PATH_AUTO),
                                      (moe.MOE_ACT_MXFP8, moe.MOE_PATH_PERSISTENT),
                                      (moe.MOE_ACT_BF16, moe.MOE_PATH_AUTO)])
@pytest.mark.parametrize("T,H,I,E,k,n,flags", [
    (8, 256, 128, 64, 8, 4, 0),                              # one launch routes every layer
    (8, 256, 128, 64, 8, 4, moe.MOE_DEBUG_SPLIT_ROUTING),    # the two general launches
    (32, 1024, 256, 1000, 16, 3, 0),                         # widest top-k, 512 assignments
    (5, 384, 128, 384, 8, 3, 0),
    (64, 256, 128, 40, 4, 3, 0),                             # T > 32: general launches
])
def test_chain_routing_arrays_bit_exact(O, T, H, I, E, k, n, flags, act, path):
    """Every layer's routing arrays of a chain, bit for bit; then the last layer's act1 rows,
    which the previous layer's combine wrote straight into its slots: with the residual on,
    the workspace keeps that layer's bf16 input, and its rows quantised by the oracle's rule
    must equal the codes at the last layer's slots."""
    Ls = [LY.Layer(f"rc{l}", H, I, E, k, T, 1300 + T + E + 11 * l) for l in range(n)]
    lgh = [LY.host_logits(L) for L in Ls]
    ws_w = [LY.device_packed_weights(L, moe.mxfp4_quantize) for L in Ls]
    x = dev(LY.host_x(Ls[0]))
    nb = moe.moe_mxfp4_workspace_size_chain(n, T, H, I, E, k, act)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_chain(x, [dev(a) for a in lgh], [w[0] for w in ws_w],
                                [w[1] for w in ws_w], [w[2] for w in ws_w], [w[3] for w in ws_w],
                                T, H, I, E, k, y, residual=True, act_mode=act, path=path,
                                workspace=ws, workspace_bytes=nb, debug_flags=flags)
    assert moe.moe_mxfp4_get_status() == 0
    pos = None
    for l in range(n):
        lay = moe.moe_mxfp4_workspace_layout_chain(n, l, T, H, I, E, k, act)
        a = _ws_arrays(ws, lay, T, H, I, E, k, act)
        pos = _check_routing(O, a, lgh[l], k)
    x_last = _region(ws, lay.x_stream[(n - 1) & 1], T * H, np.uint16).reshape(T, H)
    _check_act1(O, a, x_last, pos, act)


@pytest.mark.parametrize("act", [moe.MOE_ACT_MXFP8, moe.MOE_ACT_BF16])
@pytest.mark.parametrize("T", [8, 32, 48])
def test_chain_layer0_act1_codes(O, T, act):
    """A one-layer chain: its activation step (inside the chain's one-launch routing kernel at
    T <= 32, the activation kernel above) against the oracle's quantisation of x."""
    H, I, E, k = 512, 128, 16, 4
    L = LY.Layer("c1", H, I, E, k, T, 1500 + T)
    xh, lgh = LY.host_x(L), LY.host_logits(L)
    w = LY.device_packed_weights(L, moe.mxfp4_quantize)
    nb = moe.moe_mxfp4_workspace_size_chain(1, T, H, I, E, k, act)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_chain(dev(xh), [dev(lgh)], [w[0]], [w[1]], [w[2]], [w[3]], T, H, I, E,
                                k, y, act_mode=act, workspace=ws, workspace_bytes=nb)
    assert moe.moe_mxfp4_get_status() == 0
    lay = moe.moe_mxfp4_workspace_layout_chain(1, 0, T, H, I, E, k, act)
    a = _ws_arrays(ws, lay, T, H, I, E, k, act)
    pos = _check_routing(O, a, lgh, k)
    _check_act1(O, a, xh, pos, act)
    # and the same layer through moe_mxfp4_forward_ex gives the same y
    y1 = torch.empty_like(y)
    moe.moe_mxfp4_forward_ex(dev(xh), dev(lgh), *w, T, H, I, E, k, y1, act_mode=act)
    assert moe.moe_mxfp4_get_status() == 0
    assert torch.equal(y.view(torch.int16), y1.view(torch.int16))
    assert np.isfinite(bf16_to_f64(host_bf16(y))).all()
