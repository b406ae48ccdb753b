"""GPU parity: the CUDA library through its C ABI against the fp64 CPU oracle.

Bars: packed weights, MXFP8 activation codes and routing indices bit-exact; router weights
within 1e-6 relative; y in MXFP8 mode within rel-Frobenius 1e-2 and max|err| <= 4e-2 * rms of
the oracle's MXFP8-emulation output; y in bf16 mode within rel-Frobenius 5e-3 of the exact
oracle.  Full-size layers are checked on sampled tokens (and their experts' packed bytes).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import mxfp4_expert_layer_dflash_b300 as moe  # noqa: E402
from gpu_util import (bf16_to_f64, dev, device_layer, gpu_forward, host_bf16,  # noqa: E402
                      max_err_over_rms, rel_fro)
from synth import layers as LY  # noqa: E402
from synth import synth as S  # noqa: E402

MXFP8_FRO, MXFP8_MAX, BF16_FRO = 1e-2, 4e-2, 5e-3
SMALL = ["tiny", "mid_t8"]
FULL = ["full_t8", "full_t256", "full_t1024_zipf"]


@pytest.fixture(scope="module")
def O():
    from oracle import oracle
    return oracle


def _oracle_layer(O, L, experts=None):
    return LY.host_packed_weights(L, O.mxfp4_quantize, experts)


# ------------------------------------------------------------------ generator and packing

def test_device_generator_matches_host():
    n = 1 << 20
    t = torch.empty(n, dtype=torch.float32, device="cuda")
    for seed, tid, start in [(0, 2, 0), (3, 3, 123456789), (4, 2, 7 * 4096 * 6144 + 17)]:
        S.dev_fill_normal_f32(seed, tid, start, n, 0.02, t.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert (t.cpu().numpy() == S.normal_f32(seed, tid, start, n, 0.02)).all()


@pytest.mark.parametrize("name", SMALL)
def test_quantize_bytes_exact_all_experts(O, name):
    L = LY.LAYERS[name]
    d = LY.device_packed_weights(L, moe.mxfp4_quantize)
    h = _oracle_layer(O, L)
    for a, b in zip(d, h):
        assert (a.cpu().numpy() == b).all()


def test_quantize_edge_values(O):
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((64, 256)) * rng.choice([1e-30, 1e-3, 1.0, 1e30], (64, 1)))
    w = w.astype(np.float32)
    w[0] = 0.0
    w[1, :] = -0.0
    w[2, :32] = np.float32(2.0 ** -140)                   # clamped scale
    w[3, :32] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0] * 4   # ties and saturation
    w[4, :32] = np.float32(3.0e38)
    w[5, :] = np.float32(1e-45)
    fp4 = torch.empty((64, 128), dtype=torch.uint8, device="cuda")
    sc = torch.empty((64, 8), dtype=torch.uint8, device="cuda")
    moe.mxfp4_quantize(dev(w), 64, 256, fp4, sc)
    a, b = O.mxfp4_quantize(w)
    assert (fp4.cpu().numpy() == a).all() and (sc.cpu().numpy() == b).all()


# ------------------------------------------------------------------ activations and routing

@pytest.mark.parametrize("name", SMALL + FULL)
def test_mxfp8_activation_codes_exact(O, name):
    L = LY.LAYERS[name]
    x = LY.host_x(L)
    rows = min(L.T, 64)
    codes = torch.empty((rows, L.H), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, L.H // 32), dtype=torch.uint8, device="cuda")
    moe.moe_mxfp8_quantize_rows(dev(x[:rows]), rows, L.H, codes, scales)
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    for r in range(rows):
        rc, rs = O.mxfp8_quantize_row(bf16_to_f64(x[r]))
        assert (c[r] == rc).all() and (s[r] == rs).all()


def _route_gpu(lg, k):
    T, E = lg.shape
    out = [torch.empty(n, dtype=dt, device="cuda") for n, dt in
           [(T * k, torch.int32), (T * k, torch.float32), (E, torch.int32), (E + 1, torch.int32),
            (T * k, torch.int32), (T * k, torch.int32)]]
    moe.moe_mxfp4_route(dev(lg), T, E, k, *out)
    assert moe.moe_mxfp4_get_status() == 0
    return [o.cpu().numpy() for o in out]


def _check_route(O, lg, k):
    idx, w, cnt, off, perm, pos = _route_gpu(lg, k)
    ridx, rw = O.route(lg, k)
    assert (idx.reshape(ridx.shape) == ridx).all()
    np.testing.assert_allclose(w.reshape(rw.shape), rw, rtol=1e-6, atol=1e-7)
    rcnt, roff, rperm, rpos = O.route_arrays(ridx, lg.shape[1])
    assert (cnt == rcnt).all() and (off == roff).all()
    assert (perm == rperm).all() and (pos == rpos).all()


@pytest.mark.parametrize("name", SMALL + FULL)
def test_route_bit_exact(O, name):
    L = LY.LAYERS[name]
    _check_route(O, LY.host_logits(L), L.k)


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (13, 8, 8), (300, 2, 1), (1024, 1024, 16),
                                   (37, 64, 8), (5000, 384, 8), (511, 64, 8), (513, 64, 8)])
def test_route_ties_and_shapes(O, T, E, k):
    rng = np.random.default_rng(T + E)
    lg = (np.round(rng.standard_normal((T, E)) * 2) / 2).astype(np.float32)
    lg[0] = 0.25  # one row of exact ties
    _check_route(O, lg, k)


# ------------------------------------------------------------------ the layer

PATHS = [moe.MOE_PATH_MULTI, moe.MOE_PATH_PERSISTENT, moe.MOE_PATH_GEMMS]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name", SMALL)
def test_forward_mxfp8_small(O, name, path):
    L = LY.LAYERS[name]
    inp = device_layer(L)
    y = bf16_to_f64(host_bf16(gpu_forward(L, inp, path=path)))
    w = _oracle_layer(O, L)
    _, yref, _ = O.moe_forward(LY.host_x(L), LY.host_logits(L), *w, L.k, O.ACT_MXFP8)
    _, yex, _ = O.moe_forward(LY.host_x(L), LY.host_logits(L), *w, L.k, O.ACT_EXACT)
    f, m = rel_fro(y, yref), max_err_over_rms(y, yref)
    print(f"{name}: mxfp8 vs emulation fro={f:.3e} max/rms={m:.3e}; vs exact {rel_fro(y, yex):.3e}")
    assert f <= MXFP8_FRO and m <= MXFP8_MAX


@pytest.mark.parametrize("name", SMALL)
def test_forward_bf16_small(O, name):
    L = LY.LAYERS[name]
    inp = device_layer(L)
    y = bf16_to_f64(host_bf16(gpu_forward(L, inp, act_mode=moe.MOE_ACT_BF16)))
    w = _oracle_layer(O, L)
    _, yex, _ = O.moe_forward(LY.host_x(L), LY.host_logits(L), *w, L.k, O.ACT_EXACT)
    f = rel_fro(y, yex)
    print(f"{name}: bf16 vs exact fro={f:.3e}")
    assert f <= BF16_FRO


def _sample_tokens(T, n=4):
    return sorted(set([0, T - 1] + list(np.random.default_rng(T).choice(T, n, replace=False))))


@pytest.mark.parametrize("name", FULL)
def test_forward_full_size_sampled(O, name):
    L = LY.LAYERS[name]
    inp = device_layer(L)
    y = host_bf16(gpu_forward(L, inp))
    yb = host_bf16(gpu_forward(L, inp, act_mode=moe.MOE_ACT_BF16))
    x, lg = LY.host_x(L), LY.host_logits(L)
    toks = _sample_tokens(L.T)
    ridx, _ = O.route(lg[toks], L.k)
    experts = np.unique(ridx)
    w = _oracle_layer(O, L, experts)
    for e in experts[:: max(1, len(experts) // 4)]:       # packed bytes of sampled experts
        for dv, hv in zip(inp[2:], w):
            assert (dv[e].cpu().numpy() == hv[e]).all()
    _, yref, _ = O.moe_forward(x, lg, *w, L.k, O.ACT_MXFP8, tokens=toks)
    _, yex, _ = O.moe_forward(x, lg, *w, L.k, O.ACT_EXACT, tokens=toks)
    yt = bf16_to_f64(y[toks])
    f, m = rel_fro(yt, yref), max_err_over_rms(yt, yref)
    fb = rel_fro(bf16_to_f64(yb[toks]), yex)
    print(f"{name}: mxfp8 fro={f:.3e} max/rms={m:.3e}; bf16 vs exact fro={fb:.3e}")
    assert f <= MXFP8_FRO and m <= MXFP8_MAX
    assert fb <= BF16_FRO
    del inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T,E,seed", [(4096, 384, 8), (256, 1024, 9)])
def test_forward_extreme_sizes_sampled(O, T, E, seed):
    """The full per-expert shape at the edges of the supported range: 4096 tokens (32768
    assignments: the permutation's many passes, wide chunks at scale) and the largest expert
    count (E = 1024, 20 GB of packed weights).  Sampled tokens against the oracle, in both
    activation modes."""
    L = LY.Layer(f"edge_t{T}_e{E}", 6144, 2048, E, 8, T, seed)
    inp = device_layer(L)
    y = host_bf16(gpu_forward(L, inp))
    yb = host_bf16(gpu_forward(L, inp, act_mode=moe.MOE_ACT_BF16))
    x, lg = LY.host_x(L), LY.host_logits(L)
    toks = _sample_tokens(T)
    ridx, _ = O.route(lg[toks], L.k)
    w = _oracle_layer(O, L, np.unique(ridx))
    _, yref, _ = O.moe_forward(x, lg, *w, L.k, O.ACT_MXFP8, tokens=toks)
    _, yex, _ = O.moe_forward(x, lg, *w, L.k, O.ACT_EXACT, tokens=toks)
    yt = bf16_to_f64(y[toks])
    f, m = rel_fro(yt, yref), max_err_over_rms(yt, yref)
    fb = rel_fro(bf16_to_f64(yb[toks]), yex)
    print(f"T={T} E={E}: mxfp8 fro={f:.3e} max/rms={m:.3e}; bf16 vs exact fro={fb:.3e}")
    assert f <= MXFP8_FRO and m <= MXFP8_MAX
    assert fb <= BF16_FRO
    del inp
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ edge cases and invariants

def _layer_inputs(O, T, H, I, E, k, seed, logits=None):
    L = LY.Layer("edge", H, I, E, k, T, seed)
    x = LY.host_x(L)
    lg = LY.host_logits(L) if logits is None else logits
    w = _oracle_layer(O, L)
    return L, x, lg, w


@pytest.mark.parametrize("T,H,I,E,k,ties", [(1, 256, 128, 8, 2, False), (13, 128, 256, 5, 5, False),
                                            (200, 128, 128, 2, 1, False),
                                            (150, 256, 128, 4, 2, True), (7, 384, 384, 1, 1, False),
                                            (33, 512, 128, 16, 16, False),
                                            (600, 256, 128, 4, 2, False),
                                            (520, 128, 256, 3, 1, True)])
@pytest.mark.parametrize("act,path", [(moe.MOE_ACT_MXFP8, moe.MOE_PATH_MULTI),
                                      (moe.MOE_ACT_MXFP8, moe.MOE_PATH_PERSISTENT),
                                      (moe.MOE_ACT_MXFP8, moe.MOE_PATH_GEMMS),
                                      (moe.MOE_ACT_BF16, moe.MOE_PATH_AUTO)])
def test_forward_edge_shapes(O, T, H, I, E, k, ties, act, path):
    lg = np.zeros((T, E), np.float32) if ties else None   # ties: all tokens on experts 0..k-1
    L, x, lg, w = _layer_inputs(O, T, H, I, E, k, T + H, lg)
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_ex(dev(x), dev(lg), *(dev(a) for a in w), T, H, I, E, k, y,
                             act_mode=act, path=path)
    assert moe.moe_mxfp4_get_status() == 0
    yg = bf16_to_f64(host_bf16(y))
    if act == moe.MOE_ACT_MXFP8:
        _, yref, _ = O.moe_forward(x, lg, *w, k, O.ACT_MXFP8)
        assert rel_fro(yg, yref) <= MXFP8_FRO and max_err_over_rms(yg, yref) <= MXFP8_MAX
    else:
        _, yref, _ = O.moe_forward(x, lg, *w, k, O.ACT_EXACT)
        assert rel_fro(yg, yref) <= BF16_FRO


@pytest.mark.parametrize("name", SMALL + FULL)
def test_persistent_equals_multi_kernel_bitwise(name):
    """Every execution path runs the same arithmetic in the same order: the whole layer in
    one launch, both GEMMs in one launch, and one launch per step."""
    L = LY.LAYERS[name]
    inp = device_layer(L)
    ym = gpu_forward(L, inp, path=moe.MOE_PATH_MULTI)
    for path in (moe.MOE_PATH_PERSISTENT, moe.MOE_PATH_GEMMS):
        yp = gpu_forward(L, inp, path=path)
        assert torch.equal(ym.view(torch.int16), yp.view(torch.int16)), path
    del inp
    torch.cuda.empty_cache()


def test_auto_path_choice():
    """One launch for both GEMMs up to 110 GEMM work items per SM, two launches above."""
    sel = moe.moe_mxfp4_select_path
    assert sel(8, 2048, 1024, 64, 8) == moe.MOE_PATH_GEMMS           # 8 tokens, mid shape
    assert sel(32, 2048, 1024, 64, 8) == moe.MOE_PATH_GEMMS          # 32 tokens, mid shape
    assert sel(1, 6144, 2048, 384, 8) == moe.MOE_PATH_GEMMS
    assert sel(16, 256, 128, 8, 2) == moe.MOE_PATH_GEMMS
    assert sel(8, 6144, 2048, 384, 8) == moe.MOE_PATH_GEMMS          # full shape, 8 tokens
    assert sel(32, 6144, 2048, 384, 8) == moe.MOE_PATH_GEMMS         # 71 items per SM
    assert sel(64, 6144, 2048, 384, 8) == moe.MOE_PATH_GEMMS         # 108 items per SM
    assert sel(128, 6144, 2048, 384, 8) == moe.MOE_PATH_MULTI        # 112 items per SM
    assert sel(256, 6144, 2048, 384, 8) == moe.MOE_PATH_MULTI        # full shape, 256 tokens
    assert sel(1024, 6144, 2048, 384, 8) == moe.MOE_PATH_MULTI
    assert sel(8, 2048, 1024, 64, 8, moe.MOE_ACT_BF16) == moe.MOE_PATH_MULTI


def test_zero_weights_give_zero(O):
    L, x, lg, w = _layer_inputs(O, 16, 256, 128, 8, 2, 5)
    w = tuple(np.zeros_like(a) for a in w)
    y = torch.full((16, 256), 1.0, dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward(dev(x), dev(lg), *(dev(a) for a in w), 16, 256, 128, 8, 2, y)
    assert moe.moe_mxfp4_get_status() == 0
    assert (y.float() == 0).all()


def test_t_zero_is_noop():
    y = torch.full((4, 256), 3.0, dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(64, dtype=torch.uint8, device="cuda")
    moe.moe_mxfp4_forward(z, z, z, z, z, z, 0, 256, 128, 8, 2, y)
    assert (y.float() == 3.0).all()


@pytest.mark.parametrize("act", [moe.MOE_ACT_MXFP8, moe.MOE_ACT_BF16])
def test_deterministic_and_permutation_equivariant(O, act):
    L = LY.LAYERS["mid_t8"]
    L = LY.Layer("perm", L.H, L.I, L.E, L.k, 40, 9)
    inp = device_layer(L)
    y1 = gpu_forward(L, inp, act_mode=act)
    y2 = gpu_forward(L, inp, act_mode=act)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    p = torch.randperm(L.T, generator=torch.Generator().manual_seed(0)).cuda()
    yp = gpu_forward(L, (inp[0][p].contiguous(), inp[1][p].contiguous()) + inp[2:], act_mode=act)
    assert torch.equal(yp.view(torch.int16), y1[p].view(torch.int16))


@pytest.mark.parametrize("act", [moe.MOE_ACT_MXFP8, moe.MOE_ACT_BF16])
def test_power_of_two_scale_plumbing(O, act):
    L = LY.LAYERS["tiny"]
    inp = device_layer(L)
    y1 = gpu_forward(L, inp, act_mode=act).float()
    s2 = (inp[5] + 1)
    y2 = gpu_forward(L, inp[:5] + (s2,), act_mode=act).float()
    assert torch.equal(y2, 2 * y1)
    s13 = inp[3].clone()
    s13[:, L.I:] += 1
    y3 = gpu_forward(L, inp[:3] + (s13,) + inp[4:], act_mode=act).float()
    assert torch.equal(y3, 2 * y1)


# E8M0 codes across the range a quantiser of fp32 weights can emit (0..252), one per K block
EXTREME_CODES = [0, 1, 2, 3, 60, 125, 126, 127, 128, 129, 130, 131, 190, 240, 248, 252]


@pytest.mark.parametrize("act", [moe.MOE_ACT_MXFP8, moe.MOE_ACT_BF16])
def test_extreme_scale_codes(O, act):
    """Every K block of W13 gets one extreme scale code; token t has activations only in block
    t % 16, sized by 2^(124 - code) (kept >= 2^-106) so the layer stays finite.  Blocks a token
    does not touch still meet zeros: a decode that overflowed would turn them into NaN."""
    T, H, I, E, k = 32, 512, 256, 4, 2
    L, _, lg, w = _layer_inputs(O, T, H, I, E, k, 77)
    w13, s13, w2, s2 = (a.copy() for a in w)
    s13[...] = np.array(EXTREME_CODES, np.uint8)
    rng = np.random.default_rng(5)
    xf = np.zeros((T, H), np.float32)
    for t in range(T):
        j = t % 16
        xf[t, 32 * j:32 * j + 32] = rng.standard_normal(32) * 2.0 ** max(124 - EXTREME_CODES[j],
                                                                         -106)
    x = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_ex(dev(x), dev(lg), dev(w13), dev(s13), dev(w2), dev(s2), T, H, I, E, k,
                             y, act_mode=act)
    assert moe.moe_mxfp4_get_status() == 0
    yg = bf16_to_f64(host_bf16(y))
    assert np.isfinite(yg).all()
    mode = O.ACT_MXFP8 if act == moe.MOE_ACT_MXFP8 else O.ACT_EXACT
    _, yref, _ = O.moe_forward(x, lg, w13, s13, w2, s2, k, mode)
    for t in range(T):                                      # per token: magnitudes differ widely
        if act == moe.MOE_ACT_MXFP8:
            assert rel_fro(yg[t], yref[t]) <= MXFP8_FRO
            assert max_err_over_rms(yg[t], yref[t]) <= MXFP8_MAX
        else:
            assert rel_fro(yg[t], yref[t]) <= BF16_FRO


@pytest.mark.parametrize("act", [moe.MOE_ACT_MXFP8, moe.MOE_ACT_BF16])
@pytest.mark.parametrize("T,E,k,ties", [(1, 8, 2, False), (5, 64, 8, False), (8, 384, 8, False),
                                        (13, 5, 5, True), (16, 1000, 16, False),
                                        (31, 384, 8, True), (32, 1, 1, False), (32, 64, 16, False)])
def test_small_block_routing_matches_split_kernels(O, T, E, k, ties, act):
    """For T <= 32 routing and the activation step run as one kernel; with
    MOE_DEBUG_SPLIT_ROUTING they run as the three standalone kernels.  Same bits."""
    H, I = 256, 128
    L = LY.Layer("small", H, I, E, k, T, 900 + T + E)
    lg = np.zeros((T, E), np.float32) if ties else LY.host_logits(L)
    inp = (dev(LY.host_x(L)), dev(lg)) + tuple(LY.device_packed_weights(L, moe.mxfp4_quantize))
    ys = []
    for flags in (0, moe.MOE_DEBUG_SPLIT_ROUTING):
        y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        moe.moe_mxfp4_forward_ex(*inp, T, H, I, E, k, y, act_mode=act, debug_flags=flags)
        assert moe.moe_mxfp4_get_status() == 0
        ys.append(y)
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))
    if not ties and E <= 64:   # and against the oracle
        w = _oracle_layer(O, L)
        wd = tuple(dev(a) for a in w)
        y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        moe.moe_mxfp4_forward_ex(inp[0], inp[1], *wd, T, H, I, E, k, y, act_mode=act)
        yg = bf16_to_f64(host_bf16(y))
        mode = O.ACT_MXFP8 if act == moe.MOE_ACT_MXFP8 else O.ACT_EXACT
        _, yref, _ = O.moe_forward(LY.host_x(L), lg, *w, k, mode)
        assert rel_fro(yg, yref) <= (MXFP8_FRO if act == moe.MOE_ACT_MXFP8 else BF16_FRO)
