"""GPU parity of the chain of layers (moe_mxfp4_forward_chain) through the C ABI.

Without the residual the chain must equal successive single-layer calls bit for bit (the fused
combine + next-layer activation step keeps the unfused arithmetic and order).  With the residual
it is compared with the oracle's chain under the layer's own bars, each against the oracle mode
that applies the path's roundings: MXFP8 mode against the MXFP8-emulation oracle (rel-Frobenius
<= 1e-2, max|err| <= 4e-2 * rms), bf16 mode against the bf16-emulation oracle, which rounds h
to bf16 before GEMM2 as the mode does (rel-Frobenius <= 5e-3).  Against the exact chain those
h roundings compound over the layers and their bf16 hand-offs: the oracle's own bf16-emulation
chain already lies 4.7e-3 to 5.1e-3 from its exact chain on these cases, against 1.7e-3 for
one layer.  Those cases raise every E8M0 scale by 2 (weights x 4,
exactly) so that each layer's output is comparable to the residual stream it is added to (the
stream's rms grows from 1 to between 1.2 and 4.6 over the layers).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import mxfp4_expert_layer_dflash_b300 as moe  # noqa: E402
from gpu_util import bf16_to_f64, dev, host_bf16, max_err_over_rms, rel_fro  # noqa: E402
from synth import layers as LY  # noqa: E402

MXFP8_FRO, MXFP8_MAX, BF16_FRO = 1e-2, 4e-2, 5e-3


def _layers(T, H, I, E, k, n, seed, device_weights=True):
    Ls = [LY.Layer(f"chain{l}", H, I, E, k, T, seed + 7 * l) for l in range(n)]
    lgs = [dev(LY.host_logits(L)) for L in Ls]
    if device_weights:
        ws = [LY.device_packed_weights(L, moe.mxfp4_quantize) for L in Ls]
    else:
        from oracle import oracle as O
        ws = [tuple(dev(a) for a in LY.host_packed_weights(L, O.mxfp4_quantize)) for L in Ls]
    return Ls, lgs, ws


def _chain(x, lgs, ws, L, residual, act, path=moe.MOE_PATH_AUTO):
    y = torch.full((L.T, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_chain(x, lgs, [w[0] for w in ws], [w[1] for w in ws],
                                [w[2] for w in ws], [w[3] for w in ws], L.T, L.H, L.I, L.E, L.k,
                                y, residual=residual, act_mode=act, path=path)
    assert moe.moe_mxfp4_get_status() == 0
    return y


def _successive(x, lgs, ws, L, act, path=moe.MOE_PATH_AUTO):
    cur = x
    for lg, w in zip(lgs, ws):
        y = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
        moe.moe_mxfp4_forward_ex(cur, lg, *w, L.T, L.H, L.I, L.E, L.k, y, act_mode=act, path=path)
        assert moe.moe_mxfp4_get_status() == 0
        cur = y
    return cur


MODES = [(moe.MOE_ACT_MXFP8, moe.MOE_PATH_MULTI), (moe.MOE_ACT_MXFP8, moe.MOE_PATH_PERSISTENT),
         (moe.MOE_ACT_MXFP8, moe.MOE_PATH_GEMMS), (moe.MOE_ACT_BF16, moe.MOE_PATH_AUTO)]


@pytest.mark.parametrize("act,path", MODES)
@pytest.mark.parametrize("T,H,I,E,k,n", [(16, 256, 128, 8, 2, 3), (1, 384, 128, 4, 4, 2),
                                         (600, 256, 256, 6, 2, 2), (40, 2048, 1024, 64, 8, 4),
                                         (9, 128, 128, 1, 1, 5)])
def test_chain_without_residual_is_successive_calls(T, H, I, E, k, n, act, path):
    Ls, lgs, ws = _layers(T, H, I, E, k, n, 100 + T)
    x = dev(LY.host_x(Ls[0]))
    yc = _chain(x, lgs, ws, Ls[0], False, act, path)
    ys = _successive(x, lgs, ws, Ls[0], act, path)
    assert torch.equal(yc.view(torch.int16), ys.view(torch.int16))


@pytest.mark.parametrize("path", [moe.MOE_PATH_AUTO, moe.MOE_PATH_PERSISTENT])
def test_chain_full_shape_is_successive_calls(path):
    Ls, lgs, ws = _layers(8, 6144, 2048, 384, 8, 2, 500)
    x = dev(LY.host_x(Ls[0]))
    yc = _chain(x, lgs, ws, Ls[0], False, moe.MOE_ACT_MXFP8, path)
    ys = _successive(x, lgs, ws, Ls[0], moe.MOE_ACT_MXFP8)
    assert torch.equal(yc.view(torch.int16), ys.view(torch.int16))
    del ws
    torch.cuda.empty_cache()


@pytest.mark.parametrize("act,path", [(moe.MOE_ACT_MXFP8, moe.MOE_PATH_AUTO),
                                      (moe.MOE_ACT_MXFP8, moe.MOE_PATH_PERSISTENT),
                                      (moe.MOE_ACT_BF16, moe.MOE_PATH_AUTO)])
@pytest.mark.parametrize("T,H,I,E,k,n", [(16, 256, 128, 8, 2, 3), (5, 384, 256, 4, 2, 2)])
def test_chain_with_residual_matches_oracle(T, H, I, E, k, n, act, path):
    from oracle import oracle as O
    Ls = [LY.Layer(f"res{l}", H, I, E, k, T, 300 + l) for l in range(n)]
    xh = LY.host_x(Ls[0])
    lgh = [LY.host_logits(L) for L in Ls]
    wh = []
    for L in Ls:
        w13, s13, w2, s2 = LY.host_packed_weights(L, O.mxfp4_quantize)
        wh.append((w13, s13 + 2, w2, s2 + 2))          # every weight x 4, exactly
    y = _chain(dev(xh), [dev(a) for a in lgh], [tuple(dev(a) for a in w) for w in wh], Ls[0],
               True, act, path)
    yg = bf16_to_f64(host_bf16(y))
    mode = O.ACT_MXFP8 if act == moe.MOE_ACT_MXFP8 else O.ACT_BF16
    yref = bf16_to_f64(O.moe_chain(xh, lgh, wh, k, mode, residual=True))
    delta = yref - bf16_to_f64(xh)
    print(f"rms(x) {np.sqrt(np.mean(bf16_to_f64(xh) ** 2)):.3f} "
          f"rms(sum of layer outputs) {np.sqrt(np.mean(delta ** 2)):.3f} "
          f"fro {rel_fro(yg, yref):.2e} max/rms {max_err_over_rms(yg, yref):.2e}")
    if act == moe.MOE_ACT_MXFP8:
        assert rel_fro(yg, yref) <= MXFP8_FRO and max_err_over_rms(yg, yref) <= MXFP8_MAX
    else:
        assert rel_fro(yg, yref) <= BF16_FRO


@pytest.mark.parametrize("act", [moe.MOE_ACT_MXFP8, moe.MOE_ACT_BF16])
@pytest.mark.parametrize("T,H,I,E,k,n", [(32, 1024, 256, 40, 16, 3), (30, 6144, 128, 16, 2, 2),
                                         (7, 2048, 256, 200, 8, 3), (5, 384, 128, 600, 4, 2)])
def test_chain_small_block_routing_matches_split_kernels(T, H, I, E, k, n, act):
    """At T <= 32 the chain routes every layer, and runs layer 0's activation step, in one
    launch; MOE_DEBUG_SPLIT_ROUTING makes it use the general routing kernels instead.  Both must
    give the same routing and slot rows, so the outputs are equal bit for bit.  The residual is
    on so that x itself reaches the output too.  The shapes cover 512 assignments (T = 32,
    k = 16: no warp is free during the top-k, so all of step a4 follows the routing), a mix of
    early and late activation units (T = 30, H = 6144), and all three top-k widths (E up to
    128, up to 384, above 384)."""
    Ls, lgs, ws = _layers(T, H, I, E, k, n, 700 + T)
    x = dev(LY.host_x(Ls[0]))
    outs = []
    for flags in (0, moe.MOE_DEBUG_SPLIT_ROUTING):
        y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        moe.moe_mxfp4_forward_chain(x, lgs, [w[0] for w in ws], [w[1] for w in ws],
                                    [w[2] for w in ws], [w[3] for w in ws], T, H, I, E, k, y,
                                    residual=True, act_mode=act, debug_flags=flags)
        assert moe.moe_mxfp4_get_status() == 0
        outs.append(y)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert not torch.isnan(outs[0].float()).any()


def test_chain_residual_with_zero_weights_returns_x():
    Ls, lgs, ws = _layers(12, 256, 128, 8, 2, 3, 7)
    zero = [tuple(torch.zeros_like(a) for a in w) for w in ws]
    x = dev(LY.host_x(Ls[0]))
    for act in (moe.MOE_ACT_MXFP8, moe.MOE_ACT_BF16):
        y = _chain(x, lgs, zero, Ls[0], True, act)
        assert torch.equal(y.view(torch.int16), x.view(torch.int16))


def test_chain_output_may_alias_input():
    Ls, lgs, ws = _layers(16, 256, 128, 8, 2, 2, 11)
    x = dev(LY.host_x(Ls[0]))
    want = _chain(x, lgs, ws, Ls[0], True, moe.MOE_ACT_MXFP8)
    xa = x.clone()
    moe.moe_mxfp4_forward_chain(xa, lgs, [w[0] for w in ws], [w[1] for w in ws],
                                [w[2] for w in ws], [w[3] for w in ws], 16, 256, 128, 8, 2, xa,
                                residual=True)
    assert moe.moe_mxfp4_get_status() == 0
    assert torch.equal(xa.view(torch.int16), want.view(torch.int16))


def test_chain_with_caller_workspace_allocates_nothing():
    Ls, lgs, ws = _layers(16, 256, 128, 8, 2, 3, 13)
    x = dev(LY.host_x(Ls[0]))
    nb = moe.moe_mxfp4_workspace_size_chain(3, 16, 256, 128, 8, 2)
    wsp = torch.empty(nb, dtype=torch.uint8, device="cuda")
    y = torch.empty((16, 256), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_chain(x, lgs, [w[0] for w in ws], [w[1] for w in ws],
                                [w[2] for w in ws], [w[3] for w in ws], 16, 256, 128, 8, 2, y,
                                workspace=wsp, workspace_bytes=nb)
    assert moe.moe_mxfp4_get_status() == 0
    assert torch.equal(y.view(torch.int16),
                       _successive(x, lgs, ws, Ls[0], moe.MOE_ACT_MXFP8).view(torch.int16))


def test_chain_of_the_most_layers():
    """MOE_MAX_CHAIN layers: every layer's logits pointer travels in the routing launch's
    parameters and every routing block sits one stride further into the workspace.  Bitwise
    against successive calls; then, with zero weights in every layer but the last and the
    residual on, the block reaches the last layer unchanged, so the result depends on the last
    layer's routing block and logits: checked against the oracle's chain."""
    from oracle import oracle as O
    n = moe.MOE_MAX_CHAIN
    Ls, lgs, ws = _layers(6, 128, 128, 4, 2, n, 4000)
    x = dev(LY.host_x(Ls[0]))
    for act in (moe.MOE_ACT_MXFP8, moe.MOE_ACT_BF16):
        yc = _chain(x, lgs, ws, Ls[0], False, act)
        ys = _successive(x, lgs, ws, Ls[0], act)
        assert torch.equal(yc.view(torch.int16), ys.view(torch.int16))
    lgh = [LY.host_logits(L) for L in Ls]
    last = LY.host_packed_weights(Ls[-1], O.mxfp4_quantize)
    last = (last[0], last[1] + 2, last[2], last[3] + 2)      # x 4: comparable to the stream
    zero = tuple(np.zeros_like(a) for a in last)
    wh = [zero] * (n - 1) + [last]
    wd = [tuple(torch.zeros_like(a) for a in ws[0])] * (n - 1) + [tuple(dev(a) for a in last)]
    y = _chain(x, [dev(a) for a in lgh], wd, Ls[0], True, moe.MOE_ACT_MXFP8)
    xh = LY.host_x(Ls[0])
    yref = bf16_to_f64(O.moe_chain(xh, lgh, wh, 2, O.ACT_MXFP8, residual=True))
    yg = bf16_to_f64(host_bf16(y))
    assert float(np.abs(yref - bf16_to_f64(xh)).max()) > 0.1   # the last layer does move it
    assert rel_fro(yg, yref) <= MXFP8_FRO and max_err_over_rms(yg, yref) <= MXFP8_MAX


@pytest.mark.parametrize("T,n", [(8, 4), (40, 3), (8, 40)])
def test_chain_in_one_launch(T, n):
    """MOE_PATH_PERSISTENT runs up to 16 chained layers in one launch (after the routing of
    every layer): one launch per 16 layers plus the routing's, bit-identical to the chain of
    per-layer launches, with and without the residual stream."""
    H, I, E, k = 256, 128, 16, 4
    Ls, lgs, ws = _layers(T, H, I, E, k, n, 2600 + T + n)
    x = dev(LY.host_x(Ls[0]))
    for residual in (False, True):
        y_multi = _chain(x, lgs, ws, Ls[0], residual, moe.MOE_ACT_MXFP8, moe.MOE_PATH_MULTI)
        _chain(x, lgs, ws, Ls[0], residual, moe.MOE_ACT_MXFP8, moe.MOE_PATH_PERSISTENT)
        n0 = moe.moe_mxfp4_launch_count()
        y_one = _chain(x, lgs, ws, Ls[0], residual, moe.MOE_ACT_MXFP8, moe.MOE_PATH_PERSISTENT)
        launches = moe.moe_mxfp4_launch_count() - n0
        routing = 1 if T <= 32 else 3          # one routing launch, or two plus act1
        assert launches == routing + (n + 15) // 16
        assert torch.equal(y_one.view(torch.int16), y_multi.view(torch.int16))
        if not residual:
            ys = _successive(x, lgs, ws, Ls[0], moe.MOE_ACT_MXFP8)
            assert torch.equal(y_one.view(torch.int16), ys.view(torch.int16))


def test_chain_in_one_launch_timeout_and_recovery():
    """The chained launch's GEMM2 dependency wait forced to run out: the call reports
    MOE_ERR_DEVICE_TIMEOUT, every CTA gives up (barriers included), and the next chain on the
    same workspace is correct."""
    Ls, lgs, ws = _layers(8, 256, 128, 8, 2, 3, 2700)
    x = dev(LY.host_x(Ls[0]))
    want = _chain(x, lgs, ws, Ls[0], True, moe.MOE_ACT_MXFP8, moe.MOE_PATH_MULTI)
    y = torch.empty_like(want)
    moe.moe_mxfp4_forward_chain(x, lgs, [w[0] for w in ws], [w[1] for w in ws],
                                [w[2] for w in ws], [w[3] for w in ws], 8, 256, 128, 8, 2, y,
                                residual=True, path=moe.MOE_PATH_PERSISTENT,
                                debug_flags=moe.MOE_DEBUG_SHORT_TIMEOUT
                                | moe.MOE_DEBUG_FORCE_DEP_TIMEOUT)
    assert moe.moe_mxfp4_get_status() == moe.MOE_ERR_DEVICE_TIMEOUT
    assert moe.moe_mxfp4_get_status() == 0
    y2 = _chain(x, lgs, ws, Ls[0], True, moe.MOE_ACT_MXFP8, moe.MOE_PATH_PERSISTENT)
    assert torch.equal(y2.view(torch.int16), want.view(torch.int16))
