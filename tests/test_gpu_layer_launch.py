"""The whole layer in one persistent launch (MOE_PATH_PERSISTENT, MXFP8 mode).

For a block of T <= 32 tokens the launch routes the block (every CTA in its own shared memory),
quantises the activations, runs both GEMMs and the combine: one kernel per forward.  Above 32
tokens the routing kernels run first and the launch does the GEMMs and the combine.  Its CTAs
meet at grid-wide barriers built on scratch that need not start at zero.

Checked here, all through the C ABI:
- one launch per forward at T <= 32 (the library's launch counter), four above; one for the
  routed layer too, whose router then runs inside the launch;
- the routing arrays CTA 0 publishes and the act1 codes the CTAs write, bit for bit against the
  oracle, across top-k widths, expert counts and tie-heavy logits;
- y bit-identical to the multi-launch path (same arithmetic, same order);
- scratch holding arbitrary bytes, calls of different shapes sharing one workspace, many calls
  in a row, and CUDA-graph replays (where the host's call number is frozen) all give the same
  bits.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import mxfp4_expert_layer_dflash_b300 as moe  # noqa: E402
from gpu_util import bf16_to_f64, dev, host_bf16, max_err_over_rms, rel_fro  # noqa: E402
from synth import layers as LY  # noqa: E402
from test_gpu_routing_arrays import _check_act1, _check_routing, _ws_arrays  # noqa: E402

P, M = moe.MOE_PATH_PERSISTENT, moe.MOE_PATH_MULTI


@pytest.fixture(scope="module")
def O():
    from oracle import oracle
    return oracle


def _inputs(T, H, I, E, k, seed, ties=False):
    L = LY.Layer("ll", H, I, E, k, T, seed)
    xh = LY.host_x(L)
    lgh = LY.host_logits(L)
    if ties:
        lgh = (np.round(lgh * 2) / 2).astype(np.float32)
        lgh[T // 2] = 0.5
    w = LY.device_packed_weights(L, moe.mxfp4_quantize)
    return L, xh, lgh, (dev(xh), dev(lgh)) + tuple(w)


def _fwd(inp, L, path, ws=None, flags=0):
    y = torch.full((L.T, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    kw = {}
    if ws is not None:
        kw = dict(workspace=ws, workspace_bytes=ws.numel())
    moe.moe_mxfp4_forward_ex(*inp, L.T, L.H, L.I, L.E, L.k, y, path=path, debug_flags=flags,
                             **kw)
    assert moe.moe_mxfp4_get_status() == 0
    return y


def _eq(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("T,want", [(1, 1), (8, 1), (32, 1), (33, 4), (64, 4)])
def test_launches_per_forward(T, want):
    L, _, _, inp = _inputs(T, 256, 128, 16, 4, 40 + T)
    _fwd(inp, L, P)                                  # set-up call
    n0 = moe.moe_mxfp4_launch_count()
    _fwd(inp, L, P)
    assert moe.moe_mxfp4_launch_count() - n0 == want


@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (5, 64, 8), (8, 384, 8), (16, 1000, 16),
                                   (31, 128, 4), (32, 64, 16), (32, 1, 1), (13, 5, 5)])
def test_routing_inside_the_launch_bit_exact(O, T, E, k, ties):
    H, I = 256, 128
    L, xh, lgh, inp = _inputs(T, H, I, E, k, 2000 + T + E, ties)
    lay = moe.moe_mxfp4_workspace_layout(T, H, I, E, k)
    ws = torch.randint(0, 256, (lay.total,), dtype=torch.uint8, device="cuda")   # any bytes
    y = _fwd(inp, L, P, ws)
    a = _ws_arrays(ws, lay, T, H, I, E, k, moe.MOE_ACT_MXFP8)
    pos = _check_routing(O, a, lgh, k)
    _check_act1(O, a, xh, pos, moe.MOE_ACT_MXFP8)
    assert _eq(y, _fwd(inp, L, M))
    if not ties:
        w = LY.host_packed_weights(L, O.mxfp4_quantize)
        _, yref, _ = O.moe_forward(xh, lgh, *w, k, O.ACT_MXFP8)
        yg = bf16_to_f64(host_bf16(y))
        assert rel_fro(yg, yref) <= 1e-2 and max_err_over_rms(yg, yref) <= 4e-2


@pytest.mark.parametrize("name", ["tiny", "mid_t8", "full_t8"])
def test_configs_equal_the_multi_launch_path(name):
    L = LY.LAYERS[name]
    inp = (dev(LY.host_x(L)), dev(LY.host_logits(L))) + tuple(
        LY.device_packed_weights(L, moe.mxfp4_quantize))
    ym = _fwd(inp, L, M)
    for _ in range(3):                                # consecutive calls, one scratch
        assert _eq(_fwd(inp, L, P), ym)
    del inp
    torch.cuda.empty_cache()


def test_shapes_alternating_on_one_workspace():
    """Two shapes share one caller workspace in turn: each call's barrier words sit where the
    other shape keeps activations, so every call starts on scratch the other overwrote."""
    La, _, _, ia = _inputs(8, 512, 256, 64, 8, 77)
    Lb, _, _, ib = _inputs(24, 512, 256, 64, 8, 78)
    nb = max(moe.moe_mxfp4_workspace_size(L.T, L.H, L.I, L.E, L.k) for L in (La, Lb))
    ws = torch.randint(0, 256, (nb,), dtype=torch.uint8, device="cuda")
    ra, rb = _fwd(ia, La, M), _fwd(ib, Lb, M)
    for _ in range(3):
        assert _eq(_fwd(ia, La, P, ws), ra)
        assert _eq(_fwd(ib, Lb, P, ws), rb)


def test_graph_replays_of_the_layer_launch():
    """Replays of a captured call repeat its host-side call number; the scratch's own counter
    keeps the barriers of consecutive replays apart."""
    L, _, _, inp = _inputs(8, 1024, 512, 64, 8, 91)
    want = _fwd(inp, L, M)
    y = torch.empty_like(want)
    _fwd(inp, L, P)                                   # set-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.moe_mxfp4_forward_ex(*inp, L.T, L.H, L.I, L.E, L.k, y, path=P)
    for _ in range(5):
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert moe.moe_mxfp4_get_status() == 0
        assert _eq(y, want)


def _abs_dot(x_bits, w_bits):
    xa = np.abs(bf16_to_f64(x_bits))
    wa = np.abs(bf16_to_f64(w_bits))
    return xa @ wa.T


@pytest.mark.parametrize("T,H,E,k", [(8, 1024, 64, 8), (32, 2048, 384, 8), (3, 512, 1000, 16)])
def test_router_inside_the_layer_launch(O, T, H, E, k):
    """The routed layer on the single-launch path at T <= 32: one launch computes the logits
    (every warp one expert's row against all token rows), routes and runs the layer.  Read back
    from the workspace: the logits lie within the router's error bound of the exact ones
    (64 * 2^-24 * sum |x||w| per logit), the routing arrays are the oracle's routing of those
    logits bit for bit, and y equals the multi-launch layer fed the same logits."""
    from synth import synth as S
    I = 256
    L, xh, _, inp = _inputs(T, H, I, E, k, 95 + T)
    w_r = S.router_bf16(95 + T, E, H)
    lay = moe.moe_mxfp4_workspace_layout_routed(T, H, I, E, k)
    ws = torch.randint(0, 256, (lay.total,), dtype=torch.uint8, device="cuda")
    y1 = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_routed(inp[0], dev(w_r), *inp[2:], T, H, I, E, k, y1)   # set-up
    n0 = moe.moe_mxfp4_launch_count()
    moe.moe_mxfp4_forward_routed(inp[0], dev(w_r), *inp[2:], T, H, I, E, k, y1, path=P,
                                 workspace=ws, workspace_bytes=lay.total)
    assert moe.moe_mxfp4_get_status() == 0
    assert moe.moe_mxfp4_launch_count() - n0 == 1
    lg = ws[lay.logits:lay.logits + T * E * 4].cpu().numpy().view(np.float32).reshape(T, E)
    exact = O.router_logits(xh, w_r)
    bound = 64 * 2.0 ** -24 * _abs_dot(xh, w_r)
    assert (np.abs(lg - exact) <= bound).all()
    a = _ws_arrays(ws, lay, T, H, I, E, k, moe.MOE_ACT_MXFP8)
    pos = _check_routing(O, a, lg.copy(), k)
    _check_act1(O, a, xh, pos, moe.MOE_ACT_MXFP8)
    y2 = _fwd((inp[0], dev(lg.copy())) + inp[2:], L, M)
    assert _eq(y1, y2)
