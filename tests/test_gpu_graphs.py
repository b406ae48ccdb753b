"""The library's calls are stream-ordered device work with no host synchronisation, so after a
first (set-up) call they can be captured in a CUDA graph; replaying the graph gives the same
bits as calling the library again."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import mxfp4_expert_layer_dflash_b300 as moe  # noqa: E402
from gpu_util import dev, device_layer  # noqa: E402
from synth import layers as LY  # noqa: E402
from synth import synth as S  # noqa: E402


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()                                  # set-up: scratch sized, tensor maps, attributes
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("name,path", [("mid_t8", moe.MOE_PATH_MULTI),
                                       ("mid_t8", moe.MOE_PATH_PERSISTENT),
                                       ("mid_t8", moe.MOE_PATH_GEMMS),
                                       ("full_e32_t64", moe.MOE_PATH_AUTO)])
def test_layer_graph_replay_is_bitwise_equal(name, path):
    L = LY.LAYERS[name]
    inp = device_layer(L)
    y_eager = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    y_graph = torch.empty_like(y_eager)
    moe.moe_mxfp4_forward_ex(*inp, L.T, L.H, L.I, L.E, L.k, y_eager, path=path)
    g = _capture(lambda: moe.moe_mxfp4_forward_ex(*inp, L.T, L.H, L.I, L.E, L.k, y_graph,
                                                  path=path))
    y_graph.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert moe.moe_mxfp4_get_status() == 0
    assert torch.equal(y_eager.view(torch.int16), y_graph.view(torch.int16))
    del inp
    torch.cuda.empty_cache()


def test_routed_layer_dense_and_verify_replay():
    L = LY.LAYERS["mid_t8"]
    inp = device_layer(L)
    w_r = dev(S.router_bf16(L.seed, L.E, L.H))
    y1 = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty_like(y1)
    moe.moe_mxfp4_forward_routed(inp[0], w_r, *inp[2:], L.T, L.H, L.I, L.E, L.k, y1)
    g = _capture(lambda: moe.moe_mxfp4_forward_routed(inp[0], w_r, *inp[2:], L.T, L.H, L.I, L.E,
                                                      L.k, y2))
    g.replay()
    T, K, N = 16, 1024, 512
    x = dev(S.x_bf16(3, T, K))
    wf = dev(S.dense_w_f32(3, N, K))
    codes = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    sc = torch.empty((N, K // 32), dtype=torch.uint8, device="cuda")
    moe.mxfp8_quantize(wf, N, K, codes, sc)
    d1 = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    d2 = torch.empty_like(d1)
    moe.moe_fp8_dense_forward(x, codes, sc, T, K, N, d1)
    gd = _capture(lambda: moe.moe_fp8_dense_forward(x, codes, sc, T, K, N, d2))
    gd.replay()
    p, q, d, u, U = S.verify_inputs(4, 8, 7, 5000)
    t = [dev(a) for a in (p, q, d, u)]
    Ut = torch.from_numpy(U.view(np.int64)).cuda()
    n1 = torch.empty(8, dtype=torch.int32, device="cuda")
    k1 = torch.empty((8, 8), dtype=torch.int32, device="cuda")
    n2, k2 = torch.empty_like(n1), torch.empty_like(k1)
    moe.moe_verify_block(*t, Ut, 8, 7, 5000, n1, k1)
    gv = _capture(lambda: moe.moe_verify_block(*t, Ut, 8, 7, 5000, n2, k2))
    gv.replay()
    torch.cuda.synchronize()
    assert moe.moe_mxfp4_get_status() == 0
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(d1.view(torch.int16), d2.view(torch.int16))
    assert torch.equal(n1, n2) and torch.equal(k1, k2)
