"""GPU parity of the steps beside the expert layer: the router (split-K bf16 tcgen05 GEMM +
top-k), the layer with the router in front, MXFP8 weight packing and the dense MXFP8
projection, all through the C ABI against the fp64 oracle.

Bars: packed bytes bit-exact; router logits within an fp32-accumulation bound of the exact
logits; routing indices exact wherever the exact logits separate the top k + 1 by more than
that bound (elsewhere the GPU's choice must be the top k of its own logits); the projection
within one bf16 ulp of the oracle's bf16 output (rounding of an fp32 vs an fp64 sum).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import mxfp4_expert_layer_dflash_b300 as moe  # noqa: E402
from gpu_util import (bf16_to_f64, dev, device_layer, host_bf16, max_err_over_rms,  # noqa: E402
                      rel_fro)
from synth import layers as LY  # noqa: E402
from synth import synth as S  # noqa: E402


@pytest.fixture(scope="module")
def O():
    from oracle import oracle
    return oracle


def _abs_dot(x16, w16):
    """sum_h |x||w| per (t, e): scale of the fp32 accumulation error of a logit"""
    xa = np.abs(bf16_to_f64(x16))
    wa = np.abs(bf16_to_f64(w16))
    return xa @ wa.T


def _router_case(T, H, E, seed):
    return S.x_bf16(seed, T, H), S.router_bf16(seed, E, H)


def _gpu_router(x, w, T, H, E, k):
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    moe.moe_router_topk(dev(x), dev(w), T, H, E, k, idx, gate, logits_out=logits)
    assert moe.moe_mxfp4_get_status() == 0
    return idx.cpu().numpy(), gate.cpu().numpy(), logits.cpu().numpy()


def _separated(ref, k, tol):
    """tokens whose exact top k+1 logits are pairwise more than 2*tol apart"""
    top = -np.sort(-ref, axis=1)[:, :k + 1]
    return np.all(np.diff(-top, axis=1) > 2 * tol[:, None], axis=1)


@pytest.mark.parametrize("T,H,E,k", [(16, 256, 8, 2), (8, 2048, 64, 8), (256, 6144, 384, 8),
                                     (300, 512, 40, 4), (1, 6144, 384, 8), (1024, 1024, 130, 6)])
def test_router_topk_matches_oracle(O, T, H, E, k):
    x, w = _router_case(T, H, E, T + E)
    idx, gate, logits = _gpu_router(x, w, T, H, E, k)
    ref = O.router_logits(x, w)
    tol = 64 * 2.0 ** -24 * _abs_dot(x, w)            # fp32 accumulation of H products
    assert (np.abs(logits - ref) <= tol).all(), float(np.abs(logits - ref).max())
    tol_t = tol.max(axis=1)
    sep = _separated(ref, k, tol_t)
    ridx, rgate = O.route(ref.astype(np.float32), k)
    assert (idx[sep] == ridx[sep]).all()
    np.testing.assert_allclose(gate[sep], rgate[sep], rtol=1e-5, atol=1e-6)
    # every token: the GPU's choice is the top k of its own logits (ties: lower index)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        assert list(idx[t]) == order
    print(f"T={T} H={H} E={E}: {int(sep.sum())}/{T} tokens separated; "
          f"max |logit err| {float(np.abs(logits - ref).max()):.2e}")


def test_router_deterministic():
    T, H, E, k = 256, 6144, 384, 8
    x, w = _router_case(T, H, E, 5)
    a = _gpu_router(x, w, T, H, E, k)
    b = _gpu_router(x, w, T, H, E, k)
    assert all(np.array_equal(u, v) for u, v in zip(a, b))


@pytest.mark.parametrize("name", ["tiny", "mid_t8"])
def test_routed_layer_matches_oracle(O, name):
    L = LY.LAYERS[name]
    inp = device_layer(L)
    x = LY.host_x(L)
    w_r = S.router_bf16(L.seed, L.E, L.H)
    y = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_routed(inp[0], dev(w_r), *inp[2:], L.T, L.H, L.I, L.E, L.k, y)
    assert moe.moe_mxfp4_get_status() == 0
    ref_logits = O.router_logits(x, w_r)
    sep = _separated(ref_logits, L.k, (64 * 2.0 ** -24 * _abs_dot(x, w_r)).max(axis=1))
    w = LY.host_packed_weights(L, O.mxfp4_quantize)
    _, yref, _ = O.moe_forward(x, ref_logits.astype(np.float32), *w, L.k, O.ACT_MXFP8)
    yg = bf16_to_f64(host_bf16(y))
    assert sep.sum() >= L.T // 2
    f, m = rel_fro(yg[sep], yref[sep]), max_err_over_rms(yg[sep], yref[sep])
    print(f"{name}: routed layer vs oracle on {int(sep.sum())}/{L.T} tokens fro={f:.3e} max/rms={m:.3e}")
    assert f <= 1e-2 and m <= 4e-2


@pytest.mark.parametrize("L", [LY.LAYERS["full_t8"], LY.Layer("routed_t64", 2048, 1024, 64, 8, 64, 7),
                               LY.Layer("routed_t256", 6144, 2048, 384, 8, 256, 3)],
                         ids=["full_t8", "mid_t64", "full_t256"])
def test_routed_layer_equals_layer_on_its_logits(L):
    """The fused router changes nothing but where the logits come from: the layer fed the
    router's own fp32 logits gives the same bits (above 32 tokens the router's last kernel
    also takes the top-k the layer would)."""
    inp = device_layer(L)
    w_r = dev(S.router_bf16(L.seed, L.E, L.H))
    idx = torch.empty((L.T, L.k), dtype=torch.int32, device="cuda")
    gate = torch.empty((L.T, L.k), dtype=torch.float32, device="cuda")
    logits = torch.empty((L.T, L.E), dtype=torch.float32, device="cuda")
    moe.moe_router_topk(inp[0], w_r, L.T, L.H, L.E, L.k, idx, gate, logits_out=logits)
    y1 = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty_like(y1)
    moe.moe_mxfp4_forward_routed(inp[0], w_r, *inp[2:], L.T, L.H, L.I, L.E, L.k, y1)
    moe.moe_mxfp4_forward(inp[0], logits, *inp[2:], L.T, L.H, L.I, L.E, L.k, y2)
    assert moe.moe_mxfp4_get_status() == 0
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    del inp
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ dense MXFP8 projection

def test_mxfp8_quantize_bytes_exact(O):
    w = S.dense_w_f32(21, 96, 384)
    w[3] = 0.0
    w[5, :64] = 1e4
    codes = torch.empty((96, 384), dtype=torch.uint8, device="cuda")
    sc = torch.empty((96, 12), dtype=torch.uint8, device="cuda")
    moe.mxfp8_quantize(dev(w), 96, 384, codes, sc)
    rc, rs = O.mxfp8_quantize(w)
    assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(sc.cpu().numpy(), rs)


def _ulp_distance(a16, b16):
    """distance in bf16 ulps between bit patterns (ordered-integer mapping of the sign)"""
    def key(u):
        s = u.astype(np.int32)
        return np.where(s & 0x8000, 0x8000 - (s & 0x7FFF), 0x8000 + s)
    return np.abs(key(a16) - key(b16))


def _dense_gpu(x, T, K, N, seed):
    wf = dev(S.dense_w_f32(seed, N, K))
    codes = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    sc = torch.empty((N, K // 32), dtype=torch.uint8, device="cuda")
    moe.mxfp8_quantize(wf, N, K, codes, sc)
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    moe.moe_fp8_dense_forward(dev(x), codes, sc, T, K, N, y)
    assert moe.moe_mxfp4_get_status() == 0
    return host_bf16(y), codes.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("T,K,N", [(16, 256, 384), (8, 6144, 6144), (300, 128, 96),
                                   (1, 1024, 2048), (129, 512, 260), (33, 384, 200),
                                   (32, 256, 260)])
def test_dense_projection_within_one_ulp(O, T, K, N):
    seed = T + K + N
    x = S.x_bf16(seed, T, K)
    y, codes, sc = _dense_gpu(x, T, K, N, seed)
    rc, rs = O.mxfp8_quantize(S.dense_w_f32(seed, N, K))
    assert np.array_equal(codes, rc) and np.array_equal(sc, rs)
    y16, y64 = O.dense_forward(x, rc, rs, O.ACT_MXFP8)
    d = _ulp_distance(y, y16)
    print(f"T={T} K={K} N={N}: {int((d > 0).sum())} of {d.size} outputs one ulp off")
    assert d.max() <= 1


def test_dense_projection_full_size_sampled(O):
    T, K, N = 256, 6144, 6144
    x = S.x_bf16(77, T, K)
    y, codes, sc = _dense_gpu(x, T, K, N, 77)
    toks = np.array([0, 1, 63, 64, 127, 128, 200, 255])
    rc, rs = O.mxfp8_quantize(S.dense_w_f32(77, N, K))
    assert np.array_equal(codes, rc) and np.array_equal(sc, rs)
    y16, _ = O.dense_forward(x[toks], rc, rs, O.ACT_MXFP8)     # oracle rows are independent
    assert _ulp_distance(y[toks], y16).max() <= 1


def test_dense_projection_deterministic_and_zero_rows():
    T, K, N = 64, 1024, 512
    x = S.x_bf16(5, T, K)
    x[7] = 0
    a, _, _ = _dense_gpu(x, T, K, N, 5)
    b, _, _ = _dense_gpu(x, T, K, N, 5)
    assert np.array_equal(a, b)
    assert (bf16_to_f64(a[7]) == 0).all()


@pytest.mark.parametrize("T,H,E,k", [(1, 256, 130, 3), (3, 384, 7, 2)])
def test_router_odd_expert_counts(O, T, H, E, k):
    """T*E not a multiple of 4 (the split partials are summed one by one)"""
    x, w = _router_case(T, H, E, 40 + T)
    idx, gate, logits = _gpu_router(x, w, T, H, E, k)
    ref = O.router_logits(x, w)
    tol = 64 * 2.0 ** -24 * _abs_dot(x, w)
    assert (np.abs(logits - ref) <= tol).all()
    sep = _separated(ref, k, tol.max(axis=1))
    ridx, _ = O.route(ref.astype(np.float32), k)
    assert (idx[sep] == ridx[sep]).all()
