"""The C-ABI library loads and exports every function include/*.h declares; host-side argument
validation returns its error codes before any CUDA call (no GPU needed)."""
import glob
import os
import re

import pytest

from conftest import ROOT


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                             src, flags=re.M):
            if not m.group(0).lstrip().startswith(("typedef", "#", "return")):
                names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def moe():
    import mxfp4_expert_layer_dflash_b300 as m
    if not os.path.exists(m.LIB_PATH):
        from mxfp4_expert_layer_dflash_b300 import build
        build.build()
    m.lib()
    return m


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("moe_mxfp4_forward", "moe_mxfp4_forward_ex", "mxfp4_quantize",
                 "moe_mxfp4_workspace_size", "moe_mxfp4_get_status", "moe_mxfp4_route",
                 "moe_mxfp8_quantize_rows", "moe_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(moe):
    for name in _declared_functions():
        assert hasattr(moe.lib(), name), name


def test_status_strings(moe):
    for code, name in moe.STATUS.items():
        assert moe.moe_status_string(code) == name


def test_workspace_size(moe):
    small = moe.moe_mxfp4_workspace_size(16, 256, 128, 8, 2)
    big = moe.moe_mxfp4_workspace_size(256, 6144, 2048, 384, 8)
    assert 0 < small < big
    assert moe.moe_mxfp4_workspace_size(256, 6144, 2048, 384, 8, 1) > big
    assert moe.moe_mxfp4_workspace_size(16, 250, 128, 8, 2) == 0       # H % 32
    assert moe.moe_mxfp4_workspace_size(16, 256, 112, 8, 2) == 0       # I % 32
    assert moe.moe_mxfp4_workspace_size(16, 256, 128, 8, 9) == 0       # k > E
    assert moe.moe_mxfp4_workspace_size(16, 256, 128, 8, 2, 7) == 0    # bad act mode


def _fwd(moe, **kw):
    a = dict(x=256, lg=512, w13=1024, s13=2048, w2=4096, s2=8192, T=4, H=256, I=128, E=8, k=2,
             y=16384)
    a.update(kw)
    return moe.lib().moe_mxfp4_forward(a["x"], a["lg"], a["w13"], a["s13"], a["w2"], a["s2"],
                                       a["T"], a["H"], a["I"], a["E"], a["k"], a["y"], None)


def test_host_validation_rejects_before_launch(moe):
    # fake, never-dereferenced addresses: every case fails validation on the host
    assert _fwd(moe, x=None) == -1
    assert _fwd(moe, T=-1) == -1
    assert _fwd(moe, k=0) == -1
    assert _fwd(moe, k=9) == -1
    assert _fwd(moe, k=17, E=32) == -2
    assert _fwd(moe, E=2000, k=2) == -2
    assert _fwd(moe, H=200) == -2           # widths: multiples of 32
    assert _fwd(moe, I=80) == -2
    assert _fwd(moe, w13=1032) == -3        # every pointer 16-byte aligned
    assert _fwd(moe, w2=4100) == -3
    assert _fwd(moe, x=258) == -3
    assert _fwd(moe, T=0) == 0               # no-op, nothing launched
    L = moe.lib()
    assert L.mxfp4_quantize(None, 4, 64, 256, 512, None) == -1
    assert L.mxfp4_quantize(256, 4, 48, 256, 512, None) == -2
    assert L.mxfp4_quantize(260, 4, 64, 256, 512, None) == -3
    assert L.mxfp4_quantize(256, 0, 64, 256, 512, None) == 0
    assert L.moe_mxfp8_quantize_rows(256, 3, 40, 512, 1024, None) == -2


def test_forward_ex_rejects_small_workspace(moe):
    o = moe.moe_opts(0, 0, 256 * 1024, 16, 0, None, 0)
    import ctypes
    rc = moe.lib().moe_mxfp4_forward_ex(256, 512, 1024, 2048, 4096, 8192, 4, 256, 128, 8, 2,
                                        16384, None, ctypes.byref(o))
    assert rc == -5
    o = moe.moe_opts(3, 0, None, 0, 0, None, 0)
    rc = moe.lib().moe_mxfp4_forward_ex(256, 512, 1024, 2048, 4096, 8192, 4, 256, 128, 8, 2,
                                        16384, None, ctypes.byref(o))
    assert rc == -1


def test_select_path_validates_on_host(moe):
    L = moe.lib()
    assert L.moe_mxfp4_select_path(16, 250, 128, 8, 2, 0) == -2     # H % 32
    assert L.moe_mxfp4_select_path(16, 256, 128, 8, 9, 0) == -1     # k > E
    assert L.moe_mxfp4_select_path(16, 256, 128, 8, 2, 5) == -1     # bad act mode


def test_next_rows_validate_on_host(moe):
    L = moe.lib()
    # dense projection: K % 128, N % 4, null pointers, alignment; T == 0 is a no-op
    assert L.moe_fp8_dense_forward(256, 512, 1024, 4, 200, 64, 2048, None) == -2
    assert L.moe_fp8_dense_forward(256, 512, 1024, 4, 256, 66, 2048, None) == -2
    assert L.moe_fp8_dense_forward(None, 512, 1024, 4, 256, 64, 2048, None) == -1
    assert L.moe_fp8_dense_forward(256, 520, 1024, 4, 256, 64, 2048, None) == -3
    assert L.moe_fp8_dense_forward(256, 512, 1024, 0, 256, 64, 2048, None) == 0
    # router: shapes as the layer
    assert L.moe_router_topk(256, 512, 4, 250, 8, 2, None, 1024, 2048, None) == -2
    assert L.moe_router_topk(256, 512, 4, 160, 8, 2, None, 1024, 2048, None) == -2  # K tiles
    assert L.moe_router_topk(256, 512, 4, 256, 8, 9, None, 1024, 2048, None) == -1
    assert L.moe_router_topk(256, None, 4, 256, 8, 2, None, 1024, 2048, None) == -1
    assert L.moe_router_topk(256, 512, 0, 256, 8, 2, None, 1024, 2048, None) == 0
    assert L.mxfp8_quantize(256, 4, 48, 512, 1024, None) == -2
    assert L.mxfp8_quantize(256, 0, 64, 512, 1024, None) == 0
    # routed layer: router weights required; workspace larger than the unrouted one
    o = moe.moe_opts(0, 0, None, 0, 0, None, 0)
    import ctypes
    assert L.moe_mxfp4_forward_routed(256, None, 1024, 2048, 4096, 8192, 4, 256, 128, 8, 2,
                                      16384, None, ctypes.byref(o)) == -1
    assert (moe.moe_mxfp4_workspace_size_routed(256, 6144, 2048, 384, 8)
            > moe.moe_mxfp4_workspace_size(256, 6144, 2048, 384, 8))


def test_verify_validates_on_host(moe):
    L = moe.lib()
    a = [256, 512, 768, 1024, 1280]
    assert L.moe_verify_block(*a, 4, 0, 100, 1536, 1792, None) == -1       # g < 1
    assert L.moe_verify_block(*a, 4, 65, 100, 1536, 1792, None) == -1      # g > 64
    assert L.moe_verify_block(*a, 4, 7, 0, 1536, 1792, None) == -1         # V < 1
    assert L.moe_verify_block(256, 512, 768, 1024, 1284, 4, 7, 100, 1536, 1792, None) == -3
    assert L.moe_verify_block(*a, 0, 7, 100, 1536, 1792, None) == 0        # S = 0: no-op
    assert L.moe_verify_block(None, 512, 768, 1024, 1280, 4, 7, 100, 1536, 1792, None) == -1


def _chain(moe, n=2, layer_ptrs=None, **kw):
    """moe_mxfp4_forward_chain with fake, never-dereferenced addresses"""
    import ctypes
    a = dict(x=256, T=4, H=256, I=128, E=8, k=2, residual=0, y=16384, opts=None)
    a.update(kw)
    base = layer_ptrs or [(512, 1024, 2048, 4096, 8192)] * n
    arrs = [(ctypes.c_void_p * max(n, 1))(*[p[i] for p in base]) for i in range(5)]
    return moe.lib().moe_mxfp4_forward_chain(n, a["x"], *arrs, a["T"], a["H"], a["I"], a["E"],
                                             a["k"], a["residual"], a["y"], None, a["opts"])


def test_chain_validates_on_host(moe):
    ok = (512, 1024, 2048, 4096, 8192)
    assert _chain(moe, n=0) == -1
    assert _chain(moe, n=moe.MOE_MAX_CHAIN + 1) == -1
    assert _chain(moe, residual=2) == -1
    assert _chain(moe, layer_ptrs=[ok, (512, None, 2048, 4096, 8192)]) == -1
    assert _chain(moe, layer_ptrs=[ok, (512, 1040, 2048, 4096, 8192)]) == -3   # fp4 alignment
    assert _chain(moe, layer_ptrs=[ok, (520, 1024, 2048, 4096, 8192)]) == -3   # logits
    assert _chain(moe, H=200) == -2
    assert _chain(moe, k=9) == -1
    assert _chain(moe, y=16386) == -3
    assert _chain(moe, T=0) == 0                 # no-op, nothing launched
    import ctypes
    o = moe.moe_opts(0, 0, 256 * 1024, 16, 0, None, 0)
    assert _chain(moe, opts=ctypes.byref(o)) == -5   # workspace too small
    o = moe.moe_opts(4, 0, None, 0, 0, None, 0)
    assert _chain(moe, opts=ctypes.byref(o)) == -1   # bad act mode


def test_chain_workspace_size(moe):
    one = moe.moe_mxfp4_workspace_size(16, 256, 128, 8, 2)
    c1 = moe.moe_mxfp4_workspace_size_chain(1, 16, 256, 128, 8, 2)
    c4 = moe.moe_mxfp4_workspace_size_chain(4, 16, 256, 128, 8, 2)
    assert one < c1 < c4                          # residual buffers; a routing block per layer
    assert moe.moe_mxfp4_workspace_size_chain(0, 16, 256, 128, 8, 2) == 0
    assert moe.moe_mxfp4_workspace_size_chain(2, 16, 250, 128, 8, 2) == 0
    assert moe.moe_mxfp4_workspace_size_chain(2, 16, 160, 128, 8, 2) == 0   # no padded chains
    assert moe.moe_mxfp4_workspace_size_chain(2, 16, 256, 128, 8, 2, 9) == 0


def _regions(lay, T, H, I, E, k, act):
    """(name, offset, bytes) of every array a layout names"""
    ab = 2 if act == 1 else 1
    return [("topk_idx", lay.topk_idx, T * k * 4), ("topk_w", lay.topk_w, T * k * 4),
            ("cnt", lay.cnt, E * 4), ("off", lay.off, (E + 1) * 4),
            ("perm", lay.perm, T * k * 4), ("pos", lay.pos, T * k * 4),
            ("xq", lay.xq, T * k * H * ab), ("xs", lay.xs, T * k * H // 32),
            ("hq", lay.hq, T * k * I * ab), ("hs", lay.hs, T * k * I // 32),
            ("yp", lay.yp, T * k * H * 4)]


@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("T,H,I,E,k", [(16, 256, 128, 8, 2), (8, 6144, 2048, 384, 8),
                                       (1, 128, 128, 1, 1)])
def test_workspace_layout_is_disjoint_and_aligned(moe, T, H, I, E, k, act):
    lay = moe.moe_mxfp4_workspace_layout(T, H, I, E, k, act)
    assert lay.total == moe.moe_mxfp4_workspace_size(T, H, I, E, k, act)
    assert lay.x_stream[0] == lay.x_stream[1] == 2**64 - 1     # SIZE_MAX: single layer
    assert lay.logits == 2**64 - 1                             # no router in this layout
    rl = moe.moe_mxfp4_workspace_layout_routed(T, H, I, E, k, act)
    assert rl.total == moe.moe_mxfp4_workspace_size_routed(T, H, I, E, k, act)
    assert rl.logits % 256 == 0 and rl.logits + T * E * 4 <= rl.total
    for n, o, b in _regions(rl, T, H, I, E, k, act):
        assert o + b <= rl.logits or rl.logits + T * E * 4 <= o, n
    regs = sorted(_regions(lay, T, H, I, E, k, act), key=lambda r: r[1])
    for (n0, o0, b0), (n1, o1, b1) in zip(regs, regs[1:]):
        assert o0 + b0 <= o1, (n0, n1)
    for n, o, b in regs:
        assert o % 256 == 0 and o + b <= lay.total, n


def test_chain_workspace_layout(moe):
    n, T, H, I, E, k = 3, 8, 256, 128, 8, 2
    lays = [moe.moe_mxfp4_workspace_layout_chain(n, l, T, H, I, E, k) for l in range(n)]
    total = moe.moe_mxfp4_workspace_size_chain(n, T, H, I, E, k)
    route = ("topk_idx", "topk_w", "cnt", "off", "perm", "pos")
    for lay in lays:
        assert lay.total == total
        for name, o, b in _regions(lay, T, H, I, E, k, 0):
            assert o % 256 == 0 and o + b <= total, name
        for s in lay.x_stream:
            assert s % 256 == 0 and s + T * H * 2 <= total
    # every layer has its own routing arrays; the activation buffers are shared
    for name in route:
        assert len({getattr(l, name) for l in lays}) == n, name
    for name in ("xq", "xs", "hq", "hs", "yp"):
        assert len({getattr(l, name) for l in lays}) == 1, name
    spans = [(o, o + b) for lay in lays for nm, o, b in _regions(lay, T, H, I, E, k, 0)
             if nm in route]
    spans += [(o, o + b) for nm, o, b in _regions(lays[0], T, H, I, E, k, 0) if nm not in route]
    spans += [(s, s + T * H * 2) for s in lays[0].x_stream]
    spans.sort()
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    L = moe.lib()
    lay = moe.moe_workspace_layout()
    import ctypes
    assert L.moe_mxfp4_workspace_layout_chain(3, 3, T, H, I, E, k, 0, ctypes.byref(lay)) == -1
    assert L.moe_mxfp4_workspace_layout_chain(3, 0, T, 250, I, E, k, 0, ctypes.byref(lay)) == -2
    assert L.moe_mxfp4_workspace_layout_chain(3, 0, T, 160, I, E, k, 0, ctypes.byref(lay)) == -2
    assert L.moe_mxfp4_workspace_layout(T, H, I, E, k, 0, None) == -1


def test_noalloc_checks_arguments_before_its_scratch_limit(moe):
    """A null or misaligned pointer is reported as such even when the shape would also be
    too large for the fixed scratch array (the forward's order: arguments, then size)."""
    L = moe.lib()
    big_T = 4096                                    # far past the array at the full shape
    args = [256, 512, 1024, 2048, 4096, 8192]
    assert L.moe_mxfp4_forward_noalloc(None, *args[1:], big_T, 6144, 2048, 384, 8, 16384,
                                       None) == -1
    assert L.moe_mxfp4_forward_noalloc(*args[:2], 1032, *args[3:], big_T, 6144, 2048, 384, 8,
                                       16384, None) == -3
    assert L.moe_mxfp4_forward_noalloc(*args, big_T, 6144, 2048, 384, 8, 16384, None) == -5
    assert L.moe_mxfp4_forward_noalloc(*args, 4, 250, 128, 8, 2, 16384, None) == -2


def test_alloc_counter_is_exported(moe):
    assert moe.moe_mxfp4_alloc_count() >= 0


def test_padded_workspace_sizes(moe):
    """Widths that are multiples of 32 but not of 128 run on zero-padded copies: their scratch
    is the padded shape's layout followed by the copies of the weights, x and y."""
    T, H, I, E, k = 16, 160, 96, 8, 2
    Hp, Ip = 256, 128
    n = moe.moe_mxfp4_workspace_size(T, H, I, E, k)
    assert n == moe.moe_mxfp4_workspace_size_padded(T, H, I, E, k)
    copies = E * 2 * Ip * Hp // 2 + E * 2 * Ip * Hp // 32 + E * Hp * Ip // 2 + E * Hp * Ip // 32
    copies += 2 * T * Hp * 2
    assert n >= moe.moe_mxfp4_workspace_size(T, Hp, Ip, E, k) + copies
    nr = moe.moe_mxfp4_workspace_size_routed(T, H, I, E, k)
    assert nr == moe.moe_mxfp4_workspace_size_padded(T, H, I, E, k, routed=True)
    assert nr >= moe.moe_mxfp4_workspace_size_routed(T, Hp, Ip, E, k) + copies + E * Hp * 2
    # 16-byte aligned FP4 weights at native widths: the padded size is the larger one
    assert (moe.moe_mxfp4_workspace_size_padded(T, 256, 128, E, k)
            > moe.moe_mxfp4_workspace_size(T, 256, 128, E, k))
    assert moe.moe_mxfp4_workspace_size_padded(T, 250, 128, E, k) == 0
    assert moe.moe_mxfp4_workspace_size_padded(T, H, I, E, k, routed=2) == 0


@pytest.mark.parametrize("act", [0, 1])
def test_padded_layout_is_the_padded_shapes(moe, act):
    T, H, I, E, k = 16, 160, 96, 8, 2
    lay = moe.moe_mxfp4_workspace_layout(T, H, I, E, k, act)
    ref = moe.moe_mxfp4_workspace_layout(T, 256, 128, E, k, act)
    for name in ("topk_idx", "topk_w", "cnt", "off", "perm", "pos", "xq", "xs", "hq", "hs", "yp"):
        assert getattr(lay, name) == getattr(ref, name), name
    assert lay.total == moe.moe_mxfp4_workspace_size(T, H, I, E, k, act) > ref.total
