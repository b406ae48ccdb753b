"""Python binding of libmoe_mxfp4.so: the MXFP4 MoE expert layer on B300 (sm_103a).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
Functions carry the C ABI's names (``include/moe_mxfp4.h``) and accept torch CUDA tensors (or
raw integer device addresses).  Errors raise ``MoeError``.  There is no fallback: if the
compiled library is missing, loading fails with an error.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_MXFP4_LIB selects another build of the same library (e.g. one compiled with different
# tuning knobs); by default the in-tree build is loaded
LIB_PATH = os.environ.get("MOE_MXFP4_LIB") or os.path.join(_HERE, "libmoe_mxfp4.so")

MOE_OK = 0
MOE_ACT_MXFP8, MOE_ACT_BF16 = 0, 1
MOE_PATH_AUTO, MOE_PATH_MULTI, MOE_PATH_PERSISTENT, MOE_PATH_GEMMS = 0, 1, 2, 3
MOE_DEBUG_SHORT_TIMEOUT = 1
MOE_DEBUG_FORCE_DEP_TIMEOUT = 2
MOE_DEBUG_SPLIT_ROUTING = 4
MOE_DEBUG_STALL_DECODE = 8
MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE, MOE_ERR_ALIGNMENT = -1, -2, -3
MOE_ERR_CUDA, MOE_ERR_NO_MEMORY, MOE_ERR_DEVICE_TIMEOUT = -4, -5, -6
MOE_MAX_K, MOE_MAX_E, MOE_MAX_CHAIN = 16, 1024, 256
MOE_NOALLOC_SCRATCH_BYTES = 80 * 1024 * 1024

STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED_SHAPE",
          -3: "MOE_ERR_ALIGNMENT", -4: "MOE_ERR_CUDA", -5: "MOE_ERR_NO_MEMORY",
          -6: "MOE_ERR_DEVICE_TIMEOUT", -7: "MOE_ERR_DEVICE_FAULT", -8: "MOE_ERR_NO_DEVICE"}


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status})")
        self.status = status


class moe_opts(ctypes.Structure):
    _fields_ = [("act_mode", ctypes.c_int), ("path", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("debug_flags", ctypes.c_uint32),
                ("step_events", ctypes.POINTER(ctypes.c_void_p)),
                ("n_step_events", ctypes.c_int)]


class moe_workspace_layout(ctypes.Structure):
    """Byte offsets of a forward's intermediate arrays inside a caller workspace."""
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("topk_idx", "topk_w", "cnt", "off", "perm", "pos", "xq", "xs", "hq", "hs",
                 "yp", "logits")] + [("x_stream", ctypes.c_size_t * 2),
                                     ("total", ctypes.c_size_t)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        fwd = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp, vp]
        L.moe_mxfp4_forward.argtypes = fwd
        L.moe_mxfp4_forward.restype = i
        L.moe_mxfp4_forward_ex.argtypes = fwd + [ctypes.POINTER(moe_opts)]
        L.moe_mxfp4_forward_ex.restype = i
        L.moe_mxfp4_forward_noalloc.argtypes = fwd
        L.moe_mxfp4_forward_noalloc.restype = i
        L.moe_mxfp4_forward_routed.argtypes = fwd + [ctypes.POINTER(moe_opts)]
        L.moe_mxfp4_forward_routed.restype = i
        L.moe_mxfp4_forward_chain.argtypes = [i, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp,
                                              vp, ctypes.POINTER(moe_opts)]
        L.moe_mxfp4_forward_chain.restype = i
        L.moe_mxfp4_workspace_size_chain.argtypes = [i, i, i, i, i, i, i]
        L.moe_mxfp4_workspace_size_chain.restype = sz
        L.moe_mxfp4_workspace_size_routed.argtypes = [i, i, i, i, i, i]
        L.moe_mxfp4_workspace_size_routed.restype = sz
        L.moe_mxfp4_workspace_size_padded.argtypes = [i, i, i, i, i, i, i]
        L.moe_mxfp4_workspace_size_padded.restype = sz
        L.moe_router_topk.argtypes = [vp, vp, i, i, i, i, vp, vp, vp, vp]
        L.moe_router_topk.restype = i
        L.mxfp8_quantize.argtypes = [vp, i64, i64, vp, vp, vp]
        L.mxfp8_quantize.restype = i
        L.moe_fp8_dense_forward.argtypes = [vp, vp, vp, i, i, i, vp, vp]
        L.moe_fp8_dense_forward.restype = i
        L.moe_verify_block.argtypes = [vp, vp, vp, vp, vp, i, i, i64, vp, vp, vp]
        L.moe_verify_block.restype = i
        L.moe_mxfp4_select_path.argtypes = [i, i, i, i, i, i]
        L.moe_mxfp4_select_path.restype = i
        L.moe_mxfp4_workspace_size.argtypes = [i, i, i, i, i, i]
        L.moe_mxfp4_workspace_size.restype = sz
        L.mxfp4_quantize.argtypes = [vp, i64, i64, vp, vp, vp]
        L.mxfp4_quantize.restype = i
        L.moe_mxfp4_route.argtypes = [vp, i, i, i, vp, vp, vp, vp, vp, vp, vp]
        L.moe_mxfp4_route.restype = i
        L.moe_mxfp8_quantize_rows.argtypes = [vp, i64, i64, vp, vp, vp]
        L.moe_mxfp8_quantize_rows.restype = i
        L.moe_mxfp4_get_status.argtypes = [vp]
        L.moe_mxfp4_get_status.restype = i
        L.moe_mxfp4_launch_count.argtypes = []
        L.moe_mxfp4_launch_count.restype = ctypes.c_uint64
        L.moe_mxfp4_alloc_count.argtypes = []
        L.moe_mxfp4_alloc_count.restype = ctypes.c_uint64
        L.moe_mxfp4_workspace_layout.argtypes = [i, i, i, i, i, i,
                                                 ctypes.POINTER(moe_workspace_layout)]
        L.moe_mxfp4_workspace_layout.restype = i
        L.moe_mxfp4_workspace_layout_routed.argtypes = [i, i, i, i, i, i,
                                                        ctypes.POINTER(moe_workspace_layout)]
        L.moe_mxfp4_workspace_layout_routed.restype = i
        L.moe_mxfp4_workspace_layout_chain.argtypes = [i, i, i, i, i, i, i, i,
                                                       ctypes.POINTER(moe_workspace_layout)]
        L.moe_mxfp4_workspace_layout_chain.restype = i
        L.moe_status_string.argtypes = [i]
        L.moe_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, what: str) -> int:
    if rc != MOE_OK:
        raise MoeError(rc, what)
    return rc


def moe_mxfp4_forward(x_bf16, router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, T, H, I, E, k,
                      y_bf16, stream=None):
    return _check(lib().moe_mxfp4_forward(_ptr(x_bf16), _ptr(router_logits), _ptr(w13_fp4),
                                          _ptr(w13_e8m0), _ptr(w2_fp4), _ptr(w2_e8m0), T, H, I, E,
                                          k, _ptr(y_bf16), _stream(stream)), "moe_mxfp4_forward")


def moe_mxfp4_forward_ex(x_bf16, router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, T, H, I, E,
                         k, y_bf16, stream=None, act_mode=MOE_ACT_MXFP8, path=MOE_PATH_AUTO,
                         workspace=None, workspace_bytes=0, debug_flags=0, step_events=None):
    o = moe_opts(act_mode, path, _ptr(workspace), workspace_bytes, debug_flags)
    if step_events is not None:   # a ctypes array of cudaEvent_t handles
        o.step_events = ctypes.cast(step_events, ctypes.POINTER(ctypes.c_void_p))
        o.n_step_events = len(step_events)
    return _check(lib().moe_mxfp4_forward_ex(_ptr(x_bf16), _ptr(router_logits), _ptr(w13_fp4),
                                             _ptr(w13_e8m0), _ptr(w2_fp4), _ptr(w2_e8m0), T, H, I,
                                             E, k, _ptr(y_bf16), _stream(stream),
                                             ctypes.byref(o)), "moe_mxfp4_forward_ex")


def moe_mxfp4_forward_chain(x_bf16, router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, T, H, I,
                            E, k, y_bf16, residual=False, stream=None, act_mode=MOE_ACT_MXFP8,
                            path=MOE_PATH_AUTO, workspace=None, workspace_bytes=0,
                            debug_flags=0, step_events=None):
    """Layers back to back over one token block: router_logits and the four weight arguments
    are sequences with one device tensor per layer; x_{l+1} = bf16(y_l + residual * x_l)."""
    n = len(router_logits)
    arrs = [router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0]
    if any(len(a) != n for a in arrs):
        raise ValueError("one logits tensor and one set of weights per layer")
    ptrs = [(ctypes.c_void_p * max(n, 1))(*[_ptr(t) for t in a]) for a in arrs]
    o = moe_opts(act_mode, path, _ptr(workspace), workspace_bytes, debug_flags)
    if step_events is not None:
        o.step_events = ctypes.cast(step_events, ctypes.POINTER(ctypes.c_void_p))
        o.n_step_events = len(step_events)
    return _check(lib().moe_mxfp4_forward_chain(n, _ptr(x_bf16), *ptrs, T, H, I, E, k,
                                                int(bool(residual)), _ptr(y_bf16),
                                                _stream(stream), ctypes.byref(o)),
                  "moe_mxfp4_forward_chain")


def moe_mxfp4_workspace_size_chain(n_layers, T, H, I, E, k, act_mode=MOE_ACT_MXFP8) -> int:
    return int(lib().moe_mxfp4_workspace_size_chain(n_layers, T, H, I, E, k, act_mode))


def moe_mxfp4_forward_noalloc(x_bf16, router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, T, H,
                              I, E, k, y_bf16, stream=None):
    """moe_mxfp4_forward for callers that cannot allocate: scratch lives in a fixed-size
    device array inside the library (MOE_NOALLOC_SCRATCH_BYTES)."""
    return _check(lib().moe_mxfp4_forward_noalloc(
        _ptr(x_bf16), _ptr(router_logits), _ptr(w13_fp4), _ptr(w13_e8m0), _ptr(w2_fp4),
        _ptr(w2_e8m0), T, H, I, E, k, _ptr(y_bf16), _stream(stream)), "moe_mxfp4_forward_noalloc")


def moe_mxfp4_workspace_size(T, H, I, E, k, act_mode=MOE_ACT_MXFP8) -> int:
    return int(lib().moe_mxfp4_workspace_size(T, H, I, E, k, act_mode))


def moe_mxfp4_forward_routed(x_bf16, w_router_bf16, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, T, H,
                             I, E, k, y_bf16, stream=None, act_mode=MOE_ACT_MXFP8,
                             path=MOE_PATH_AUTO, workspace=None, workspace_bytes=0,
                             debug_flags=0, step_events=None):
    """The layer with the router in front: router weights [E, H] bf16 instead of logits."""
    o = moe_opts(act_mode, path, _ptr(workspace), workspace_bytes, debug_flags)
    if step_events is not None:
        o.step_events = ctypes.cast(step_events, ctypes.POINTER(ctypes.c_void_p))
        o.n_step_events = len(step_events)
    return _check(lib().moe_mxfp4_forward_routed(
        _ptr(x_bf16), _ptr(w_router_bf16), _ptr(w13_fp4), _ptr(w13_e8m0), _ptr(w2_fp4),
        _ptr(w2_e8m0), T, H, I, E, k, _ptr(y_bf16), _stream(stream), ctypes.byref(o)),
        "moe_mxfp4_forward_routed")


def moe_mxfp4_workspace_size_routed(T, H, I, E, k, act_mode=MOE_ACT_MXFP8) -> int:
    return int(lib().moe_mxfp4_workspace_size_routed(T, H, I, E, k, act_mode))


def moe_mxfp4_workspace_size_padded(T, H, I, E, k, act_mode=MOE_ACT_MXFP8, routed=False) -> int:
    return int(lib().moe_mxfp4_workspace_size_padded(T, H, I, E, k, act_mode, int(routed)))


def moe_router_topk(x_bf16, w_router_bf16, T, H, E, k, topk_idx, topk_w, logits_out=None,
                    stream=None):
    return _check(lib().moe_router_topk(_ptr(x_bf16), _ptr(w_router_bf16), T, H, E, k,
                                        _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w),
                                        _stream(stream)), "moe_router_topk")


def mxfp8_quantize(w, rows, K, out_e4m3, out_e8m0, stream=None):
    return _check(lib().mxfp8_quantize(_ptr(w), rows, K, _ptr(out_e4m3), _ptr(out_e8m0),
                                       _stream(stream)), "mxfp8_quantize")


def moe_fp8_dense_forward(x_bf16, w_e4m3, w_e8m0, T, K, N, y_bf16, stream=None):
    return _check(lib().moe_fp8_dense_forward(_ptr(x_bf16), _ptr(w_e4m3), _ptr(w_e8m0), T, K, N,
                                              _ptr(y_bf16), _stream(stream)),
                  "moe_fp8_dense_forward")


def moe_verify_block(p, q, draft, u, U, S, g, V, n_acc, tokens, stream=None):
    """Rejection-sampling verification of a drafted block per sequence (see the header)."""
    return _check(lib().moe_verify_block(_ptr(p), _ptr(q), _ptr(draft), _ptr(u), _ptr(U), S, g,
                                         V, _ptr(n_acc), _ptr(tokens), _stream(stream)),
                  "moe_verify_block")


def moe_mxfp4_select_path(T, H, I, E, k, act_mode=MOE_ACT_MXFP8) -> int:
    """The path MOE_PATH_AUTO takes on the current device (MOE_PATH_MULTI or
    MOE_PATH_GEMMS)."""
    rc = int(lib().moe_mxfp4_select_path(T, H, I, E, k, act_mode))
    if rc < 0:
        raise MoeError(rc, "moe_mxfp4_select_path")
    return rc


def mxfp4_quantize(w, rows, K, out_fp4, out_e8m0, stream=None):
    return _check(lib().mxfp4_quantize(_ptr(w), rows, K, _ptr(out_fp4), _ptr(out_e8m0),
                                       _stream(stream)), "mxfp4_quantize")


def moe_mxfp4_route(router_logits, T, E, k, topk_idx, topk_w, cnt, off, perm, pos, stream=None):
    return _check(lib().moe_mxfp4_route(_ptr(router_logits), T, E, k, _ptr(topk_idx),
                                        _ptr(topk_w), _ptr(cnt), _ptr(off), _ptr(perm), _ptr(pos),
                                        _stream(stream)), "moe_mxfp4_route")


def moe_mxfp8_quantize_rows(x_bf16, rows, K, codes, scales, stream=None):
    return _check(lib().moe_mxfp8_quantize_rows(_ptr(x_bf16), rows, K, _ptr(codes),
                                                _ptr(scales), _stream(stream)),
                  "moe_mxfp8_quantize_rows")


def moe_mxfp4_get_status(stream=None) -> int:
    """Synchronizes the stream and returns (and clears) the device status word."""
    return int(lib().moe_mxfp4_get_status(_stream(stream)))


def moe_mxfp4_launch_count() -> int:
    return int(lib().moe_mxfp4_launch_count())


def moe_mxfp4_alloc_count() -> int:
    return int(lib().moe_mxfp4_alloc_count())


def moe_mxfp4_workspace_layout(T, H, I, E, k, act_mode=MOE_ACT_MXFP8) -> moe_workspace_layout:
    out = moe_workspace_layout()
    _check(lib().moe_mxfp4_workspace_layout(T, H, I, E, k, act_mode, ctypes.byref(out)),
           "moe_mxfp4_workspace_layout")
    return out


def moe_mxfp4_workspace_layout_routed(T, H, I, E, k, act_mode=MOE_ACT_MXFP8) -> moe_workspace_layout:
    out = moe_workspace_layout()
    _check(lib().moe_mxfp4_workspace_layout_routed(T, H, I, E, k, act_mode, ctypes.byref(out)),
           "moe_mxfp4_workspace_layout_routed")
    return out


def moe_mxfp4_workspace_layout_chain(n_layers, layer, T, H, I, E, k,
                                     act_mode=MOE_ACT_MXFP8) -> moe_workspace_layout:
    out = moe_workspace_layout()
    _check(lib().moe_mxfp4_workspace_layout_chain(n_layers, layer, T, H, I, E, k, act_mode,
                                                  ctypes.byref(out)),
           "moe_mxfp4_workspace_layout_chain")
    return out


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


# --------------------------------------------------------------- tensor-level convenience

def quantize_weights(w_f32):
    """fp32 CUDA tensor [..., K] -> (packed uint8 [..., K/2], E8M0 uint8 [..., K/32])."""
    import torch
    K = w_f32.shape[-1]
    rows = w_f32.numel() // K
    fp4 = torch.empty(w_f32.shape[:-1] + (K // 2,), dtype=torch.uint8, device=w_f32.device)
    sc = torch.empty(w_f32.shape[:-1] + (K // 32,), dtype=torch.uint8, device=w_f32.device)
    mxfp4_quantize(w_f32, rows, K, fp4, sc)
    return fp4, sc


def layer_forward(x_bf16, router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, k, y=None,
                  act_mode=MOE_ACT_MXFP8, path=MOE_PATH_AUTO, stream=None):
    """Shape-inferring wrapper of moe_mxfp4_forward_ex over torch CUDA tensors."""
    import torch
    T, H = x_bf16.shape
    E = router_logits.shape[1]
    I = w2_fp4.shape[-1] * 2
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=x_bf16.device)
    moe_mxfp4_forward_ex(x_bf16, router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, T, H, I, E, k,
                         y, stream, act_mode=act_mode, path=path)
    return y
