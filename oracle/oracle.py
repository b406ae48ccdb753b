"""ctypes binding of the fp64 CPU oracle (``liboracle.so``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py``.  The CUDA library never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "liboracle.so")

ACT_EXACT, ACT_MXFP8, ACT_BF16 = 0, 1, 2


def build() -> None:
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fopenmp",
                           "-shared", "-fPIC", "-o", LIB, os.path.join(_HERE, "oracle.c"), "-lm"])


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            build()
        L = ctypes.CDLL(LIB)
        vp, i64, i32, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        for name in ("oracle_e2m1_value", "oracle_e8m0_value", "oracle_e4m3_value"):
            getattr(L, name).restype = d
            getattr(L, name).argtypes = [i32]
        L.oracle_bf16_value.restype = d
        L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        L.oracle_floor_log2_f32.restype = i32
        L.oracle_floor_log2_f32.argtypes = [ctypes.c_float]
        L.oracle_e2m1_encode.restype = i32
        L.oracle_e2m1_encode.argtypes = [d]
        L.oracle_e4m3_encode.restype = i32
        L.oracle_e4m3_encode.argtypes = [d]
        L.oracle_bf16_from_double.restype = ctypes.c_uint16
        L.oracle_bf16_from_double.argtypes = [d]
        L.oracle_mxfp4_quantize.restype = None
        L.oracle_mxfp4_quantize.argtypes = [vp, i64, i64, vp, vp]
        L.oracle_mxfp8_quantize_row.restype = None
        L.oracle_mxfp8_quantize_row.argtypes = [vp, i64, vp, vp]
        L.oracle_route.restype = None
        L.oracle_route.argtypes = [vp, i64, i64, i32, vp, vp]
        L.oracle_route_arrays.restype = None
        L.oracle_route_arrays.argtypes = [vp, i64, i32, i64, vp, vp, vp, vp]
        L.oracle_moe_forward.restype = i32
        L.oracle_moe_forward.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, i32,
                                         vp, i64, vp, vp, vp, i32]
        L.oracle_moe_chain.restype = i32
        L.oracle_moe_chain.argtypes = [i32, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, i32,
                                       i32, vp, i32]
        L.oracle_router_logits.restype = None
        L.oracle_router_logits.argtypes = [vp, vp, i64, i64, i64, vp]
        L.oracle_mxfp8_quantize.restype = None
        L.oracle_mxfp8_quantize.argtypes = [vp, i64, i64, vp, vp]
        L.oracle_verify.restype = i32
        L.oracle_verify.argtypes = [vp, vp, vp, vp, vp, i64, i32, i64, vp, vp]
        L.oracle_dense_forward.restype = i32
        L.oracle_dense_forward.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, vp]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def e2m1_value(c): return lib().oracle_e2m1_value(int(c))
def e8m0_value(c): return lib().oracle_e8m0_value(int(c))
def e4m3_value(c): return lib().oracle_e4m3_value(int(c))
def bf16_value(b): return lib().oracle_bf16_value(int(b))
def floor_log2_f32(a): return lib().oracle_floor_log2_f32(float(a))
def e2m1_encode(q): return lib().oracle_e2m1_encode(float(q))
def e4m3_encode(q): return lib().oracle_e4m3_encode(float(q))
def bf16_from_double(v): return lib().oracle_bf16_from_double(float(v))


def mxfp4_quantize(w: np.ndarray):
    """fp32 [R, K] -> (packed E2M1 [R, K/2] uint8, E8M0 [R, K/32] uint8)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    K = w.shape[-1]
    R = w.size // K
    fp4 = np.empty(w.shape[:-1] + (K // 2,), dtype=np.uint8)
    sc = np.empty(w.shape[:-1] + (K // 32,), dtype=np.uint8)
    lib().oracle_mxfp4_quantize(_p(w), R, K, _p(fp4), _p(sc))
    return fp4, sc


def mxfp8_quantize_row(v: np.ndarray):
    v = np.ascontiguousarray(v, dtype=np.float64)
    codes = np.empty(v.shape[0], dtype=np.uint8)
    sc = np.empty(v.shape[0] // 32, dtype=np.uint8)
    lib().oracle_mxfp8_quantize_row(_p(v), v.shape[0], _p(codes), _p(sc))
    return codes, sc


def route(logits: np.ndarray, k: int):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    gate = np.empty((T, k), dtype=np.float64)
    lib().oracle_route(_p(logits), T, E, k, _p(idx), _p(gate))
    return idx, gate


def route_arrays(idx: np.ndarray, E: int):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    cnt = np.empty(E, dtype=np.int32)
    off = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    pos = np.empty(T * k, dtype=np.int32)
    lib().oracle_route_arrays(_p(idx), T, k, E, _p(cnt), _p(off), _p(perm), _p(pos))
    return cnt, off, perm, pos


def moe_forward(x_bf16, logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, k, act_mode=ACT_EXACT,
                tokens=None, want_h=False, n_threads=0):
    """Returns (y_bf16 uint16 [n, H], y_f64 [n, H], h [n, k, I] or None)."""
    x_bf16 = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, H = x_bf16.shape
    E = logits.shape[1]
    I = w2_fp4.shape[-1] * 2
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    n = T if tok is None else tok.shape[0]
    y16 = np.empty((n, H), dtype=np.uint16)
    y64 = np.empty((n, H), dtype=np.float64)
    h = np.empty((n, k, I), dtype=np.float64) if want_h else None
    arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (w13_fp4, w13_e8m0, w2_fp4, w2_e8m0)]
    rc = lib().oracle_moe_forward(_p(x_bf16), _p(logits), *(_p(a) for a in arrs), T, H, I, E, k,
                                  act_mode, _p(tok), n, _p(y64), _p(y16), _p(h), n_threads)
    if rc != 0:
        raise ValueError(f"oracle_moe_forward rejected the arguments ({rc})")
    return y16, y64, h


def moe_chain(x_bf16, logits_list, weights_list, k, act_mode=ACT_EXACT, residual=False,
              n_threads=0):
    """Layers back to back: x_{l+1} = bf16_RNE(y_l + residual * x_l); returns x_L (uint16
    bf16 bits [T, H]).  logits_list[l] is [T, E] f32, weights_list[l] = (w13, s13, w2, s2)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T, H = x.shape
    n = len(logits_list)
    assert n == len(weights_list) and n >= 1
    lg = [np.ascontiguousarray(a, dtype=np.float32) for a in logits_list]
    ws = [[np.ascontiguousarray(a, dtype=np.uint8) for a in w] for w in weights_list]
    E = lg[0].shape[1]
    I = ws[0][2].shape[-1] * 2

    def ptrs(arrs):
        return (ctypes.c_void_p * n)(*[a.ctypes.data for a in arrs])
    out = np.empty((T, H), dtype=np.uint16)
    rc = lib().oracle_moe_chain(n, _p(x), ptrs(lg), *(ptrs([w[i] for w in ws]) for i in range(4)),
                                T, H, I, E, k, act_mode, int(bool(residual)), _p(out), n_threads)
    if rc != 0:
        raise ValueError(f"oracle_moe_chain rejected the arguments ({rc})")
    return out


def router_logits(x_bf16: np.ndarray, w_bf16: np.ndarray) -> np.ndarray:
    """Router logits [T, E] in fp64 from x [T, H] and W_r [E, H] (bf16 bit patterns)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    T, H = x.shape
    E = w.shape[0]
    assert w.shape[1] == H
    out = np.empty((T, E), dtype=np.float64)
    lib().oracle_router_logits(_p(x), _p(w), T, H, E, _p(out))
    return out


def mxfp8_quantize(w: np.ndarray):
    """fp32 [R, K] -> (E4M3 codes [R, K] uint8, E8M0 scales [R, K/32] uint8)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    K = w.shape[-1]
    R = w.size // K
    codes = np.empty(w.shape, dtype=np.uint8)
    sc = np.empty(w.shape[:-1] + (K // 32,), dtype=np.uint8)
    lib().oracle_mxfp8_quantize(_p(w), R, K, _p(codes), _p(sc))
    return codes, sc


def dense_forward(x_bf16, w_e4m3, w_e8m0, act_mode=ACT_MXFP8):
    """Dense FP8 projection: returns (y_bf16 uint16 [T, N], y_f64 [T, N])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    w = np.ascontiguousarray(w_e4m3, dtype=np.uint8)
    s = np.ascontiguousarray(w_e8m0, dtype=np.uint8)
    T, K = x.shape
    N = w.shape[0]
    y16 = np.empty((T, N), dtype=np.uint16)
    y64 = np.empty((T, N), dtype=np.float64)
    rc = lib().oracle_dense_forward(_p(x), _p(w), _p(s), T, K, N, act_mode, _p(y64), _p(y16))
    if rc != 0:
        raise ValueError("oracle_dense_forward: invalid arguments")
    return y16, y64


def verify(p, q, draft, u, U):
    """Rejection-sampling verification: p [S, g+1, V], q [S, g, V] fp32, draft [S, g] int32,
    u [S, g] fp32, U [S] uint64 -> (n_acc [S] int32, tokens [S, g+1] int32)."""
    p = np.ascontiguousarray(p, dtype=np.float32)
    q = np.ascontiguousarray(q, dtype=np.float32)
    draft = np.ascontiguousarray(draft, dtype=np.int32)
    u = np.ascontiguousarray(u, dtype=np.float32)
    U = np.ascontiguousarray(U, dtype=np.uint64)
    S, g, V = q.shape
    assert p.shape == (S, g + 1, V) and draft.shape == (S, g) and u.shape == (S, g)
    n_acc = np.empty(S, dtype=np.int32)
    tok = np.empty((S, g + 1), dtype=np.int32)
    if lib().oracle_verify(_p(p), _p(q), _p(draft), _p(u), _p(U), S, g, V, _p(n_acc),
                           _p(tok)) != 0:
        raise ValueError("oracle_verify: invalid arguments")
    return n_acc, tok
