"""Seeded synthetic inputs for the MXFP4 MoE layer (test and benchmark infrastructure).

The generator is counter-based (definitions in ``synth_core.h``): SplitMix64 streams, and
standard normal draws by Marsaglia's polar method in a fixed sequence of correctly rounded
fp32 operations, so the host library (``libsynth.so``) and the device library
(``libsynth_dev.so``) produce the same bits.  It holds none of the layer's arithmetic; packing the fp32 weights to MXFP4 is done by
whichever side (the oracle or the CUDA library) is under test.

Workload recipe (shapes and value distributions of the layers this repository measures):
  x       [T, H]  bf16 RNE of an N(0, 1) draw                (tensor id 0)
  logits  [T, E]  fp32 N(0, 1) draw, optional Zipf bias      (tensor id 1)
  w13     [E, 2I, H] fp32 N(0, 0.02^2) draw before packing   (tensor id 2)
  w2      [E, H, I]  fp32 N(0, 0.02^2) draw before packing   (tensor id 3)
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libsynth.so")
DEV_LIB = os.path.join(_HERE, "libsynth_dev.so")

ID_X, ID_LOGITS, ID_W13, ID_W2, ID_WROUTER, ID_WDENSE = 0, 1, 2, 3, 4, 5
ID_VERIFY_Z, ID_VERIFY_N, ID_VERIFY_D, ID_VERIFY_U, ID_VERIFY_R = 6, 7, 8, 9, 10
W_SIGMA = 0.02


def build(device: bool = True) -> None:
    """Compile the host generator (gcc) and, if ``device``, its CUDA twin (nvcc, sm_103a)."""
    src = os.path.join(_HERE, "synth.c")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-shared",
                           "-fPIC", "-o", HOST_LIB, src, "-lm"])
    if device:
        subprocess.check_call(["nvcc", "-O3", "-std=c++17", "-gencode",
                               "arch=compute_103a,code=sm_103a", "-lineinfo", "-shared",
                               "-Xcompiler", "-fPIC", "-cudart", "shared", "-o", DEV_LIB,
                               os.path.join(_HERE, "synth_dev.cu")])


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            build(device=False)
        lib = ctypes.CDLL(HOST_LIB)
        u64, u32, i64 = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64
        lib.synth_splitmix_out.restype = u64
        lib.synth_splitmix_out.argtypes = [u64, u64]
        lib.synth_std_normal.restype = ctypes.c_float
        lib.synth_std_normal.argtypes = [u64, u32, u64]
        lib.synth_ln_f32.restype = ctypes.c_float
        lib.synth_ln_f32.argtypes = [ctypes.c_float]
        lib.synth_fill_normal_f32.restype = None
        lib.synth_fill_normal_f32.argtypes = [u64, u32, u64, u64, ctypes.c_float, ctypes.c_void_p]
        lib.synth_fill_x_bf16.restype = None
        lib.synth_fill_x_bf16.argtypes = [u64, i64, i64, ctypes.c_void_p]
        lib.synth_fill_bf16.restype = None
        lib.synth_fill_bf16.argtypes = [u64, u32, u64, u64, ctypes.c_float, ctypes.c_void_p]
        lib.synth_fill_verify.restype = None
        lib.synth_fill_verify.argtypes = [u64, i64, ctypes.c_int, i64, ctypes.c_float,
                                          ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_fill_logits.restype = None
        lib.synth_fill_logits.argtypes = [u64, i64, i64, ctypes.c_int, ctypes.c_void_p]
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_LIB):
            raise RuntimeError(f"{DEV_LIB} is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(DEV_LIB)
        lib.synth_dev_fill_normal_f32.restype = ctypes.c_int
        lib.synth_dev_fill_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint32,
                                                  ctypes.c_uint64, ctypes.c_uint64,
                                                  ctypes.c_float, ctypes.c_void_p,
                                                  ctypes.c_void_p]
        _dev = lib
    return _dev


def splitmix_out(seed: int, n: int) -> int:
    """n-th output (n >= 1) of SplitMix64 seeded with ``seed``."""
    return int(_host_lib().synth_splitmix_out(seed, n))


def std_normal(seed: int, tensor_id: int, i: int) -> np.float32:
    """Draw i of the (seed, tensor id) stream: a standard normal value in fp32."""
    return np.float32(_host_lib().synth_std_normal(seed, tensor_id, i))


def ln_f32(s: float) -> np.float32:
    """The generator's own fp32 natural logarithm (positive normal arguments)."""
    return np.float32(_host_lib().synth_ln_f32(s))


def normal_f32(seed: int, tensor_id: int, start: int, n: int, sigma: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    if n:
        _host_lib().synth_fill_normal_f32(seed, tensor_id, start, n, sigma,
                                          out.ctypes.data_as(ctypes.c_void_p))
    return out


def x_bf16(seed: int, T: int, H: int) -> np.ndarray:
    """[T, H] bf16 bit patterns (uint16)."""
    out = np.empty((T, H), dtype=np.uint16)
    if T * H:
        _host_lib().synth_fill_x_bf16(seed, T, H, out.ctypes.data_as(ctypes.c_void_p))
    return out


def router_sigma(H: int) -> float:
    """Router weight scale: the power of two nearest below 1/sqrt(H), so that logits of
    N(0, 1) x have a standard deviation in [0.5, 1)."""
    s = 1.0
    while s * s * H > 1.0:
        s *= 0.5
    return s


def router_bf16(seed: int, E: int, H: int) -> np.ndarray:
    """Router weights [E, H] as bf16 bit patterns (uint16): bf16(router_sigma(H) * z)."""
    out = np.empty((E, H), dtype=np.uint16)
    if E * H:
        _host_lib().synth_fill_bf16(seed, ID_WROUTER, 0, E * H, router_sigma(H),
                                    out.ctypes.data_as(ctypes.c_void_p))
    return out


def dense_w_f32(seed: int, N: int, K: int) -> np.ndarray:
    """fp32 dense-projection weights [N, K] (before MXFP8 packing)."""
    out = np.empty((N, K), dtype=np.float32)
    if N * K:
        _host_lib().synth_fill_normal_f32(seed, ID_WDENSE, 0, N * K, W_SIGMA,
                                          out.ctypes.data_as(ctypes.c_void_p))
    return out


def logits(seed: int, T: int, E: int, zipf: bool = False) -> np.ndarray:
    out = np.empty((T, E), dtype=np.float32)
    if T * E:
        _host_lib().synth_fill_logits(seed, T, E, int(zipf), out.ctypes.data_as(ctypes.c_void_p))
    return out


def w13_f32(seed: int, E: int, I: int, H: int, experts=None) -> np.ndarray:
    """fp32 gate/up weights [E, 2I, H] (only ``experts`` filled if given, rest zero)."""
    out = np.zeros((E, 2 * I, H), dtype=np.float32)
    for e in (range(E) if experts is None else experts):
        n = 2 * I * H
        _host_lib().synth_fill_normal_f32(seed, ID_W13, e * n, n, W_SIGMA,
                                          out[e].ctypes.data_as(ctypes.c_void_p))
    return out


def w2_f32(seed: int, E: int, H: int, I: int, experts=None) -> np.ndarray:
    """fp32 down weights [E, H, I] (only ``experts`` filled if given, rest zero)."""
    out = np.zeros((E, H, I), dtype=np.float32)
    for e in (range(E) if experts is None else experts):
        n = H * I
        _host_lib().synth_fill_normal_f32(seed, ID_W2, e * n, n, W_SIGMA,
                                          out[e].ctypes.data_as(ctypes.c_void_p))
    return out


def dev_fill_normal_f32(seed: int, tensor_id: int, start: int, n: int, sigma: float,
                        dev_ptr: int, stream: int = 0) -> None:
    """Device twin of ``normal_f32``: writes n fp32 values to device memory at ``dev_ptr``."""
    rc = _dev_lib().synth_dev_fill_normal_f32(seed, tensor_id, start, n, sigma,
                                              ctypes.c_void_p(dev_ptr), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"synth_dev_fill_normal_f32 failed ({rc})")


def verify_inputs(seed: int, S: int, g: int, V: int, sigma_t: float = 3.0, sigma_n: float = 0.2):
    """(p [S, g+1, V], q [S, g, V] fp32, draft [S, g] int32, u [S, g] fp32, U [S] uint64): the
    probabilities and uniforms of a speculative verification (see synth_fill_verify).  The
    default drafter noise accepts about 5.2 of 7 drafted tokens (6.2 emitted per round, near
    the coding acceptance length the pages report)."""
    p = np.empty((S, g + 1, V), dtype=np.float32)
    q = np.empty((S, g, V), dtype=np.float32)
    d = np.empty((S, g), dtype=np.int32)
    u = np.empty((S, g), dtype=np.float32)
    U = np.empty(S, dtype=np.uint64)
    _host_lib().synth_fill_verify(seed, S, g, V, sigma_t, sigma_n,
                                  *(a.ctypes.data_as(ctypes.c_void_p) for a in (p, q, d, u, U)))
    return p, q, d, u, U
