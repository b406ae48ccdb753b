"""Seeded synthetic MoE layers: the workloads this repository tests and measures.

Each layer is fixed by its dimensions and seed; values follow the recipe in ``synth.py``
(x ~ unit draw as bf16, logits ~ unit draw (+ Zipf bias for the skewed layer), fp32 weights
~ draw * 0.02 packed to MXFP4).  Packing is done by a caller-supplied quantize function (the
oracle's or the CUDA library's), so this module holds none of the layer's arithmetic.

Token counts are sequences x 8 because a DFlash verification pass scores a block of up to 8
drafted positions per sequence in one forward (techllm.github.io, "2. DFlash").
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import synth as S


@dataclass(frozen=True)
class Layer:
    name: str
    H: int
    I: int
    E: int
    k: int
    T: int
    seed: int
    zipf: bool = False

    @property
    def desc(self) -> str:
        return (f"H={self.H} I={self.I} E={self.E} top-{self.k} T={self.T}"
                + (" zipf-skewed routing" if self.zipf else "") + f" seed={self.seed}")


LAYERS = {
    "tiny": Layer("tiny", 256, 128, 8, 2, 16, 0),
    "mid_t8": Layer("mid_t8", 2048, 1024, 64, 8, 8, 1),
    "full_t8": Layer("full_t8", 6144, 2048, 384, 8, 8, 2),
    "full_t256": Layer("full_t256", 6144, 2048, 384, 8, 256, 3),
    "full_t1024_zipf": Layer("full_t1024_zipf", 6144, 2048, 384, 8, 1024, 4, zipf=True),
    # full per-expert shape with 32 experts (0.64 GB of packed weights, larger than L2):
    # the case detailed ncu captures run on
    "full_e32_t64": Layer("full_e32_t64", 6144, 2048, 32, 8, 64, 5),
    # the skewed 1024-token layer's regime (top experts near 1024 tokens each) on 32 experts:
    # the case for detailed captures of the tensor-bound GEMMs
    "zipf_e32_t1024": Layer("zipf_e32_t1024", 6144, 2048, 32, 8, 1024, 6, zipf=True),
}


def host_x(L: Layer) -> np.ndarray:
    return S.x_bf16(L.seed, L.T, L.H)


def host_logits(L: Layer) -> np.ndarray:
    return S.logits(L.seed, L.T, L.E, zipf=L.zipf)


def host_packed_weights(L: Layer, quantize, experts=None):
    """(w13_fp4, w13_e8m0, w2_fp4, w2_e8m0) as numpy arrays, packed with ``quantize``
    (fp32 [R, K] -> (fp4, e8m0)).  Only ``experts`` are filled when given (others zero)."""
    E, H, I = L.E, L.H, L.I
    w13 = np.zeros((E, 2 * I, H // 2), np.uint8)
    s13 = np.zeros((E, 2 * I, H // 32), np.uint8)
    w2 = np.zeros((E, H, I // 2), np.uint8)
    s2 = np.zeros((E, H, I // 32), np.uint8)
    for e in (range(E) if experts is None else sorted(set(int(v) for v in experts))):
        a = S.normal_f32(L.seed, S.ID_W13, e * 2 * I * H, 2 * I * H, S.W_SIGMA).reshape(2 * I, H)
        w13[e], s13[e] = quantize(a)
        b = S.normal_f32(L.seed, S.ID_W2, e * H * I, H * I, S.W_SIGMA).reshape(H, I)
        w2[e], s2[e] = quantize(b)
    return w13, s13, w2, s2


def device_packed_weights(L: Layer, quantize_into, device="cuda", experts_per_batch=16):
    """Packed weights generated and packed on the GPU: fp32 weights are drawn by the device
    twin of the generator, ``experts_per_batch`` experts at a time, and packed by
    ``quantize_into(w_f32, rows, K, out_fp4, out_e8m0)``."""
    import torch
    E, H, I = L.E, L.H, L.I
    w13 = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=device)
    s13 = torch.empty((E, 2 * I, H // 32), dtype=torch.uint8, device=device)
    w2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device=device)
    s2 = torch.empty((E, H, I // 32), dtype=torch.uint8, device=device)
    nb = min(E, experts_per_batch)
    tmp = torch.empty(nb * 2 * I * H, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream().cuda_stream
    for e0 in range(0, E, nb):
        ne = min(nb, E - e0)
        n = ne * 2 * I * H
        S.dev_fill_normal_f32(L.seed, S.ID_W13, e0 * 2 * I * H, n, S.W_SIGMA, tmp.data_ptr(),
                              stream)
        quantize_into(tmp[:n], ne * 2 * I, H, w13[e0:e0 + ne], s13[e0:e0 + ne])
        n = ne * H * I
        S.dev_fill_normal_f32(L.seed, S.ID_W2, e0 * H * I, n, S.W_SIGMA, tmp.data_ptr(), stream)
        quantize_into(tmp[:n], ne * H, I, w2[e0:e0 + ne], s2[e0:e0 + ne])
    del tmp
    return w13, s13, w2, s2
