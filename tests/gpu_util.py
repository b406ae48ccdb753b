"""Helpers shared by the GPU tests: host<->device marshalling and error metrics."""
import numpy as np
import torch

import mxfp4_expert_layer_dflash_b300 as moe
from synth import layers as LY


def dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bf16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rel_fro(y, ref):
    return float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300))


def max_err_over_rms(y, ref):
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(np.abs(y - ref).max() / max(rms, 1e-300))


def device_layer(L):
    """(x, logits, w13, s13, w2, s2) on the GPU for layer L (weights drawn and packed there)."""
    x = dev(LY.host_x(L))
    lg = dev(LY.host_logits(L))
    w = LY.device_packed_weights(L, moe.mxfp4_quantize)
    return (x, lg) + tuple(w)


def gpu_forward(L, inputs, act_mode=moe.MOE_ACT_MXFP8, path=moe.MOE_PATH_AUTO, T=None):
    x, lg, w13, s13, w2, s2 = inputs
    T = L.T if T is None else T
    y = torch.full((T, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_ex(x, lg, w13, s13, w2, s2, T, L.H, L.I, L.E, L.k, y,
                             act_mode=act_mode, path=path)
    assert moe.moe_mxfp4_get_status() == 0
    return y
