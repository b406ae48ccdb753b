"""Failure detection on the GPU without a fault: a bounded device wait that runs out.

MOE_DEBUG_FORCE_DEP_TIMEOUT makes the single-launch path's GEMM2 items wait for a GEMM1
completion count that is never reached; with MOE_DEBUG_SHORT_TIMEOUT the wait gives up after
about a millisecond.  The kernel must then report MOE_ERR_DEVICE_TIMEOUT through the status
word, shut down cleanly (every role sees the abort flag), and leave the context usable: the
next normal call on the same stream is correct.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import mxfp4_expert_layer_dflash_b300 as moe  # noqa: E402
from gpu_util import bf16_to_f64, device_layer, gpu_forward, host_bf16, rel_fro  # noqa: E402
from synth import layers as LY  # noqa: E402


@pytest.fixture(scope="module")
def O():
    from oracle import oracle
    return oracle


@pytest.mark.parametrize("path", [moe.MOE_PATH_PERSISTENT, moe.MOE_PATH_GEMMS])
@pytest.mark.parametrize("name", ["tiny", "full_e32_t64"])
def test_dependency_wait_times_out_and_context_survives(O, name, path):
    L = LY.LAYERS[name]
    inp = device_layer(L)
    x, lg, w13, s13, w2, s2 = inp
    y = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    assert moe.moe_mxfp4_get_status() == 0
    moe.moe_mxfp4_forward_ex(x, lg, w13, s13, w2, s2, L.T, L.H, L.I, L.E, L.k, y,
                             path=path,
                             debug_flags=moe.MOE_DEBUG_SHORT_TIMEOUT
                             | moe.MOE_DEBUG_FORCE_DEP_TIMEOUT)
    assert moe.moe_mxfp4_get_status() == moe.MOE_ERR_DEVICE_TIMEOUT
    assert moe.moe_mxfp4_get_status() == 0          # reading the status clears it
    # the context survives: the same call without the flags is correct
    if name == "tiny":
        y2 = bf16_to_f64(host_bf16(gpu_forward(L, inp, path=path)))
        w = LY.host_packed_weights(L, O.mxfp4_quantize)
        _, yref, _ = O.moe_forward(LY.host_x(L), LY.host_logits(L), *w, L.k, O.ACT_MXFP8)
        assert rel_fro(y2, yref) <= 1e-2
    else:
        ym = gpu_forward(L, inp, path=moe.MOE_PATH_MULTI)
        yp = gpu_forward(L, inp, path=path)
        assert torch.equal(ym.view(torch.int16), yp.view(torch.int16))
    del inp
    torch.cuda.empty_cache()


def test_flag_is_ignored_by_the_two_launch_path():
    L = LY.LAYERS["tiny"]
    inp = device_layer(L)
    y = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_ex(*inp, L.T, L.H, L.I, L.E, L.k, y, path=moe.MOE_PATH_MULTI,
                             debug_flags=moe.MOE_DEBUG_SHORT_TIMEOUT
                             | moe.MOE_DEBUG_FORCE_DEP_TIMEOUT)
    assert moe.moe_mxfp4_get_status() == 0
    ref = gpu_forward(L, inp, path=moe.MOE_PATH_MULTI)
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    assert np.isfinite(bf16_to_f64(host_bf16(y))).all()


def test_bf16_decode_wait_times_out_and_context_survives(O):
    """The bf16 mode's GEMM: decoders whose buffers are never handed back give up after the
    short timeout; every role sees the abort flag, the status reads MOE_ERR_DEVICE_TIMEOUT,
    and the next normal call is correct."""
    L = LY.LAYERS["mid_t8"]                  # 16 K steps per item: the decoders need a buffer back
    inp = device_layer(L)
    y = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    assert moe.moe_mxfp4_get_status() == 0
    moe.moe_mxfp4_forward_ex(*inp, L.T, L.H, L.I, L.E, L.k, y, act_mode=moe.MOE_ACT_BF16,
                             debug_flags=moe.MOE_DEBUG_SHORT_TIMEOUT | moe.MOE_DEBUG_STALL_DECODE)
    assert moe.moe_mxfp4_get_status() == moe.MOE_ERR_DEVICE_TIMEOUT
    assert moe.moe_mxfp4_get_status() == 0
    yb = gpu_forward(L, inp, act_mode=moe.MOE_ACT_BF16)
    toks = [0, 3, 7]
    w = LY.host_packed_weights(L, O.mxfp4_quantize, None)
    _, yref, _ = O.moe_forward(LY.host_x(L), LY.host_logits(L), *w, L.k, O.ACT_EXACT,
                               tokens=np.array(toks))
    assert rel_fro(bf16_to_f64(host_bf16(yb))[toks], yref) <= 5e-3
    del inp
    torch.cuda.empty_cache()
