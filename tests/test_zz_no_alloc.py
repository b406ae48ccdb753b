"""moe_mxfp4_forward_noalloc: the forward for callers that cannot allocate device memory
(plugin interfaces that only hand over input and output buffers, runtimes whose memory belongs
to another allocator, services that forbid allocation while serving).  Its scratch is a
fixed-size device array inside the library, so these checks compare it, through the C ABI,
with moe_mxfp4_forward on two calls in a row (the second call reuses the array the first one
left behind), and check that oversized shapes are refused before anything runs.

This file is collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import mxfp4_expert_layer_dflash_b300 as moe  # noqa: E402
from gpu_util import bf16_to_f64, device_layer, host_bf16, max_err_over_rms, rel_fro  # noqa: E402
from synth import layers as LY  # noqa: E402

MXFP8_FRO, MXFP8_MAX = 1e-2, 4e-2


@pytest.mark.parametrize("name", ["tiny", "mid_t8", "full_t256"])
def test_noalloc_matches_forward_on_two_calls(name):
    L = LY.LAYERS[name]
    x, lg, w13, s13, w2, s2 = device_layer(L)
    args = (x, lg, w13, s13, w2, s2, L.T, L.H, L.I, L.E, L.k)
    y_ref = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward(*args, y_ref)
    assert moe.moe_mxfp4_get_status() == 0
    ref = bf16_to_f64(host_bf16(y_ref))
    for _ in range(2):
        y = torch.full((L.T, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        moe.moe_mxfp4_forward_noalloc(*args, y)
        assert moe.moe_mxfp4_get_status() == 0
        got = bf16_to_f64(host_bf16(y))
        assert np.isfinite(got).all()
        assert rel_fro(got, ref) <= MXFP8_FRO and max_err_over_rms(got, ref) <= MXFP8_MAX
    del x, lg, w13, s13, w2, s2
    torch.cuda.empty_cache()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    L = LY.LAYERS["full_t256"]
    big_T = 1024
    need = moe.moe_mxfp4_workspace_size(big_T, L.H, L.I, L.E, L.k)
    assert need > moe.MOE_NOALLOC_SCRATCH_BYTES
    z = torch.zeros(64, dtype=torch.uint8, device="cuda")
    y = torch.zeros(64, dtype=torch.uint8, device="cuda")
    rc = moe.lib().moe_mxfp4_forward_noalloc(z.data_ptr(), z.data_ptr(), z.data_ptr(),
                                             z.data_ptr(), z.data_ptr(), z.data_ptr(), big_T, L.H,
                                             L.I, L.E, L.k, y.data_ptr(), None)
    assert rc == -5  # MOE_ERR_NO_MEMORY, nothing launched
    assert (y == 0).all()
