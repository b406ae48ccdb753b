"""moe_mxfp4_forward_noalloc: the forward for callers that cannot allocate device memory
(plugin interfaces that only hand over input and output buffers, runtimes whose memory belongs
to another allocator, services that forbid allocation while serving).  Its scratch is a
fixed-size device array inside the library.

The checks, all through the C ABI:
- two calls in a row (the second reuses the array the first one left behind) give exactly the
  bits moe_mxfp4_forward gives: the same kernels run on the same inputs, only the scratch
  memory differs;
- the calls allocate nothing: the library's allocation counter does not move, checked also in
  a fresh process, where the library's scratch cache is still empty (so any fall-through to
  it would have to allocate);
- shapes that need more scratch than the array holds are refused before anything runs.

This file is collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

import mxfp4_expert_layer_dflash_b300 as moe  # noqa: E402
from gpu_util import device_layer  # noqa: E402
from synth import layers as LY  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("name", ["tiny", "mid_t8", "full_t256"])
def test_noalloc_matches_forward_on_two_calls(name):
    L = LY.LAYERS[name]
    x, lg, w13, s13, w2, s2 = device_layer(L)
    args = (x, lg, w13, s13, w2, s2, L.T, L.H, L.I, L.E, L.k)
    y_ref = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward(*args, y_ref)
    assert moe.moe_mxfp4_get_status() == 0
    allocs = moe.moe_mxfp4_alloc_count()
    for _ in range(2):
        y = torch.full((L.T, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        moe.moe_mxfp4_forward_noalloc(*args, y)
        assert moe.moe_mxfp4_get_status() == 0
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    assert moe.moe_mxfp4_alloc_count() == allocs
    del x, lg, w13, s13, w2, s2
    torch.cuda.empty_cache()


_FRESH = r"""
import sys, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import mxfp4_expert_layer_dflash_b300 as moe
from gpu_util import device_layer
from synth import layers as LY
L = LY.LAYERS["mid_t8"]
inp = device_layer(L)
args = inp + (L.T, L.H, L.I, L.E, L.k)
assert moe.moe_mxfp4_alloc_count() == 0
ys = []
for _ in range(2):
    y = torch.full((L.T, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_mxfp4_forward_noalloc(*args, y)
    assert moe.moe_mxfp4_get_status() == 0
    ys.append(y)
assert moe.moe_mxfp4_alloc_count() == 0, "the no-allocation forward allocated"
y_ref = torch.empty_like(ys[0])
moe.moe_mxfp4_forward(*args, y_ref)       # this one grows the library's cache
assert moe.moe_mxfp4_get_status() == 0
assert moe.moe_mxfp4_alloc_count() == 1
for y in ys:
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
print("fresh-process no-allocation check ok")
"""


def test_noalloc_allocates_nothing_in_a_fresh_process():
    r = subprocess.run([sys.executable, "-c", _FRESH, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "check ok" in r.stdout


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
