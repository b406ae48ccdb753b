"""bench.py's host-side model (CPU): the algorithmic bytes the roofline divides by, and the
names of the steps it times.

Per expert at the full shape (H=6144, I=2048): w13 2I x H/2 packed bytes + 2I x H/32 scales,
w2 H x I/2 + H x I/32 — 12,582,912 + 786,432 + 6,291,456 + 393,216 = 20,054,016 bytes; plus
the token-side bytes x (T x H bf16), logits (T x E fp32) and y (T x H bf16).
"""
import numpy as np

import bench
from synth import layers as LY


def test_full_shape_bytes_per_expert():
    L = LY.LAYERS["full_t256"]
    cnt = np.ones(L.E, dtype=np.int32)
    touched, b1, b2, total = bench.layer_bytes(L, cnt)
    assert touched == 384
    assert b1 == 384 * (12_582_912 + 786_432)
    assert b2 == 384 * (6_291_456 + 393_216)
    assert total == 384 * 20_054_016 + 256 * 6144 * 2 + 256 * 384 * 4 + 256 * 6144 * 2


def test_only_touched_experts_count():
    L = LY.LAYERS["full_t8"]
    cnt = np.zeros(L.E, dtype=np.int32)
    cnt[[3, 7, 300]] = [5, 1, 2]
    touched, b1, b2, total = bench.layer_bytes(L, cnt)
    assert touched == 3 and b1 + b2 == 3 * 20_054_016


def test_step_names_follow_the_launch_sequence():
    assert bench.step_names(1, 256) == ["route_topk", "route_permute", "act_quant", "gemm1",
                                        "gemm2", "combine"]
    assert bench.step_names(2, 256) == ["route_topk", "route_permute", "act_quant",
                                        "gemm1+gemm2+combine"]
    assert bench.step_names(1, 8) == ["route_act", "gemm1", "gemm2", "combine"]
    assert bench.step_names(2, 32) == ["layer"]          # the whole layer in one launch
    assert bench.step_names(3, 8) == ["route_act", "gemm1+gemm2", "combine"]
