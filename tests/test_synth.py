"""The seeded input generator: published SplitMix64 outputs, the normal law of its draws, the
polar method's steps, determinism, shapes."""
import math

import numpy as np

from conftest import read_golden


def test_splitmix64_published_outputs(synth_mod):
    for n, hexv in read_golden("splitmix64_seed0.txt"):
        assert synth_mod.splitmix_out(0, int(n)) == int(hexv, 16)


def test_normal_draws_follow_the_standard_normal(synth_mod):
    """400k draws against the N(0, 1) law: moments, the Kolmogorov-Smirnov distance to the
    normal CDF (scipy), and the two-sided 3-sigma tail mass 0.0027."""
    from scipy import stats
    z = synth_mod.normal_f32(5, 2, 0, 400000, 1.0).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.var() - 1.0) < 0.01
    k = ((z ** 4).mean()) / z.var() ** 2
    assert abs(k - 3.0) < 0.05
    assert stats.kstest(z, "norm").statistic < 0.003
    assert abs((np.abs(z) > 3.0).mean() - 2 * stats.norm.sf(3.0)) < 4e-4


def test_log_within_two_ulps(synth_mod):
    """The generator's own fp32 logarithm against math.log over (2^-46, 1] and the
    range-reduction edges (m near sqrt(2), powers of two)."""
    rng = np.random.default_rng(0)
    xs = np.concatenate([np.float32(2.0) ** -rng.uniform(0, 46, 4000).astype(np.float32),
                         np.float32([1 - 2.0 ** -24, 0.5, 0.70710677, 0.7071068, 2.0 ** -46,
                                     2.0 ** -23])]).astype(np.float32)
    for x in xs:
        got, ref = float(synth_mod.ln_f32(float(x))), math.log(float(x))
        assert abs(got - ref) <= 2 * float(np.spacing(np.float32(abs(ref)))), (float(x), got, ref)
    assert synth_mod.ln_f32(1.0) == 0.0


def test_polar_method_by_hand(synth_mod):
    """Draws recomputed from the published steps of the polar method in numpy fp32 (one RN
    rounding per operation; the logarithm is the generator's, pinned above): the 23-bit
    fields of each attempt's SplitMix64 output, v = (2u + 1 - 2^23) 2^-23, the first
    attempt with s = v1^2 + v2^2 < 1, then v1 sqrt(-2 ln(s) / s)."""
    f32 = np.float32
    seed, tid = 7, 3
    key = synth_mod.splitmix_out(seed, tid + 1)
    tries = []
    for i in range(200):
        for a in range(40):
            r = synth_mod.splitmix_out(key, 64 * i + a + 1)
            v1 = f32(2 * (r >> 41) + 1 - 2 ** 23) * f32(2.0 ** -23)
            v2 = f32(2 * ((r >> 18) & 0x7FFFFF) + 1 - 2 ** 23) * f32(2.0 ** -23)
            s = f32(f32(v1 * v1) + f32(v2 * v2))
            if s < f32(1.0):
                q = f32(f32(f32(-2.0) * synth_mod.ln_f32(float(s))) / s)
                want = f32(v1 * np.sqrt(q, dtype=np.float32))
                break
        tries.append(a + 1)
        assert synth_mod.std_normal(seed, tid, i) == want
    assert max(tries) > 1          # rejections happen (acceptance pi/4)


def test_streams_are_counter_based(synth_mod):
    a = synth_mod.normal_f32(3, 2, 1000, 50, 0.02)
    b = synth_mod.normal_f32(3, 2, 0, 1050, 0.02)[1000:]
    assert (a == b).all()
    assert not (synth_mod.normal_f32(3, 3, 1000, 50, 0.02) == a).all()
    assert not (synth_mod.normal_f32(4, 2, 1000, 50, 0.02) == a).all()
    assert a[0] == np.float32(synth_mod.std_normal(3, 2, 1000) * np.float32(0.02))


def test_x_is_bf16_of_unit_draw(synth_mod):
    x = synth_mod.x_bf16(1, 4, 64)
    z = synth_mod.normal_f32(1, 0, 0, 256, 1.0).reshape(4, 64)
    back = (x.astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.abs(back - z) <= np.abs(z) * 2.0 ** -8 + 1e-30)


def test_zipf_bias(synth_mod):
    E = 384
    a = synth_mod.logits(4, 8, E, zipf=False)
    b = synth_mod.logits(4, 8, E, zipf=True)
    bias = np.array([3.0 * math.log(1.0 / (e + 1)) for e in range(E)])
    assert np.allclose(b - a, bias[None, :], atol=1e-5)
    assert b[:, 0].mean() > b[:, -1].mean()


def test_router_and_dense_weight_draws(synth_mod):
    """The bf16 router fill is bf16_RNE(sigma * z) of the pinned z draws (tensor id 4); the
    dense weight fill is sigma * z in fp32 (tensor id 5)."""
    import torch
    E, H, seed = 3, 256, 9
    sigma = synth_mod.router_sigma(H)
    assert sigma == 2.0 ** -4
    w = synth_mod.router_bf16(seed, E, H)
    z = np.array([synth_mod.std_normal(seed, synth_mod.ID_WROUTER, i) for i in range(E * H)],
                 dtype=np.float32)
    want = torch.from_numpy((np.float32(sigma) * z).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(w.ravel(), want)
    d = synth_mod.dense_w_f32(seed, 2, 64)
    zd = np.array([synth_mod.std_normal(seed, synth_mod.ID_WDENSE, i) for i in range(128)],
                  dtype=np.float32)
    assert np.array_equal(d.ravel(), (np.float32(synth_mod.W_SIGMA) * zd))
    assert synth_mod.router_sigma(6144) == 2.0 ** -7 and synth_mod.router_sigma(2048) == 2.0 ** -6


def test_verify_inputs(synth_mod):
    p, q, d, u, U = synth_mod.verify_inputs(3, 4, 7, 1000)
    assert p.shape == (4, 8, 1000) and q.shape == (4, 7, 1000)
    np.testing.assert_allclose(p.sum(axis=2), 1.0, atol=1e-5)
    np.testing.assert_allclose(q.sum(axis=2), 1.0, atol=1e-5)
    assert ((d >= 0) & (d < 1000)).all()
    assert ((u >= 0) & (u < 1)).all() and np.array_equal(u * 2.0 ** 24, np.floor(u * 2.0 ** 24))
    assert U[0] == synth_mod.splitmix_out(synth_mod.splitmix_out(3, synth_mod.ID_VERIFY_R + 1), 0)
    again = synth_mod.verify_inputs(3, 4, 7, 1000)
    assert all(np.array_equal(a, b) for a, b in zip((p, q, d, u, U), again))
