"""GPU parity of the rejection-sampling verification of a drafted block: accept counts and
tokens bit-exact against the oracle (the uniforms are inputs; draws use exact integer masses),
at the verify step's full size and on small and forced cases."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import mxfp4_expert_layer_dflash_b300 as moe  # noqa: E402
from gpu_util import dev  # noqa: E402
from synth import synth as S  # noqa: E402


@pytest.fixture(scope="module")
def O():
    from oracle import oracle
    return oracle


def _gpu_verify(p, q, d, u, U):
    Sq, g, V = q.shape
    n = torch.empty(Sq, dtype=torch.int32, device="cuda")
    tok = torch.empty((Sq, g + 1), dtype=torch.int32, device="cuda")
    Ud = torch.from_numpy(U.view(np.int64)).cuda()
    moe.moe_verify_block(dev(p), dev(q), dev(d), dev(u), Ud, Sq, g, V, n, tok)
    return n.cpu().numpy(), tok.cpu().numpy()


@pytest.mark.parametrize("Sq,g,V,seed", [(32, 7, 152064, 1), (1, 1, 5, 2), (64, 3, 1000, 3),
                                         (4, 7, 32000, 4), (300, 7, 4099, 5), (2, 16, 65537, 6)])
def test_verify_bit_exact(O, Sq, g, V, seed):
    p, q, d, u, U = S.verify_inputs(seed, Sq, g, V)
    n, tok = _gpu_verify(p, q, d, u, U)
    assert moe.moe_mxfp4_get_status() == 0
    rn, rtok = O.verify(p, q, d, u, U)
    assert np.array_equal(n, rn)
    assert np.array_equal(tok, rtok)
    print(f"S={Sq} g={g} V={V}: mean accepted {n.mean():.2f}")


def test_verify_forced_cases(O):
    Sq, g, V = 6, 4, 3000
    rng = np.random.default_rng(9)
    p = rng.dirichlet(np.ones(V), size=(Sq, g + 1)).astype(np.float32)
    q = p[:, :g].copy()                                     # p == q: everything accepted ...
    d = rng.integers(0, V, (Sq, g)).astype(np.int32)
    u = (rng.integers(0, 2 ** 24, (Sq, g)) / 2.0 ** 24).astype(np.float32)
    U = rng.integers(0, 2 ** 64, Sq, dtype=np.uint64)
    p[1, 2, d[1, 2]] = 0.0                                  # ... but an impossible draft rejects
    q[1, 2, d[1, 2]] = 0.0                                  # (and leaves no residual: draw from p)
    p[2, 0, :] = 0.0
    p[2, 0, 17] = 1.0                                       # residual all on token 17
    d[2, 0] = 18
    U[3] = 0
    U[4] = 2 ** 64 - 1
    n, tok = _gpu_verify(p, q, d, u, U)
    rn, rtok = O.verify(p, q, d, u, U)
    assert np.array_equal(n, rn) and np.array_equal(tok, rtok)
    assert n[1] == 2 and n[2] == 0 and tok[2, 0] == 17
    assert (n[[0, 3, 4, 5]] == g).all()


def test_verify_deterministic_and_bad_draft(O):
    p, q, d, u, U = S.verify_inputs(11, 16, 7, 20000)
    a = _gpu_verify(p, q, d, u, U)
    b = _gpu_verify(p, q, d, u, U)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    d2 = d.copy()
    d2[5, 0] = 20000                      # outside the vocabulary: checked before any read
    n, tok = _gpu_verify(p, q, d2, u, U)
    assert moe.moe_mxfp4_get_status() == -7                    # MOE_ERR_DEVICE_FAULT
    assert n[5] == 0
    assert np.array_equal(np.delete(n, 5), np.delete(a[0], 5))
