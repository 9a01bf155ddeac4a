"""Pins of the oracle's LayerNorm (forward and backward) to facts outside
itself: hand-worked values, torch's float64 layer_norm and its autograd,
central finite differences, and the identities of the definition (a constant
row gives beta; shift and scale invariance at eps = 0; dx sums to zero along
the row and is orthogonal to xhat at eps = 0).  A plausible slip -- the
sample variance (N - 1), the variance taken about zero, eps outside the
square root, a dropped mean term or a wrong sign in dx, beta added before
the scaling -- fails at least one of them."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import GOLDEN, eval_expr


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def test_hand_examples():
    with open(os.path.join(GOLDEN, "layernorm_hand_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        x, g, b = _f32([c["x"]]), _f32(c["gamma"]), _f32(c["beta"])
        fw = oracle.layernorm_fwd(x, g, b, c["eps"], "f32", "f32")
        np.testing.assert_allclose(fw["y64"][0], [eval_expr(v) for v in c["y"]], rtol=1e-14,
                                   atol=1e-15)
        assert abs(fw["mean64"][0] - eval_expr(c["mean"])) < 1e-15
        assert abs(fw["rstd64"][0] - eval_expr(c["rstd"])) < 1e-15
        bw = oracle.layernorm_bwd(_f32([c["dy"]]), x, None, None, g, c["eps"], "f32", "f32")
        np.testing.assert_allclose(bw["dx64"][0], [eval_expr(v) for v in c["dx"]], rtol=1e-14,
                                   atol=1e-15)
        np.testing.assert_allclose(bw["dgamma64"], [eval_expr(v) for v in c["dgamma"]],
                                   rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(bw["dbeta64"], [eval_expr(v) for v in c["dbeta"]], atol=0)


@pytest.mark.parametrize("N", [1, 7, 64, 513])
@pytest.mark.parametrize("eps", [0.0, 1e-5, 0.3])
@pytest.mark.parametrize("with_beta", [True, False])
def test_forward_matches_torch_float64(N, eps, with_beta):
    if N == 1 and eps == 0.0:
        pytest.skip("0/0: a one-element row has zero variance")
    rng = np.random.default_rng(N)
    x = _f32(rng.standard_normal((5, N)) * 3 + 1.5)
    g = _f32(rng.uniform(0.5, 1.5, N))
    b = _f32(rng.standard_normal(N)) if with_beta else None
    out = oracle.layernorm_fwd(x, g, b, eps, "f32", "f32")
    ref = torch.nn.functional.layer_norm(
        torch.from_numpy(x).double(), (N,), torch.from_numpy(g).double(),
        torch.from_numpy(b).double() if with_beta else None, eps).numpy()
    np.testing.assert_allclose(out["y64"], ref, rtol=1e-12, atol=1e-12)
    # and the stored outputs are those values rounded once
    assert np.array_equal(out["y"], ref.astype(np.float32))


@pytest.mark.parametrize("N", [2, 9, 128])
@pytest.mark.parametrize("eps", [0.0, 1e-5])
def test_backward_matches_torch_autograd_float64(N, eps):
    rng = np.random.default_rng(10 + N)
    x = _f32(rng.standard_normal((4, N)) + 0.5)
    g = _f32(rng.uniform(0.5, 1.5, N))
    b = _f32(rng.standard_normal(N))
    dy = _f32(rng.standard_normal((4, N)))
    out = oracle.layernorm_bwd(dy, x, None, None, g, eps, "f32", "f32")
    xt = torch.from_numpy(x).double().requires_grad_()
    gt = torch.from_numpy(g).double().requires_grad_()
    bt = torch.from_numpy(b).double().requires_grad_()
    y = torch.nn.functional.layer_norm(xt, (N,), gt, bt, eps)
    (y * torch.from_numpy(dy).double()).sum().backward()
    np.testing.assert_allclose(out["dx64"], xt.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(out["dgamma64"], gt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["dbeta64"], bt.grad.numpy(), rtol=1e-12, atol=1e-12)


def _loss(x, g, b, dy, eps):
    return float((oracle.layernorm_fwd(x, g, b, eps, "f32", "f32")["y64"] * dy).sum())


@pytest.mark.parametrize("N", [2, 5, 16])
def test_backward_matches_central_differences(N):
    # inputs on a 2^-8 grid and steps of 2^-10, 2^-11: every perturbed input is
    # exact in fp32; Richardson extrapolation leaves an O(h^4) truncation error
    eps = 1e-3
    rng = np.random.default_rng(200 + N)
    M = 3
    x = _f32(np.round(rng.uniform(-2.0, 2.0, (M, N)) * 256) / 256)
    g = _f32(np.round(rng.uniform(0.5, 1.5, N) * 256) / 256)
    b = _f32(np.round(rng.standard_normal(N) * 256) / 256)
    dy = _f32(np.round(rng.standard_normal((M, N)) * 256) / 256).astype(np.float64)
    out = oracle.layernorm_bwd(_f32(dy), x, None, None, g, eps, "f32", "f32")

    def central(f, a, idx, h):
        ap, am = a.copy(), a.copy()
        ap[idx] += np.float32(h)
        am[idx] -= np.float32(h)
        return (f(ap) - f(am)) / (2 * h)

    def rich(f, a, idx):
        h = 2.0 ** -10
        return (4 * central(f, a, idx, h / 2) - central(f, a, idx, h)) / 3

    fd_dx = np.array([[rich(lambda xx: _loss(xx, g, b, dy, eps), x, (i, j)) for j in range(N)]
                      for i in range(M)])
    fd_dg = np.array([rich(lambda gg: _loss(x, gg, b, dy, eps), g, (j,)) for j in range(N)])
    fd_db = np.array([rich(lambda bb: _loss(x, g, bb, dy, eps), b, (j,)) for j in range(N)])
    scale = max(1.0, np.abs(fd_dx).max())
    assert np.abs(out["dx64"] - fd_dx).max() <= 1e-7 * scale
    assert np.abs(out["dgamma64"] - fd_dg).max() <= 1e-7 * max(1.0, np.abs(fd_dg).max())
    assert np.abs(out["dbeta64"] - fd_db).max() <= 1e-7 * max(1.0, np.abs(fd_db).max())


def test_constant_row_gives_beta():
    x = _f32(np.full((3, 32), 2.75))
    g = _f32(np.linspace(0.5, 1.5, 32))
    b = _f32(np.linspace(-1, 1, 32))
    out = oracle.layernorm_fwd(x, g, b, 1e-5, "f32", "f32")
    assert np.array_equal(out["y64"], np.broadcast_to(b.astype(np.float64), (3, 32)))


def test_shift_and_scale_invariance_at_eps_zero():
    # x on an integer grid; 4x + 3 is exact in fp32, so y(4x + 3) = y(x) and
    # y(-2x) = -y(x) up to the rounding of the double sums
    rng = np.random.default_rng(5)
    x = _f32(rng.integers(-50, 50, (4, 40)))
    g, b = _f32(np.ones(40)), None
    base = oracle.layernorm_fwd(x, g, b, 0.0, "f32", "f32")["y64"]
    for a, c in ((4.0, 3.0), (-2.0, 0.0), (0.5, -7.0)):
        y = oracle.layernorm_fwd(_f32(x * a + c), g, b, 0.0, "f32", "f32")["y64"]
        np.testing.assert_allclose(y, np.sign(a) * base, rtol=1e-13, atol=1e-13)
    # normalised rows: mean 0 and population variance 1
    assert np.abs(base.mean(axis=1)).max() < 1e-13
    np.testing.assert_allclose((base ** 2).mean(axis=1), 1.0, rtol=1e-13)


def test_backward_identities():
    rng = np.random.default_rng(6)
    x = _f32(rng.standard_normal((6, 96)) + 2)
    g = _f32(rng.uniform(0.5, 1.5, 96))
    dy = _f32(rng.standard_normal((6, 96)))
    for eps in (0.0, 1e-2):
        out = oracle.layernorm_bwd(dy, x, None, None, g, eps, "f32", "f32")
        fw = oracle.layernorm_fwd(x, g, None, eps, "f32", "f32")
        xhat = (x.astype(np.float64) - fw["mean64"][:, None]) * fw["rstd64"][:, None]
        scale = np.abs(out["dx64"]).sum(axis=1)
        assert np.all(np.abs(out["dx64"].sum(axis=1)) <= 1e-13 * scale)
        if eps == 0.0:
            assert np.all(np.abs((out["dx64"] * xhat).sum(axis=1)) <= 1e-12 * scale)
        else:   # eps leaks a part proportional to eps / (var + eps)
            assert np.all(np.abs((out["dx64"] * xhat).sum(axis=1)) > 1e-8 * scale)


def test_backward_with_saved_statistics_uses_them():
    # the saved fp32 mean and rstd, not recomputed ones: perturbing the saved
    # rstd scales dx's row accordingly
    rng = np.random.default_rng(7)
    x = _f32(rng.standard_normal((3, 64)))
    g = _f32(np.ones(64))
    dy = _f32(rng.standard_normal((3, 64)))
    fw = oracle.layernorm_fwd(x, g, None, 1e-5, "f32", "f32")
    a = oracle.layernorm_bwd(dy, x, fw["mean"], fw["rstd"], g, 1e-5, "f32", "f32")
    r2 = _f32(fw["rstd"] * 2)
    b = oracle.layernorm_bwd(dy, x, fw["mean"], r2, g, 1e-5, "f32", "f32")
    assert not np.allclose(a["dx64"], b["dx64"])
    with pytest.raises(ValueError):
        oracle.layernorm_bwd(dy, x, fw["mean"], None, g, 1e-5, "f32", "f32")
