"""Pins of the double-precision oracle to facts outside itself.

Each test fixes the oracle against something it cannot merely restate: values
worked out by hand, closed forms, invariants of the definition, central finite
differences of the forward, and library routines on the special cases they
cover (torch's CPU rms_norm and its autograd in float64, torch's fp32->bf16
conversion).  A plausible slip in the oracle -- eps outside the square root, a
sum instead of a mean, a dropped term or wrong sign in dx, gamma indexed by row,
a double rounding through fp32 -- fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import GOLDEN, eval_expr


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_rounding_boundary_fixtures():
    with open(os.path.join(GOLDEN, "bf16_rne.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        v = -0.0 if c["value"] == "-0" else eval_expr(c["value"])
        got = oracle.round_bf16(v)
        assert got == int(c["bits"], 16), (c, hex(got))


def test_bf16_rounding_matches_torch_on_fp32_values():
    # For values exactly representable in fp32, fp32->bf16 (torch, RNE) and the
    # oracle's double->bf16 must agree bit for bit.
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e30).astype(np.float32),
        (rng.standard_normal(5000) * 1e-38).astype(np.float32),     # subnormal range
        # exact ties: bf16 value plus half its spacing
        ((rng.integers(0, 1 << 15, 5000, dtype=np.uint32) << 16) | 0x8000).view(np.float32),
    ])
    vals = vals[np.isfinite(vals)]
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.round_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_outputs_round_once_from_double():
    # Build y64 values that lie strictly between a bf16 tie T and the next fp32
    # above/below it: rounding through fp32 first would land on T and then go to
    # even; the single rounding from double must go to the nearer side.
    c = 3.0 * math.sqrt(2.0) / 5.0          # x = [3, 4, 3, 4, ...], eps = 0: y = x r gamma
    cands = []
    for k in range(200):
        t = 1.0 + (2 * k + 1) * 2.0 ** -8    # a tie between two bf16 values in [1, 2)
        g0 = np.float32(t / c)
        for d in range(-3, 4):
            cands.append(np.float32(g0 + d * np.float32(2.0 ** -24)))
    g = _f32(cands)
    N = len(g)
    x = _f32(np.tile([3.0, 4.0], N // 2 + 1)[:N])
    g[1::2] = g[1::2] * np.float32(0.75)    # odd columns: x = 4, keep y near the same ties
    out = oracle.fwd(x[None, :], g, 0.0, "f32", "f32")
    y64 = out["y64"][0]
    f32 = y64.astype(np.float32).astype(np.float64)
    bits32 = y64.astype(np.float32).view(np.uint32)
    sensitive = (bits32 & 0xFFFF == 0x8000) & (y64 != f32)
    assert sensitive.sum() >= 5
    xb = np.array([oracle.round_bf16(v) for v in x], np.uint16)
    yb = oracle.fwd(xb[None, :], g, 0.0, "bf16", "f32")
    assert np.array_equal(yb["y64"][0], y64)
    for j in np.nonzero(sensitive)[0]:
        lower = int(bits32[j] >> 16)
        want = lower + 1 if y64[j] > f32[j] else lower
        assert int(yb["y"][0, j]) == want


def test_bf16_decode_is_exact():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    dec = oracle.bf16_array_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    same = (dec == ref) | (np.isnan(dec) & np.isnan(ref))
    assert same.all()
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0x0001) == 2.0 ** -133


# ---------------------------------------------------------------- hand examples

def _hand():
    with open(os.path.join(GOLDEN, "rmsnorm_hand_examples.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _hand()["forward"], ids=lambda c: c["work"][:30])
def test_forward_hand_examples(case):
    x = _f32([case["x"]])
    g = _f32(case["gamma"])
    out = oracle.fwd(x, g, case["eps"], "f32", "f32")
    want_y = np.array([eval_expr(v) for v in case["y"]])
    assert np.allclose(out["y64"][0], want_y, rtol=1e-15, atol=1e-300)
    assert math.isclose(out["rstd64"][0], eval_expr(case["rstd"]), rel_tol=1e-15)


@pytest.mark.parametrize("case", _hand()["backward"], ids=lambda c: c["work"][:30])
def test_backward_hand_examples(case):
    x = _f32([case["x"]])
    dy = _f32([case["dy"]])
    g = _f32(case["gamma"])
    out = oracle.bwd(dy, x, None, g, case["eps"], "f32", "f32")
    want_dx = np.array([eval_expr(v) for v in case["dx"]])
    want_dg = np.array([eval_expr(v) for v in case["dgamma"]])
    assert np.allclose(out["dx64"][0], want_dx, rtol=1e-14, atol=1e-15)
    assert np.allclose(out["dgamma64"], want_dg, rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("c", [1e-3, -1e-3, 1.0, -1.0, 37.0, -37.0])
@pytest.mark.parametrize("eps", [1e-6, 1e-2, 0.5])
def test_constant_row_closed_form(c, eps):
    # x_j = c for all j: mean(x^2) = c^2, so y_j = c / sqrt(c^2 + eps) * gamma_j
    N = 37
    g = _f32(np.linspace(-2, 3, N))
    x = _f32(np.full((1, N), c))
    cf = float(np.float32(c))
    out = oracle.fwd(x, g, eps, "f32", "f32")
    want = cf / math.sqrt(cf * cf + eps) * g.astype(np.float64)
    assert np.allclose(out["y64"][0], want, rtol=1e-14, atol=1e-300)


def test_scale_invariance_and_unit_mean_square_eps0():
    rng = np.random.default_rng(1)
    M, N = 5, 64
    x = _f32(rng.standard_normal((M, N)))
    g = _f32(rng.uniform(0.5, 1.5, N))
    base = oracle.fwd(x, g, 0.0, "f32", "f32")["y64"]
    # y / gamma has unit mean square per row
    ms = np.mean((base / g.astype(np.float64)) ** 2, axis=1)
    assert np.allclose(ms, 1.0, rtol=0, atol=1e-14)
    for alpha in (2.0 ** -10, 8.0, -2.0):   # exact fp32 scalings of x
        xs = _f32(x * np.float32(alpha))
        ys = oracle.fwd(xs, g, 0.0, "f32", "f32")["y64"]
        assert np.allclose(ys, math.copysign(1.0, alpha) * base, rtol=1e-14, atol=1e-300)


@pytest.mark.parametrize("eps", [0.0, 1e-3, 0.7])
def test_backward_orthogonality_identity(eps):
    # sum_j dx_j x_j = r * sum_j(gamma_j dy_j x_j) * eps / (mean(x^2) + eps); zero for eps = 0
    rng = np.random.default_rng(2)
    M, N = 6, 33
    x = _f32(rng.standard_normal((M, N)))
    dy = _f32(rng.standard_normal((M, N)))
    g = _f32(rng.normal(1.0, 0.1, N))
    out = oracle.bwd(dy, x, None, g, eps, "f32", "f32")
    x64, dy64, g64 = x.astype(np.float64), dy.astype(np.float64), g.astype(np.float64)
    ms = np.mean(x64 ** 2, axis=1)
    r = 1.0 / np.sqrt(ms + eps)
    dot = np.sum(g64 * dy64 * x64, axis=1)
    lhs = np.sum(out["dx64"] * x64, axis=1)
    rhs = r * dot * eps / (ms + eps)
    scale = r * np.sum(np.abs(g64 * dy64 * x64), axis=1)
    assert np.all(np.abs(lhs - rhs) <= 1e-13 * scale)


def test_n_equals_one():
    x = _f32([[-3.0], [0.5], [2.0 ** -20]])
    g = _f32([1.75])
    for eps in (0.0, 0.25):
        out = oracle.fwd(x, g, eps, "f32", "f32")
        xv = x[:, 0].astype(np.float64)
        want = xv / np.sqrt(xv * xv + eps) * 1.75
        assert np.allclose(out["y64"][:, 0], want, rtol=1e-15)
    out = oracle.fwd(x, g, 0.0, "f32", "f32")
    assert np.array_equal(out["y64"][:, 0], np.sign(x[:, 0]) * 1.75)


def test_zero_row_and_nan_propagation():
    g = _f32([1.0, 2.0])
    out = oracle.fwd(_f32([[0.0, 0.0]]), g, 0.25, "f32", "f32")
    assert out["rstd64"][0] == 2.0 and np.all(out["y64"] == 0.0)
    out = oracle.fwd(_f32([[0.0, 0.0]]), g, 0.0, "f32", "f32")
    assert np.all(np.isnan(out["y64"]))


# ---------------------------------------------------------------- finite differences

def _loss(x, g, dy, eps):
    return float(np.sum(dy.astype(np.float64) * oracle.fwd(x, g, eps, "f32", "f32")["y64"]))


@pytest.mark.parametrize("N", [1, 2, 3, 8, 17])
@pytest.mark.parametrize("eps", [0.0, 0.25])
def test_backward_matches_central_differences(N, eps):
    # Inputs on a 2^-8 grid and steps of 2^-10, 2^-11, so every perturbed input is
    # exact in fp32; Richardson extrapolation of two central differences leaves an
    # O(h^4) ~ 1e-12 truncation error.
    rng = np.random.default_rng(100 + N)
    M = 3
    x = _f32(np.round(rng.uniform(0.25, 2.0, (M, N)) * rng.choice([-1, 1], (M, N)) * 256) / 256)
    g = _f32(np.round(rng.uniform(0.5, 1.5, N) * 256) / 256)
    dy = _f32(np.round(rng.standard_normal((M, N)) * 256) / 256)
    out = oracle.bwd(dy, x, None, g, eps, "f32", "f32")

    def central(f, a, idx, h):
        ap, am = a.copy(), a.copy()
        ap[idx] += np.float32(h)
        am[idx] -= np.float32(h)
        return (f(ap) - f(am)) / (2 * h)

    def rich(f, a, idx):
        h = 2.0 ** -10
        return (4 * central(f, a, idx, h / 2) - central(f, a, idx, h)) / 3

    fd_dx = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            fd_dx[i, j] = rich(lambda xx: _loss(xx, g, dy, eps), x, (i, j))
    fd_dg = np.array([rich(lambda gg: _loss(x, gg, dy, eps), g, (j,)) for j in range(N)])
    scale = max(1.0, np.abs(fd_dx).max())
    assert np.abs(out["dx64"] - fd_dx).max() <= 1e-8 * scale
    scale = max(1.0, np.abs(fd_dg).max())
    assert np.abs(out["dgamma64"] - fd_dg).max() <= 1e-8 * scale


def test_backward_uses_given_rstd():
    # With rstd passed in, r is that value (eps not used): compare against the
    # closed form evaluated with the given r.
    rng = np.random.default_rng(3)
    M, N = 4, 16
    x = _f32(rng.standard_normal((M, N)))
    dy = _f32(rng.standard_normal((M, N)))
    g = _f32(rng.normal(1.0, 0.1, N))
    rstd = _f32(rng.uniform(0.5, 2.0, M))
    a = oracle.bwd(dy, x, rstd, g, 123.0, "f32", "f32")
    b = oracle.bwd(dy, x, rstd, g, 0.0, "f32", "f32")
    assert np.array_equal(a["dx64"], b["dx64"])
    r = rstd.astype(np.float64)[:, None]
    dot = np.sum(g * dy.astype(np.float64) * x, axis=1, keepdims=True)
    # the identity sum(dx x) = r dot (1 - r^2 mean(x^2)) holds for any r
    lhs = np.sum(a["dx64"] * x, axis=1, keepdims=True)
    rhs = r * dot * (1 - r * r * np.mean(x.astype(np.float64) ** 2, axis=1, keepdims=True))
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
    assert np.allclose(a["dgamma64"], np.sum(dy.astype(np.float64) * x * r, axis=0), rtol=1e-13)


# ---------------------------------------------------------------- library routines

@pytest.mark.parametrize("eps", [1e-6, 0.1])
def test_forward_matches_torch_rms_norm_f64(eps):
    rng = np.random.default_rng(4)
    M, N = 7, 129
    x = _f32(rng.standard_normal((M, N)) * 3)
    g = _f32(rng.normal(1.0, 0.2, N))
    out = oracle.fwd(x, g, eps, "f32", "f32")
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x).double(), (N,),
                                       torch.from_numpy(g).double(), eps).numpy()
    assert np.allclose(out["y64"], ref, rtol=1e-13, atol=0)


@pytest.mark.parametrize("eps", [0.0, 1e-5, 0.3])
def test_backward_matches_torch_autograd_f64(eps):
    rng = np.random.default_rng(5)
    M, N = 5, 64
    x = _f32(rng.standard_normal((M, N)))
    g = _f32(rng.normal(1.0, 0.1, N))
    dy = _f32(rng.standard_normal((M, N)))
    xt = torch.from_numpy(x).double().requires_grad_()
    gt = torch.from_numpy(g).double().requires_grad_()
    y = torch.nn.functional.rms_norm(xt, (N,), gt, eps)
    y.backward(torch.from_numpy(dy).double())
    out = oracle.bwd(dy, x, None, g, eps, "f32", "f32")
    assert np.allclose(out["dx64"], xt.grad.numpy(), rtol=1e-12, atol=1e-13)
    assert np.allclose(out["dgamma64"], gt.grad.numpy(), rtol=1e-12, atol=1e-13)


def test_bf16_path_equals_f32_path_on_decoded_values():
    # The bf16 input path decodes exactly, so it matches the fp32 path fed with
    # the decoded values; outputs are the oracle's bf16 rounding of y64.
    rng = np.random.default_rng(6)
    M, N = 4, 40
    xb = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).to(torch.bfloat16)
    gb = torch.from_numpy(rng.normal(1, 0.1, N).astype(np.float32)).to(torch.bfloat16)
    xbits = xb.view(torch.int16).numpy().view(np.uint16)
    gbits = gb.view(torch.int16).numpy().view(np.uint16)
    a = oracle.fwd(xbits, gbits, 1e-5, "bf16", "bf16")
    b = oracle.fwd(_f32(xb.float().numpy()), _f32(gb.float().numpy()), 1e-5, "f32", "f32")
    assert np.array_equal(a["y64"], b["y64"])
    want = np.array([oracle.round_bf16(v) for v in a["y64"].ravel()], np.uint16).reshape(M, N)
    assert np.array_equal(a["y"], want)
    c = oracle.fwd(xbits, _f32(gb.float().numpy()), 1e-5, "bf16", "f32")
    assert np.array_equal(c["y64"], a["y64"])


# ---------------------------------------------------------------- fused add

def test_fused_add_reduces_to_forward():
    rng = np.random.default_rng(8)
    M, N = 3, 24
    x = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).to(torch.bfloat16)
    g = torch.from_numpy(rng.normal(1, 0.1, N).astype(np.float32)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    gb = g.view(torch.int16).numpy().view(np.uint16)
    zero = np.zeros((M, N), np.uint16)
    f = oracle.fwd(xb, gb, 1e-6, "bf16")
    a = oracle.fused_add_fwd(xb, zero, gb, 1e-6, "bf16")     # r = 0
    b = oracle.fused_add_fwd(zero, xb, gb, 1e-6, "bf16")     # x = 0
    for o in (a, b):
        assert np.array_equal(o["h"], xb)
        assert np.array_equal(o["y"], f["y"])
        assert np.array_equal(o["rstd"], f["rstd"])


def test_fused_add_residual_matches_torch_bf16_add():
    # h = residual + x stored in bf16: torch adds bf16 tensors in fp32 and rounds
    # to nearest even, which is the correctly rounded sum for bf16 operands.
    rng = np.random.default_rng(9)
    M, N = 8, 100
    r = torch.from_numpy((rng.standard_normal((M, N)) * 30).astype(np.float32)).to(torch.bfloat16)
    x = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).to(torch.bfloat16)
    g = torch.ones(N, dtype=torch.bfloat16)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    out = oracle.fused_add_fwd(bits(x), bits(r), bits(g), 1e-6, "bf16")
    assert np.array_equal(out["h"], bits(r + x))
    # y is the forward of the stored h, not of the unrounded sum
    f = oracle.fwd(bits(r + x), bits(g), 1e-6, "bf16")
    assert np.array_equal(out["y64"], f["y64"])


# ---------------------------------------------------------------- fused add, backward

@pytest.mark.parametrize("eps", [0.0, 1e-5, 0.3])
def test_fused_add_backward_matches_torch_autograd_f64(eps):
    # h = r + x, y = rms_norm(h) * gamma; loss = sum(dy y) + sum(dres h): the
    # gradient of r and of x is dh = dx_rms(h) + dres
    rng = np.random.default_rng(21)
    M, N = 5, 48
    r = _f32(rng.standard_normal((M, N)))
    x = _f32(rng.standard_normal((M, N)))
    g = _f32(rng.normal(1.0, 0.1, N))
    dy = _f32(rng.standard_normal((M, N)))
    dres = _f32(rng.standard_normal((M, N)))
    h = _f32(r.astype(np.float64) + x)       # the stored h
    rt = torch.from_numpy(r).double().requires_grad_()
    xt = torch.from_numpy(x).double().requires_grad_()
    gt = torch.from_numpy(g).double().requires_grad_()
    s_ = rt + xt
    # value: the stored h (fp32 rounding of the sum); gradient: that of h = r + x
    ht = s_.detach().float().double() + (s_ - s_.detach())
    y = torch.nn.functional.rms_norm(ht, (N,), gt, eps)
    loss = (torch.from_numpy(dy).double() * y).sum() + (torch.from_numpy(dres).double() * ht).sum()
    loss.backward()
    out = oracle.fused_add_bwd(dy, h, None, g, dres, eps, "f32", "f32")
    assert np.allclose(out["dh64"], xt.grad.numpy(), rtol=1e-11, atol=1e-12)
    assert np.allclose(out["dh64"], rt.grad.numpy(), rtol=1e-11, atol=1e-12)
    assert np.allclose(out["dgamma64"], gt.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_fused_add_backward_reduces_to_backward():
    rng = np.random.default_rng(22)
    M, N = 4, 40
    h = _f32(rng.standard_normal((M, N)))
    g = _f32(rng.normal(1.0, 0.1, N))
    dy = _f32(rng.standard_normal((M, N)))
    zero = np.zeros((M, N), np.float32)
    a = oracle.fused_add_bwd(dy, h, None, g, zero, 1e-5, "f32", "f32")
    b = oracle.bwd(dy, h, None, g, 1e-5, "f32", "f32")
    assert np.array_equal(a["dh64"], b["dx64"]) and np.array_equal(a["dgamma64"], b["dgamma64"])
    # and the residual gradient passes straight through where dy = 0
    dres = _f32(rng.standard_normal((M, N)))
    c = oracle.fused_add_bwd(np.zeros_like(dy), h, None, g, dres, 1e-5, "f32", "f32")
    assert np.array_equal(c["dh64"], dres.astype(np.float64))


def test_fused_add_backward_weight_dtype_gradient_is_rounded_once():
    rng = np.random.default_rng(23)
    M, N = 6, 24
    bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    h = bits(rng.standard_normal((M, N)).astype(np.float32))
    dy = bits(rng.standard_normal((M, N)).astype(np.float32))
    dres = bits(rng.standard_normal((M, N)).astype(np.float32))
    g = bits(rng.normal(1, 0.1, N).astype(np.float32))
    out = oracle.fused_add_bwd(dy, h, None, g, dres, 1e-5, "bf16", "bf16")
    want = np.array([oracle.round_bf16(v) for v in out["dgamma64"]], np.uint16)
    assert np.array_equal(out["dgamma_w"], want)
    want_dh = np.array([oracle.round_bf16(v) for v in out["dh64"].ravel()], np.uint16)
    assert np.array_equal(out["dh"].ravel(), want_dh)


# ---------------------------------------------------------------- strided rows

def test_strided_rows_equal_contiguous_rows_and_torch():
    # q of a fused QKV projection: [T, Hq, D] rows inside a [T, (Hq + 2 Hk) D] buffer
    rng = np.random.default_rng(31)
    T, Hq, Hk, D = 5, 3, 1, 16
    width = (Hq + 2 * Hk) * D
    buf = _f32(rng.standard_normal((T, width)))
    g = _f32(rng.normal(1.0, 0.1, D))
    out = oracle.fwd_strided(buf, width, D, g, T, Hq, D, 1e-5, "f32", "f32")
    q = buf[:, :Hq * D].reshape(T * Hq, D)
    ref = oracle.fwd(np.ascontiguousarray(q), g, 1e-5, "f32", "f32")
    assert np.array_equal(out["y64"], ref["y64"])
    assert np.array_equal(out["rstd"], ref["rstd"])
    yq = out["y"].reshape(-1)[: T * width].reshape(T, width)[:, :Hq * D].reshape(T * Hq, D)
    assert np.array_equal(yq, ref["y"])
    # untouched elements (the k and v columns) stay zero in the output buffer
    assert (out["y"].reshape(-1)[: T * width].reshape(T, width)[:, Hq * D:] == 0).all()
    t = torch.nn.functional.rms_norm(torch.from_numpy(buf).double().view(T, -1, D)[:, :Hq],
                                     (D,), torch.from_numpy(g).double(), 1e-5)
    assert np.allclose(out["y64"].reshape(T, Hq, D), t.numpy(), rtol=1e-13, atol=0)


def test_strided_rows_follow_both_strides():
    # output rows at different strides than the input rows
    rng = np.random.default_rng(32)
    T, H, D = 3, 4, 8
    x = _f32(rng.standard_normal((T, H, D)))
    g = _f32(rng.uniform(0.5, 1.5, D))
    out = oracle.fwd_strided(x, H * D, D, g, T, H, D, 0.0, "f32", "f32", y_st=D, y_sh=T * D)
    ref = oracle.fwd(x.reshape(T * H, D), g, 0.0, "f32", "f32")["y"].reshape(T, H, D)
    y = out["y"].reshape(H, T, D)      # y[h, t] holds row (t, h)
    assert np.array_equal(y.transpose(1, 0, 2), ref)
