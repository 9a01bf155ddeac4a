"""Pins of the oracle's quantised outputs (FP8 E4M3 per-row scale, NVFP4
blocks of 16 with E4M3 scales) to facts outside themselves: torch's
float8_e4m3fn conversion, the E2M1 value table with a brute-force nearest
search, hand-worked examples, and invariants of the definitions (scale
invariance, exact powers of two, all-zero rows and blocks, the error bound of
the formats against the pinned forward)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import GOLDEN

E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # magnitudes of codes 0..7


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _torch_e4m3(vals):
    return torch.from_numpy(_f32(vals)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ---------------------------------------------------------------- E4M3

def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_values()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_rounding_matches_torch_within_range():
    # every finite value, every midpoint between neighbours (the ties) and
    # random fp32 values over the whole range, subnormals included
    vals = oracle.e4m3_values()
    pos = np.unique(vals[np.isfinite(vals) & (vals >= 0)])
    mids = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(3)
    rnd = np.exp2(rng.uniform(-12, np.log2(448.0), 20000)) * rng.choice([-1, 1], 20000)
    x = _f32(np.concatenate([pos, -pos, mids, -mids, rnd]))
    x = x[np.abs(x) <= 448]
    got = np.array([oracle.round_e4m3(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, _torch_e4m3(x))


def test_e4m3_saturates_and_keeps_nan():
    # the finite-saturating conversion: beyond 448 the code stays at +-448
    for v in (449.0, 464.0, 479.9, 480.0, 1e6, float("inf")):
        assert oracle.round_e4m3(v) == 0x7E and oracle.round_e4m3(-v) == 0xFE
    assert oracle.round_e4m3(float("nan")) == 0x7F
    assert oracle.round_e4m3(-0.0) == 0x80 and oracle.round_e4m3(0.0) == 0x00


# ---------------------------------------------------------------- E2M1

def test_e2m1_decode_table():
    got = oracle.e2m1_values()
    assert list(got[:8]) == E2M1_TABLE
    assert list(got[8:]) == [-v for v in E2M1_TABLE]


def _nearest_e2m1(v):
    """Brute force: the table entry nearest to |v| (ties: the even code),
    saturating at 6."""
    a = min(abs(v), 6.0)
    d = [abs(a - t) for t in E2M1_TABLE]
    best = min(d)
    cands = [c for c in range(8) if d[c] == best]
    c = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
    return c | (8 if np.signbit(v) else 0)


def test_e2m1_rounding_against_brute_force():
    mids = [(a + b) / 2 for a, b in zip(E2M1_TABLE[:-1], E2M1_TABLE[1:])]
    rng = np.random.default_rng(5)
    vals = E2M1_TABLE + mids + list(rng.uniform(-8, 8, 5000)) + [7.0, 100.0, 1e30]
    vals += [-v for v in vals]
    for v in vals:
        assert oracle.round_e2m1(v) == _nearest_e2m1(v), v
    # the ties by name: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for v, c in ties.items():
        assert oracle.round_e2m1(v) == c


# ---------------------------------------------------------------- hand examples

def _golden():
    with open(os.path.join(GOLDEN, "quant_hand_examples.json")) as f:
        return json.load(f)


def test_fp8_hand_example():
    for c in _golden()["fp8"]:
        out = oracle.fwd_fp8(_f32(c["x"]), _f32(c["gamma"]), c["eps"], "f32", "f32")
        assert out["q"].tolist() == c["q"]
        np.testing.assert_allclose(out["scale64"], c["scale"], rtol=1e-15)


def test_nvfp4_hand_examples():
    for c in _golden()["nvfp4"]:
        out = oracle.fwd_nvfp4(_f32(c["x"]), _f32(c["gamma"]), c["gs"], c["eps"], "f32", "f32")
        assert out["sf"].tolist() == c["sf"], c["note"]
        assert out["q"].tolist() == c["q"], c["note"]


# ---------------------------------------------------------------- invariants

def _rows(M, N, seed, dtype="bf16"):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, N))
    g = 1.0 + 0.1 * rng.standard_normal(N)
    if dtype == "bf16":
        return (np.array([oracle.round_bf16(v) for v in x.reshape(-1)], np.uint16).reshape(M, N),
                np.array([oracle.round_bf16(v) for v in g], np.uint16))
    return _f32(x), _f32(g)


def test_fp8_row_maximum_maps_to_448_and_error_bound():
    x, g = _rows(6, 96, 1)
    out = oracle.fwd_fp8(x, g, 1e-6, "bf16", "bf16")
    y64 = oracle.fwd(x, g, 1e-6, "bf16", "bf16")["y64"]
    jmax = np.abs(y64).argmax(axis=1)
    for i, j in enumerate(jmax):
        assert out["q"][i, j] in (0x7E, 0xFE)
        assert (out["q"][i, j] == 0xFE) == (y64[i, j] < 0)
    np.testing.assert_allclose(out["scale64"], np.abs(y64).max(axis=1) / 448, rtol=1e-15)
    deq = oracle.e4m3_values()[out["q"]] * out["scale64"][:, None]
    # E4M3: half a spacing is 2^-4 of the value for normals, 2^-10 below 2^-6
    bound = np.maximum(np.abs(y64) * 2.0 ** -4, 2.0 ** -10 * out["scale64"][:, None])
    assert np.all(np.abs(deq - y64) <= bound * (1 + 1e-12))


def test_fp8_constant_rows_closed_form():
    N = 64
    for c in (1e-3, 1.0, -37.0):
        x = _f32(np.full((1, N), c))
        g = _f32(np.full(N, 0.75))
        eps = 1e-6
        out = oracle.fwd_fp8(x, g, eps, "f32", "f32")
        assert np.all(out["q"] == (0xFE if c < 0 else 0x7E))
        y = float(np.float32(c)) / np.sqrt(float(np.float32(c)) ** 2 + eps) * 0.75
        np.testing.assert_allclose(out["scale64"][0], abs(y) / 448, rtol=1e-14)


@pytest.mark.parametrize("alpha", [2.0 ** -10, 8.0, -2.0, -0.5])
def test_fp8_and_nvfp4_scale_invariance_at_eps_zero(alpha):
    # powers of two scale x exactly, so y(alpha x) = sign(alpha) y(x) exactly
    x, g = _f32(np.random.default_rng(2).standard_normal((4, 64))), _f32(np.ones(64) * 1.25)
    xa = _f32(x * np.float32(alpha))
    flip = 0x80 if alpha < 0 else 0
    a, b = oracle.fwd_fp8(x, g, 0.0, "f32", "f32"), oracle.fwd_fp8(xa, g, 0.0, "f32", "f32")
    assert np.array_equal(b["q"], a["q"] ^ flip)
    np.testing.assert_allclose(b["scale64"], a["scale64"], rtol=1e-15)
    a, b = (oracle.fwd_nvfp4(x, g, 448.0, 0.0, "f32", "f32"),
            oracle.fwd_nvfp4(xa, g, 448.0, 0.0, "f32", "f32"))
    assert np.array_equal(b["sf"], a["sf"])
    codes_a, codes_b = oracle.unpack_e2m1(a["q"]), oracle.unpack_e2m1(b["q"])
    nz = (codes_a & 7) != 0
    assert np.array_equal(codes_b[nz], codes_a[nz] ^ (8 if alpha < 0 else 0))


def test_nvfp4_global_scale_power_of_two_shifts_only_the_block_exponent():
    # doubling gs doubles every gs * amax / 6 exactly: the E4M3 block codes
    # move up one binade (code + 8 for normals) and the E2M1 codes stay
    x, g = _rows(4, 128, 8)
    a = oracle.fwd_nvfp4(x, g, 100.0, 1e-6, "bf16", "bf16")
    b = oracle.fwd_nvfp4(x, g, 200.0, 1e-6, "bf16", "bf16")
    normal = (a["sf"] & 0x78) != 0
    assert normal.all()
    assert np.array_equal(b["sf"].astype(int), a["sf"].astype(int) + 8)
    assert np.array_equal(b["q"], a["q"])


def test_nvfp4_block_maximum_error_bound_and_scales():
    x, g = _rows(5, 256, 9)
    gs = 448.0 * 6 / 5.0
    out = oracle.fwd_nvfp4(x, g, gs, 1e-6, "bf16", "bf16")
    y64 = oracle.fwd(x, g, 1e-6, "bf16", "bf16")["y64"]
    M, N = y64.shape
    blocks = y64.reshape(M, N // 16, 16)
    amax = np.abs(blocks).max(axis=2)
    np.testing.assert_allclose(out["sfv64"], gs * amax / 6, rtol=1e-15)
    S = oracle.e4m3_values()[out["sf"]]
    assert np.array_equal(out["sf"], np.vectorize(oracle.round_e4m3)(_f32(gs * amax / 6)))
    codes = oracle.unpack_e2m1(out["q"]).reshape(M, N // 16, 16)
    # the element of largest magnitude lands on +-6
    jm = np.abs(blocks).argmax(axis=2)
    top = np.take_along_axis(codes, jm[..., None], axis=2)[..., 0]
    assert np.all((top & 7) == 7)
    # dequantised error: at most half an E2M1 spacing at the scaled value
    deq = oracle.e2m1_values()[codes] * (S / gs)[..., None]
    v = np.abs(blocks) * (gs / S)[..., None]
    half = np.where(v < 2, 0.25, np.where(v < 4, 0.5, 1.0)) + np.maximum(v - 6, 0)
    assert np.all(np.abs(deq - blocks) <= half * (S / gs)[..., None] * (1 + 1e-12))


@pytest.mark.parametrize("eps", [0.0, 1e-6])
def test_zero_rows_and_blocks_quantise_to_zero(eps):
    x = _f32(np.zeros((2, 32)))
    x[1, 16:] = 1.0                                # row 1: block 0 zero, block 1 not
    g = _f32(np.ones(32))
    f8 = oracle.fwd_fp8(x, g, eps, "f32", "f32")
    assert np.all(f8["q"][0] == 0) and f8["scale"][0] == 0.0
    f4 = oracle.fwd_nvfp4(x, g, 6.0, eps, "f32", "f32")
    assert np.all(f4["q"][0] == 0) and np.all(f4["sf"][0] == 0)
    assert np.all(f4["q"][1, :8] == 0) and f4["sf"][1, 0] == 0 and f4["sf"][1, 1] != 0


def test_fused_add_reduces_to_the_plain_forward():
    x, g = _rows(3, 64, 11)
    zero = np.zeros_like(x)
    for fn, kw in ((oracle.fwd_fp8, {}), (oracle.fwd_nvfp4, {"gs": 300.0})):
        args = (lambda a, r=None: fn(a, g, eps=1e-6, x_dtype="bf16", w_dtype="bf16", residual=r,
                                     **kw))
        plain = args(x)
        for a, r in ((x, zero), (zero, x)):
            fused = args(a, r)
            assert np.array_equal(fused["q"], plain["q"])
            assert np.array_equal(fused["h"], x)
    # and h is the fused-add forward's stored sum
    r, _ = _rows(3, 64, 12)
    out = oracle.fwd_fp8(x, g, 1e-6, "bf16", "bf16", residual=r)
    assert np.array_equal(out["h"], oracle.fused_add_fwd(x, r, g, 1e-6, "bf16", "bf16")["h"])


def test_quantised_oracles_reject_bad_arguments():
    x, g = _f32(np.ones((2, 24))), _f32(np.ones(24))
    with pytest.raises(ValueError):
        oracle.fwd_nvfp4(x, g, 6.0, 1e-6, "f32", "f32")          # N not a multiple of 16
    x, g = _f32(np.ones((2, 32))), _f32(np.ones(32))
    for gs in (0.0, -1.0, float("nan")):
        with pytest.raises(ValueError):
            oracle.fwd_nvfp4(x, g, gs, 1e-6, "f32", "f32")
