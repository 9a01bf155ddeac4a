"""GPU LayerNorm forward and backward against the oracle, element by element.

Bounds (those of the RMSNorm parity tests): bf16 outputs within 2 bf16 ulp of
the oracle's once-rounded value, fp32 outputs within 1e-5 (1 + |ref|), the
weight gradients within 1e-4 of max(|ref|, sqrt(sum of squared terms)).  Two
sums can cancel: y = t * gamma + beta and dx = rstd (g - mean(g) - xhat
mean(g xhat)), and so can x - mean inside both; where they do, an fp32
evaluation is bounded by a few fp32 roundings of the terms (x r gamma,
mean(|x|) r gamma for the computed mean's own rounding, beta; the three dx
terms with xhat's own) plus, in the forward,
rstd's relative error (the 1e-5 its own check allows) times |t gamma| -- not
by roundings of the result -- so a bf16 element beyond 2 ulp is accepted only
within 2 ulp plus that floor, and the test counts how many needed it.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity_util as pu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import row_wise_normalization_02_gb300 as rn  # noqa: E402

U32 = 2.0 ** -24


def f32(v):
    return float(np.float32(v))


def inputs(M, N, xd, wd, seed, beta=True, mean=0.0):
    x = si.fill((M, N), seed=seed, tensor_id=1, dtype=xd, p0=mean)
    g = si.fill(N, seed=seed, tensor_id=3, p0=1.0, p1=0.1, dtype=wd)
    b = si.fill(N, seed=seed, tensor_id=5, p0=0.0, p1=0.1, dtype=wd) if beta else None
    dy = si.fill((M, N), seed=seed, tensor_id=4, dtype=xd)
    return x, g, b, dy


# ---------------------------------------------------------------- runners

def run_fwd(x, g, b, eps, xd, wd, offsets=None):
    M, N = x.shape
    o = offsets or {}
    bx, bg = pu.dev(x, o.get("x", 0)), pu.dev(g, o.get("gamma", 0))
    bb = pu.dev(b, o.get("beta", 0)) if b is not None else None
    by = pu.empty(M * N, xd, o.get("y", 0))
    bm, br = pu.empty(M, "f32"), pu.empty(M, "f32")
    rn.layernorm_fwd(bx.ptr, bg.ptr, bb.ptr if bb else None, by.ptr, bm.ptr, br.ptr, M, N, eps,
                     xd, wd)
    torch.cuda.synchronize()
    for buf in (bx, bg, bb, by, bm, br):
        if buf is not None:
            assert buf.guards_ok(), "write outside a buffer"
    return {"y": by.download(pu.np_dtype(xd)).reshape(M, N), "mean": bm.download(np.float32),
            "rstd": br.download(np.float32)}


def run_bwd(dy, x, mean, rstd, g, eps, xd, wd, want=(True, True), offsets=None):
    M, N = x.shape
    o = offsets or {}
    bdy, bx, bg = pu.dev(dy, o.get("dy", 0)), pu.dev(x, o.get("x", 0)), pu.dev(g, o.get("gamma", 0))
    bm = pu.dev(mean) if mean is not None else None
    br = pu.dev(rstd) if rstd is not None else None
    bdx = pu.empty(M * N, xd, o.get("dx", 0))
    bdg = pu.empty(N, "f32") if want[0] else None
    bdb = pu.empty(N, "f32") if want[1] else None
    ws = rn.layernorm_bwd_workspace_size(M, N, xd, wd)
    bws = pu.Buf(max(ws, 16))
    rn.layernorm_bwd(bdy.ptr, bx.ptr, bm.ptr if bm else None, br.ptr if br else None, bg.ptr,
                     bdx.ptr, bdg.ptr if bdg else None, bdb.ptr if bdb else None, bws.ptr, ws,
                     M, N, eps, xd, wd)
    torch.cuda.synchronize()
    for buf in (bdy, bx, bg, bm, br, bdx, bdg, bdb, bws):
        if buf is not None:
            assert buf.guards_ok(), "write outside a buffer"
    out = {"dx": bdx.download(pu.np_dtype(xd)).reshape(M, N)}
    if bdg:
        out["dgamma"] = bdg.download(np.float32)
    if bdb:
        out["dbeta"] = bdb.download(np.float32)
    return out


# ---------------------------------------------------------------- checks

def _bf16_with_floor(gpu_bits, ref_bits, ref64, floor, what):
    d = pu.bf16_ulp_dist(gpu_bits, ref_bits)
    strict = d > 2
    if strict.any():
        gv = oracle.bf16_array_to_f64(gpu_bits)
        ok = np.abs(gv - ref64) <= 2 * pu.bf16_ulp_of(ref64) + floor
        bad = strict & ~ok
        assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond 2 ulp and the "
                               f"cancellation floor, at {np.argwhere(bad)[:5].tolist()}")
        # rows shorter than 32 cancel by construction (N = 1: x - mean = 0 and
        # dx = 0 exactly; N = 2: xhat = +-sqrt(var / (var + eps)), so dx is an
        # eps-sized sliver of its terms), so the count is capped for longer
        # rows only, as for the RMSNorm dx
        N = d.shape[-1] if d.ndim > 1 else d.size
        assert N < 32 or strict.sum() <= max(2, 1e-4 * d.size), (
            f"{what}: {int(strict.sum())} of {d.size} elements needed the cancellation floor")
    return int(strict.sum())


def check_fwd(out, x, g, b, eps, xd, wd):
    ref = oracle.layernorm_fwd(x, g, b, eps, xd, wd)
    pu.check_f32(out["mean"], ref["mean64"], what="mean")
    pu.check_f32(out["rstd"], ref["rstd64"], what="rstd")
    if xd == "bf16":
        # y = (x - mean) r gamma + beta: the terms are x r gamma, mean r gamma
        # and beta, and both sums can cancel.  A computed row mean rounds on
        # the scale of the row's mean |x| (the sum of magnitudes), not of
        # |mean|; rstd's own fp32 error (bounded by the 1e-5 checked above)
        # scales the term t gamma = y - beta.
        bv = oracle.to_f64(b, wd) if b is not None else np.zeros(x.shape[1])
        x64 = oracle.to_f64(x, xd)
        rg = ref["rstd64"][:, None] * np.abs(oracle.to_f64(g, wd))[None, :]
        floor = (16 * U32 * (rg * (np.abs(x64) + np.abs(x64).mean(axis=1, keepdims=True))
                             + np.abs(bv)[None, :]) +
                 1e-5 * np.abs(ref["y64"] - bv[None, :]))
        return _bf16_with_floor(out["y"], ref["y"], ref["y64"], floor, "y")
    pu.check_f32(out["y"], ref["y64"], what="y")
    return 0


def check_bwd(out, dy, x, mean, rstd, g, eps, xd, wd):
    ref = oracle.layernorm_bwd(dy, x, mean, rstd, g, eps, xd, wd)
    x64, dy64, g64 = oracle.to_f64(x, xd), oracle.to_f64(dy, xd), oracle.to_f64(g, wd)
    if mean is None:
        fw = oracle.layernorm_fwd(x, g, None, eps, xd, wd)
        mu, r = fw["mean64"], fw["rstd64"]
    else:
        mu, r = mean.astype(np.float64), rstd.astype(np.float64)
    xh = (x64 - mu[:, None]) * r[:, None]
    gg = dy64 * g64[None, :]
    n = 0
    N = x.shape[1]
    # xhat = (x - mean) r itself carries the cancellation of x - mean
    xh_mag = np.abs(xh) + r[:, None] * (np.abs(x64) + np.abs(x64).mean(axis=1, keepdims=True))
    floor = 64 * U32 * r[:, None] * (np.abs(gg) + np.abs(gg).sum(1, keepdims=True) / N +
                                     xh_mag * np.abs(gg * xh).sum(1, keepdims=True) / N)
    if xd == "bf16":
        n = _bf16_with_floor(out["dx"], ref["dx"], ref["dx64"], floor, "dx")
    elif N < 32:
        # rows shorter than 32 cancel by construction (N = 1: dx = 0 exactly,
        # its terms r dy gamma with r up to eps^-1/2): the floor on the terms'
        # scale joins 1e-5 (1 + |ref|) there (reading R22)
        err = np.abs(out["dx"].astype(np.float64) - ref["dx64"])
        lim = 1e-5 * (1 + np.abs(ref["dx64"])) + floor
        assert (err <= lim).all(), (f"dx: {int((err > lim).sum())} elements beyond "
                                    f"1e-5(1+|ref|) and the cancellation floor")
    else:
        pu.check_f32(out["dx"], ref["dx64"], what="dx")
    if "dgamma" in out:
        # recomputed statistics: the kernel's fp32 mean rounds on the scale of
        # the row's magnitudes, so each term dy * xhat carries up to a few fp32
        # units of mean(|x|) r |dy| (the forward's 16-unit floor, reading R22);
        # it shows where few rows are summed and xhat is near zero
        dg_floor = None
        if mean is None:
            dg_floor = (16 * U32 * np.abs(dy64) * (r[:, None] *
                        np.abs(x64).mean(axis=1, keepdims=True))).sum(0)
        pu.check_dgamma(out["dgamma"], ref["dgamma64"], ((dy64 * xh) ** 2).sum(0),
                        floor=dg_floor)
    if "dbeta" in out:
        pu.check_dgamma(out["dbeta"], ref["dbeta64"], (dy64 ** 2).sum(0))
    return n


PAIRS = [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32")]


# ---------------------------------------------------------------- forward

@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N", [16, 128, 1000, 4096, 8192, 2049])
@pytest.mark.parametrize("beta", [True, False])
def test_forward(xd, wd, N, beta):
    x, g, b, _ = inputs(300, N, xd, wd, seed=N, beta=beta, mean=0.5)
    out = run_fwd(x, g, b, f32(1e-5), xd, wd)
    check_fwd(out, x, g, b, f32(1e-5), xd, wd)


@pytest.mark.parametrize("force", ["subwarp:g=16:vpt=1:cps=1", "subwarp:g=32:vpt=1:pf=0:cps=1",
                                   "subwarp:g=8:vpt=2:cps=1", "cta:vpt=1:cps=1",
                                   "cta:vpt=2:t=64:cps=1", "cta:vpt=4:t=32:pf=0:cps=1",
                                   "generic:cps=1"])
def test_forward_forced_variants_walk_many_rows(debug_env, force):
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    x, g, b, _ = inputs(2000, 128, "bf16", "bf16", seed=3)
    check_fwd(run_fwd(x, g, b, f32(1e-5), "bf16", "bf16"), x, g, b, f32(1e-5), "bf16", "bf16")


def test_forward_unaligned_pointers_and_constant_rows():
    x, g, b, _ = inputs(40, 256, "bf16", "bf16", seed=4)
    x[3] = x[3, 0]                      # a constant row: y = beta
    out = run_fwd(x, g, b, f32(1e-5), "bf16", "bf16", offsets={"x": 2, "y": 2})
    check_fwd(out, x, g, b, f32(1e-5), "bf16", "bf16")
    assert np.array_equal(out["y"][3], b)


def test_forward_large_mean_small_spread():
    # mean 64, unit spread: the two-pass variance keeps rstd accurate
    x, g, b, _ = inputs(64, 4096, "f32", "f32", seed=5, mean=64.0)
    check_fwd(run_fwd(x, g, b, f32(1e-5), "f32", "f32"), x, g, b, f32(1e-5), "f32", "f32")


# ---------------------------------------------------------------- backward

@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N", [16, 128, 1000, 4096, 8192, 2049])
@pytest.mark.parametrize("saved", [True, False])
def test_backward(xd, wd, N, saved):
    x, g, _, dy = inputs(300, N, xd, wd, seed=N + 1)
    eps = f32(1e-5)
    fw = oracle.layernorm_fwd(x, g, None, eps, xd, wd) if saved else None
    mean, rstd = (fw["mean"], fw["rstd"]) if saved else (None, None)
    out = run_bwd(dy, x, mean, rstd, g, eps, xd, wd)
    check_bwd(out, dy, x, mean, rstd, g, eps, xd, wd)


@pytest.mark.parametrize("force", ["subwarp:g=16:vpt=1:cps=1", "subwarp:g=32:vpt=1:pf=0:cps=1",
                                   "subwarp:g=4:vpt=1:cps=1", "cta:vpt=1:cps=1",
                                   "cta:vpt=2:t=64:cps=1", "cta:vpt=2:t=64:pf=0:cps=1",
                                   "staged:vpt=1:st=2:cps=1", "staged:vpt=2:t=64:st=3:cps=1",
                                   "staged:vpt=4:t=32:st=8:cps=1", "generic:cps=1", "generic",
                                   # short rows through the ring, 256 / g rows per stage
                                   "staged:g=32:vpt=4:cps=1", "staged:g=32:vpt=3:st=2:cps=1",
                                   "staged:g=16:vpt=2:st=4:cps=1", "staged:g=8:vpt=1:st=3:cps=1"])
@pytest.mark.parametrize("N", [128, 32, 1024, 760])
def test_backward_forced_variants_walk_many_rows(debug_env, force, N):
    if "g=4" in force and N != 32:
        pytest.skip("4 lanes hold at most 4 vectors")
    if N >= 760 and "staged:g=" not in force:
        pytest.skip("the short-row sizes are for the ring forms")
    import re
    m = re.search(r"g=(\d+):vpt=(\d+)", force)
    if m and int(m.group(1)) * int(m.group(2)) * 8 < N:
        pytest.skip("the forced lanes do not hold the row")
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    x, g, _, dy = inputs(3000, N, "bf16", "bf16", seed=6)
    fw = oracle.layernorm_fwd(x, g, None, f32(1e-5), "bf16", "bf16")
    out = run_bwd(dy, x, fw["mean"], fw["rstd"], g, f32(1e-5), "bf16", "bf16")
    check_bwd(out, dy, x, fw["mean"], fw["rstd"], g, f32(1e-5), "bf16", "bf16")


@pytest.mark.parametrize("saved,force,N", [(True, "staged:vpt=4:st=3", 8192),
                                           (False, "staged:vpt=4:st=3", 8192),
                                           (True, "staged:g=32:vpt=4:st=3", 1024),
                                           (False, "staged:g=32:vpt=4:st=3", 1024)])
def test_backward_staged_wait_timeout_is_reported_and_the_context_survives(debug_env, saved,
                                                                           force, N):
    # a negative wait limit: every wait for a row gives up at once; the kernel
    # stores nothing more, drains its copies and raises the flag that
    # rmsnorm_check_device reports and clears
    x, g, _, dy = inputs(1024 if N > 1024 else 4000, N, "bf16", "bf16", seed=44)
    fw = oracle.layernorm_fwd(x, g, None, f32(1e-5), "bf16", "bf16")
    mean, rstd = (fw["mean"], fw["rstd"]) if saved else (None, None)
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    rn.rmsnorm_check_device()
    debug_env.set("RMSNORM_WAIT_LIMIT_CYCLES", "-1")
    run_bwd(dy, x, mean, rstd, g, f32(1e-5), "bf16", "bf16")
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_check_device()
    assert e.value.status == 6
    rn.rmsnorm_check_device()
    debug_env.delete("RMSNORM_WAIT_LIMIT_CYCLES")
    out = run_bwd(dy, x, mean, rstd, g, f32(1e-5), "bf16", "bf16")
    check_bwd(out, dy, x, mean, rstd, g, f32(1e-5), "bf16", "bf16")
    rn.rmsnorm_check_device()


def test_backward_weight_gradients_are_deterministic_and_optional():
    x, g, _, dy = inputs(4096, 1024, "bf16", "bf16", seed=7)
    a = run_bwd(dy, x, None, None, g, f32(1e-5), "bf16", "bf16")
    b = run_bwd(dy, x, None, None, g, f32(1e-5), "bf16", "bf16")
    assert np.array_equal(a["dgamma"], b["dgamma"]) and np.array_equal(a["dbeta"], b["dbeta"])
    only = run_bwd(dy, x, None, None, g, f32(1e-5), "bf16", "bf16", want=(False, True))
    assert np.array_equal(only["dbeta"], a["dbeta"]) and np.array_equal(only["dx"], a["dx"])
    none = run_bwd(dy, x, None, None, g, f32(1e-5), "bf16", "bf16", want=(False, False))
    assert np.array_equal(none["dx"], a["dx"])


def test_backward_unaligned_pointers():
    x, g, _, dy = inputs(50, 384, "bf16", "bf16", seed=8)
    out = run_bwd(dy, x, None, None, g, f32(1e-5), "bf16", "bf16",
                  offsets={"x": 2, "dy": 4, "dx": 6})
    check_bwd(out, dy, x, None, None, g, f32(1e-5), "bf16", "bf16")


def test_zero_rows():
    rn.layernorm_fwd(None, None, None, None, None, None, 0, 64, 1e-5, "bf16", "bf16")
    dg, db = torch.full((64,), 7.0, device="cuda"), torch.full((64,), 7.0, device="cuda")
    rn.layernorm_bwd(None, None, None, None, None, None, dg.data_ptr(), db.data_ptr(), None, 0, 0,
                     64, 1e-5, "bf16", "bf16")
    torch.cuda.synchronize()
    assert float(dg.abs().sum()) == 0.0 and float(db.abs().sum()) == 0.0


def check_workload(wl, inp):
    """A LayerNorm workload at full size through the default dispatch."""
    x, g = inp["x"], inp["gamma"]
    eps = f32(wl.eps)
    if wl.op == "ln_fwd":
        b = inp.get("beta")
        n = check_fwd(run_fwd(x, g, b, eps, wl.x_dtype, wl.w_dtype), x, g, b, eps, wl.x_dtype,
                      wl.w_dtype)
    else:
        fw = oracle.layernorm_fwd(x, g, None, eps, wl.x_dtype, wl.w_dtype)
        out = run_bwd(inp["dy"], x, fw["mean"], fw["rstd"], g, eps, wl.x_dtype, wl.w_dtype)
        n = check_bwd(out, inp["dy"], x, fw["mean"], fw["rstd"], g, eps, wl.x_dtype, wl.w_dtype)
    print(wl.name, {"floor": n})


@pytest.mark.parametrize("N", [20000, 32768])
def test_long_rows(N):
    # beyond 2048 vectors per row (the forward) and 1024 (the backward): the
    # wide kernels; the backward's two partial rows fit in shared memory up to
    # about 28 K columns, the scalar kernel takes longer rows
    x, g, b, dy = inputs(24, N, "bf16", "bf16", seed=N % 97)
    eps = f32(1e-5)
    assert "/wide/" in rn.rmsnorm_describe_plan(rn.OP_LAYERNORM_FWD, 24, N, "bf16", "bf16")
    fam = "/wide/" if N == 20000 else "/generic/"
    assert fam in rn.rmsnorm_describe_plan(rn.OP_LAYERNORM_BWD, 24, N, "bf16", "bf16")
    check_fwd(run_fwd(x, g, b, eps, "bf16", "bf16"), x, g, b, eps, "bf16", "bf16")
    out = run_bwd(dy, x, None, None, g, eps, "bf16", "bf16")
    check_bwd(out, dy, x, None, None, g, eps, "bf16", "bf16")


# ---------------------------------------------------------------- the wide kernels:
# operands at any offsets, rows of any length (the backward: rows a multiple
# of 16 bytes), forced onto shapes that walk several rows per CTA

def _es(xd):
    return 4 if xd == "f32" else 2


def _scaled(off, xd, wd):
    return {k: v * (_es(wd) if k in ("gamma", "beta") else _es(xd)) % 16 for k, v in off.items()}


LN_FWD_OFFSETS = [{}, {"x": 1}, {"y": 3}, {"x": 5, "y": 2, "gamma": 1, "beta": 3}]


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N", [1, 7, 129, 1000, 2049, 8192, 20001])
@pytest.mark.parametrize("k", range(len(LN_FWD_OFFSETS)))
def test_wide_forward(debug_env, xd, wd, N, k):
    if xd == "f32" and N == 20001:
        N = 10003
    debug_env.set("RMSNORM_FORCE_VARIANT", "wide:cps=1")
    M = 37 if N > 8192 else 300
    x, g, b, _ = inputs(M, N, xd, wd, seed=N + 90 + k, beta=k != 1, mean=0.5)
    out = run_fwd(x, g, b, f32(1e-5), xd, wd, offsets=_scaled(LN_FWD_OFFSETS[k], xd, wd))
    check_fwd(out, x, g, b, f32(1e-5), xd, wd)


LN_BWD_OFFSETS = [{}, {"x": 1}, {"dy": 3}, {"dx": 1}, {"x": 5, "dy": 2, "dx": 7, "gamma": 1}]


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N", [8, 1032, 4096, 20000])
@pytest.mark.parametrize("k", range(len(LN_BWD_OFFSETS)))
def test_wide_backward(debug_env, xd, wd, N, k):
    if xd == "f32":
        N = N // 2 if N > 8 else 4
    debug_env.set("RMSNORM_FORCE_VARIANT", "wide:cps=1")
    M = 37 if N >= 10000 else 500
    x, g, _, dy = inputs(M, N, xd, wd, seed=N + 91 + k)
    eps = f32(1e-5)
    o = _scaled(LN_BWD_OFFSETS[k], xd, wd)
    fw = oracle.layernorm_fwd(x, g, None, eps, xd, wd)
    out = run_bwd(dy, x, fw["mean"], fw["rstd"], g, eps, xd, wd, offsets=o)
    check_bwd(out, dy, x, fw["mean"], fw["rstd"], g, eps, xd, wd)
    if k % 2 == 0:   # statistics recomputed from x
        out = run_bwd(dy, x, None, None, g, eps, xd, wd, offsets=o)
        check_bwd(out, dy, x, None, None, g, eps, xd, wd)


def test_wide_backward_is_deterministic_and_gradients_optional(debug_env):
    debug_env.set("RMSNORM_FORCE_VARIANT", "wide")
    x, g, _, dy = inputs(2000, 4096, "bf16", "bf16", seed=92)
    o = {"x": 2, "dy": 6, "dx": 4}
    a = run_bwd(dy, x, None, None, g, f32(1e-5), "bf16", "bf16", offsets=o)
    b = run_bwd(dy, x, None, None, g, f32(1e-5), "bf16", "bf16", offsets=o)
    for key in ("dx", "dgamma", "dbeta"):
        assert np.array_equal(a[key], b[key]), key
    none = run_bwd(dy, x, None, None, g, f32(1e-5), "bf16", "bf16", want=(False, False),
                   offsets=o)
    assert np.array_equal(none["dx"], a["dx"])


def test_wide_plans():
    def plan(op, N, a=True, M=4096):
        return rn.rmsnorm_describe_plan(op, M, N, "bf16", "bf16", a)
    fwd, bwd = rn.OP_LAYERNORM_FWD, rn.OP_LAYERNORM_BWD
    for N in (2049, 1001, 40001):            # rows off 16 bytes
        assert "/wide/" in plan(fwd, N), plan(fwd, N)
    assert "/generic/" in plan(bwd, 2049)    # the backward's split would move per row
    for N in (1024, 8192):                   # operands off 16 bytes
        assert "/wide/" in plan(fwd, N, False) and "/wide/" in plan(bwd, N, False)
    assert "/wide/" in plan(fwd, 32768) and "/wide/" in plan(bwd, 12288)
