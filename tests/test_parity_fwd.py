"""GPU forward and fused-add forward against the oracle, element by element.

Shapes span every kernel family (short rows packed per warp, one row per CTA,
ragged rows, the generic fallback), several tiles and ragged tails, and the
persistent loops (forced to few CTAs per SM so every CTA walks several rows).
"""
import os

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity_util as pu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

PAIRS = [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")]


def f32(v):
    return float(np.float32(v))


def make(M, N, xd, wd, seed, gamma=("normal", 1.0, 0.2), xscale=1.0):
    x = si.fill((M, N), seed=seed, tensor_id=1, dtype=xd, p1=xscale)
    g = si.fill(N, seed=seed, tensor_id=3, dist=gamma[0], p0=gamma[1], p1=gamma[2], dtype=wd)
    return x, g


def check_fwd(x, g, eps, xd, wd, out, want_rstd=True):
    ref = oracle.fwd(x, g, eps, xd, wd)
    if xd == "bf16":
        pu.check_bf16_ulp(out["y"], ref["y"], what="y")
    else:
        pu.check_f32(out["y"], ref["y64"], what="y")
    if want_rstd:
        pu.check_f32(out["rstd"], ref["rstd64"], what="rstd")
    return ref


def check_fused(x, r, g, eps, xd, wd, out, want_rstd=False):
    ref = oracle.fused_add_fwd(x, r, g, eps, xd, wd)
    assert np.array_equal(out["h"], ref["h"]), "h differs from the correctly rounded sum"
    if xd == "bf16":
        pu.check_bf16_ulp(out["y"], ref["y"], what="y")
    else:
        pu.check_f32(out["y"], ref["y64"], what="y")
    if want_rstd:
        pu.check_f32(out["rstd"], ref["rstd64"], what="rstd")


# N values per family for bf16 (E = 8) and fp32 (E = 4)
N_BF16 = [8, 16, 24, 40, 128, 256, 512, 768, 1024,          # short rows, packed
          1032, 2048, 4096, 5120, 7168, 8192, 16384, 32768,  # one row per CTA
          1, 2, 7, 9, 127, 129, 255, 1023, 1025, 2049, 4095,  # ragged
          40000]                                             # clusters of CTAs
N_F32 = [4, 12, 128, 512, 1024, 4096, 8192, 16384, 1, 3, 5, 1023, 2049, 40000]


def _cases():
    out = []
    for xd, wd in PAIRS:
        for N in (N_F32 if xd == "f32" else N_BF16):
            M = 37 if N >= 16384 else 129 if N >= 1024 else 300
            out.append((xd, wd, M, N))
    return out


@pytest.mark.parametrize("xd,wd,M,N", _cases())
def test_fwd_matches_oracle(xd, wd, M, N):
    x, g = make(M, N, xd, wd, seed=N)
    eps = f32(1e-5)
    out = pu.run_fwd(x, g, eps, xd, wd)
    check_fwd(x, g, eps, xd, wd, out)


@pytest.mark.parametrize("xd,wd,M,N", [c for c in _cases() if c[3] in (8, 128, 768, 2049, 5120,
                                                                           8192, 40000)])
def test_fused_add_matches_oracle(xd, wd, M, N):
    x, g = make(M, N, xd, wd, seed=N + 1)
    r = si.fill((M, N), seed=N + 1, tensor_id=2, dtype=xd, p1=3.0)
    eps = f32(1e-6)
    out = pu.run_fused(x, r, g, eps, xd, wd, want_rstd=True)
    check_fused(x, r, g, eps, xd, wd, out, want_rstd=True)


@pytest.mark.parametrize("op", ["fwd", "fused"])
@pytest.mark.parametrize("force,N", [
    ("subwarp:g=8:vpt=2:pf=1:cps=1", 128), ("subwarp:g=8:vpt=2:pf=0:cps=1", 128),
    ("subwarp:g=16:vpt=1:pf=1:cps=1", 128), ("subwarp:g=32:vpt=3:pf=1:cps=1", 768),
    ("subwarp:g=32:vpt=4:pf=0:cps=1", 1024),
    ("cta:vpt=4:pf=1:cps=1", 8192), ("cta:vpt=4:pf=0:cps=1", 8192),
    ("cta:vpt=2:pf=1:cps=1", 4096), ("cta:vpt=8:pf=0:cps=1", 8192),
    ("cta:vpt=1:pf=1:cps=1", 2048), ("cta:vpt=4:pf=1:t=512:cps=1", 5120),
    ("ragged:vpt=2:pf=1:cps=1", 2049), ("ragged:vpt=1:pf=0:cps=1", 2049),
    ("ragged:vpt=4:pf=0:cps=1", 4096), ("ragged:vpt=2:pf=1:cps=2", 1025), ("generic:cps=1", 8192), ("generic:cps=1", 2049),
    ("wide:cps=1", 8192), ("wide:cps=1", 2049), ("wide:t=64:cps=1", 1025),
    ("staged:vpt=4:st=3:cps=1", 8192), ("staged:vpt=4:st=2:cps=1", 8192),
    ("staged:vpt=2:st=5:cps=1", 4096), ("staged:vpt=8:st=2:cps=1", 16384),
    ("staged:vpt=1:st=8:cps=1", 2048), ("staged:vpt=4:t=512:st=2:cps=1", 5120),
    ("staged:vpt=4:st=4:cps=1", 1032),
])
def test_forced_variants_walk_several_rows(debug_env, op, force, N):
    # one CTA per SM: each CTA walks several rows, exercising the persistent
    # loop, the next-row prefetch and the alternating reduction buffers
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    M = 2000 if N <= 1024 else 700
    x, g = make(M, N, "bf16", "bf16", seed=7)
    eps = f32(1e-6)
    if op == "fwd":
        check_fwd(x, g, eps, "bf16", "bf16", pu.run_fwd(x, g, eps, "bf16", "bf16"))
    else:
        r = si.fill((M, N), seed=7, tensor_id=2, dtype="bf16")
        out = pu.run_fused(x, r, g, eps, "bf16", "bf16", want_rstd=True)
        check_fused(x, r, g, eps, "bf16", "bf16", out, want_rstd=True)


@pytest.mark.parametrize("offsets,N", [
    ({"x": 2, "y": 2}, 4096),              # same residue: ragged rows
    ({"x": 2, "y": 2, "gamma": 2}, 2048),
    ({"x": 6, "y": 6, "residual": 6}, 1000),
    ({"x": 2, "y": 4}, 4096),              # residues differ: x off y (fused: y off h, wide)
    ({"gamma": 2}, 8192),                  # only gamma unaligned: ragged
    ({"x": 14, "y": 14, "residual": 14, "rstd": 4}, 129),
])
def test_unaligned_pointers(offsets, N):
    M = 65
    x, g = make(M, N, "bf16", "bf16", seed=3)
    eps = f32(1e-5)
    check_fwd(x, g, eps, "bf16", "bf16", pu.run_fwd(x, g, eps, "bf16", "bf16", offsets=offsets))
    r = si.fill((M, N), seed=3, tensor_id=2, dtype="bf16")
    out = pu.run_fused(x, r, g, eps, "bf16", "bf16", want_rstd=True, offsets=offsets)
    check_fused(x, r, g, eps, "bf16", "bf16", out, want_rstd=True)


def test_unaligned_f32_pointers():
    M, N = 40, 1030
    x, g = make(M, N, "f32", "f32", seed=4)
    eps = f32(1e-5)
    out = pu.run_fwd(x, g, eps, "f32", "f32", offsets={"x": 4, "y": 4, "gamma": 8})
    check_fwd(x, g, eps, "f32", "f32", out)


@pytest.mark.parametrize("N", [128, 4096, 2049])
def test_no_rstd_output(N):
    x, g = make(50, N, "bf16", "bf16", seed=5)
    eps = f32(1e-6)
    out = pu.run_fwd(x, g, eps, "bf16", "bf16", want_rstd=False)
    check_fwd(x, g, eps, "bf16", "bf16", out, want_rstd=False)


@pytest.mark.parametrize("N", [128, 8192, 2049])
def test_special_rows(N):
    # constant rows, zero rows (eps > 0), rows with huge and tiny scales
    M = 8
    x, g = make(M, N, "bf16", "bf16", seed=6)
    x = x.copy()
    x[0] = oracle.round_bf16(37.0)
    x[1] = oracle.round_bf16(-1e-3)
    x[2] = 0
    x[3] = (si.fill(N, seed=9, tensor_id=1, dtype="bf16", p1=1e15))
    x[4] = (si.fill(N, seed=9, tensor_id=2, dtype="bf16", p1=1e-15))
    x[5, ::3] = 0
    eps = f32(1e-5)
    check_fwd(x, g, eps, "bf16", "bf16", pu.run_fwd(x, g, eps, "bf16", "bf16"))


def test_zero_row_with_zero_eps_gives_nan():
    x = np.zeros((2, 256), np.uint16)
    x[1] = oracle.round_bf16(1.0)
    g = si.fill(256, seed=1, tensor_id=3, dtype="bf16")
    out = pu.run_fwd(x, g, 0.0, "bf16", "bf16")
    y = oracle.bf16_array_to_f64(out["y"])
    ref = oracle.fwd(x, g, 0.0, "bf16", "bf16")
    # rstd = 1/sqrt(0) = +inf and y = 0 * inf = NaN, on both sides
    assert np.isinf(ref["rstd64"][0]) and np.isnan(ref["y64"][0]).all()
    assert np.isposinf(out["rstd"][0]) and np.isnan(y[0]).all()
    assert np.isfinite(y[1]).all()


def test_outlier_residual_and_input():
    wl = si.WORKLOADS["fadd_bf16_m32768_n4096"]
    M, N = 512, wl.N
    x = si.fill((M, N), seed=wl.seed, tensor_id=1, dtype="bf16", outlier_fraction=1e-3,
                outlier_scale=100.0)
    r = si.fill((M, N), seed=wl.seed, tensor_id=2, dtype="bf16", outlier_fraction=1e-3,
                outlier_scale=100.0)
    g = si.fill(N, seed=wl.seed, tensor_id=3, dtype="bf16", p0=1.0, p1=0.1)
    eps = f32(wl.eps)
    out = pu.run_fused(x, r, g, eps, "bf16", "bf16", want_rstd=True)
    check_fused(x, r, g, eps, "bf16", "bf16", out, want_rstd=True)


def test_results_are_deterministic_and_stream_independent():
    M, N = 1000, 4096
    x, g = make(M, N, "bf16", "bf16", seed=8)
    eps = f32(1e-5)
    a = pu.run_fwd(x, g, eps, "bf16", "bf16")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = pu.run_fwd(x, g, eps, "bf16", "bf16", stream=s)
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["rstd"], b["rstd"])


def test_plan_families():
    import row_wise_normalization_02_gb300 as rn
    assert "/subwarp/" in rn.rmsnorm_describe_plan(rn.OP_FWD, 262144, 128, "bf16", "bf16")
    assert "/cta/" in rn.rmsnorm_describe_plan(rn.OP_FWD, 16384, 8192, "bf16", "bf16")
    assert "/cta/" in rn.rmsnorm_describe_plan(rn.OP_FUSED_ADD, 32768, 4096, "bf16", "bf16")
    assert "/ragged/" in rn.rmsnorm_describe_plan(rn.OP_FWD, 4096, 2049, "bf16", "bf16")
    assert "/cluster/" in rn.rmsnorm_describe_plan(rn.OP_FWD, 16, 40000, "bf16", "bf16")
    assert "/cluster/" in rn.rmsnorm_describe_plan(rn.OP_BWD, 16, 40000, "bf16", "bf16")
    assert "/cluster/" in rn.rmsnorm_describe_plan(rn.OP_FUSED_ADD_BWD, 16, 32768, "bf16", "bf16")
    assert "/wide/" in rn.rmsnorm_describe_plan(rn.OP_FWD, 16, 40001, "bf16", "bf16")
    assert "/wide/" in rn.rmsnorm_describe_plan(rn.OP_FWD, 16, 1 << 19, "bf16", "bf16")
    assert "/staged/" in rn.rmsnorm_describe_plan(rn.OP_BWD, 16384, 8192, "bf16", "f32")
    assert "/subwarp/" in rn.rmsnorm_describe_plan(rn.OP_BWD, 262144, 128, "bf16", "bf16")
    assert "/staged/g32/vpt3/" in rn.rmsnorm_describe_plan(rn.OP_BWD, 65536, 768, "bf16", "bf16")
