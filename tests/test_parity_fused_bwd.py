"""GPU fused-add backward (dh = dx(h) + dres, written over dres; dgamma in
fp32 or in the weight dtype) against the oracle, element by element."""
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


def f32(v):
    return float(np.float32(v))


def make(M, N, xd, wd, seed):
    h = si.fill((M, N), seed=seed, tensor_id=1, dtype=xd, p1=2.0)
    dy = si.fill((M, N), seed=seed, tensor_id=4, dtype=xd)
    dres = si.fill((M, N), seed=seed, tensor_id=2, dtype=xd)
    g = si.fill(N, seed=seed, tensor_id=3, p0=1.0, p1=0.1, dtype=wd)
    return h, dy, dres, g


def run(h, dy, dres, g, rstd, eps, xd, wd, dg_dtype="f32", offsets=None, stream=None):
    M, N = h.shape
    o = offsets or {}
    bh, bdy, bg = pu.dev(h, o.get("h", 0)), pu.dev(dy, o.get("dy", 0)), pu.dev(g, o.get("gamma", 0))
    bres = pu.dev(dres, o.get("dres", 0))
    brs = pu.dev(rstd) if rstd is not None else None
    bdg = pu.empty(N, dg_dtype)
    ws = rn.rmsnorm_bwd_workspace_size(M, N, xd, wd)
    bws = pu.Buf(max(16, ws))
    rn.rmsnorm_fused_add_bwd(bdy.ptr, bh.ptr, brs.ptr if brs else None, bg.ptr, bres.ptr, bdg.ptr,
                             dg_dtype, bws.ptr, ws, M, N, eps, xd, wd, stream=stream)
    torch.cuda.synchronize()
    for b in (bh, bdy, bg, bres, bdg, bws):
        assert b.guards_ok()
    return {"dh": bres.download(pu.np_dtype(xd), (M, N)),
            "dgamma": bdg.download(pu.np_dtype(dg_dtype), (N,))}


def check(h, dy, dres, g, rstd, eps, xd, wd, out, dg_dtype="f32"):
    ref = oracle.fused_add_bwd(dy, h, rstd, g, dres, eps, xd, wd)
    aux = oracle.bwd(dy, h, rstd, g, eps, xd, wd)     # error scales of the dx part
    h64, dy64, g64 = oracle.to_f64(h, xd), oracle.to_f64(dy, xd), oracle.to_f64(g, wd)
    r = rstd.astype(np.float64) if rstd is not None else 1.0 / np.sqrt(np.mean(h64 ** 2, 1) + eps)
    if xd == "bf16":
        n_floor, _ = pu.check_dx_bf16(out["dh"], ref["dh"], ref["dh64"], h64, dy64, g64, r,
                                      aux["c64"], aux["dot_abs64"], what="dh")
    else:
        n_floor = 0
        pu.check_f32(out["dh"], ref["dh64"], what="dh")
    if dg_dtype == "f32":
        pu.check_dgamma(out["dgamma"], ref["dgamma64"], aux["dgamma_sq64"])
    else:
        # rounded once to bf16 from the fp32 sum: within 1 ulp of the oracle's
        # rounding of the exact sum, unless that sum sits within the fp32
        # error of a bf16 tie or cancels -- then within the fp32 sum's bound
        # (1e-4 of max(|sum|, sqrt(sum of squared terms))) plus one bf16 ulp
        d = pu.bf16_ulp_dist(out["dgamma"], ref["dgamma_w"])
        far = d > 1
        if far.any():
            from oracle import bf16_array_to_f64
            gv = bf16_array_to_f64(out["dgamma"])
            ex = ref["dgamma64"]
            scale = np.maximum(np.abs(ex), np.sqrt(aux["dgamma_sq64"]))
            ok = np.abs(gv - ex) <= 1e-4 * scale + pu.bf16_ulp_of(ex)
            assert (ok | ~far).all(), (f"dgamma (bf16): {int((far & ~ok).sum())} columns beyond "
                                       f"1 ulp and the sum's bound, max {int(d.max())} ulp")
    return {"floor": n_floor}


PAIRS = [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")]
N_LIST = [8, 128, 768, 1024, 2048, 4096, 8192, 16384, 32768, 2049, 7, 40000]


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N", N_LIST)
def test_fused_add_bwd_matches_oracle(xd, wd, N):
    if xd == "f32" and N in (7, 2049):
        N += 1  # keep the fp32 list to aligned and one odd size below
    M = 33 if N >= 16384 else 300 if N >= 1024 else 1100
    h, dy, dres, g = make(M, N, xd, wd, seed=N + 31)
    eps = f32(1e-5)
    rstd = oracle.fwd(h, g, eps, xd, wd)["rstd"]
    out = run(h, dy, dres, g, rstd, eps, xd, wd)
    check(h, dy, dres, g, rstd, eps, xd, wd, out)


@pytest.mark.parametrize("N", [128, 4096, 2049])
def test_dgamma_in_weight_dtype_and_no_rstd(N):
    h, dy, dres, g = make(400, N, "bf16", "bf16", seed=N + 32)
    eps = f32(1e-4)
    out = run(h, dy, dres, g, None, eps, "bf16", "bf16", dg_dtype="bf16")
    check(h, dy, dres, g, None, eps, "bf16", "bf16", out, dg_dtype="bf16")


@pytest.mark.parametrize("force,N", [
    ("staged:vpt=4:st=2:cps=1", 8192), ("staged:vpt=2:st=3:cps=1", 4096),
    ("staged:vpt=4:st=2:cps=1", 5120), ("subwarp:g=8:vpt=2:pf=1:cps=1", 128),
    ("subwarp:g=32:vpt=3:pf=0:cps=1", 768), ("ragged:vpt=2:pf=1:cps=1", 2049),
    ("ragged:vpt=1:pf=0:cps=1", 2049), ("generic:cps=1", 4096), ("wide:cps=1", 4096),
    ("staged:g=32:vpt=3:cps=1", 768), ("staged:g=8:vpt=2:st=4:cps=1", 128),
    ("staged:g=32:vpt=4:st=2:cps=1", 1024),
])
def test_forced_variants(debug_env, force, N):
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    M = 2500 if N <= 1024 else 600
    h, dy, dres, g = make(M, N, "bf16", "f32", seed=33)
    eps = f32(1e-5)
    rstd = oracle.fwd(h, g, eps, "bf16", "f32")["rstd"]
    out = run(h, dy, dres, g, rstd, eps, "bf16", "f32")
    check(h, dy, dres, g, rstd, eps, "bf16", "f32", out)


@pytest.mark.parametrize("offsets,N", [({"h": 2, "dy": 2, "dres": 2}, 4096),
                                       ({"h": 2, "dy": 4, "dres": 2}, 1000)])
def test_unaligned(offsets, N):
    h, dy, dres, g = make(100, N, "bf16", "bf16", seed=34)
    eps = f32(1e-5)
    rstd = oracle.fwd(h, g, eps, "bf16", "bf16")["rstd"]
    out = run(h, dy, dres, g, rstd, eps, "bf16", "bf16", offsets=offsets)
    check(h, dy, dres, g, rstd, eps, "bf16", "bf16", out)


def test_bitwise_reproducible():
    h, dy, dres, g = make(700, 4096, "bf16", "bf16", seed=35)
    eps = f32(1e-5)
    rstd = oracle.fwd(h, g, eps, "bf16", "bf16")["rstd"]
    a = run(h, dy, dres, g, rstd, eps, "bf16", "bf16", dg_dtype="bf16")
    b = run(h, dy, dres, g, rstd, eps, "bf16", "bf16", dg_dtype="bf16")
    assert np.array_equal(a["dh"], b["dh"]) and np.array_equal(a["dgamma"], b["dgamma"])
