"""GPU forward with quantised outputs (FP8 E4M3 per row, NVFP4 blocks of 16)
against the oracle.

The codes are integers decided by floating point.  The oracle decides on the
fp32 rounding of the exact quotient; the kernels on their own fp32 values,
which differ from the exact ones by a few fp32 roundings (FP8: rstd cancels)
plus, for NVFP4, the fp32 error of rstd.  So a code must equal the oracle's,
except that where the exact value lies within that error of the midpoint
between two neighbouring codes either neighbour is correct: the test accepts
the other neighbour there and nowhere else, and reports how often it did.
An NVFP4 block whose scale took the other neighbour is checked against the
codes the exact values give under that scale.  Scales (fp32) and rstd use the
1e-5 relative bound of the other fp32 outputs; h is bit-exact.
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
FP8_WINDOW = 8 * U32            # four fp32 roundings, doubled
RSTD_REL = 1e-5                 # bound on the fp32 rstd (checked below)
FP4_WINDOW = RSTD_REL + 8 * U32

E4M3 = oracle.e4m3_values()
E2M1 = oracle.e2m1_values()


def f32(v):
    return float(np.float32(v))


# ---------------------------------------------------------------- runners

def run(kind, x, g, eps, xd, wd, residual=None, gs=None, offsets=None, q_offset=0):
    """Launch rmsnorm_fwd_fp8 / rmsnorm_fwd_nvfp4 on copies of the inputs;
    returns the downloaded outputs (q, scales, rstd, h)."""
    M, N = x.shape
    o = offsets or {}
    bx, bg = pu.dev(x, o.get("x", 0)), pu.dev(g, o.get("gamma", 0))
    br = pu.dev(residual, o.get("residual", 0)) if residual is not None else None
    brs = pu.empty(M, "f32")
    if kind == "fp8":
        bq, bs = pu.Buf(M * N, q_offset), pu.empty(M, "f32")
        rn.rmsnorm_fwd_fp8(bx.ptr, br.ptr if br else None, bg.ptr, bq.ptr, bs.ptr, brs.ptr, M, N,
                           eps, xd, wd)
    else:
        bq, bs = pu.Buf(M * N // 2, q_offset), pu.Buf(M * N // 16)
        rn.rmsnorm_fwd_nvfp4(bx.ptr, br.ptr if br else None, bg.ptr, gs, bq.ptr, bs.ptr, brs.ptr,
                             M, N, eps, xd, wd)
    torch.cuda.synchronize()
    for b in (bx, bg, br, brs, bq, bs):
        if b is not None:
            assert b.guards_ok(), "write outside a buffer"
    out = {"q": bq.download(np.uint8).reshape(M, -1), "rstd": brs.download(np.float32)}
    out["scale"] = (bs.download(np.float32) if kind == "fp8"
                    else bs.download(np.uint8).reshape(M, N // 16))
    if br is not None:
        out["h"] = br.download(pu.np_dtype(xd)).reshape(M, N)
    return out


# ---------------------------------------------------------------- checks

def _ambiguous(codes_a, codes_b, exact, table, window):
    """True where codes a and b are neighbours of the same sign and the exact
    value lies within `window` (relative) of the midpoint between them."""
    sign_bit = np.uint8(table.size // 2)
    sign_a, sign_b = codes_a & sign_bit, codes_b & sign_bit
    mag_a = codes_a.astype(np.int64) - sign_a.astype(np.int64)
    mag_b = codes_b.astype(np.int64) - sign_b.astype(np.int64)
    neighbours = (sign_a == sign_b) & (np.abs(mag_a - mag_b) == 1)
    mid = (np.abs(table[codes_a]) + np.abs(table[codes_b])) / 2
    near = np.abs(np.abs(exact) - mid) <= window * np.abs(exact)
    return neighbours & near


def check_rstd_and_h(out, x, g, eps, xd, wd, residual):
    if residual is None:
        ref = oracle.fwd(x, g, eps, xd, wd)
    else:
        ref = oracle.fused_add_fwd(x, residual, g, eps, xd, wd)
        assert np.array_equal(out["h"], ref["h"]), "h differs"
    pu.check_f32(out["rstd"], ref["rstd64"], rtol=RSTD_REL, what="rstd")


def check_fp8(out, x, g, eps, xd, wd, residual=None):
    ref = oracle.fwd_fp8(x, g, eps, xd, wd, residual=residual)
    check_rstd_and_h(out, x, g, eps, xd, wd, residual)
    s64 = ref["scale64"]
    assert np.all(np.abs(out["scale"] - s64) <= RSTD_REL * np.abs(s64)), "scale"
    diff = out["q"] != ref["q"]
    ok = _ambiguous(out["q"][diff], ref["q"][diff], ref["v64"][diff], E4M3, FP8_WINDOW)
    assert ok.all(), (f"{(~ok).sum()} FP8 codes differ outside the rounding window; first: "
                      f"gpu {out['q'][diff][~ok][:5]} ref {ref['q'][diff][~ok][:5]} "
                      f"exact {ref['v64'][diff][~ok][:5]}")
    return {"codes": out["q"].size, "tie_window": int(diff.sum())}


def _e2m1_codes(v):
    return np.vectorize(oracle.round_e2m1, otypes=[np.uint8])(v.astype(np.float32))


def check_nvfp4(out, x, g, eps, xd, wd, gs, residual=None):
    ref = oracle.fwd_nvfp4(x, g, gs, eps, xd, wd, residual=residual)
    check_rstd_and_h(out, x, g, eps, xd, wd, residual)
    M, N = x.shape
    nb = N // 16
    # block scales
    sf_gpu, sf_ref = out["scale"], ref["sf"]
    sdiff = sf_gpu != sf_ref
    ok = _ambiguous(sf_gpu[sdiff], sf_ref[sdiff], ref["sfv64"][sdiff], E4M3, FP4_WINDOW)
    assert ok.all(), (f"{(~ok).sum()} block scales differ outside the rounding window: gpu "
                      f"{sf_gpu[sdiff][~ok][:5]} ref {sf_ref[sdiff][~ok][:5]} exact "
                      f"{ref['sfv64'][sdiff][~ok][:5]}")
    # codes: the oracle's, or under the GPU's (validated) scale where it differs
    q_gpu = oracle.unpack_e2m1(out["q"]).reshape(M, nb, 16)
    q_ref = oracle.unpack_e2m1(ref["q"]).reshape(M, nb, 16).copy()
    exact = ref["v64"].reshape(M, nb, 16).copy()
    if sdiff.any():
        S_ref, S_gpu = E4M3[sf_ref[sdiff]], E4M3[sf_gpu[sdiff]]
        y64 = exact[sdiff] * (S_ref / gs)[:, None]
        exact[sdiff] = np.where(S_gpu[:, None] > 0, y64 * gs / S_gpu[:, None], 0.0)
        q_ref[sdiff] = _e2m1_codes(exact[sdiff])
    diff = q_gpu != q_ref
    ok = _ambiguous(q_gpu[diff], q_ref[diff], exact[diff], E2M1, FP4_WINDOW)
    assert ok.all(), (f"{(~ok).sum()} FP4 codes differ outside the rounding window: gpu "
                      f"{q_gpu[diff][~ok][:5]} ref {q_ref[diff][~ok][:5]} exact "
                      f"{exact[diff][~ok][:5]}")
    return {"codes": q_gpu.size, "tie_window": int(diff.sum()), "scales_tie": int(sdiff.sum())}


# ---------------------------------------------------------------- inputs

def inputs(M, N, xd, wd, seed, fused=False, outliers=False):
    kw = dict(outlier_fraction=1e-3, outlier_scale=100.0) if outliers else {}
    x = si.fill((M, N), seed=seed, tensor_id=1, dtype=xd, **kw)
    g = si.fill(N, seed=seed, tensor_id=3, p0=1.0, p1=0.1, dtype=wd)
    r = si.fill((M, N), seed=seed, tensor_id=2, dtype=xd, **kw) if fused else None
    return x, g, r


PAIRS = [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32")]
GS = 448.0 * 6 / 8.0        # global scale for |y| up to about 8


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N", [16, 128, 1024, 4096, 2064])
@pytest.mark.parametrize("fused", [False, True])
def test_fp8(xd, wd, N, fused):
    x, g, r = inputs(300, N, xd, wd, seed=N, fused=fused, outliers=fused)
    eps = f32(1e-6)
    out = run("fp8", x, g, eps, xd, wd, residual=r)
    check_fp8(out, x, g, eps, xd, wd, residual=r)


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N", [16, 128, 1024, 4096, 2064])
@pytest.mark.parametrize("fused", [False, True])
def test_nvfp4(xd, wd, N, fused):
    x, g, r = inputs(300, N, xd, wd, seed=N + 1, fused=fused, outliers=fused)
    eps = f32(1e-6)
    out = run("nvfp4", x, g, eps, xd, wd, residual=r, gs=GS)
    check_nvfp4(out, x, g, eps, xd, wd, GS, residual=r)


@pytest.mark.parametrize("N", [1000, 24, 8200])
def test_fp8_rows_that_are_not_16_byte_aligned_or_long(N):
    # an x base 2 bytes off 16: the scalar kernel, at short, medium and long rows
    x, g, _ = inputs(70, N, "bf16", "bf16", seed=3)
    out = run("fp8", x, g, f32(1e-5), "bf16", "bf16", offsets={"x": 2})
    check_fp8(out, x, g, f32(1e-5), "bf16", "bf16")


@pytest.mark.parametrize("kind", ["fp8", "nvfp4"])
def test_unaligned_pointers_take_the_scalar_kernel(kind):
    x, g, r = inputs(50, 256, "bf16", "bf16", seed=4, fused=True)
    offs = {"x": 2, "residual": 4, "gamma": 2}
    out = run(kind, x, g, f32(1e-6), "bf16", "bf16", residual=r, gs=GS, offsets=offs, q_offset=1)
    if kind == "fp8":
        check_fp8(out, x, g, f32(1e-6), "bf16", "bf16", residual=r)
    else:
        check_nvfp4(out, x, g, f32(1e-6), "bf16", "bf16", GS, residual=r)


FORCED = ["subwarp:g=32:vpt=2:cps=1", "subwarp:g=8:vpt=2:cps=1", "subwarp:g=16:vpt=1:cps=1",
          "subwarp:g=32:vpt=1:cps=1", "subwarp:g=16:vpt=1:pf=0:cps=1", "cta:vpt=1:cps=1",
          "cta:vpt=2:t=64:cps=1", "cta:vpt=4:t=32:cps=1", "cta:vpt=4:t=32:pf=0:cps=1",
          "cta:vpt=8:t=32:pf=0:cps=1", "staged:vpt=1:st=2:cps=1", "staged:vpt=2:t=64:st=3:cps=1",
          "staged:vpt=4:t=32:st=8:cps=1", "generic:cps=1"]


@pytest.mark.parametrize("force", FORCED)
@pytest.mark.parametrize("kind", ["fp8", "nvfp4"])
def test_forced_variants_walk_many_rows(debug_env, force, kind):
    # N = 128 bf16: 16 vectors per row; one CTA per SM, so every CTA loops
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    x, g, r = inputs(2000, 128, "bf16", "bf16", seed=5, fused=True)
    out = run(kind, x, g, f32(1e-6), "bf16", "bf16", residual=r, gs=GS)
    if kind == "fp8":
        check_fp8(out, x, g, f32(1e-6), "bf16", "bf16", residual=r)
    else:
        check_nvfp4(out, x, g, f32(1e-6), "bf16", "bf16", GS, residual=r)


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N", [2064, 8192])
@pytest.mark.parametrize("kind", ["fp8", "nvfp4"])
@pytest.mark.parametrize("fused", [False, True])
def test_staged_ring_long_rows(debug_env, xd, wd, N, kind, fused):
    # rows arrive through the bulk-copy ring; two stages, so it wraps often
    debug_env.set("RMSNORM_FORCE_VARIANT", "staged:st=2")
    x, g, r = inputs(200, N, xd, wd, seed=N + 9, fused=fused, outliers=fused)
    out = run(kind, x, g, f32(1e-6), xd, wd, residual=r, gs=GS)
    if kind == "fp8":
        check_fp8(out, x, g, f32(1e-6), xd, wd, residual=r)
    else:
        check_nvfp4(out, x, g, f32(1e-6), xd, wd, GS, residual=r)


@pytest.mark.parametrize("kind", ["fp8", "nvfp4"])
def test_staged_wait_timeout_is_reported_and_the_context_survives(debug_env, kind):
    # a negative wait limit: every wait for a row gives up at once; the kernel
    # stores nothing more, drains its copies and raises the flag that
    # rmsnorm_check_device reports and clears
    x, g, r = inputs(1024, 8192, "bf16", "bf16", seed=43, fused=True)
    debug_env.set("RMSNORM_FORCE_VARIANT", "staged:vpt=4:st=4")
    rn.rmsnorm_check_device()
    debug_env.set("RMSNORM_WAIT_LIMIT_CYCLES", "-1")
    run(kind, x, g, f32(1e-6), "bf16", "bf16", residual=r, gs=GS)
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_check_device()
    assert e.value.status == 6
    rn.rmsnorm_check_device()
    debug_env.delete("RMSNORM_WAIT_LIMIT_CYCLES")
    out = run(kind, x, g, f32(1e-6), "bf16", "bf16", residual=r, gs=GS)
    if kind == "fp8":
        check_fp8(out, x, g, f32(1e-6), "bf16", "bf16", residual=r)
    else:
        check_nvfp4(out, x, g, f32(1e-6), "bf16", "bf16", GS, residual=r)
    rn.rmsnorm_check_device()


@pytest.mark.parametrize("eps", [0.0, 1e-6])
@pytest.mark.parametrize("force", ["", "generic", "staged:st=2"])
def test_zero_rows_and_blocks(debug_env, eps, force):
    if force:
        debug_env.set("RMSNORM_FORCE_VARIANT", force)
    x, g, _ = inputs(8, 64, "bf16", "bf16", seed=6)
    x[2] = 0                  # an all-zero row
    x[5, 16:32] = 0           # an all-zero block
    # (with eps = 0 the zero row's rstd is infinite, so only its codes and
    # scales are compared; the other rows go through the full check)
    keep = np.array([i for i in range(8) if eps > 0 or i != 2])
    for kind in ("fp8", "nvfp4"):
        out = run(kind, x, g, f32(eps), "bf16", "bf16", gs=GS)
        assert np.all(out["q"][2] == 0)
        part = {k: v[keep] for k, v in out.items()}
        if kind == "fp8":
            assert out["scale"][2] == 0.0
            check_fp8(part, x[keep], g, f32(eps), "bf16", "bf16")
        else:
            assert np.all(out["scale"][2] == 0) and out["scale"][5, 1] == 0
            assert np.all(out["q"][5, 8:16] == 0)
            check_nvfp4(part, x[keep], g, f32(eps), "bf16", "bf16", GS)


def test_global_scale_extremes_saturate_and_underflow():
    # a large gs drives block scales to 448 (saturation), a small one into the
    # E4M3 subnormals; both stay within the reading's rounding
    x, g, _ = inputs(64, 256, "bf16", "bf16", seed=7)
    sf = {}
    for gs in (1e5, 0.05, 1.0):
        out = run("nvfp4", x, g, f32(1e-6), "bf16", "bf16", gs=gs)
        check_nvfp4(out, x, g, f32(1e-6), "bf16", "bf16", gs)
        sf[gs] = out["scale"]
    assert (sf[1e5] == 0x7E).any()       # saturated block scales
    assert (sf[0.05] < 8).any()          # subnormal block scales


def test_single_row_and_empty():
    x, g, _ = inputs(1, 4096, "bf16", "bf16", seed=8)
    check_fp8(run("fp8", x, g, f32(1e-6), "bf16", "bf16"), x, g, f32(1e-6), "bf16", "bf16")
    rn.rmsnorm_fwd_fp8(None, None, None, None, None, None, 0, 4096, 1e-6, "bf16", "bf16")
    rn.rmsnorm_fwd_nvfp4(None, None, None, 1.0, None, None, None, 0, 4096, 1e-6, "bf16", "bf16")


def check_workload(wl, inp):
    """A quantised workload at full size through the default dispatch."""
    x, g = inp["x"], inp["gamma"]
    r = inp.get("residual")
    eps = f32(wl.eps)
    kind = "fp8" if "fp8" in wl.op else "nvfp4"
    out = run(kind, x, g, eps, wl.x_dtype, wl.w_dtype, residual=r, gs=wl.global_scale)
    if kind == "fp8":
        info = check_fp8(out, x, g, eps, wl.x_dtype, wl.w_dtype, residual=r)
    else:
        info = check_nvfp4(out, x, g, eps, wl.x_dtype, wl.w_dtype, wl.global_scale, residual=r)
    print(wl.name, info)


@pytest.mark.parametrize("kind", ["fp8", "nvfp4"])
@pytest.mark.parametrize("N", [20000, 32768])
def test_long_rows(kind, N):
    # up to 4096 vectors per row: CTA form with 8 vectors per thread
    x, g, r = inputs(24, N, "bf16", "bf16", seed=N % 89, fused=True)
    out = run(kind, x, g, f32(1e-6), "bf16", "bf16", residual=r, gs=GS)
    if kind == "fp8":
        check_fp8(out, x, g, f32(1e-6), "bf16", "bf16", residual=r)
    else:
        check_nvfp4(out, x, g, f32(1e-6), "bf16", "bf16", GS, residual=r)
