"""GPU forward over strided per-head rows (q/k norm on slices of a fused QKV
projection output) against the oracle, element by element; elements outside
the rows must stay untouched."""
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


def run_case(T, Hq, Hk, D, xd, wd, which="q", in_place=True, seed=0, eps=1e-6, offset=0):
    width = (Hq + 2 * Hk) * D
    buf = si.fill((T, width), seed=seed, tensor_id=1, dtype=xd)
    g = si.fill(D, seed=seed, tensor_id=3, p0=1.0, p1=0.1, dtype=wd)
    H = Hq if which == "q" else Hk
    col0 = 0 if which == "q" else Hq * D
    check(buf, g, T, H, D, width, col0, xd, wd, eps, in_place, offset)


def check_workload(wl, inp):
    """A strided workload at full size: its q slice normalised in place."""
    check(inp["x"], inp["gamma"], wl.M // wl.heads, wl.heads, wl.N, wl.stride_token, 0,
          wl.x_dtype, wl.w_dtype, wl.eps, True, 0)


def check(buf, g, T, H, D, width, col0, xd, wd, eps, in_place, offset):
    eps = f32(eps)
    es = pu.esize(xd)
    bx = pu.dev(buf, offset)
    bg = pu.dev(g)
    br = pu.empty(T * H, "f32")
    if in_place:
        yb, y_st, y_sh, yptr = bx, width, D, bx.ptr + col0 * es
    else:
        yb = pu.empty(T * H * D, xd, offset)
        y_st, y_sh, yptr = H * D, D, yb.ptr
    rn.rmsnorm_fwd_strided(bx.ptr + col0 * es, width, D, bg.ptr, yptr, y_st, y_sh, br.ptr, T, H, D,
                           eps, xd, wd)
    torch.cuda.synchronize()
    for b in (bx, bg, br, yb):
        assert b.guards_ok()
    flat = buf.reshape(-1)
    ref = oracle.fwd_strided(flat[col0:], width, D, g, T, H, D, eps, xd, wd)
    got_rows = (yb.download(pu.np_dtype(xd)).reshape(-1)[col0:] if in_place else
                yb.download(pu.np_dtype(xd))).reshape(-1)
    ref_rows = ref["y"].reshape(-1)
    # gather the rows of both sides
    st = width if in_place else H * D
    idx = (np.arange(T)[:, None, None] * st + np.arange(H)[None, :, None] * D +
           np.arange(D)[None, None, :]).reshape(-1)
    ridx = (np.arange(T)[:, None, None] * width + np.arange(H)[None, :, None] * D +
            np.arange(D)[None, None, :]).reshape(-1)
    g_rows, r_rows = got_rows[idx], ref_rows[ridx]
    if xd == "bf16":
        pu.check_bf16_ulp(g_rows, r_rows, what="y")
    else:
        pu.check_f32(g_rows, ref["y64"].reshape(-1), what="y")
    pu.check_f32(br.download(np.float32), ref["rstd"].astype(np.float64), what="rstd")
    if in_place:
        # every element outside the normalised rows is unchanged
        mask = np.ones(T * width, bool)
        mask[col0 + ridx] = False
        after = bx.download(pu.np_dtype(xd)).reshape(-1)
        assert np.array_equal(after[mask], flat[mask])


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("which", ["q", "k"])
def test_qk_norm_in_place_bf16(D, which):
    run_case(257, 8, 2, D, "bf16", "bf16", which=which, seed=D)


@pytest.mark.parametrize("xd,wd", [("f32", "f32"), ("bf16", "f32")])
def test_qk_norm_other_dtypes_out_of_place(xd, wd):
    run_case(100, 6, 2, 128, xd, wd, in_place=False, seed=7)


@pytest.mark.parametrize("D", [100, 2048, 1])
def test_unaligned_and_wide_heads_take_the_scalar_path(D):
    run_case(33, 4, 1, D, "bf16", "bf16", seed=D)


def test_unaligned_base_pointer():
    run_case(40, 4, 2, 64, "bf16", "bf16", seed=9, offset=2)


def test_single_head_rows_with_a_token_stride():
    run_case(500, 1, 1, 128, "bf16", "bf16", seed=10)


@pytest.mark.parametrize("force", ["subwarp:g=16:vpt=1:pf=1:cps=1", "subwarp:g=8:vpt=2:pf=0:cps=1",
                                   "subwarp:g=32:vpt=1:pf=1:cps=1", "generic:cps=1"])
def test_forced_variants_walk_many_rows(debug_env, force):
    # few CTAs: every thread steps (token, head) across many rows and wraps
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    run_case(3001, 7, 1, 128, "bf16", "bf16", seed=11)
