"""rmsnorm_bwd_noalloc: the backward for callers that cannot allocate device
memory (for example a serving runtime whose memory pool owns the whole GPU, or
a plugin interface that offers no allocator), so they cannot hand rmsnorm_bwd
the workspace it asks for.  The entry point keeps the dgamma partial rows in a
scratch array inside the library's device image instead.

Checked through the C ABI against rmsnorm_bwd (with a workspace) on two calls
in a row with different shapes and data -- bit for bit, since both run the
same kernels -- and against the oracle; also on ragged rows (whose grid is
whole residue classes of the row alignment) and fp32 operands, on operands
off 16 bytes whose wide kernel wants more partial rows than the scratch holds
(its grid is bounded to it), and for the rejection of a shape whose partial
rows do not fit the scratch.  This file is
collected last; it passes alone in a fresh process and after the other tests.
"""
import re

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
from tests.test_parity_bwd import check_bwd  # noqa: E402


def _inputs(M, N, xd, wd, seed):
    x = si.fill((M, N), seed=seed, tensor_id=1, dtype=xd)
    dy = si.fill((M, N), seed=seed, tensor_id=4, dtype=xd)
    g = si.fill(N, seed=seed, tensor_id=3, p0=1.0, p1=0.1, dtype=wd)
    rstd = oracle.fwd(x, g, float(np.float32(1e-5)), xd, wd, want64=False)["rstd"]
    return x, dy, g, rstd


def _compare_with_workspace_entry_point(M, N, xd, wd, seed):
    x, dy, g, rstd = _inputs(M, N, xd, wd, seed)
    eps = float(np.float32(1e-5))
    bx, bdy, bg, brs = pu.dev(x), pu.dev(dy), pu.dev(g), pu.dev(rstd)

    # the entry point with a caller-provided workspace
    ws = rn.rmsnorm_bwd_workspace_size(M, N, xd, wd)
    assert ws <= rn.NOALLOC_SCRATCH_BYTES
    bws = pu.Buf(ws)
    dx_a, dg_a = pu.empty(M * N, xd), pu.empty(N, "f32")
    rn.rmsnorm_bwd(bdy.ptr, bx.ptr, brs.ptr, bg.ptr, dx_a.ptr, dg_a.ptr, bws.ptr, ws, M, N, eps,
                   xd, wd)

    # the allocation-free entry point
    dx_b, dg_b = pu.empty(M * N, xd), pu.empty(N, "f32")
    rn.rmsnorm_bwd_noalloc(bdy.ptr, bx.ptr, brs.ptr, bg.ptr, dx_b.ptr, dg_b.ptr, M, N, eps, xd,
                           wd)
    torch.cuda.synchronize()
    for b in (dx_a, dg_a, dx_b, dg_b, bws):
        assert b.guards_ok()

    npd = pu.np_dtype(xd)
    a_dx, b_dx = dx_a.download(npd, (M, N)), dx_b.download(npd, (M, N))
    a_dg, b_dg = dg_a.download(np.float32), dg_b.download(np.float32)
    # both calls run the same kernels over the same rows in the same order,
    # so anything short of bit equality is a fault
    assert np.array_equal(a_dx.view(np.uint8), b_dx.view(np.uint8)), "dx differs"
    assert np.array_equal(a_dg.view(np.uint32), b_dg.view(np.uint32)), "dgamma differs"
    # and the result is the backward's, within the parity tolerances
    check_bwd(x, dy, g, rstd, eps, xd, wd, {"dx": b_dx, "dgamma": b_dg})


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    # two calls in a row with different shapes and data: the second finds the
    # first call's partial rows in the scratch and must not depend on them
    _compare_with_workspace_entry_point(4096, 8192, "bf16", "f32", seed=31)
    _compare_with_workspace_entry_point(3000, 2048, "bf16", "bf16", seed=32)


@pytest.mark.parametrize("M,N,xd,wd", [(4096, 2049, "bf16", "bf16"),   # ragged rows
                                       (1024, 4096, "f32", "f32")])
def test_noalloc_ragged_and_fp32_shapes(M, N, xd, wd):
    _compare_with_workspace_entry_point(M, N, xd, wd, seed=34)


def test_noalloc_bounds_the_wide_grid_to_its_scratch():
    # x off 16 bytes at 32768 bf16 columns: the wide backward, one CTA per SM,
    # wants more partial rows than the scratch holds; the aligned plan's
    # (clusters) fit, and the call runs with fewer CTAs
    M, N = 2048, 32768
    ws = rn.rmsnorm_bwd_workspace_size(M, N, "bf16", "bf16")
    aligned = rn.rmsnorm_describe_plan(rn.OP_BWD, M, N, "bf16", "bf16", True)
    grid = int(aligned.split("/grid")[1].split("/")[0])
    m = re.search(r"/cl(\d+)/", aligned)
    cl = int(m.group(1)) if m else 1
    if ws <= rn.NOALLOC_SCRATCH_BYTES or (grid // cl) * N * 4 > rn.NOALLOC_SCRATCH_BYTES:
        pytest.skip("this device's grids do not give the case")
    assert "/wide/" in rn.rmsnorm_describe_plan(rn.OP_BWD, M, N, "bf16", "bf16", "mixed")
    x, dy, g, rstd = _inputs(M, N, "bf16", "bf16", seed=35)
    eps = float(np.float32(1e-5))
    bx, bdy, bg, brs = pu.dev(x, 2), pu.dev(dy), pu.dev(g), pu.dev(rstd)
    dx_a, dg_a = pu.empty(M * N, "bf16"), pu.empty(N, "f32")
    bws = pu.Buf(ws)
    rn.rmsnorm_bwd(bdy.ptr, bx.ptr, brs.ptr, bg.ptr, dx_a.ptr, dg_a.ptr, bws.ptr, ws, M, N, eps,
                   "bf16", "bf16")
    dx_b, dg_b = pu.empty(M * N, "bf16"), pu.empty(N, "f32")
    rn.rmsnorm_bwd_noalloc(bdy.ptr, bx.ptr, brs.ptr, bg.ptr, dx_b.ptr, dg_b.ptr, M, N, eps,
                           "bf16", "bf16")
    torch.cuda.synchronize()
    for b in (dx_a, dg_a, dx_b, dg_b, bws):
        assert b.guards_ok()
    npd = pu.np_dtype("bf16")
    a_dx, b_dx = dx_a.download(npd, (M, N)), dx_b.download(npd, (M, N))
    # dx does not depend on the grid; dgamma's summation order does
    assert np.array_equal(a_dx.view(np.uint8), b_dx.view(np.uint8)), "dx differs"
    check_bwd(x, dy, g, rstd, eps, "bf16", "bf16", {"dx": b_dx, "dgamma": dg_b.download(np.float32)})


def test_noalloc_rejects_shapes_beyond_its_scratch():
    M, N = 8, 1 << 20         # 8 partial rows of 1M fp32 columns: 32 MiB > 16 MiB
    assert rn.rmsnorm_bwd_workspace_size(M, N, "bf16", "bf16") > rn.NOALLOC_SCRATCH_BYTES
    x = si.fill((M, N), seed=33, tensor_id=1, dtype="bf16")
    g = si.fill(N, seed=33, tensor_id=3, dtype="bf16")
    bx, bdy, bg = pu.dev(x), pu.dev(x), pu.dev(g)
    bdx, bdg = pu.empty(M * N, "bf16"), pu.empty(N, "f32")
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_bwd_noalloc(bdy.ptr, bx.ptr, None, bg.ptr, bdx.ptr, bdg.ptr, M, N, 1e-5,
                               "bf16", "bf16")
    assert e.value.status == 4     # RMSNORM_ERR_WORKSPACE
    torch.cuda.synchronize()
    # rejected before any launch: the outputs still hold the canary pattern
    assert (bdx.view().cpu().numpy() == pu.CANARY).all()
    assert (bdg.view().cpu().numpy() == pu.CANARY).all()
    # without dgamma no scratch is needed, and the call goes through
    rn.rmsnorm_bwd_noalloc(bdy.ptr, bx.ptr, None, bg.ptr, bdx.ptr, None, M, N, 1e-5, "bf16",
                           "bf16")
    torch.cuda.synchronize()
    assert bdx.guards_ok()
