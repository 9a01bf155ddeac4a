"""The L2 lookahead of the register kernels: one bulk prefetch per CTA
iteration asks for the rows two iterations ahead to be brought into L2.  It is
a hint, so it must change no bit of any output, with or without it and at any
distance, including the last iterations where the rows ahead run past the end
and are clipped; and the dispatch turns it on exactly where it was measured
to pay (the LayerNorm CTA kernels, the sub-warp backward kernels with next-row
prefetch, the ragged kernels) and nowhere else -- not in the ring kernels,
whose stages keep the rows in flight.  The wide kernel sizes its lookahead
to the grid: as many rows ahead (at most two) as keep 12 MB of requests in
flight."""
import numpy as np
import pytest

import oracle
from tests import parity_util as pu
from tests import test_parity_fused_bwd as fb
from tests import test_parity_layernorm as tl
from tests.test_parity_bwd import check_bwd

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import row_wise_normalization_02_gb300 as rn  # noqa: E402


@pytest.mark.parametrize("op,M,N,on", [
    (rn.OP_LAYERNORM_FWD, 16384, 8192, True),
    (rn.OP_LAYERNORM_BWD, 16384, 8192, True),
    (rn.OP_LAYERNORM_BWD, 65536, 1024, False),   # short rows: through the bulk-copy ring
    (rn.OP_LAYERNORM_FWD, 65536, 1024, False),   # the sub-warp forward lost with it
    (rn.OP_BWD, 262144, 128, True),
    (rn.OP_FUSED_ADD_BWD, 262144, 128, True),
    (rn.OP_BWD, 65536, 768, False),              # full-warp rows: no next-row prefetch
    (rn.OP_BWD, 16384, 8192, False),             # staged: the ring keeps rows in flight
    (rn.OP_FWD, 16384, 8192, False),
    (rn.OP_FUSED_ADD, 32768, 4096, False),
    (rn.OP_FWD, 262144, 128, False),
    (rn.OP_FWD, 4096, 2049, True),               # ragged rows: the aligned interior
    (rn.OP_BWD, 4096, 2049, True),
])
def test_dispatch(op, M, N, on):
    plan = rn.rmsnorm_describe_plan(op, M, N, "bf16", "bf16")
    assert ("/l2ahead2" in plan) == on, plan


def _bits(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint32)


def _same(runs):
    base = runs[0]
    for other in runs[1:]:
        assert base.keys() == other.keys()
        for k in base:
            assert np.array_equal(_bits(base[k]), _bits(other[k])), k


def _over_distances(debug_env, fn):
    runs = []
    for l2 in (None, 0, 1, 3):
        if l2 is None:
            debug_env.delete("RMSNORM_FORCE_VARIANT", raising=False)
        else:
            debug_env.set("RMSNORM_FORCE_VARIANT", f"keep:l2={l2}")
        runs.append(fn())
    debug_env.delete("RMSNORM_FORCE_VARIANT", raising=False)
    _same(runs)
    return runs[0]


@pytest.mark.parametrize("M,N", [(3001, 8192), (20001, 1024)])
def test_layernorm_forward_bits_do_not_depend_on_it(debug_env, M, N):
    eps = tl.f32(1e-5)
    x, g, b, _ = tl.inputs(M, N, "bf16", "bf16", seed=61)
    out = _over_distances(debug_env, lambda: tl.run_fwd(x, g, b, eps, "bf16", "bf16"))
    tl.check_fwd(out, x, g, b, eps, "bf16", "bf16")


@pytest.mark.parametrize("M,N,saved", [(3001, 8192, True), (20001, 1024, True),
                                       (20001, 1024, False)])
def test_layernorm_backward_bits_do_not_depend_on_it(debug_env, M, N, saved):
    eps = tl.f32(1e-5)
    x, g, _, dy = tl.inputs(M, N, "bf16", "bf16", seed=62)
    fw = oracle.layernorm_fwd(x, g, None, eps, "bf16", "bf16")
    mean, rstd = (fw["mean"], fw["rstd"]) if saved else (None, None)
    out = _over_distances(
        debug_env, lambda: tl.run_bwd(dy, x, mean, rstd, g, eps, "bf16", "bf16"))
    tl.check_bwd(out, dy, x, mean, rstd, g, eps, "bf16", "bf16")


def test_rmsnorm_short_row_backward_bits_do_not_depend_on_it(debug_env):
    M, N, eps = 50001, 128, tl.f32(1e-6)
    x, g, _, dy = tl.inputs(M, N, "bf16", "bf16", seed=63, beta=False)
    rstd = oracle.fwd(x, g, eps, "bf16", "bf16", want64=False)["rstd"]
    out = _over_distances(debug_env, lambda: pu.run_bwd(dy, x, rstd, g, eps, "bf16", "bf16"))
    check_bwd(x, dy, g, rstd, eps, "bf16", "bf16", out)


def test_fused_add_short_row_backward_bits_do_not_depend_on_it(debug_env):
    M, N, eps = 50001, 128, tl.f32(1e-6)
    h, g, _, dy = tl.inputs(M, N, "bf16", "bf16", seed=64, beta=False)
    dres = tl.inputs(M, N, "bf16", "bf16", seed=65, beta=False)[3]
    rstd = oracle.fwd(h, g, eps, "bf16", "bf16", want64=False)["rstd"]
    out = _over_distances(
        debug_env, lambda: fb.run(h, dy, dres, g, rstd, eps, "bf16", "bf16"))
    fb.check(h, dy, dres, g, rstd, eps, "bf16", "bf16", out)


def test_ragged_rows_bits_do_not_depend_on_it(debug_env):
    M, N, eps = 1001, 2049, tl.f32(1e-6)
    x, g, _, dy = tl.inputs(M, N, "bf16", "bf16", seed=66, beta=False)
    fwd = _over_distances(debug_env, lambda: pu.run_fwd(x, g, eps, "bf16", "bf16"))
    rstd = oracle.fwd(x, g, eps, "bf16", "bf16", want64=False)["rstd"]
    bwd = _over_distances(debug_env, lambda: pu.run_bwd(dy, x, rstd, g, eps, "bf16", "bf16"))
    ref = oracle.fwd(x, g, eps, "bf16", "bf16")
    pu.check_bf16_ulp(fwd["y"], ref["y"], what="y")
    check_bwd(x, dy, g, rstd, eps, "bf16", "bf16", bwd)


@pytest.mark.parametrize("op,M,N,aligned,ahead", [
    (rn.OP_FUSED_ADD, 32768, 4096, False, 1),    # 608 CTAs x 2 rows of 8 KB: one step
    (rn.OP_FUSED_ADD, 32768, 2048, False, None),
    (rn.OP_BWD, 32768, 4096, False, None),
    (rn.OP_FWD, 8192, 20000, "mixed", 0),        # 608 x 40 KB: none
    (rn.OP_BWD, 8192, 20000, "mixed", 0),
])
def test_wide_dispatch(op, M, N, aligned, ahead):
    plan = rn.rmsnorm_describe_plan(op, M, N, "bf16", "bf16", aligned)
    assert "/wide/" in plan, plan
    grid = int(plan.split("/grid")[1].split("/")[0])
    inputs = 1 if op == rn.OP_FWD else 2
    want = min(2, (12 << 20) // (grid * inputs * N * 2))
    if ahead is not None:
        assert want == ahead, plan
    assert (f"/l2ahead{want}" in plan) if want else ("/l2ahead" not in plan), plan


def test_wide_rows_bits_do_not_depend_on_it(debug_env):
    import seeded_inputs as si
    from tests.test_parity_fwd import check_fused
    M, N, eps = 3001, 4096, tl.f32(1e-6)
    x, g, _, dy = tl.inputs(M, N, "bf16", "bf16", seed=67, beta=False)
    r = si.fill((M, N), seed=67, tensor_id=2, dtype="bf16")
    # y off the residual: the fused add's wide form
    fused = _over_distances(debug_env, lambda: pu.run_fused(
        x, r, g, eps, "bf16", "bf16", want_rstd=True, offsets={"y": 2}))
    check_fused(x, r, g, eps, "bf16", "bf16", fused, want_rstd=True)
    # x off dy and dx: the wide backward's shifted reads
    rstd = oracle.fwd(x, g, eps, "bf16", "bf16", want64=False)["rstd"]
    runs = []
    for l2 in (0, 1, 3):
        debug_env.set("RMSNORM_FORCE_VARIANT", f"wide:l2={l2}")
        runs.append(pu.run_bwd(dy, x, rstd, g, eps, "bf16", "bf16", offsets={"x": 6}))
    debug_env.delete("RMSNORM_FORCE_VARIANT", raising=False)
    _same(runs)
    check_bwd(x, dy, g, rstd, eps, "bf16", "bf16", runs[0])
