"""GPU parity of the mixed-alignment forms: inputs (x, dy, the fused-add
backward's h) whose rows start at another offset modulo 16 bytes than the
outputs' (for example x a view at an odd element offset of a larger buffer),
against the oracle, element by element.

The outputs set the row split (scalar head, 16-byte body, scalar tail); each
shifted input is read in aligned chunks and realigned across lanes.  Shapes
cover rows on 16 bytes (one split for every row), odd rows (the split moves
with the row), rows too short for a body, several CTAs per SM and forced
shapes whose CTAs walk many rows.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity_util as pu
from tests.test_parity_bwd import check_bwd, make as make_bwd
from tests.test_parity_fused_bwd import check as check_fused_bwd, make as make_fused_bwd
from tests.test_parity_fused_bwd import run as run_fused_bwd
from tests.test_parity_fwd import check_fused, check_fwd, make as make_fwd

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import row_wise_normalization_02_gb300 as rn  # noqa: E402


def f32(v):
    return float(np.float32(v))


def rows_for(N):
    return 37 if N >= 16384 else 129 if N >= 4096 else 300


# byte offsets of the operands from a 256-byte boundary: every shift of x
# against the outputs is a multiple of the element size
FWD_OFFSETS = {
    "bf16": [{"x": 2}, {"x": 14}, {"x": 8}, {"x": 6, "y": 4, "residual": 4},
             {"y": 2, "residual": 2}, {"x": 10, "y": 12, "residual": 12, "gamma": 4}],
    "f32": [{"x": 4}, {"x": 12, "y": 8, "residual": 8}, {"y": 4, "residual": 4}],
}
N_BF16 = [8192, 4096, 16384, 2049, 1000, 129, 9, 7, 1]
N_F32 = [4096, 8192, 1030, 5, 3]
PAIRS = [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")]


def _fwd_cases():
    out = []
    for xd, wd in PAIRS:
        for N in (N_F32 if xd == "f32" else N_BF16):
            for o in FWD_OFFSETS[xd]:
                out.append((xd, wd, N, o))
    return out


@pytest.mark.parametrize("xd,wd,N,offsets", _fwd_cases())
def test_mixed_fwd(xd, wd, N, offsets):
    M = rows_for(N)
    x, g = make_fwd(M, N, xd, wd, seed=N + 71)
    eps = f32(1e-5)
    out = pu.run_fwd(x, g, eps, xd, wd, offsets=offsets)
    check_fwd(x, g, eps, xd, wd, out)


@pytest.mark.parametrize("xd,wd,N,offsets", [c for c in _fwd_cases()
                                             if c[2] in (8192, 2049, 129, 7, 1030, 5)])
def test_mixed_fused_add(xd, wd, N, offsets):
    M = rows_for(N)
    x, g = make_fwd(M, N, xd, wd, seed=N + 72)
    r = si.fill((M, N), seed=N + 72, tensor_id=2, dtype=xd, p1=3.0)
    eps = f32(1e-6)
    out = pu.run_fused(x, r, g, eps, xd, wd, want_rstd=True, offsets=offsets)
    check_fused(x, r, g, eps, xd, wd, out, want_rstd=True)


BWD_OFFSETS = {
    "bf16": [{"x": 2}, {"dy": 6}, {"x": 2, "dy": 10}, {"x": 4, "dy": 4},
             {"dx": 2}, {"x": 14, "dy": 12, "dx": 8, "gamma": 4}],
    "f32": [{"x": 4}, {"dy": 8, "x": 12}, {"dx": 4}],
}


def _bwd_cases():
    out = []
    for xd, wd in PAIRS:
        for N in (N_F32 if xd == "f32" else N_BF16):
            for o in BWD_OFFSETS[xd]:
                out.append((xd, wd, N, o))
    return out


@pytest.mark.parametrize("xd,wd,N,offsets", _bwd_cases())
def test_mixed_bwd(xd, wd, N, offsets):
    M = rows_for(N)
    x, dy, g = make_bwd(M, N, xd, wd, seed=N + 73)
    eps = f32(1e-5)
    rstd = oracle.fwd(x, g, eps, xd, wd)["rstd"]
    out = pu.run_bwd(dy, x, rstd, g, eps, xd, wd, offsets=offsets)
    check_bwd(x, dy, g, rstd, eps, xd, wd, out)


@pytest.mark.parametrize("N", [8192, 2049, 9])
def test_mixed_bwd_recomputed_rstd(N):
    M = rows_for(N)
    x, dy, g = make_bwd(M, N, "bf16", "f32", seed=N + 74)
    eps = f32(1e-5)
    out = pu.run_bwd(dy, x, None, g, eps, "bf16", "f32", offsets={"x": 6, "dy": 2})
    check_bwd(x, dy, g, None, eps, "bf16", "f32", out)


@pytest.mark.parametrize("xd,wd", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32")])
@pytest.mark.parametrize("N", [4096, 2049, 7])
@pytest.mark.parametrize("which", ["h", "dy", "both"])
def test_mixed_fused_add_bwd(xd, wd, N, which):
    if xd == "f32" and N in (7, 2049):
        N += 1
    s = 4 if xd == "f32" else 2
    offsets = {"h": {"h": s}, "dy": {"dy": 3 * s}, "both": {"h": s, "dy": 2 * s}}[which]
    M = rows_for(N)
    h, dy, dres, g = make_fused_bwd(M, N, xd, wd, seed=N + 75)
    eps = f32(1e-5)
    rstd = oracle.fwd(h, g, eps, xd, wd)["rstd"]
    out = run_fused_bwd(h, dy, dres, g, rstd, eps, xd, wd, offsets=offsets)
    check_fused_bwd(h, dy, dres, g, rstd, eps, xd, wd, out)


@pytest.mark.parametrize("force,N", [
    ("ragged:vpt=2:pf=1:cps=1", 2049), ("ragged:vpt=2:pf=0:cps=1", 4096),
    ("ragged:vpt=1:pf=1:cps=1", 1000), ("ragged:vpt=1:pf=0:cps=2", 2049),
    ("ragged:vpt=4:pf=0:cps=1", 8192), ("ragged:vpt=4:pf=0:t=96:cps=1", 2049),
])
def test_mixed_forced_shapes_walk_several_rows(debug_env, force, N):
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    M = 700
    eps = f32(1e-5)
    x, g = make_fwd(M, N, "bf16", "bf16", seed=N + 76)
    check_fwd(x, g, eps, "bf16", "bf16", pu.run_fwd(x, g, eps, "bf16", "bf16", offsets={"x": 6}))
    r = si.fill((M, N), seed=N + 76, tensor_id=2, dtype="bf16")
    out = pu.run_fused(x, r, g, eps, "bf16", "bf16", want_rstd=True, offsets={"x": 10})
    check_fused(x, r, g, eps, "bf16", "bf16", out, want_rstd=True)
    x, dy, g = make_bwd(M, N, "bf16", "f32", seed=N + 77)
    rstd = oracle.fwd(x, g, eps, "bf16", "f32")["rstd"]
    out = pu.run_bwd(dy, x, rstd, g, eps, "bf16", "f32", offsets={"x": 2, "dy": 12})
    check_bwd(x, dy, g, rstd, eps, "bf16", "f32", out)


def test_mixed_dgamma_is_bitwise_reproducible():
    x, dy, g = make_bwd(600, 4096, "bf16", "f32", seed=78)
    eps = f32(1e-5)
    rstd = oracle.fwd(x, g, eps, "bf16", "f32")["rstd"]
    outs = pu.run_bwd(dy, x, rstd, g, eps, "bf16", "f32", offsets={"x": 2, "dy": 6}, repeat=3)
    for o in outs[1:]:
        assert np.array_equal(o["dgamma"].view(np.uint32), outs[0]["dgamma"].view(np.uint32))
        assert np.array_equal(o["dx"], outs[0]["dx"])


@pytest.mark.parametrize("force,N,dres", [
    ("staged:vpt=4:st=2:cps=1", 8192, False), ("staged:vpt=2:st=3:cps=1", 4096, False),
    ("staged:vpt=1:st=2:cps=1", 2048, False), ("staged:vpt=4:st=3:cps=1", 4096, True),
    ("staged:vpt=2:st=2:cps=1", 1032, True),
])
def test_mixed_staged_backward_walks_several_rows(debug_env, force, N, dres):
    # dx (and dres) and gamma on 16 bytes, x / h and dy off them: the ring
    # copies their rows' enclosing spans
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    M, eps = 700, f32(1e-5)
    if dres:
        h, dy, dr, g = make_fused_bwd(M, N, "bf16", "f32", seed=N + 79)
        rstd = oracle.fwd(h, g, eps, "bf16", "f32")["rstd"]
        out = run_fused_bwd(h, dy, dr, g, rstd, eps, "bf16", "f32", offsets={"h": 14, "dy": 4})
        check_fused_bwd(h, dy, dr, g, rstd, eps, "bf16", "f32", out)
        return
    x, dy, g = make_bwd(M, N, "bf16", "f32", seed=N + 79)
    rstd = oracle.fwd(x, g, eps, "bf16", "f32")["rstd"]
    for off in ({"x": 2}, {"dy": 10}, {"x": 6, "dy": 12}):
        out = pu.run_bwd(dy, x, rstd, g, eps, "bf16", "f32", offsets=off)
        check_bwd(x, dy, g, rstd, eps, "bf16", "f32", out)


def test_mixed_plans():
    def plan(op, N, M=4096):
        return rn.rmsnorm_describe_plan(op, M, N, "bf16", "bf16", "mixed")
    for op in (0, 1):
        for N in (8192, 2049, 128, 15000):
            assert "/ragged_mix/" in plan(op, N), plan(op, N)
    for op in (2, 3):
        # rows a multiple of 16 bytes, 129-2048 vectors: the ring backward
        for N in (8192, 4096, 15000, 1032):
            assert "/staged_mix/" in plan(op, N), plan(op, N)
        for N in (2049, 128, 1000):
            assert "/ragged_mix/" in plan(op, N), plan(op, N)
    for op in (0, 1, 2, 3):
        # beyond four vectors per thread in 512 threads: the wide two-pass
        # kernel, or the scalar one for backward rows off 16 bytes
        for N in (16385, 40001, 20000):
            fam = "/wide/" if op < 2 or N == 20000 else "/generic/"
            assert fam in plan(op, N, 64), plan(op, N, 64)
    # 1024 vectors at 31 per warp and slot: four vectors per thread, 9 warps
    assert "/vpt4/t288/pf1/" in plan(0, 8192), plan(0, 8192)
