"""GPU parity of the wide kernel (two passes of 16-byte vectors per row, each
pass in the frame of one operand's alignment, the other operands realigned to
it) against the oracle, element by element.

It serves what the register, ring and cluster kernels do not take: outputs
that disagree modulo 16 bytes (y off the residual in the fused add), rows
beyond the mixed-alignment tiers, rows off 16 bytes beyond the ragged tier.
Forced shapes put every operation and dtype pair through it at offsets of
every operand, rows too short for a body, one-vector bodies and rows that
several CTAs walk in turn; the default dispatch reaches it on long rows.
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

PAIRS = [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")]


def f32(v):
    return float(np.float32(v))


def es(xd):
    return 4 if xd == "f32" else 2


# byte offsets from a 256-byte boundary, in element units of the activation
# dtype (gamma in its own): outputs off each other, inputs off the outputs,
# everything off
FWD_OFFSETS = [{}, {"x": 1}, {"y": 1}, {"y": 3, "residual": 0, "x": 5},
               {"x": 7, "y": 2, "residual": 6, "gamma": 1}, {"residual": 1}]


def scaled(offsets, xd, wd):
    return {k: v * (es(wd) if k == "gamma" else es(xd)) % 16 for k, v in offsets.items()}


def _fwd_cases():
    out = []
    for xd, wd in PAIRS:
        for N in ((1, 3, 4, 129, 1000, 4100, 20000) if xd == "f32" else
                  (1, 7, 9, 129, 1000, 2049, 8192, 20001)):
            for k, o in enumerate(FWD_OFFSETS):
                if (N + k) % 2 == 0 or N in (1, 20000, 20001):
                    out.append((xd, wd, N, k))
    return out


@pytest.mark.parametrize("xd,wd,N,k", _fwd_cases())
def test_wide_fwd_and_fused_add(debug_env, xd, wd, N, k):
    debug_env.set("RMSNORM_FORCE_VARIANT", "wide:cps=1")
    M = 37 if N >= 16384 else 300
    o = scaled(FWD_OFFSETS[k], xd, wd)
    x, g = make_fwd(M, N, xd, wd, seed=N + 80 + k)
    eps = f32(1e-5)
    check_fwd(x, g, eps, xd, wd, pu.run_fwd(x, g, eps, xd, wd, offsets=o))
    r = si.fill((M, N), seed=N + 80 + k, tensor_id=2, dtype=xd, p1=3.0)
    out = pu.run_fused(x, r, g, eps, xd, wd, want_rstd=True, offsets=o)
    check_fused(x, r, g, eps, xd, wd, out, want_rstd=True)


BWD_OFFSETS = [{}, {"x": 1}, {"dy": 3}, {"dx": 1}, {"x": 5, "dy": 2, "dx": 7, "gamma": 1},
               {"x": 1, "dy": 1, "dx": 1}]


def _bwd_cases():
    out = []
    for xd, wd in PAIRS:
        # rows a multiple of 16 bytes (dx's split the same for every row)
        for N in ((4, 8, 1032, 4096, 20000) if xd == "f32" else (8, 16, 1032, 8192, 20000)):
            for k in range(len(BWD_OFFSETS)):
                out.append((xd, wd, N, k))
    return out


@pytest.mark.parametrize("xd,wd,N,k", _bwd_cases())
def test_wide_bwd(debug_env, xd, wd, N, k):
    debug_env.set("RMSNORM_FORCE_VARIANT", "wide:cps=1")
    M = 37 if N >= 16384 else 700
    o = scaled(BWD_OFFSETS[k], xd, wd)
    x, dy, g = make_bwd(M, N, xd, wd, seed=N + 81 + k)
    eps = f32(1e-5)
    rstd = oracle.fwd(x, g, eps, xd, wd)["rstd"]
    check_bwd(x, dy, g, rstd, eps, xd, wd, pu.run_bwd(dy, x, rstd, g, eps, xd, wd, offsets=o))
    if k % 2 == 0:   # rstd recomputed from x and eps
        check_bwd(x, dy, g, None, eps, xd, wd,
                  pu.run_bwd(dy, x, None, g, eps, xd, wd, offsets=o))


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N", [1032, 20000])
@pytest.mark.parametrize("offsets", [{}, {"h": 1}, {"dy": 3, "dres": 1}, {"h": 2, "dy": 5}])
def test_wide_fused_add_bwd(debug_env, xd, wd, N, offsets):
    debug_env.set("RMSNORM_FORCE_VARIANT", "wide:cps=1")
    M = 37 if N >= 16384 else 500
    o = scaled(offsets, xd, wd)
    h, dy, dres, g = make_fused_bwd(M, N, xd, wd, seed=N + 82)
    eps = f32(1e-5)
    rstd = oracle.fwd(h, g, eps, xd, wd)["rstd"]
    out = run_fused_bwd(h, dy, dres, g, rstd, eps, xd, wd, offsets=o)
    check_fused_bwd(h, dy, dres, g, rstd, eps, xd, wd, out)


def test_wide_dgamma_is_bitwise_reproducible(debug_env):
    debug_env.set("RMSNORM_FORCE_VARIANT", "wide")
    x, dy, g = make_bwd(600, 4096, "bf16", "f32", seed=83)
    eps = f32(1e-5)
    rstd = oracle.fwd(x, g, eps, "bf16", "f32")["rstd"]
    outs = pu.run_bwd(dy, x, rstd, g, eps, "bf16", "f32", offsets={"x": 2, "dy": 6, "dx": 4},
                      repeat=3)
    for o in outs[1:]:
        assert np.array_equal(o["dgamma"].view(np.uint32), outs[0]["dgamma"].view(np.uint32))
        assert np.array_equal(o["dx"], outs[0]["dx"])


def test_wide_rejects_backward_rows_off_16_bytes(debug_env):
    # dx's split would move from row to row: the forced plan is refused
    debug_env.set("RMSNORM_FORCE_VARIANT", "wide")
    with pytest.raises(rn.RMSNormError):
        rn.rmsnorm_describe_plan(rn.OP_BWD, 64, 2049, "bf16", "bf16", False)
    assert "/wide/" in rn.rmsnorm_describe_plan(rn.OP_FWD, 64, 2049, "bf16", "bf16", False)


def test_wide_plans():
    def plan(op, N, a, M=4096, xd="bf16"):
        return rn.rmsnorm_describe_plan(op, M, N, xd, xd, a)
    # outputs off each other (or x off y with rows beyond the mixed tiers)
    for N in (4096, 2049, 128):
        assert "/wide/" in plan(rn.OP_FUSED_ADD, N, False), plan(rn.OP_FUSED_ADD, N, False)
    for op in (rn.OP_FWD, rn.OP_FUSED_ADD):
        for N in (20000, 40001, 1 << 19):
            assert "/wide/" in plan(op, N, "mixed", 64), plan(op, N, "mixed", 64)
    # rows off 16 bytes beyond the ragged tier (the forward)
    assert "/wide/" in plan(rn.OP_FWD, 40001, True, 64)
    # the backward with rows a multiple of 16 bytes; the dgamma partial row
    # must fit in shared memory
    for op in (rn.OP_BWD, rn.OP_FUSED_ADD_BWD):
        assert "/wide/" in plan(op, 20000, "mixed", 64), plan(op, 20000, "mixed", 64)
        assert "/wide/" in plan(op, 4096, False), plan(op, 4096, False)
        assert "/generic/" in plan(op, 40001, "mixed", 64), plan(op, 40001, "mixed", 64)
        assert "/generic/" in plan(op, 65536, "mixed", 64), plan(op, 65536, "mixed", 64)
