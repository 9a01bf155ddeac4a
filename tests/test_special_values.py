"""Rows with special values through the backward and LayerNorm kernels: a
constant row, a zero row (eps > 0), rows scaled by 1e15 and by 1e-15, and a
row with every third element zero, at the row lengths of the sub-warp,
staged, ragged and generic families, compared with the oracle."""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity_util as pu
from tests import test_parity_layernorm as tl
from tests.test_parity_bwd import check_bwd

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _special_rows(M, N, seed, xd="bf16"):
    x = si.fill((M, N), seed=seed, tensor_id=1, dtype=xd).copy()
    x[0] = oracle.round_bf16(37.0) if xd == "bf16" else np.float32(37.0)
    x[1] = 0
    x[2] = si.fill(N, seed=seed + 1, tensor_id=1, dtype=xd, p1=1e15)
    x[3] = si.fill(N, seed=seed + 1, tensor_id=2, dtype=xd, p1=1e-15)
    x[4, ::3] = 0
    return x


@pytest.mark.parametrize("N", [128, 8192, 2049, 40000])
@pytest.mark.parametrize("saved", [True, False])
def test_rmsnorm_backward_special_rows(N, saved):
    M, eps = 7, float(np.float32(1e-5))
    x = _special_rows(M, N, seed=80)
    g = si.fill(N, seed=80, tensor_id=3, p0=1.0, p1=0.1, dtype="f32")
    dy = si.fill((M, N), seed=80, tensor_id=4, dtype="bf16")
    rstd = oracle.fwd(x, g, eps, "bf16", "f32", want64=False)["rstd"] if saved else None
    out = pu.run_bwd(dy, x, rstd, g, eps, "bf16", "f32")
    check_bwd(x, dy, g, rstd, eps, "bf16", "f32", out)


@pytest.mark.parametrize("N", [128, 1024, 8192, 2049])
def test_layernorm_special_rows(N):
    M, eps = 7, tl.f32(1e-5)
    x = _special_rows(M, N, seed=81)
    _, g, b, dy = tl.inputs(M, N, "bf16", "bf16", seed=81)
    tl.check_fwd(tl.run_fwd(x, g, b, eps, "bf16", "bf16"), x, g, b, eps, "bf16", "bf16")
    fw = oracle.layernorm_fwd(x, g, b, eps, "bf16", "bf16")
    for mean, rstd in ((fw["mean"], fw["rstd"]), (None, None)):
        out = tl.run_bwd(dy, x, mean, rstd, g, eps, "bf16", "bf16")
        tl.check_bwd(out, dy, x, mean, rstd, g, eps, "bf16", "bf16")
