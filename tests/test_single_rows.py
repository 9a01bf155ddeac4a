"""One and two rows, at the row lengths of every kernel family: the grid then
has far more CTAs than rows (most walk no row at all), no row has a successor
to prefetch or to request into L2, and the backward's partial rows come from
one or two CTAs.  Every operation is compared with the oracle."""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity_util as pu
from tests import test_parity_fused_bwd as fb
from tests import test_parity_layernorm as tl
from tests import test_parity_quant as tq
from tests.test_parity_bwd import check_bwd
from tests.test_parity_fwd import check_fused, check_fwd, make

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

# sub-warp, CTA (and staged backward), ragged, beyond the register tiers
N_RMS = [128, 1024, 8192, 2049, 40000]
EPS = float(np.float32(1e-6))


def _dy(M, N, xd, seed):
    return si.fill((M, N), seed=seed, tensor_id=4, dtype=xd)


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N", N_RMS)
def test_rmsnorm_forward_and_fused_add(M, N):
    x, g = make(M, N, "bf16", "bf16", seed=70 + N)
    check_fwd(x, g, EPS, "bf16", "bf16", pu.run_fwd(x, g, EPS, "bf16", "bf16"))
    r = make(M, N, "bf16", "bf16", seed=71 + N)[0]
    check_fused(x, r, g, EPS, "bf16", "bf16", pu.run_fused(x, r, g, EPS, "bf16", "bf16"))


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N", N_RMS)
@pytest.mark.parametrize("saved", [True, False])
def test_rmsnorm_backward(M, N, saved):
    x, g = make(M, N, "bf16", "f32", seed=72 + N)
    dy = _dy(M, N, "bf16", 72 + N)
    rstd = oracle.fwd(x, g, EPS, "bf16", "f32", want64=False)["rstd"] if saved else None
    out = pu.run_bwd(dy, x, rstd, g, EPS, "bf16", "f32")
    check_bwd(x, dy, g, rstd, EPS, "bf16", "f32", out)


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N", [128, 4096, 2049])
def test_fused_add_backward(M, N):
    h, g = make(M, N, "bf16", "bf16", seed=73 + N)
    dy, dres = _dy(M, N, "bf16", 73 + N), _dy(M, N, "bf16", 74 + N)
    rstd = oracle.fwd(h, g, EPS, "bf16", "bf16", want64=False)["rstd"]
    out = fb.run(h, dy, dres, g, rstd, EPS, "bf16", "bf16")
    fb.check(h, dy, dres, g, rstd, EPS, "bf16", "bf16", out)


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N", [128, 1024, 8192, 2049])
def test_layernorm(M, N):
    eps = tl.f32(1e-5)
    x, g, b, dy = tl.inputs(M, N, "bf16", "bf16", seed=75 + N)
    tl.check_fwd(tl.run_fwd(x, g, b, eps, "bf16", "bf16"), x, g, b, eps, "bf16", "bf16")
    fw = oracle.layernorm_fwd(x, g, b, eps, "bf16", "bf16")
    for mean, rstd in ((fw["mean"], fw["rstd"]), (None, None)):
        out = tl.run_bwd(dy, x, mean, rstd, g, eps, "bf16", "bf16")
        tl.check_bwd(out, dy, x, mean, rstd, g, eps, "bf16", "bf16")


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N", [128, 8192, 2064])
@pytest.mark.parametrize("kind", ["fp8", "nvfp4"])
def test_quantised_outputs(M, N, kind):
    x, g, r = tq.inputs(M, N, "bf16", "bf16", seed=76 + N, fused=True)
    for res in (None, r):
        out = tq.run(kind, x, g, EPS, "bf16", "bf16", residual=res, gs=tq.GS)
        if kind == "fp8":
            tq.check_fp8(out, x, g, EPS, "bf16", "bf16", residual=res)
        else:
            tq.check_nvfp4(out, x, g, EPS, "bf16", "bf16", tq.GS, residual=res)
