"""The measured workloads at full size, through the same default dispatch the
bench times, compared with the oracle on every output element."""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity_util as pu
from tests.test_parity_bwd import check_bwd
from tests.test_parity_fwd import check_fused, check_fwd
from tests import test_parity_fused_bwd as fb

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.mark.parametrize("name", list(si.WORKLOADS))
def test_workload_matches_oracle(name):
    wl = si.WORKLOADS[name]
    inp = si.make_inputs(wl)
    eps = float(np.float32(wl.eps))
    x, g = inp["x"], inp["gamma"]
    off = dict(wl.offsets)
    if wl.op == "fwd":
        out = pu.run_fwd(x, g, eps, wl.x_dtype, wl.w_dtype, want_rstd=wl.store_rstd,
                         offsets=off)
        check_fwd(x, g, eps, wl.x_dtype, wl.w_dtype, out, want_rstd=wl.store_rstd)
    elif wl.op == "fused_add":
        r = inp["residual"]
        out = pu.run_fused(x, r, g, eps, wl.x_dtype, wl.w_dtype, want_rstd=wl.store_rstd,
                           offsets=off)
        check_fused(x, r, g, eps, wl.x_dtype, wl.w_dtype, out, want_rstd=wl.store_rstd)
    elif wl.offsets and wl.op != "bwd":
        raise AssertionError(f"operand offsets are not wired for {wl.op}")
    elif wl.op in ("ln_fwd", "ln_bwd"):
        from tests import test_parity_layernorm as tl
        tl.check_workload(wl, inp)
    elif wl.op in ("fwd_fp8", "fused_add_fp8", "fwd_nvfp4", "fused_add_nvfp4"):
        from tests import test_parity_quant as tq
        tq.check_workload(wl, inp)
    elif wl.op == "fwd_strided":
        from tests import test_parity_strided as ts
        ts.check_workload(wl, inp)
    elif wl.op == "fused_add_bwd":
        # x plays the stored sum h; the saved rstd comes from the oracle forward;
        # dgamma in the weight dtype
        rstd = oracle.fwd(x, g, eps, wl.x_dtype, wl.w_dtype, want64=False)["rstd"]
        out = fb.run(x, inp["dy"], inp["residual"], g, rstd, eps, wl.x_dtype, wl.w_dtype,
                     dg_dtype=wl.w_dtype)
        info = fb.check(x, inp["dy"], inp["residual"], g, rstd, eps, wl.x_dtype, wl.w_dtype,
                        out, dg_dtype=wl.w_dtype)
        print("FLOOR", name, info["floor"], wl.M * wl.N)
    else:
        # the saved rstd comes from the oracle forward
        rstd = oracle.fwd(x, g, eps, wl.x_dtype, wl.w_dtype, want64=False)["rstd"]
        out = pu.run_bwd(inp["dy"], x, rstd, g, eps, wl.x_dtype, wl.w_dtype, offsets=off)
        info = check_bwd(x, inp["dy"], g, rstd, eps, wl.x_dtype, wl.w_dtype, out)
        # elements that needed the cancellation floor, of the tensor's size
        print("FLOOR", name, info.get("floor", 0), wl.M * wl.N, info)
