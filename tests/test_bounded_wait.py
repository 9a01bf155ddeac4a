"""The bounded waits of the bulk-copy staged kernels, exercised without any
fault: a negative wait limit (RMSNORM_WAIT_LIMIT_CYCLES=-1) makes every wait
for a row give up at once, whether or not the row has arrived.  The kernel
must then store nothing more, wait (with its own bound) for the copies it has
in flight, raise the timeout flag and return; rmsnorm_check_device reports
it, clears it, and the context stays usable for a normal call."""
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


def _data(M, N, seed):
    x = si.fill((M, N), seed=seed, tensor_id=1, dtype="bf16")
    dy = si.fill((M, N), seed=seed, tensor_id=4, dtype="bf16")
    g = si.fill(N, seed=seed, tensor_id=3, p0=1.0, p1=0.1, dtype="bf16")
    return x, dy, g


FORCE = {"bwd_short_rows": "staged:g=8:vpt=2:st=4"}


@pytest.mark.parametrize("op", ["fwd", "fused", "bwd", "bwd_short_rows"])
def test_timeout_is_reported_and_the_context_survives(debug_env, op):
    M, N, eps = 1024, 8192, float(np.float32(1e-5))
    if op == "bwd_short_rows":     # 32 rows of 128 per stage of the ring
        M, N = 8192, 128
    x, dy, g = _data(M, N, seed=41)
    debug_env.set("RMSNORM_FORCE_VARIANT", FORCE.get(op, "staged:vpt=4:st=4"))
    rn.rmsnorm_check_device()                    # start from a clear flag
    debug_env.set("RMSNORM_WAIT_LIMIT_CYCLES", "-1")
    if op == "fwd":
        pu.run_fwd(x, g, eps, "bf16", "bf16")
    elif op == "fused":
        pu.run_fused(x, dy, g, eps, "bf16", "bf16")
    else:
        pu.run_bwd(dy, x, None, g, eps, "bf16", "bf16")
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_check_device()
    assert e.value.status == 6                   # RMSNORM_ERR_TIMEOUT
    rn.rmsnorm_check_device()                    # the flag was cleared

    # same variant, normal limit: correct results, no flag
    debug_env.delete("RMSNORM_WAIT_LIMIT_CYCLES")
    if op in FORCE:
        from tests.test_parity_bwd import check_bwd
        out = pu.run_bwd(dy, x, None, g, eps, "bf16", "bf16")
        check_bwd(x, dy, g, None, eps, "bf16", "bf16", out)
    else:
        out = pu.run_fwd(x, g, eps, "bf16", "bf16")
        ref = oracle.fwd(x, g, eps, "bf16", "bf16")
        pu.check_bf16_ulp(out["y"], ref["y"])
    rn.rmsnorm_check_device()


def test_check_device_is_quiet_after_normal_work():
    M, N, eps = 256, 4096, float(np.float32(1e-5))
    x, dy, g = _data(M, N, seed=42)
    pu.run_fwd(x, g, eps, "bf16", "bf16")
    pu.run_bwd(dy, x, None, g, eps, "bf16", "bf16")
    rn.rmsnorm_check_device()
