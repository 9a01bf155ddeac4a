"""Rows too long for one CTA, on thread-block clusters: forward, fused add,
backward and fused-add backward against the oracle, element by element.

Shapes cover every cluster size (2, 4, 8 CTAs), slices that do not divide the
row evenly, one and two rows (far fewer clusters than the device holds),
persistent walks of many rows per cluster (forced to one CTA per SM), the
two dtype pairs with 16-bit activations and fp32, the saved and the
recomputed rstd, and the bounded bulk-copy waits voted across a cluster.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity_util as pu
from tests import test_parity_fused_bwd as fb
from tests.test_parity_bwd import check_bwd
from tests.test_parity_fwd import check_fused, check_fwd, make

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import row_wise_normalization_02_gb300 as rn  # noqa: E402

PAIRS = [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")]
EPS = float(np.float32(1e-5))


def plan(op, M, N, xd, wd):
    return rn.rmsnorm_describe_plan(op, M, N, xd, wd)


# bf16 row lengths: the fused add on clusters from 4097 vectors on
# (N > 32768), the forward and the backward from 2049 (N > 16384); fp32 rows
# hold half as many elements
N_FWD = {"bf16": [32776, 40000, 65536, 131072, 262144], "f32": [16388, 40000, 65536]}
N_BWD = {"bf16": [16392, 20000, 24576, 40000, 65536, 131072], "f32": [8196, 40000, 65536]}


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("i", range(5))
def test_forward_and_fused_add(xd, wd, i):
    if i >= len(N_FWD[xd]):
        pytest.skip("no such length for this dtype")
    N = N_FWD[xd][i]
    M = 24
    assert "/cluster/" in plan(0, M, N, xd, wd) and "/cluster/" in plan(1, M, N, xd, wd)
    x, g = make(M, N, xd, wd, seed=N + 3)
    check_fwd(x, g, EPS, xd, wd, pu.run_fwd(x, g, EPS, xd, wd))
    r = si.fill((M, N), seed=N + 4, tensor_id=2, dtype=xd, p1=2.0)
    out = pu.run_fused(x, r, g, EPS, xd, wd, want_rstd=True)
    check_fused(x, r, g, EPS, xd, wd, out, want_rstd=True)


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("i", range(6))
@pytest.mark.parametrize("saved", [True, False])
def test_backward(xd, wd, i, saved):
    if i >= len(N_BWD[xd]):
        pytest.skip("no such length for this dtype")
    N = N_BWD[xd][i]
    M = 24
    assert "/cluster/" in plan(2, M, N, xd, wd)
    x, g = make(M, N, xd, wd, seed=N + 5)
    dy = si.fill((M, N), seed=N + 5, tensor_id=4, dtype=xd)
    rstd = oracle.fwd(x, g, EPS, xd, wd, want64=False)["rstd"] if saved else None
    out = pu.run_bwd(dy, x, rstd, g, EPS, xd, wd)
    check_bwd(x, dy, g, rstd, EPS, xd, wd, out)


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N", [16392, 32768, 40000])
@pytest.mark.parametrize("dg", ["f32", "w"])
def test_fused_add_backward(xd, wd, N, dg):
    if xd == "f32":
        N //= 2
    M = 20
    assert "/cluster/" in plan(3, M, N, xd, wd)
    h, g = make(M, N, xd, wd, seed=N + 6)
    dy = si.fill((M, N), seed=N + 6, tensor_id=4, dtype=xd)
    dres = si.fill((M, N), seed=N + 6, tensor_id=2, dtype=xd)
    rstd = oracle.fwd(h, g, EPS, xd, wd, want64=False)["rstd"]
    dgd = "f32" if dg == "f32" else wd
    out = fb.run(h, dy, dres, g, rstd, EPS, xd, wd, dg_dtype=dgd)
    fb.check(h, dy, dres, g, rstd, EPS, xd, wd, out, dg_dtype=dgd)


@pytest.mark.parametrize("M", [1, 2, 3])
@pytest.mark.parametrize("N", [24576, 40000, 65536])
def test_one_to_three_rows(M, N):
    x, g = make(M, N, "bf16", "bf16", seed=M + N)
    check_fwd(x, g, EPS, "bf16", "bf16", pu.run_fwd(x, g, EPS, "bf16", "bf16"))
    dy = si.fill((M, N), seed=M + N, tensor_id=4, dtype="bf16")
    for rstd in (oracle.fwd(x, g, EPS, "bf16", "bf16", want64=False)["rstd"], None):
        out = pu.run_bwd(dy, x, rstd, g, EPS, "bf16", "bf16")
        check_bwd(x, dy, g, rstd, EPS, "bf16", "bf16", out)


@pytest.mark.parametrize("force,N", [
    ("cluster:cl=2:cps=1", 40000), ("cluster:cl=4:cps=1", 40000), ("cluster:cl=8:cps=1", 40000),
    ("cluster:cl=2:vpt=8:pf=0:cps=1", 65536), ("cluster:cl=8:vpt=2:cps=1", 32776),
    ("cluster:cl=4:pf=0:cps=1", 65536), ("cluster:cl=2:cps=1", 16384),
    ("cluster:cl=4:t=512:cps=1", 40000),
])
def test_forward_forced_clusters_walk_many_rows(debug_env, force, N):
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    M = 300
    assert "/cluster/" in plan(0, M, N, "bf16", "bf16")
    x, g = make(M, N, "bf16", "bf16", seed=N + 7)
    check_fwd(x, g, EPS, "bf16", "bf16", pu.run_fwd(x, g, EPS, "bf16", "bf16"))
    r = si.fill((M, N), seed=N + 8, tensor_id=2, dtype="bf16")
    out = pu.run_fused(x, r, g, EPS, "bf16", "bf16", want_rstd=True)
    check_fused(x, r, g, EPS, "bf16", "bf16", out, want_rstd=True)


@pytest.mark.parametrize("force,N", [
    ("cluster:cl=2:cps=1", 16392), ("cluster:cl=4:cps=1", 40000), ("cluster:cl=8:cps=1", 40000),
    ("cluster:cl=8:st=3:cps=1", 65536), ("cluster:cl=8:vpt=2:st=2:cps=1", 32776),
    ("cluster:cl=2:cps=1", 8192), ("cluster:cl=4:st=4:cps=1", 24576),
])
def test_backward_forced_clusters_walk_many_rows(debug_env, force, N):
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    M = 300
    assert "/cluster/" in plan(2, M, N, "bf16", "f32")
    x, g = make(M, N, "bf16", "f32", seed=N + 9)
    dy = si.fill((M, N), seed=N + 9, tensor_id=4, dtype="bf16")
    rstd = oracle.fwd(x, g, EPS, "bf16", "f32", want64=False)["rstd"]
    out = pu.run_bwd(dy, x, rstd, g, EPS, "bf16", "f32")
    check_bwd(x, dy, g, rstd, EPS, "bf16", "f32", out)
    h = x
    dres = si.fill((M, N), seed=N + 10, tensor_id=2, dtype="bf16")
    out = fb.run(h, dy, dres, g, rstd, EPS, "bf16", "f32")
    fb.check(h, dy, dres, g, rstd, EPS, "bf16", "f32", out)


def test_dgamma_is_bitwise_reproducible():
    M, N = 600, 40000
    x, g = make(M, N, "bf16", "f32", seed=11)
    dy = si.fill((M, N), seed=11, tensor_id=4, dtype="bf16")
    rstd = oracle.fwd(x, g, EPS, "bf16", "f32", want64=False)["rstd"]
    outs = pu.run_bwd(dy, x, rstd, g, EPS, "bf16", "f32", repeat=3)
    for o in outs[1:]:
        assert np.array_equal(o["dgamma"].view(np.uint32), outs[0]["dgamma"].view(np.uint32))
        assert np.array_equal(o["dx"], outs[0]["dx"])


@pytest.mark.parametrize("dres", [False, True])
def test_wait_timeout_is_voted_across_the_cluster(debug_env, dres):
    # every wait gives up at once in every CTA: the cluster agrees through its
    # exchange, all CTAs stop at the first row, drain their copies and leave
    M, N = 256, 40000
    x, g = make(M, N, "bf16", "bf16", seed=12)
    dy = si.fill((M, N), seed=12, tensor_id=4, dtype="bf16")
    rn.rmsnorm_check_device()
    debug_env.set("RMSNORM_WAIT_LIMIT_CYCLES", "-1")
    if dres:
        fb.run(x, dy, dy, g, None, EPS, "bf16", "bf16")
    else:
        pu.run_bwd(dy, x, None, g, EPS, "bf16", "bf16")
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_check_device()
    assert e.value.status == 6
    rn.rmsnorm_check_device()
    debug_env.delete("RMSNORM_WAIT_LIMIT_CYCLES")
    rstd = oracle.fwd(x, g, EPS, "bf16", "bf16", want64=False)["rstd"]
    out = pu.run_bwd(dy, x, rstd, g, EPS, "bf16", "bf16")
    check_bwd(x, dy, g, rstd, EPS, "bf16", "bf16", out)
    rn.rmsnorm_check_device()
