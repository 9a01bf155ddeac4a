"""The PyTorch training functions (row_wise_normalization_02_gb300.autograd)
are marshalling over the C ABI: their outputs and gradients must carry the
same bits as the direct calls on the same inputs (whose parity with the
oracle the other tests establish), with weight gradients in the weight
dtype; the fused add must leave the caller's residual untouched and chain
through several layers."""
import numpy as np
import pytest

import seeded_inputs as si
from tests import parity_util as pu
from tests import test_parity_fused_bwd as fb
from tests import test_parity_layernorm as tl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from row_wise_normalization_02_gb300 import autograd as ag  # noqa: E402

TD = {"bf16": torch.bfloat16, "f32": torch.float32}


def _t(a, dt, grad=False):
    t = torch.from_numpy(a.view(np.int16) if dt == "bf16" else a).cuda()
    t = t.view(torch.bfloat16) if dt == "bf16" else t
    return t.clone().requires_grad_(grad)


def _np(t, dt):
    t = t.detach().contiguous().cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def _cast_like(a32, dt):
    """fp32 array -> the weight dtype as torch rounds it (autograd's cast)."""
    return _np(torch.from_numpy(a32).to(TD[dt]), dt)


PAIRS = [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32")]


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N", [128, 4096, 2049])
def test_rms_norm_matches_the_abi(xd, wd, N):
    M, eps = 300, float(np.float32(1e-6))
    x = si.fill((M, N), seed=90, tensor_id=1, dtype=xd)
    g = si.fill(N, seed=90, tensor_id=3, p0=1.0, p1=0.1, dtype=wd)
    dy = si.fill((M, N), seed=90, tensor_id=4, dtype=xd)
    tx, tg = _t(x, xd, True), _t(g, wd, True)
    y = ag.rms_norm(tx, tg, eps)
    y.backward(_t(dy, xd))
    fw = pu.run_fwd(x, g, eps, xd, wd)
    bw = pu.run_bwd(dy, x, fw["rstd"], g, eps, xd, wd)
    assert np.array_equal(_np(y, xd), fw["y"])
    assert np.array_equal(_np(tx.grad, xd), bw["dx"])
    assert tg.grad.dtype == TD[wd]
    assert np.array_equal(_np(tg.grad, wd), _cast_like(bw["dgamma"], wd))


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N", [128, 4096, 2049])
def test_fused_add_rms_norm_matches_the_abi(xd, wd, N):
    M, eps = 300, float(np.float32(1e-6))
    x = si.fill((M, N), seed=91, tensor_id=1, dtype=xd)
    r = si.fill((M, N), seed=91, tensor_id=2, dtype=xd)
    g = si.fill(N, seed=91, tensor_id=3, p0=1.0, p1=0.1, dtype=wd)
    dy = si.fill((M, N), seed=91, tensor_id=4, dtype=xd)
    dh = si.fill((M, N), seed=92, tensor_id=4, dtype=xd)
    tx, tr, tg = _t(x, xd, True), _t(r, xd, True), _t(g, wd, True)
    r_before = _np(tr, xd).copy()
    y, h = ag.fused_add_rms_norm(tx, tr, tg, eps)
    assert np.array_equal(_np(tr, xd), r_before), "the caller's residual was modified"
    torch.autograd.backward([y, h], [_t(dy, xd), _t(dh, xd)])
    fw = pu.run_fused(x, r, g, eps, xd, wd, want_rstd=True)
    assert np.array_equal(_np(y, xd), fw["y"]) and np.array_equal(_np(h, xd), fw["h"])
    bw = fb.run(fw["h"], dy, dh, g, fw["rstd"], eps, xd, wd, dg_dtype=wd)
    assert np.array_equal(_np(tx.grad, xd), bw["dh"])
    assert np.array_equal(_np(tr.grad, xd), bw["dh"])
    assert tg.grad.dtype == TD[wd]
    assert np.array_equal(_np(tg.grad, wd), bw["dgamma"])


def test_fused_add_layers_chain_through_the_residual():
    # three pre-norm layers sharing one residual stream: the h each layer
    # saves stays valid while the next layers run (no in-place reuse)
    M, N, eps = 256, 1024, 1e-6
    torch.manual_seed(0)
    xs = [torch.randn(M, N, device="cuda", dtype=torch.bfloat16, requires_grad=True)
          for _ in range(3)]
    gs = [torch.ones(N, device="cuda", dtype=torch.bfloat16, requires_grad=True)
          for _ in range(3)]
    h = torch.randn(M, N, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    loss = 0
    for x, g in zip(xs, gs):
        y, h = ag.fused_add_rms_norm(x, h, g, eps)
        loss = loss + (y.float() ** 2).mean()
    loss.backward()
    for t in xs + gs:
        assert t.grad is not None and torch.isfinite(t.grad.float()).all()


@pytest.mark.parametrize("xd,wd", PAIRS)
@pytest.mark.parametrize("N,beta", [(128, True), (8192, True), (2049, False), (1024, True)])
def test_layer_norm_matches_the_abi(xd, wd, N, beta):
    M, eps = 300, tl.f32(1e-5)
    x, g, b, dy = tl.inputs(M, N, xd, wd, seed=93, beta=beta)
    tx, tg = _t(x, xd, True), _t(g, wd, True)
    tb = _t(b, wd, True) if beta else None
    y = ag.layer_norm(tx, tg, tb, eps)
    y.backward(_t(dy, xd))
    fw = tl.run_fwd(x, g, b, eps, xd, wd)
    bw = tl.run_bwd(dy, x, fw["mean"], fw["rstd"], g, eps, xd, wd)
    assert np.array_equal(_np(y, xd), fw["y"])
    assert np.array_equal(_np(tx.grad, xd), bw["dx"])
    assert np.array_equal(_np(tg.grad, wd), _cast_like(bw["dgamma"], wd))
    if beta:
        assert np.array_equal(_np(tb.grad, wd), _cast_like(bw["dbeta"], wd))


def test_weight_gradients_can_be_skipped():
    M, N, eps = 64, 512, 1e-6
    x = torch.randn(M, N, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    g = torch.ones(N, device="cuda", dtype=torch.bfloat16)          # frozen weight
    ag.rms_norm(x, g, eps).sum().backward()
    assert x.grad is not None and g.grad is None
    x2 = x.detach().clone().requires_grad_(True)
    ag.layer_norm(x2, g, None, eps).sum().backward()
    assert x2.grad is not None


def test_bad_inputs_are_rejected():
    x = torch.randn(4, 64, device="cuda", dtype=torch.float16)
    g = torch.ones(64, device="cuda", dtype=torch.float16)
    with pytest.raises(TypeError):
        ag.rms_norm(x, g)
    x = torch.randn(4, 64, device="cuda")
    with pytest.raises(ValueError):
        ag.rms_norm(x, torch.ones(32, device="cuda"))
    with pytest.raises(ValueError):
        ag.rms_norm(x.t(), torch.ones(4, device="cuda"))


def test_residual_on_another_device_is_rejected_before_any_launch(monkeypatch):
    import row_wise_normalization_02_gb300.autograd as agm
    calls = []
    monkeypatch.setattr(agm, "rmsnorm_fused_add_fwd", lambda *a, **k: calls.append(a))
    x = torch.randn(4, 64, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ag.fused_add_rms_norm(x, x.cpu(), g)
    assert not calls


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs two GPUs")
def test_calls_follow_the_tensors_device():
    M, N, eps = 64, 1024, 1e-6
    x1 = torch.randn(M, N, device="cuda:1", dtype=torch.bfloat16)
    g1 = torch.rand(N, device="cuda:1", dtype=torch.bfloat16) + 0.5
    with torch.cuda.device(0):
        y1 = ag.rms_norm(x1, g1, eps)
    torch.cuda.synchronize(1)
    with torch.cuda.device(1):
        y_ref = ag.rms_norm(x1, g1, eps)
    torch.cuda.synchronize(1)
    assert y1.device == x1.device
    assert torch.equal(y1.view(torch.int16), y_ref.view(torch.int16))
