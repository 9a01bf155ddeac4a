"""Calls captured in a CUDA graph: every entry point only enqueues work on the
given stream (no allocation, no synchronisation), so a training step's norm
calls can be captured once and replayed.  A replay must give the same bits as
the same calls launched directly, for every kernel family the shapes reach
(short rows, one row per CTA, the bulk-copy ring, ragged rows, inputs off the
outputs' alignment, clusters), and replaying twice must not change them.
"""
import numpy as np
import pytest

import seeded_inputs as si

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import row_wise_normalization_02_gb300 as rn  # noqa: E402


def dev(a, off=0):
    """A device copy of a host array, `off` bytes past a 16-byte boundary."""
    a = a.view(np.int16) if a.dtype == np.uint16 else a
    t = torch.from_numpy(a)
    if not off:
        return t.cuda()
    e = t.element_size()
    buf = torch.empty(t.numel() + 16 // e, dtype=t.dtype, device="cuda")
    v = buf[off // e: off // e + t.numel()].view(t.shape)
    v.copy_(t.cuda())
    return v


def outputs(M, N, xd, wd, ws_bytes, dres0):
    act = torch.int16 if xd == "bf16" else torch.float32
    wdt = torch.int16 if wd == "bf16" else torch.float32
    return {"y": torch.empty((M, N), dtype=act, device="cuda"),
            "rstd": torch.empty(M, dtype=torch.float32, device="cuda"),
            "h": torch.empty((M, N), dtype=act, device="cuda"),
            "y2": torch.empty((M, N), dtype=act, device="cuda"),
            "dx": torch.empty((M, N), dtype=act, device="cuda"),
            "dg": torch.empty(N, dtype=torch.float32, device="cuda"),
            "dh": torch.empty_like(dres0),
            "dg2": torch.empty(N, dtype=wdt, device="cuda"),
            "ws": torch.empty(max(16, ws_bytes), dtype=torch.uint8, device="cuda")}


@pytest.mark.parametrize("M,N,x_off", [(2000, 128, 0), (300, 768, 0), (129, 8192, 0),
                                       (300, 2049, 0), (129, 8192, 2), (300, 1000, 6),
                                       (37, 40000, 0)])
def test_graph_replay_matches_direct_calls(M, N, x_off):
    xd, wd = "bf16", "bf16"
    eps = float(np.float32(1e-5))
    X = dev(si.fill((M, N), seed=N + 90, tensor_id=1, dtype=xd), x_off)
    R = dev(si.fill((M, N), seed=N + 90, tensor_id=2, dtype=xd))
    DY = dev(si.fill((M, N), seed=N + 90, tensor_id=4, dtype=xd))
    G = dev(si.fill(N, seed=N + 90, tensor_id=3, p0=1.0, p1=0.1, dtype=wd))
    ws = rn.rmsnorm_bwd_workspace_size(M, N, xd, wd)
    s = torch.cuda.Stream()

    def step(o):
        # forward with rstd; fused add over a fresh copy of the residual;
        # backward with dgamma; fused-add backward over a fresh copy of dres
        rn.rmsnorm_fwd(X, G, o["y"], o["rstd"], M, N, eps, xd, wd, s)
        o["h"].copy_(R)
        rn.rmsnorm_fused_add_fwd(X, o["h"], G, o["y2"], None, M, N, eps, xd, wd, s)
        rn.rmsnorm_bwd(DY, X, o["rstd"], G, o["dx"], o["dg"], o["ws"], ws, M, N, eps, xd, wd, s)
        o["dh"].copy_(R)
        rn.rmsnorm_fused_add_bwd(DY, o["h"], o["rstd"], G, o["dh"], o["dg2"], wd, o["ws"], ws,
                                 M, N, eps, xd, wd, s)

    direct = outputs(M, N, xd, wd, ws, R)
    with torch.cuda.stream(s):
        step(direct)
    s.synchronize()

    cap = outputs(M, N, xd, wd, ws, R)
    with torch.cuda.stream(s):
        step(cap)   # plans and kernel attributes settled before capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(cap)
    for k in ("y", "rstd", "y2", "dx", "dg", "dg2"):
        cap[k].zero_()
    torch.cuda.synchronize()
    for _ in range(2):
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        for k in ("y", "rstd", "h", "y2", "dx", "dg", "dh", "dg2"):
            a, b = direct[k].cpu().numpy(), cap[k].cpu().numpy()
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f"{k} differs after replay"
    rn.rmsnorm_check_device(s)   # no bounded wait gave up
