"""GPU backward (dx and dgamma) against the oracle, element by element, plus
run-to-run bit reproducibility of dgamma."""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity_util as pu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

PAIRS = [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")]


def f32(v):
    return float(np.float32(v))


def make(M, N, xd, wd, seed):
    x = si.fill((M, N), seed=seed, tensor_id=1, dtype=xd)
    dy = si.fill((M, N), seed=seed, tensor_id=4, dtype=xd)
    g = si.fill(N, seed=seed, tensor_id=3, p0=1.0, p1=0.1, dtype=wd)
    return x, dy, g


def check_bwd(x, dy, g, rstd, eps, xd, wd, out, want_dgamma=True):
    ref = oracle.bwd(dy, x, rstd, g, eps, xd, wd)
    x64, dy64, g64 = oracle.to_f64(x, xd), oracle.to_f64(dy, xd), oracle.to_f64(g, wd)
    if rstd is not None:
        r = rstd.astype(np.float64)
    else:
        r = 1.0 / np.sqrt(np.mean(x64 ** 2, axis=1) + eps)
    info = {}
    if xd == "bf16":
        info["floor"], info["max_ulp"] = pu.check_dx_bf16(out["dx"], ref["dx"], ref["dx64"], x64,
                                                          dy64, g64, r, ref["c64"],
                                                          ref["dot_abs64"])
    else:
        pu.check_f32(out["dx"], ref["dx64"], what="dx")
    if want_dgamma:
        info["dgamma_rel"] = pu.check_dgamma(out["dgamma"], ref["dgamma64"], ref["dgamma_sq64"])
    return info


N_BF16 = [8, 16, 40, 128, 256, 768, 1024, 1032, 2048, 4096, 5120, 7168, 8192, 16384, 1, 7, 9,
          127, 255, 1025, 2049, 4095, 40000]
N_F32 = [4, 12, 128, 512, 1024, 4096, 8192, 1, 3, 1023, 2049, 40000]


def _cases():
    out = []
    for xd, wd in PAIRS:
        for N in (N_F32 if xd == "f32" else N_BF16):
            M = 37 if N >= 16384 else 257 if N >= 1024 else 1100
            out.append((xd, wd, M, N))
    return out


@pytest.mark.parametrize("xd,wd,M,N", _cases())
def test_bwd_matches_oracle(xd, wd, M, N):
    x, dy, g = make(M, N, xd, wd, seed=N + 11)
    eps = f32(1e-5)
    rstd = oracle.fwd(x, g if wd == xd else g, eps, xd, wd)["rstd"]
    out = pu.run_bwd(dy, x, rstd, g, eps, xd, wd)
    check_bwd(x, dy, g, rstd, eps, xd, wd, out)


@pytest.mark.parametrize("N", [128, 4096, 2049, 40000])
def test_bwd_recomputes_rstd_when_absent(N):
    x, dy, g = make(300, N, "bf16", "f32", seed=N + 12)
    eps = f32(1e-3)
    out = pu.run_bwd(dy, x, None, g, eps, "bf16", "f32")
    check_bwd(x, dy, g, None, eps, "bf16", "f32", out)


@pytest.mark.parametrize("force", ["staged:vpt=4:st=3:cps=1", "staged:vpt=2:st=2:cps=1"])
def test_staged_bwd_recomputes_rstd_and_skips_dgamma(debug_env, force):
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    x, dy, g = make(500, 4096, "bf16", "f32", seed=14)
    eps = f32(1e-4)
    out = pu.run_bwd(dy, x, None, g, eps, "bf16", "f32")
    check_bwd(x, dy, g, None, eps, "bf16", "f32", out)
    out = pu.run_bwd(dy, x, None, g, eps, "bf16", "f32", want_dgamma=False)
    check_bwd(x, dy, g, None, eps, "bf16", "f32", out, want_dgamma=False)


@pytest.mark.parametrize("N", [128, 8192, 2049])
def test_bwd_without_dgamma(N):
    x, dy, g = make(200, N, "bf16", "bf16", seed=N + 13)
    eps = f32(1e-5)
    rstd = oracle.fwd(x, g, eps, "bf16", "bf16")["rstd"]
    out = pu.run_bwd(dy, x, rstd, g, eps, "bf16", "bf16", want_dgamma=False)
    check_bwd(x, dy, g, rstd, eps, "bf16", "bf16", out, want_dgamma=False)


@pytest.mark.parametrize("force,N", [
    ("subwarp:g=8:vpt=2:pf=1:cps=1", 128), ("subwarp:g=8:vpt=2:pf=0:cps=1", 128),
    ("subwarp:g=4:vpt=1:pf=1:cps=1", 32), ("subwarp:g=32:vpt=3:pf=1:cps=1", 768),
    ("subwarp:g=32:vpt=4:pf=0:cps=1", 1024),
    ("cta:vpt=4:pf=0:acc=1:cps=1", 8192), ("cta:vpt=4:pf=1:acc=1:cps=1", 8192),
    ("cta:vpt=2:pf=1:acc=0:cps=1", 8192), ("cta:vpt=2:pf=0:acc=0:cps=1", 4096),
    ("cta:vpt=4:pf=0:acc=0:cps=1", 8192), ("cta:vpt=8:pf=0:acc=1:cps=1", 16384),
    ("cta:vpt=1:pf=1:acc=0:cps=1", 2048),
    ("ragged:vpt=2:pf=1:cps=1", 2049), ("ragged:vpt=1:pf=0:cps=1", 2049),
    ("ragged:vpt=4:pf=0:cps=1", 2049), ("ragged:vpt=2:pf=1:mr=0", 1025),
    ("ragged:vpt=1:pf=1:cps=2", 4095),
    ("generic:cps=1", 8192), ("generic:cps=1", 2049),
    ("wide:cps=1", 8192), ("wide:t=64:cps=1", 1032),
    ("staged:vpt=4:st=3:cps=1", 8192), ("staged:vpt=4:st=2:cps=1", 8192),
    ("staged:vpt=2:st=4:cps=1", 4096), ("staged:vpt=1:st=2:cps=1", 2048),
    ("staged:vpt=4:st=2:cps=1", 5120), ("staged:vpt=4:st=3:cps=1", 1032),
    # short rows through the ring, 256 / g rows per stage (a partial last stage)
    ("staged:g=32:vpt=3:cps=1", 768), ("staged:g=32:vpt=3:st=2:cps=1", 520),
    ("staged:g=8:vpt=2:cps=1", 128), ("staged:g=4:vpt=1:st=3:cps=1", 32),
    ("staged:g=16:vpt=2:st=8:cps=1", 256), ("staged:g=32:vpt=4:st=2:cps=1", 1024),
    ("staged:g=32:vpt=1:cps=1", 200),
])
def test_forced_variants_walk_several_rows(debug_env, force, N):
    debug_env.set("RMSNORM_FORCE_VARIANT", force)
    M = 3000 if N <= 1024 else 700
    x, dy, g = make(M, N, "bf16", "f32", seed=21)
    eps = f32(1e-5)
    rstd = oracle.fwd(x, g, eps, "bf16", "f32")["rstd"]
    out = pu.run_bwd(dy, x, rstd, g, eps, "bf16", "f32")
    check_bwd(x, dy, g, rstd, eps, "bf16", "f32", out)


@pytest.mark.parametrize("offsets,N", [
    ({"x": 2, "dy": 2, "dx": 2}, 4096),                 # ragged
    ({"x": 2, "dy": 2, "dx": 2, "gamma": 4}, 1000),
    ({"x": 2, "dy": 4, "dx": 2}, 4096),                 # dy off x and dx: ragged mixed form
    ({"gamma": 4, "rstd": 4, "dgamma": 4}, 8192),       # ragged (gamma unaligned)
])
def test_bwd_unaligned_pointers(offsets, N):
    x, dy, g = make(130, N, "bf16", "f32", seed=22)
    eps = f32(1e-5)
    rstd = oracle.fwd(x, g, eps, "bf16", "f32")["rstd"]
    out = pu.run_bwd(dy, x, rstd, g, eps, "bf16", "f32", offsets=offsets)
    check_bwd(x, dy, g, rstd, eps, "bf16", "f32", out)


@pytest.mark.parametrize("N", [128, 8192, 2049])
def test_dgamma_is_bitwise_reproducible(N):
    M = 3000 if N == 128 else 600
    x, dy, g = make(M, N, "bf16", "f32", seed=23)
    eps = f32(1e-5)
    rstd = oracle.fwd(x, g, eps, "bf16", "f32")["rstd"]
    outs = pu.run_bwd(dy, x, rstd, g, eps, "bf16", "f32", repeat=3)
    for o in outs[1:]:
        assert np.array_equal(o["dgamma"].view(np.uint32), outs[0]["dgamma"].view(np.uint32))
        assert np.array_equal(o["dx"], outs[0]["dx"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o = pu.run_bwd(dy, x, rstd, g, eps, "bf16", "f32", stream=s)
    assert np.array_equal(o["dgamma"].view(np.uint32), outs[0]["dgamma"].view(np.uint32))


def test_workspace_too_small_is_rejected():
    import row_wise_normalization_02_gb300 as rn
    M, N = 512, 4096
    x, dy, g = make(M, N, "bf16", "bf16", seed=24)
    need = rn.rmsnorm_bwd_workspace_size(M, N, "bf16", "bf16")
    assert need > 0 and need % 16 == 0
    bx, bdy, bg = pu.dev(x), pu.dev(dy), pu.dev(g)
    bdx, bdg = pu.empty(M * N, "bf16"), pu.empty(N, "f32")
    ws = pu.Buf(need)
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_bwd(bdy.ptr, bx.ptr, None, bg.ptr, bdx.ptr, bdg.ptr, ws.ptr, need - 16, M, N,
                       1e-5, "bf16", "bf16")
    assert e.value.status == 4
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_bwd(bdy.ptr, bx.ptr, None, bg.ptr, bdx.ptr, bdg.ptr, None, need, M, N, 1e-5,
                       "bf16", "bf16")
    assert e.value.status == 4
    torch.cuda.synchronize()
    assert bdx.guards_ok() and bdg.guards_ok() and ws.guards_ok()
    # nothing was launched: the output still holds the canary pattern
    assert (bdx.view().cpu().numpy() == pu.CANARY).all()


def test_zero_rows_zero_dgamma():
    import row_wise_normalization_02_gb300 as rn
    N = 256
    g = si.fill(N, seed=1, tensor_id=3, dtype="bf16")
    bg, bdg = pu.dev(g), pu.empty(N, "f32")
    dummy = pu.Buf(16)
    rn.rmsnorm_bwd(dummy.ptr, dummy.ptr, None, bg.ptr, dummy.ptr, bdg.ptr, None, 0, 0, N, 1e-5,
                   "bf16", "bf16")
    torch.cuda.synchronize()
    assert (bdg.download(np.float32) == 0).all()


def test_shared_memory_limit_is_never_lowered():
    # The staged kernels need more than 48 KB of dynamic shared memory.  A
    # query that caches a large launch, then a smaller launch of the same
    # kernel, then the large launch again must all work (the kernel's limit
    # may only grow).
    import row_wise_normalization_02_gb300 as rn
    big, small = 8192, 7168
    rn.rmsnorm_bwd_workspace_size(16384, big, "bf16", "f32")
    for N in (small, big, small, big):
        x, dy, g = make(64, N, "bf16", "f32", seed=25)
        eps = f32(1e-5)
        rstd = oracle.fwd(x, g, eps, "bf16", "f32")["rstd"]
        out = pu.run_bwd(dy, x, rstd, g, eps, "bf16", "f32")
        check_bwd(x, dy, g, rstd, eps, "bf16", "f32", out)
