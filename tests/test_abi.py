"""The C ABI library: it loads, it exports every entry point the header
declares, and argument errors are reported before any CUDA call (so these run
without a GPU).  The GPU-side error paths are at the end, marked gpu."""
import ctypes
import os
import re

import pytest

import row_wise_normalization_02_gb300 as rn
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "rmsnorm.h")


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b((?:rmsnorm|layernorm)_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from row_wise_normalization_02_gb300 import _build
    _build.build()
    return rn.load_library()


def test_header_and_binding_agree():
    assert header_functions() == sorted(rn.EXPORTED_SYMBOLS)


def test_library_exports_every_header_symbol(lib):
    raw = ctypes.CDLL(rn.library_path())
    for name in header_functions():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    assert rn.rmsnorm_status_string(0) == "ok"
    assert "workspace" in rn.rmsnorm_status_string(4)
    assert rn.rmsnorm_status_string(99) == "unknown status"


FAKE = 1 << 40     # an address never dereferenced: these calls fail validation first


@pytest.mark.parametrize("args,status", [
    (dict(M=-1), 1), (dict(N=0), 1), (dict(N=(1 << 30) + 1), 1), (dict(eps=-1.0), 1),
    (dict(eps=float("nan")), 1), (dict(x=None), 1), (dict(gamma=None), 1), (dict(y=None), 1),
    (dict(x_dtype=rn.F32, w_dtype=rn.BF16), 2), (dict(x_dtype=7), 2),
    (dict(x=FAKE + 1), 3), (dict(rstd=FAKE + 2), 3),
    (dict(y=FAKE), 1),   # y overlaps x
])
def test_fwd_argument_errors_without_gpu(lib, args, status):
    a = dict(x=FAKE, gamma=FAKE + (1 << 32), y=FAKE + (2 << 32), rstd=None, M=4, N=64, eps=1e-5,
             x_dtype=rn.BF16, w_dtype=rn.BF16)
    a.update(args)
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_fwd(a["x"], a["gamma"], a["y"], a["rstd"], a["M"], a["N"], a["eps"],
                       a["x_dtype"], a["w_dtype"])
    assert e.value.status == status


def test_fused_and_bwd_argument_errors_without_gpu(lib):
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_fused_add_fwd(FAKE, None, FAKE + (1 << 32), FAKE + (2 << 32), None, 4, 64,
                                 1e-5, rn.BF16, rn.BF16)
    assert e.value.status == 1
    with pytest.raises(rn.RMSNormError) as e:    # residual aliases y
        rn.rmsnorm_fused_add_fwd(FAKE, FAKE + (3 << 32), FAKE + (1 << 32), FAKE + (3 << 32), None,
                                 4, 64, 1e-5, rn.BF16, rn.BF16)
    assert e.value.status == 1
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_bwd(None, FAKE, None, FAKE, FAKE, None, None, 0, 4, 64, 1e-5, rn.BF16,
                       rn.BF16)
    assert e.value.status == 1
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_bwd(FAKE, FAKE + (1 << 32), None, FAKE + (2 << 32), FAKE + (3 << 32), None,
                       None, 0, 4, 64, 1e-5, rn.F32, rn.BF16)
    assert e.value.status == 2
    with pytest.raises(rn.RMSNormError) as e:   # dgamma misaligned
        rn.rmsnorm_bwd(FAKE, FAKE + (1 << 32), None, FAKE + (2 << 32), FAKE + (3 << 32),
                       FAKE + (4 << 32) + 2, None, 0, 4, 64, 1e-5, rn.BF16, rn.BF16)
    assert e.value.status == 3
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_bwd_workspace_size(-3, 64, rn.BF16, rn.BF16)
    assert e.value.status == 1


@pytest.mark.parametrize("args,status", [
    (dict(x_sh=64), 1),                 # heads overlap (head stride < D)
    (dict(x_st=200), 1),                # tokens overlap (token stride < H * head stride)
    (dict(y_st=-1), 1), (dict(T=-1), 1), (dict(D=0), 1),
    (dict(x=FAKE + 1), 3),
    (dict(y=FAKE, y_st=256, y_sh=128), 1),    # y overlaps x without being the same layout
    (dict(x_dtype=rn.F32, w_dtype=rn.BF16), 2),
])
def test_strided_argument_errors_without_gpu(lib, args, status):
    a = dict(x=FAKE, x_st=384, x_sh=128, gamma=FAKE + (1 << 32), y=FAKE + (2 << 32), y_st=256,
             y_sh=128, rstd=None, T=4, H=2, D=128, x_dtype=rn.BF16, w_dtype=rn.BF16)
    a.update(args)
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_fwd_strided(a["x"], a["x_st"], a["x_sh"], a["gamma"], a["y"], a["y_st"],
                               a["y_sh"], a["rstd"], a["T"], a["H"], a["D"], 1e-6, a["x_dtype"],
                               a["w_dtype"])
    assert e.value.status == status


@pytest.mark.parametrize("kind,args,status", [
    ("nvfp4", dict(N=72), 1),                    # N not a multiple of 16
    ("nvfp4", dict(gs=0.0), 1), ("nvfp4", dict(gs=-2.0), 1), ("nvfp4", dict(gs=float("inf")), 1),
    ("nvfp4", dict(gs=float("nan")), 1),
    ("fp8", dict(q=None), 1), ("fp8", dict(qs=None), 1), ("nvfp4", dict(x=None), 1),
    ("fp8", dict(qs=FAKE + (4 << 32) + 2), 3),   # fp32 scales not 4-byte aligned
    ("fp8", dict(x=FAKE + 1), 3),
    ("fp8", dict(q=FAKE + 64), 1),               # codes overlap x
    ("nvfp4", dict(qs=FAKE + (3 << 32) + 8), 1),  # scales overlap the codes
    ("fp8", dict(residual=FAKE + 128), 1),       # residual overlaps x
    ("fp8", dict(x_dtype=rn.F32, w_dtype=rn.BF16), 2),
    ("nvfp4", dict(M=-1), 1), ("fp8", dict(eps=-1.0), 1),
])
def test_quantised_argument_errors_without_gpu(lib, kind, args, status):
    a = dict(x=FAKE, residual=None, gamma=FAKE + (1 << 32), q=FAKE + (3 << 32),
             qs=FAKE + (4 << 32), gs=6.0, rstd=None, M=4, N=64, eps=1e-6, x_dtype=rn.BF16,
             w_dtype=rn.BF16)
    a.update(args)
    with pytest.raises(rn.RMSNormError) as e:
        if kind == "fp8":
            rn.rmsnorm_fwd_fp8(a["x"], a["residual"], a["gamma"], a["q"], a["qs"], a["rstd"],
                               a["M"], a["N"], a["eps"], a["x_dtype"], a["w_dtype"])
        else:
            rn.rmsnorm_fwd_nvfp4(a["x"], a["residual"], a["gamma"], a["gs"], a["q"], a["qs"],
                                 a["rstd"], a["M"], a["N"], a["eps"], a["x_dtype"],
                                 a["w_dtype"])
    assert e.value.status == status


@pytest.mark.parametrize("args,status", [
    (dict(mean=FAKE + (5 << 32)), 1),            # mean without rstd
    (dict(x=None), 1), (dict(N=0), 1), (dict(eps=-1.0), 1),
    (dict(x_dtype=rn.F32, w_dtype=rn.BF16), 2),
    (dict(x=FAKE + 1), 3), (dict(dgamma=FAKE + (6 << 32) + 2), 3),
    (dict(dx=FAKE + 64), 1),                     # dx overlaps x
    (dict(dgamma=FAKE + (6 << 32), dbeta=FAKE + (6 << 32) + 16), 1),   # dgamma overlaps dbeta
    (dict(workspace=None), 4), (dict(workspace=FAKE + (8 << 32) + 4), 4),
])
def test_layernorm_bwd_argument_errors_without_gpu(lib, args, status):
    a = dict(dy=FAKE + (1 << 32), x=FAKE, mean=None, rstd=None, gamma=FAKE + (2 << 32),
             dx=FAKE + (3 << 32), dgamma=FAKE + (6 << 32), dbeta=FAKE + (7 << 32),
             workspace=FAKE + (8 << 32), ws_bytes=1 << 30, M=4, N=64, eps=1e-5,
             x_dtype=rn.BF16, w_dtype=rn.BF16)
    a.update(args)
    with pytest.raises(rn.RMSNormError) as e:
        rn.layernorm_bwd(a["dy"], a["x"], a["mean"], a["rstd"], a["gamma"], a["dx"], a["dgamma"],
                         a["dbeta"], a["workspace"], a["ws_bytes"], a["M"], a["N"], a["eps"],
                         a["x_dtype"], a["w_dtype"])
    assert e.value.status == status


@pytest.mark.parametrize("args,status", [
    (dict(y=None), 1), (dict(y=FAKE + 32), 1), (dict(beta=FAKE + (2 << 32) + 1), 3),
    (dict(mean=FAKE + (3 << 32), rstd=FAKE + (3 << 32)), 1),   # mean and rstd alias
    (dict(N=-4), 1),
])
def test_layernorm_fwd_argument_errors_without_gpu(lib, args, status):
    a = dict(x=FAKE, gamma=FAKE + (1 << 32), beta=None, y=FAKE + (4 << 32), mean=None, rstd=None,
             M=4, N=64)
    a.update(args)
    with pytest.raises(rn.RMSNormError) as e:
        rn.layernorm_fwd(a["x"], a["gamma"], a["beta"], a["y"], a["mean"], a["rstd"], a["M"],
                         a["N"], 1e-5, rn.BF16, rn.BF16)
    assert e.value.status == status


def test_zero_rows_is_a_no_op(lib):
    # M == 0: nothing to do, no pointer is touched and no CUDA call is made
    rn.rmsnorm_fwd(None, None, None, None, 0, 64, 1e-5, rn.BF16, rn.BF16)
    rn.rmsnorm_fused_add_fwd(None, None, None, None, None, 0, 64, 1e-5, rn.BF16, rn.BF16)
    rn.rmsnorm_bwd(None, None, None, None, None, None, None, 0, 0, 64, 1e-5, rn.BF16, rn.BF16)
    assert rn.rmsnorm_bwd_workspace_size(0, 64, rn.BF16, rn.BF16) == 0
    rn.rmsnorm_fwd_strided(None, 0, 0, None, None, 0, 0, None, 0, 8, 128, 1e-6, rn.BF16,
                           rn.BF16)
    rn.rmsnorm_fwd_fp8(None, None, None, None, None, None, 0, 64, 1e-6, rn.BF16, rn.BF16)
    rn.rmsnorm_fwd_nvfp4(None, None, None, 1.0, None, None, None, 0, 64, 1e-6, rn.BF16, rn.BF16)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import row_wise_normalization_02_gb300 as mod
    monkeypatch.setattr(mod, "_LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(ImportError):
        mod.rmsnorm_fwd(1, 1, 1, None, 1, 8, 1e-5, "bf16", "bf16")


@pytest.mark.gpu
def test_workspace_size_matches_plan_on_gpu(lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    for M, N in [(16384, 8192), (262144, 128), (4096, 2049), (1, 1), (3, 40000)]:
        b = rn.rmsnorm_bwd_workspace_size(M, N, "bf16", "f32")
        assert b > 0 and b % 16 == 0
        # at most one partial row per resident CTA, at least one per residue
        # class of ragged rows (16 classes at most)
        assert b <= max(min(M, 152 * 32), 16) * ((N + 3) // 4 * 4) * 4 * 2


def test_autograd_functions_reject_host_tensors_before_any_call():
    torch = pytest.importorskip("torch")
    from row_wise_normalization_02_gb300 import autograd as ag
    x, g = torch.randn(4, 8), torch.ones(8)
    for call in (lambda: ag.rms_norm(x, g), lambda: ag.layer_norm(x, g),
                 lambda: ag.fused_add_rms_norm(x, torch.randn(4, 8), g)):
        with pytest.raises(ValueError):
            call()
