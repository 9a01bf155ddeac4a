"""Seeded random shapes, dtypes and operand offsets through the default
dispatch, against the oracle.  Every case draws the operation (forward, fused
add, backward with saved or recomputed rstd, fused-add backward), the dtype
pair, M, N (log-uniform or a multiple of 64, so short, CTA-sized, ragged and
cluster rows all occur) and a layout class with byte offsets of the operands
on the element grid (all aligned, all on one residue modulo 16, inputs off
the outputs' alignment, every operand anywhere), so the families and their
boundaries are crossed in combinations no hand-written list enumerates.
LayerNorm (forward, backward with saved or recomputed statistics) and the
quantised outputs (FP8, NVFP4; plain or fused add) get their own draws.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity_util as pu
from tests.test_parity_bwd import check_bwd
from tests.test_parity_fused_bwd import check as check_fused_bwd
from tests.test_parity_fused_bwd import run as run_fused_bwd
from tests.test_parity_fwd import check_fused, check_fwd

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

PAIRS = [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")]
OPS = ["fwd", "fused", "bwd", "bwd_norstd", "fused_bwd"]
CASES = 120


def draw(i):
    rng = np.random.default_rng(1000 + i)
    op = OPS[rng.integers(len(OPS))]
    xd, wd = PAIRS[rng.integers(len(PAIRS))]
    if rng.random() < 0.5:   # anywhere, log-uniform
        N = max(1, int(np.exp(rng.uniform(0.0, np.log(70000.0)))))
    else:                    # hidden sizes of models: multiples of 64
        N = 64 * int(rng.integers(16, 257))
    # keep each case to a few million elements
    M = int(rng.integers(1, max(2, min(700, 4_000_000 // N + 1))))
    es = 4 if xd == "f32" else 2
    ws = 4 if wd == "f32" else 2

    def off():   # a byte offset on the element grid within 16 bytes
        return int(rng.integers(0, 16 // es)) * es
    outs = {"fwd": ["y"], "fused": ["residual", "y"], "bwd": ["dx"], "bwd_norstd": ["dx"],
            "fused_bwd": ["dres"]}[op]
    ins = {"fwd": ["x"], "fused": ["x"], "bwd": ["x", "dy"], "bwd_norstd": ["x", "dy"],
           "fused_bwd": ["h", "dy"]}[op]
    # the layout class: all aligned, all on one residue, inputs off the
    # outputs (which agree), or every operand anywhere
    cls = int(rng.integers(4))
    base = off()
    offsets = {}
    for k in outs + ins:
        if cls == 0:
            offsets[k] = 0
        elif cls == 1:
            offsets[k] = base
        elif cls == 2:
            offsets[k] = base if k in outs else off()
        else:
            offsets[k] = off()
    offsets["gamma"] = 0 if cls == 0 else int(rng.integers(0, 16 // ws)) * ws
    return op, xd, wd, M, N, offsets


@pytest.mark.parametrize("i", range(CASES))
def test_random_case_matches_oracle(i):
    op, xd, wd, M, N, offsets = draw(i)
    eps = float(np.float32(1e-5))
    seed = 5000 + i
    x = si.fill((M, N), seed=seed, tensor_id=1, dtype=xd)
    g = si.fill(N, seed=seed, tensor_id=3, p0=1.0, p1=0.2, dtype=wd)
    if op == "fwd":
        out = pu.run_fwd(x, g, eps, xd, wd, offsets=offsets)
        check_fwd(x, g, eps, xd, wd, out)
    elif op == "fused":
        r = si.fill((M, N), seed=seed, tensor_id=2, dtype=xd, p1=2.0)
        out = pu.run_fused(x, r, g, eps, xd, wd, want_rstd=True, offsets=offsets)
        check_fused(x, r, g, eps, xd, wd, out, want_rstd=True)
    elif op in ("bwd", "bwd_norstd"):
        dy = si.fill((M, N), seed=seed, tensor_id=4, dtype=xd)
        rstd = oracle.fwd(x, g, eps, xd, wd)["rstd"] if op == "bwd" else None
        out = pu.run_bwd(dy, x, rstd, g, eps, xd, wd, offsets=offsets)
        check_bwd(x, dy, g, rstd, eps, xd, wd, out)
    else:
        dy = si.fill((M, N), seed=seed, tensor_id=4, dtype=xd)
        dres = si.fill((M, N), seed=seed, tensor_id=2, dtype=xd)
        rstd = oracle.fwd(x, g, eps, xd, wd)["rstd"]
        out = run_fused_bwd(x, dy, dres, g, rstd, eps, xd, wd, offsets=offsets)
        check_fused_bwd(x, dy, dres, g, rstd, eps, xd, wd, out)


def test_draws_cover_the_families():
    """The seeded draws reach every layout class the dispatch tells apart."""
    seen = set()
    for i in range(CASES):
        op, xd, wd, M, N, o = draw(i)
        es = 4 if xd == "f32" else 2
        acts = [v for k, v in o.items() if k != "gamma"]
        rows16 = (N * es) % 16 == 0
        if all(v == 0 for v in acts):
            seen.add("aligned" if rows16 else "ragged")
        elif len(set(acts)) == 1:
            seen.add("same residue")
        else:
            seen.add("mixed")
        seen.add("short" if N * es <= 2048 else ("long" if N * es > 65536 else "cta"))
    assert {"aligned", "ragged", "same residue", "mixed", "short", "cta", "long"} <= seen, seen


# ---------------------------------------------------------------- LayerNorm
# and quantised outputs: the same seeded draws for their own entry points

from tests import test_parity_layernorm as tl  # noqa: E402
from tests import test_parity_quant as tq  # noqa: E402

LN_CASES = 40
Q_CASES = 40


def draw_ln(i):
    rng = np.random.default_rng(3000 + i)
    xd, wd = PAIRS[rng.integers(len(PAIRS))]
    bwd = bool(rng.integers(2))
    saved = bool(rng.integers(2))
    N = (max(1, int(np.exp(rng.uniform(0.0, np.log(40000.0))))) if rng.random() < 0.5
         else 64 * int(rng.integers(2, 257)))
    M = int(rng.integers(1, max(2, min(600, 3_000_000 // N + 1))))
    es = 4 if xd == "f32" else 2
    aligned = rng.random() < 0.6
    offsets = {} if aligned else {k: int(rng.integers(0, 16 // es)) * es
                                  for k in (["x", "dy", "dx"] if bwd else ["x", "y"])}
    return xd, wd, bwd, saved, M, N, offsets


@pytest.mark.parametrize("i", range(LN_CASES))
def test_random_layernorm_case_matches_oracle(i):
    xd, wd, bwd, saved, M, N, offsets = draw_ln(i)
    eps = float(np.float32(1e-5))
    x, g, b, dy = tl.inputs(M, N, xd, wd, seed=7000 + i, beta=not bwd)
    if not bwd:
        out = tl.run_fwd(x, g, b, eps, xd, wd, offsets=offsets)
        tl.check_fwd(out, x, g, b, eps, xd, wd)
        return
    mean = rstd = None
    if saved:
        fw = oracle.layernorm_fwd(x, g, None, eps, xd, wd)
        mean, rstd = fw["mean"], fw["rstd"]
    out = tl.run_bwd(dy, x, mean, rstd, g, eps, xd, wd, offsets=offsets)
    tl.check_bwd(out, dy, x, mean, rstd, g, eps, xd, wd)


def draw_q(i):
    rng = np.random.default_rng(4000 + i)
    xd, wd = PAIRS[rng.integers(len(PAIRS))]
    kind = "fp8" if rng.integers(2) else "nvfp4"
    fused = bool(rng.integers(2))
    N = 16 * int(np.exp(rng.uniform(0.0, np.log(2500.0))))   # NVFP4 blocks of 16
    if kind == "fp8" and rng.random() < 0.3:
        N += int(rng.integers(1, 16))
    M = int(rng.integers(1, max(2, min(500, 2_000_000 // N + 1))))
    es = 4 if xd == "f32" else 2
    offsets = {} if rng.random() < 0.6 else {"x": int(rng.integers(0, 16 // es)) * es}
    return xd, wd, kind, fused, M, N, offsets


@pytest.mark.parametrize("i", range(Q_CASES))
def test_random_quantised_case_matches_oracle(i):
    xd, wd, kind, fused, M, N, offsets = draw_q(i)
    eps = float(np.float32(1e-6))
    x, g, r = tq.inputs(M, N, xd, wd, seed=8000 + i, fused=fused)
    if kind == "fp8":
        out = tq.run("fp8", x, g, eps, xd, wd, residual=r, offsets=offsets)
        tq.check_fp8(out, x, g, eps, xd, wd, residual=r)
    else:
        out = tq.run("nvfp4", x, g, eps, xd, wd, residual=r, gs=tq.GS, offsets=offsets)
        tq.check_nvfp4(out, x, g, eps, xd, wd, tq.GS, residual=r)
