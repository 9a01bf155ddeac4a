"""The synthetic workloads: shapes, dtypes, value recipes, eps and seeds.

Sizes and value distributions follow the RMSNorm workloads this library is
measured on (forward, fused residual-add forward, backward, and a shape sweep
that includes a per-head q/k-norm row length and a ragged row length).
"""
from __future__ import annotations

from dataclasses import dataclass, field

# stream ids of the tensors (each tensor draws from its own sub-stream)
TENSOR_IDS = {"x": 1, "residual": 2, "gamma": 3, "dy": 4, "beta": 5}


@dataclass(frozen=True)
class Workload:
    name: str
    op: str                 # "fwd", "fused_add", "bwd", "fused_add_bwd", "fwd_strided",
                            # "fwd_fp8", "fused_add_fp8", "fwd_nvfp4", "fused_add_nvfp4",
                            # "ln_fwd", "ln_bwd"
    M: int
    N: int
    x_dtype: str            # "f32" | "bf16"
    w_dtype: str            # gamma dtype
    eps: float
    seed: int
    store_rstd: bool = True
    gamma_dist: tuple = ("normal", 1.0, 0.1)
    outlier_fraction: float = 0.0
    outlier_scale: float = 1.0
    tags: tuple = field(default_factory=tuple)
    heads: int = 0          # strided rows: M = tokens * heads, x is [tokens, stride_token]
    stride_token: int = 0
    global_scale: float = 0.0   # NVFP4 outputs: the per-tensor scale gs
    offsets: tuple = ()     # ((operand, bytes past a 256-byte boundary), ...): operands
                            # placed off 16 bytes (x a view at an odd element offset)


def tensor_recipes(wl: Workload) -> dict:
    """name -> keyword arguments of ``seeded_inputs.fill`` for that tensor."""
    act = dict(dist="normal", p0=0.0, p1=1.0, dtype=wl.x_dtype,
               outlier_fraction=wl.outlier_fraction, outlier_scale=wl.outlier_scale)
    g = dict(dist=wl.gamma_dist[0], p0=wl.gamma_dist[1], p1=wl.gamma_dist[2], dtype=wl.w_dtype)
    rec = {"x": act, "gamma": g}
    if wl.op == "fwd_strided":
        rec["x"] = dict(act, shape=(wl.M // wl.heads, wl.stride_token))
    if wl.op.startswith("fused_add") and wl.op != "fused_add_bwd":
        rec["residual"] = dict(act)
    if wl.op in ("bwd", "fused_add_bwd", "ln_bwd"):
        rec["dy"] = dict(dist="normal", p0=0.0, p1=1.0, dtype=wl.x_dtype)
    if wl.op == "ln_fwd":
        rec["beta"] = dict(dist="normal", p0=0.0, p1=0.1, dtype=wl.w_dtype)
    if wl.op == "fused_add_bwd":
        rec["residual"] = dict(dist="normal", p0=0.0, p1=1.0, dtype=wl.x_dtype)  # dres
    return rec


_SWEEP = [(262144, 128), (65536, 768), (16384, 5120), (8192, 7168), (4096, 16384),
          (4096, 2049)]

WORKLOADS = {
    # small fp32 forward: the oracle finishes it in well under a second
    "fwd_f32_m64_n1024": Workload("fwd_f32_m64_n1024", "fwd", 64, 1024, "f32", "f32", 1e-6, 0,
                                  gamma_dist=("uniform", 0.5, 1.5), tags=("small",)),
    # bf16 forward with per-row rstd
    "fwd_bf16_m16384_n8192": Workload("fwd_bf16_m16384_n8192", "fwd", 16384, 8192, "bf16",
                                      "bf16", 1e-5, 1, tags=("headline",)),
    # fused residual add: h = r + x written back over r, y = RMSNorm(h) * gamma;
    # 0.1 % of the entries of r and of x scaled by 100
    "fadd_bf16_m32768_n4096": Workload("fadd_bf16_m32768_n4096", "fused_add", 32768, 4096,
                                       "bf16", "bf16", 1e-6, 2, store_rstd=False,
                                       outlier_fraction=1e-3, outlier_scale=100.0,
                                       tags=("headline",)),
    # backward of the fused residual add at the fused-add shape: h (the stored
    # sum), dy and the residual-path gradient dres; dgamma in the weight dtype
    "fadd_bwd_bf16_m32768_n4096": Workload("fadd_bwd_bf16_m32768_n4096", "fused_add_bwd", 32768,
                                           4096, "bf16", "bf16", 1e-6, 2, tags=("next",)),
    # per-head q norm in place on a fused QKV projection output: 32768 tokens,
    # 32 q heads and 8 kv heads of 128 (row width 6144)
    "qnorm_bf16_t32768_h32_d128": Workload("qnorm_bf16_t32768_h32_d128", "fwd_strided",
                                           32768 * 32, 128, "bf16", "bf16", 1e-6, 5,
                                           store_rstd=False, heads=32, stride_token=6144,
                                           tags=("next",)),
    # quantised outputs at the forward and fused-add shapes (same inputs):
    # FP8 E4M3 with a scale per row; NVFP4 with E4M3 scales per 16 elements
    # and a global scale sized for |y| up to 8 (forward) or 128 (fused add,
    # whose outliers reach |y| ~ 70): gs = 448 * 6 / that bound
    "fwd_fp8_bf16_m16384_n8192": Workload("fwd_fp8_bf16_m16384_n8192", "fwd_fp8", 16384, 8192,
                                          "bf16", "bf16", 1e-5, 1, store_rstd=False,
                                          tags=("next",)),
    "fwd_nvfp4_bf16_m16384_n8192": Workload("fwd_nvfp4_bf16_m16384_n8192", "fwd_nvfp4", 16384,
                                            8192, "bf16", "bf16", 1e-5, 1, store_rstd=False,
                                            global_scale=448.0 * 6 / 8, tags=("next",)),
    "fadd_fp8_bf16_m32768_n4096": Workload("fadd_fp8_bf16_m32768_n4096", "fused_add_fp8", 32768,
                                           4096, "bf16", "bf16", 1e-6, 2, store_rstd=False,
                                           outlier_fraction=1e-3, outlier_scale=100.0,
                                           tags=("next",)),
    "fadd_nvfp4_bf16_m32768_n4096": Workload("fadd_nvfp4_bf16_m32768_n4096", "fused_add_nvfp4",
                                             32768, 4096, "bf16", "bf16", 1e-6, 2,
                                             store_rstd=False, outlier_fraction=1e-3,
                                             outlier_scale=100.0, global_scale=448.0 * 6 / 128,
                                             tags=("next",)),
    # LayerNorm at the forward / backward shape: bf16 activations and
    # weights, beta ~ N(0, 0.1); the backward reads the oracle forward's saved
    # mean and rstd, and writes dx, dgamma and dbeta
    "ln_fwd_bf16_m16384_n8192": Workload("ln_fwd_bf16_m16384_n8192", "ln_fwd", 16384, 8192,
                                         "bf16", "bf16", 1e-5, 6, tags=("next",)),
    "ln_bwd_bf16_m16384_n8192": Workload("ln_bwd_bf16_m16384_n8192", "ln_bwd", 16384, 8192,
                                         "bf16", "bf16", 1e-5, 6, tags=("next",)),
    # the same at a short hidden size (1024: the forward's rows handled by lane groups)
    "ln_fwd_bf16_m65536_n1024": Workload("ln_fwd_bf16_m65536_n1024", "ln_fwd", 65536, 1024,
                                         "bf16", "bf16", 1e-5, 6, tags=("next",)),
    "ln_bwd_bf16_m65536_n1024": Workload("ln_bwd_bf16_m65536_n1024", "ln_bwd", 65536, 1024,
                                         "bf16", "bf16", 1e-5, 6, tags=("next",)),
    # backward: bf16 activations, fp32 gamma; rstd from the oracle forward
    "bwd_bf16_m16384_n8192": Workload("bwd_bf16_m16384_n8192", "bwd", 16384, 8192, "bf16",
                                      "f32", 1e-5, 3, tags=("headline",)),
}
# fp32 activations and weights at the forward / backward size class
# (256 MiB per activation tensor; gamma ~ N(1, 0.1), dy ~ N(0, 1))
for _op in ("fwd", "bwd"):
    _name = f"sweep_{_op}_f32_m8192_n8192"
    WORKLOADS[_name] = Workload(_name, _op, 8192, 8192, "f32", "f32", 1e-6, 7, tags=("sweep",))
for _m, _n in _SWEEP:
    for _op in ("fwd", "bwd"):
        _name = f"sweep_{_op}_bf16_m{_m}_n{_n}"
        WORKLOADS[_name] = Workload(_name, _op, _m, _n, "bf16", "bf16", 1e-6, 4,
                                    tags=("sweep",))
# rows longer than one CTA holds (65536 bf16: 128 KiB per row), forward and
# backward, and the fused-add backward at 32768 (64 KiB rows of three operands)
for _op in ("fwd", "bwd"):
    _name = f"long_{_op}_bf16_m2048_n65536"
    WORKLOADS[_name] = Workload(_name, _op, 2048, 65536, "bf16", "bf16", 1e-6, 8,
                                tags=("sweep",))
WORKLOADS["fadd_bwd_bf16_m8192_n32768"] = Workload("fadd_bwd_bf16_m8192_n32768", "fused_add_bwd",
                                                   8192, 32768, "bf16", "bf16", 1e-6, 9,
                                                   tags=("next",))
# inputs off the outputs' 16-byte alignment: x (forward) or x (backward) one
# bf16 element past a 16-byte boundary -- a view at an odd element offset --
# while y, dy and dx are aligned
for _op in ("fwd", "bwd"):
    for _m, _n in ((16384, 8192), (32768, 4096)):
        _name = f"mixed_{_op}_bf16_m{_m}_n{_n}"
        WORKLOADS[_name] = Workload(_name, _op, _m, _n, "bf16", "bf16", 1e-6, 10,
                                    offsets=(("x", 2),), tags=("mixed",))
# the fused add with x off the residual's (and y's) alignment
WORKLOADS["mixed_fadd_bf16_m32768_n4096"] = Workload(
    "mixed_fadd_bf16_m32768_n4096", "fused_add", 32768, 4096, "bf16", "bf16", 1e-6, 10,
    store_rstd=False, offsets=(("x", 2),), tags=("mixed",))
# what neither the register nor the ring kernels take, served by the wide
# two-pass kernel: outputs that disagree modulo 16 (y one element past 16
# bytes, the residual aligned), and rows beyond the mixed-alignment tiers (x
# one element off, 20000 bf16 columns; forward and backward)
WORKLOADS["wide_fadd_bf16_m32768_n4096"] = Workload(
    "wide_fadd_bf16_m32768_n4096", "fused_add", 32768, 4096, "bf16", "bf16", 1e-6, 11,
    store_rstd=False, offsets=(("y", 2),), tags=("wide",))
WORKLOADS["wide_fwd_bf16_m8192_n20000"] = Workload(
    "wide_fwd_bf16_m8192_n20000", "fwd", 8192, 20000, "bf16", "bf16", 1e-6, 11,
    offsets=(("x", 2),), tags=("wide",))
# LayerNorm rows beyond its register tiers (forward 2048 vectors, backward
# 1024): the wide kernels, aligned operands
WORKLOADS["ln_wide_fwd_bf16_m4096_n32768"] = Workload(
    "ln_wide_fwd_bf16_m4096_n32768", "ln_fwd", 4096, 32768, "bf16", "bf16", 1e-5, 12,
    tags=("wide",))
WORKLOADS["ln_wide_bwd_bf16_m8192_n12288"] = Workload(
    "ln_wide_bwd_bf16_m8192_n12288", "ln_bwd", 8192, 12288, "bf16", "bf16", 1e-5, 12,
    tags=("wide",))
WORKLOADS["wide_bwd_bf16_m8192_n20000"] = Workload(
    "wide_bwd_bf16_m8192_n20000", "bwd", 8192, 20000, "bf16", "bf16", 1e-6, 11,
    offsets=(("x", 2),), tags=("wide",))
