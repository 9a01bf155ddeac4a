"""The synthetic workloads: shapes, dtypes, value recipes, eps and seeds.

Sizes and value distributions follow the RMSNorm workloads this library is
measured on (forward, fused residual-add forward, backward, and a shape sweep
that includes a per-head q/k-norm row length and a ragged row length).
"""
from __future__ import annotations

from dataclasses import dataclass, field

# stream ids of the tensors (each tensor draws from its own sub-stream)
TENSOR_IDS = {"x": 1, "residual": 2, "gamma": 3, "dy": 4}


@dataclass(frozen=True)
class Workload:
    name: str
    op: str                 # "fwd", "fused_add", "bwd", "fused_add_bwd", "fwd_strided"
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


def tensor_recipes(wl: Workload) -> dict:
    """name -> keyword arguments of ``seeded_inputs.fill`` for that tensor."""
    act = dict(dist="normal", p0=0.0, p1=1.0, dtype=wl.x_dtype,
               outlier_fraction=wl.outlier_fraction, outlier_scale=wl.outlier_scale)
    g = dict(dist=wl.gamma_dist[0], p0=wl.gamma_dist[1], p1=wl.gamma_dist[2], dtype=wl.w_dtype)
    rec = {"x": act, "gamma": g}
    if wl.op == "fwd_strided":
        rec["x"] = dict(act, shape=(wl.M // wl.heads, wl.stride_token))
    if wl.op == "fused_add":
        rec["residual"] = dict(act)
    if wl.op in ("bwd", "fused_add_bwd"):
        rec["dy"] = dict(dist="normal", p0=0.0, p1=1.0, dtype=wl.x_dtype)
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
    # backward: bf16 activations, fp32 gamma; rstd from the oracle forward
    "bwd_bf16_m16384_n8192": Workload("bwd_bf16_m16384_n8192", "bwd", 16384, 8192, "bf16",
                                      "f32", 1e-5, 3, tags=("headline",)),
}
for _m, _n in _SWEEP:
    for _op in ("fwd", "bwd"):
        _name = f"sweep_{_op}_bf16_m{_m}_n{_n}"
        WORKLOADS[_name] = Workload(_name, _op, _m, _n, "bf16", "bf16", 1e-6, 4,
                                    tags=("sweep",))
