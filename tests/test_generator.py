"""The seeded input generator: its published stream definition and properties."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from seeded_inputs.workloads import WORKLOADS


def test_splitmix64_reference_values():
    # SplitMix64 seeded with 0 (Steele, Lea & Flood; Vigna's reference code):
    # the first three outputs.
    s = 0
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    got = []
    for _ in range(3):
        got.append(si.splitmix64_next(s))
        s = (s + 0x9E3779B97F4A7C15) & (2 ** 64 - 1)
    assert got == want


def test_uniform_and_normal_moments():
    u = np.array([si.uniform_at(11, 1, i) for i in range(20000)])
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.01
    z = si.fill(200000, seed=11, tensor_id=1, dtype="f32").astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.var() - 1.0) < 0.01
    assert abs(np.mean(z ** 4) - 3.0) < 0.05          # normal kurtosis


def test_fill_is_counter_based_and_thread_independent():
    a = si.fill((64, 100), seed=5, tensor_id=1, dtype="bf16", threads=1)
    b = si.fill((64, 100), seed=5, tensor_id=1, dtype="bf16", threads=7)
    c = si.fill((10, 100), seed=5, tensor_id=1, dtype="bf16")
    assert np.array_equal(a, b)
    assert np.array_equal(a[:10], c)
    d = si.fill((64, 100), seed=5, tensor_id=2, dtype="bf16")
    assert not np.array_equal(a, d)


def test_bf16_fill_is_rne_of_the_double_draw():
    # the generator's bf16 rounding agrees with the oracle's independent one
    a = si.fill(3000, seed=3, tensor_id=4, dist="normal", p0=1.0, p1=0.1, dtype="bf16")
    want = [oracle.round_bf16(1.0 + 0.1 * si.normal_at(3, 4, i)) for i in range(3000)]
    assert np.array_equal(a, np.array(want, np.uint16))
    f = si.fill(3000, seed=3, tensor_id=4, dist="normal", p0=1.0, p1=0.1, dtype="f32")
    assert np.array_equal(f, np.array([1.0 + 0.1 * si.normal_at(3, 4, i) for i in range(3000)],
                                      np.float32))


def test_outliers_exact_count_distinct_and_scaled():
    n, k = 100000, 100
    pos = si.outlier_positions(n, k, seed=2, tensor_id=1)
    assert len(pos) == k and len(np.unique(pos)) == k and pos.min() >= 0 and pos.max() < n
    base = si.fill(n, seed=2, tensor_id=1, dtype="f32")
    out = si.fill(n, seed=2, tensor_id=1, dtype="f32", outlier_fraction=1e-3,
                  outlier_scale=100.0)
    diff = np.nonzero(out != base)[0]
    assert set(diff.tolist()) <= set(pos.tolist())
    assert np.allclose(out[pos], np.float32(100.0) * base[pos].astype(np.float64), rtol=1e-6)
    # positions spread over the whole range
    assert np.histogram(pos, bins=4, range=(0, n))[0].min() > 10


def test_workload_recipes():
    wl = WORKLOADS["fadd_bf16_m32768_n4096"]
    assert (wl.M, wl.N, wl.eps, wl.seed, wl.x_dtype) == (32768, 4096, 1e-6, 2, "bf16")
    small = si.make_inputs(WORKLOADS["fwd_f32_m64_n1024"])
    assert small["x"].dtype == np.float32 and small["x"].shape == (64, 1024)
    g = small["gamma"]
    assert g.min() >= 0.5 and g.max() < 1.5
    bwd = si.make_inputs(WORKLOADS["bwd_bf16_m16384_n8192"], rows=4)
    assert bwd["gamma"].dtype == np.float32 and bwd["dy"].dtype == np.uint16
    sweep = [w for w in WORKLOADS.values() if "sweep" in w.tags]
    # fwd and bwd at six bf16 sizes, one long-row bf16 size and one fp32 size
    assert len(sweep) == 16
    assert sorted({(w.x_dtype, w.w_dtype) for w in sweep}) == [("bf16", "bf16"), ("f32", "f32")]
    assert sum(w.x_dtype == "f32" for w in sweep) == 2


def test_generator_values_decode_like_torch_bf16():
    a = si.fill((4, 33), seed=1, tensor_id=1, dtype="bf16")
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.bf16_array_to_f64(a), t)
