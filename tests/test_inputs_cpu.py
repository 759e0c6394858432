"""The seeded input generators on CPU (host logic shared by the oracle's
tests, the CUDA path's tests and the bench).

* The counter-based generator is SplitMix64 (Steele, Lea & Flood, OOPSLA
  2014): with key 0 its counters give that generator's sequence from seed 0,
  whose first outputs are 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
  0x06C45D188009454F.
* Generation is order independent: any chunking of the counter range gives
  the same bits.
* Rounding to bf16 is round-to-nearest-even, checked bit for bit against
  torch's own float32 -> bfloat16 conversion; f16 likewise against torch.
* The workload recipe: N(0, 1) for u, B, C, z, dy; N(0, 0.5^2) for delta;
  A = -(n + 1); D in (0.5, 1.5); softplus(delta_bias) log-uniform in
  [1e-3, 1e-1]; io tensors exactly representable in their precision.
"""

import numpy as np
import pytest
import torch

from mamba_selective_scan_fwd_gb300 import inputs
from mamba_selective_scan_fwd_gb300.inputs import Workload, make_inputs, normal, round_bf16, round_io, uniform


def test_splitmix64_known_answers():
    got = inputs._bits(np.uint64(0), 0, 3)
    assert [int(v) for v in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_ranges_are_order_independent(monkeypatch):
    key = inputs._key(5, 2)
    whole = inputs._bits(key, 0, 1000)
    assert np.array_equal(inputs._bits(key, 300, 200), whole[300:500])
    ref_u, ref_n = uniform(9, 4, 1001), normal(9, 4, 1001, 0.5)
    # many small chunks, filled by a thread pool
    monkeypatch.setattr(inputs, "_CHUNK", 7)
    assert np.array_equal(uniform(9, 4, 1001), ref_u)
    assert np.array_equal(normal(9, 4, 1001, 0.5), ref_n)


def test_streams_and_seeds_differ():
    a = uniform(1, 0, 64)
    assert not np.array_equal(a, uniform(1, 1, 64))
    assert not np.array_equal(a, uniform(2, 0, 64))
    assert np.array_equal(a, uniform(1, 0, 64))


def test_uniform_and_normal_moments():
    n = 400_000
    u = uniform(3, 0, n)
    assert u.min() > 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 5 * np.sqrt(1 / 12 / n)
    assert abs(u.var() - 1 / 12) < 0.002
    z = normal(3, 1, n, 2.0)
    assert abs(z.mean()) < 5 * 2.0 / np.sqrt(n)
    assert abs(z.std() - 2.0) < 0.01
    # the fraction within one sigma of a normal: 0.6827
    assert abs(np.mean(np.abs(z) < 2.0) - 0.6827) < 0.005


def _edge_floats():
    rng = np.random.default_rng(0)
    x = rng.normal(size=20000).astype(np.float32) * np.float32(3.0)
    bits = np.array([0x3F808000, 0x3F818000, 0x3F80FFFF, 0x3F817FFF, 0x7F7FFFFF, 0x00000001, 0x807FFFFF,
                     0x7F800000, 0xFF800000, 0x00000000, 0x80000000, 0x3F7FFFFF, 0x477FE000],
                    dtype=np.uint32)
    return np.concatenate([x, bits.view(np.float32)])


def test_round_bf16_matches_torch():
    x = _edge_floats()
    ours = round_bf16(x).view(np.uint32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy().view(np.uint32)
    assert np.array_equal(ours, ref)
    nan = round_bf16(np.array([np.nan], dtype=np.float32))
    assert np.isnan(nan[0])


@pytest.mark.filterwarnings("ignore:overflow encountered in cast")  # values past the f16 range become inf
def test_round_f16_matches_torch():
    x = _edge_floats()
    finite = np.isfinite(x)
    ours = round_io(x[finite], "f16")
    ref = torch.from_numpy(x[finite]).to(torch.float16).to(torch.float32).numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
def test_workload_recipe(io):
    w = Workload("probe", 2, 300, 96, 8, io, seed=11)
    x = make_inputs(w, with_dy=True)
    assert x["u"].shape == (2, 300, 96) and x["B"].shape == (2, 300, 8) and x["A"].shape == (96, 8)
    for k in ("u", "delta", "B", "C", "z", "dy", "A", "D", "delta_bias"):
        assert x[k].dtype == np.float32, k
    for k in ("u", "delta", "B", "C", "z", "dy"):
        assert np.array_equal(round_io(x[k], io), x[k]), k  # exactly representable in the io type
    assert np.array_equal(x["A"], -np.broadcast_to(np.arange(1, 9, dtype=np.float32), (96, 8)))
    assert x["D"].min() > 0.5 and x["D"].max() < 1.5
    dt = np.log1p(np.exp(x["delta_bias"].astype(np.float64)))
    assert dt.min() >= 1e-3 * (1 - 1e-5) and dt.max() <= 1e-1 * (1 + 1e-5)
    assert abs(x["delta"].std() - 0.5) < 0.02 and abs(x["u"].std() - 1.0) < 0.03
    # the same workload draws the same values; optional terms can be left out
    y = make_inputs(w, with_dy=True)
    assert all(np.array_equal(x[k], y[k]) for k in x)
    w2 = Workload("probe", 2, 300, 96, 8, io, seed=11, has_D=False, has_z=False, has_bias=False)
    x2 = make_inputs(w2, with_dy=False)
    assert x2["D"] is None and x2["z"] is None and x2["delta_bias"] is None and x2["dy"] is None
    assert np.array_equal(x2["u"], x["u"])
