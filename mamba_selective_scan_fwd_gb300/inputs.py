"""Seeded, counter-based synthetic inputs for the Mamba-1 selective scan.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and bench.  It draws random numbers and rounds them to the I/O precision; it
holds none of the scan's own arithmetic.

Generator
---------
Every element ``i`` of input stream ``k`` under seed ``s`` is a pure function
of ``(s, k, i)``: the SplitMix64 output function (Steele, Lea & Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014) applied to the
counter ``key(s, k) + (i + 1) * 0x9E3779B97F4A7C15``.  Generation is therefore
order independent and can be split across threads.  Uniforms take the top 53
bits, offset by half an ulp so they lie in the open interval (0, 1).  Normals
use the Box-Muller transform on the uniforms of counters ``2i`` and ``2i+1``.

Distributions (the Mamba-1 selective-scan workload recipe)
----------------------------------------------------------
* ``u``, ``B``, ``C``, ``z``, ``dy`` ~ N(0, 1)
* raw ``delta`` ~ N(0, 0.5^2)
* ``A[d, n] = -(n + 1)`` for every channel ``d``
* ``D`` ~ U(0.5, 1.5)
* ``delta_bias = softplus^{-1}(dt)`` with ``dt`` log-uniform in [1e-3, 1e-1];
  the inverse is ``dt + log(-expm1(-dt))``.

Tensors in the I/O precision (``u, delta, B, C, z, dy``) are rounded to that
precision here (bf16: round to nearest even from f32), so that the oracle and
the CUDA path consume bit-identical values.  ``A``, ``D`` and ``delta_bias``
are always f32.  Everything is returned as numpy ``float32`` arrays whose
values are exactly representable in the I/O precision.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stream ids: one per generated tensor, fixed forever so that stored values
# keep their meaning.
STREAM = {"u": 0, "delta": 1, "B": 2, "C": 3, "z": 4, "dy": 5, "D": 6, "dt": 7}

_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([(seed & 0xFFFFFFFF) << 16 | (stream & 0xFFFF)], dtype=np.uint64)
        return _mix(base * _GOLDEN + _GOLDEN)[0]


def _bits(key: np.uint64, start: int, count: int) -> np.ndarray:
    ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + ctr * _GOLDEN)


def _to_unit(bits: np.ndarray) -> np.ndarray:
    return ((bits >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def _fill(n: int, fn) -> np.ndarray:
    """Evaluate ``fn(start, count) -> float64 array`` over [0, n) in chunks, in parallel."""
    out = np.empty(n, dtype=np.float64)
    starts = list(range(0, n, _CHUNK))

    def work(s):
        c = min(_CHUNK, n - s)
        out[s:s + c] = fn(s, c)

    if len(starts) <= 1:
        for s in starts:
            work(s)
    else:
        workers = min(len(starts), os.cpu_count() or 1, 32)
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(work, starts))
    return out


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """n uniforms in (0, 1), float64."""
    key = _key(seed, stream)
    return _fill(n, lambda s, c: _to_unit(_bits(key, s, c)))


def normal(seed: int, stream: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """n standard normals (Box-Muller on counters 2i, 2i+1), times sigma, float64."""
    key = _key(seed, stream)

    def fn(s, c):
        u = _to_unit(_bits(key, 2 * s, 2 * c))
        u1, u2 = u[0::2], u[1::2]
        return sigma * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)

    return _fill(n, fn)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even); returns float32 holding bf16 values."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    b = f.view(np.uint32)
    # NaN stays NaN (quiet); finite values round to nearest even on the top 16 bits.
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    nan = np.isnan(f)
    if nan.any():
        r = np.where(nan, (b | np.uint32(0x00400000)) & np.uint32(0xFFFF0000), r)
    return r.view(np.float32)


def to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """float32 array holding bf16 values -> uint16 bit patterns."""
    return (np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def round_io(x: np.ndarray, io: str) -> np.ndarray:
    if io == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if io == "bf16":
        return round_bf16(x)
    if io == "f16":
        return x.astype(np.float16).astype(np.float32)  # round to nearest, ties to even
    raise ValueError(f"unknown io dtype {io!r}")


@dataclass(frozen=True)
class Workload:
    """One selective-scan problem: sizes, I/O precision, which terms are present."""

    name: str
    Bsz: int
    L: int
    Dch: int
    N: int
    io: str = "f32"
    seed: int = 0
    backward: bool = True
    softplus: bool = True
    has_D: bool = True
    has_z: bool = True
    has_bias: bool = True

    @property
    def bld(self) -> int:
        return self.Bsz * self.L * self.Dch


# The five workloads the method is measured on.  Seeds: 0 for the tiny case,
# then the workload's index.
WORKLOADS = [
    Workload("tiny-f32", 1, 64, 8, 4, "f32", seed=0, backward=True),
    Workload("mamba130m-layer-bf16-fwd", 8, 2048, 1536, 16, "bf16", seed=1, backward=False),
    Workload("mamba130m-layer-f32", 8, 2048, 1536, 16, "f32", seed=2, backward=True),
    Workload("mamba2.8b-layer-bf16", 4, 4096, 5120, 16, "bf16", seed=3, backward=True),
    Workload("long-seq-bf16", 1, 131072, 1024, 16, "bf16", seed=4, backward=True),
]


def make_inputs(w: Workload, with_dy: bool | None = None) -> dict:
    """Generate the inputs of workload ``w`` as float32 numpy arrays.

    Keys: u, delta, A, B, C, D, z, delta_bias, dy (absent terms are None).
    Shapes: u/delta/z/dy [Bsz, L, Dch]; A [Dch, N]; B/C [Bsz, L, N]; D and
    delta_bias [Dch].
    """
    if with_dy is None:
        with_dy = w.backward
    s = w.seed
    bld = (w.Bsz, w.L, w.Dch)
    bln = (w.Bsz, w.L, w.N)
    n_bld = w.Bsz * w.L * w.Dch
    n_bln = w.Bsz * w.L * w.N
    out = {}
    out["u"] = round_io(normal(s, STREAM["u"], n_bld), w.io).reshape(bld)
    out["delta"] = round_io(normal(s, STREAM["delta"], n_bld, 0.5), w.io).reshape(bld)
    out["B"] = round_io(normal(s, STREAM["B"], n_bln), w.io).reshape(bln)
    out["C"] = round_io(normal(s, STREAM["C"], n_bln), w.io).reshape(bln)
    out["z"] = round_io(normal(s, STREAM["z"], n_bld), w.io).reshape(bld) if w.has_z else None
    out["dy"] = round_io(normal(s, STREAM["dy"], n_bld), w.io).reshape(bld) if with_dy else None
    out["A"] = np.ascontiguousarray(
        np.broadcast_to(-(np.arange(w.N, dtype=np.float32) + 1.0), (w.Dch, w.N)), dtype=np.float32)
    out["D"] = (0.5 + uniform(s, STREAM["D"], w.Dch)).astype(np.float32) if w.has_D else None
    if w.has_bias:
        lo, hi = np.log(1e-3), np.log(1e-1)
        dt = np.exp(lo + (hi - lo) * uniform(s, STREAM["dt"], w.Dch))
        out["delta_bias"] = (dt + np.log(-np.expm1(-dt))).astype(np.float32)
    else:
        out["delta_bias"] = None
    return out


def small_inputs(Bsz, L, Dch, N, io="f32", seed=0, softplus=True, has_D=True, has_z=True,
                 has_bias=True, with_dy=True) -> dict:
    """Inputs with the workload distributions at an arbitrary (small) size."""
    w = Workload("custom", Bsz, L, Dch, N, io, seed=seed, backward=with_dy, softplus=softplus,
                 has_D=has_D, has_z=has_z, has_bias=has_bias)
    return make_inputs(w, with_dy=with_dy)
