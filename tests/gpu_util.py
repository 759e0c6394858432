"""Helpers shared by the GPU parity tests: move seeded inputs to the GPU, run
the CUDA path through the C ABI binding, run the oracle on the same values,
and compare.

Tolerances (Mamba-1 selective scan accuracy targets):
* f32 I/O: forward (y, last_state) max normwise relative error <= 1e-5,
  gradients <= 1e-4;
* bf16 I/O with f32 state: <= 2e-2 against the oracle fed the same
  bf16-rounded inputs, with the oracle's y rounded to bf16.

"Normwise relative error" of a tensor is max|got - ref| / max|ref| (a
reference tensor that is all zero is compared absolutely).  An elementwise
ratio is not used because y = sum_n h C cancels: near-zero outputs would
measure the cancellation, not the kernel.  The parity gates take that measure
per row -- each (b, d) row of the [B, L, D] outputs, each batch row of dB / dC
-- and bound the worst row, so that an error confined to rows of small
magnitude is not hidden under the largest row's scale.
"""

from __future__ import annotations

import json
import os

import numpy as np
import torch

import mamba_selective_scan_fwd_gb300 as ss
from mamba_selective_scan_fwd_gb300.inputs import round_bf16

# f16 I/O: both sides see the same f16 inputs, so the gradients (f32 outputs)
# differ only by f32 arithmetic and keep the f32 bound; y is rounded to f16 on
# both sides, so it may differ by one f16 ulp (2^-10 relative) where the two
# unrounded values straddle a rounding boundary: 2e-3 normwise.
TOL = {"f32": {"fwd": 1e-5, "bwd": 1e-4}, "bf16": {"fwd": 2e-2, "bwd": 2e-2}, "f16": {"fwd": 2e-3, "bwd": 1e-4}}
IO_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
IO_KEYS = ("u", "delta", "B", "C", "z", "dy")


def to_device(x: dict, io: str, dev="cuda"):
    out = {}
    for k, v in x.items():
        if v is None:
            out[k] = None
            continue
        t = torch.from_numpy(np.ascontiguousarray(v))
        if k in IO_KEYS:
            t = t.to(IO_DTYPE[io])
        out[k] = t.to(dev)
    return out


def normwise(got, ref) -> float:
    if isinstance(got, torch.Tensor):
        got = got.detach().float().cpu().double().numpy()
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    if not np.all(np.isfinite(got)) and not np.array_equal(np.isfinite(got), np.isfinite(ref)):
        return float("inf")  # a non-finite output where the reference is finite fails every tolerance
    scale = np.max(np.abs(ref))
    err = np.max(np.abs(got - ref))
    return float(err / scale) if scale > 0 else float(err)


def normwise_rows(got, ref, rows_axis) -> float:
    """The worst per-row normwise error: rows_axis names the axes that index a row
    (the others are reduced within it): (0, 2) for the (b, d) rows of [B, L, D],
    (0,) for the batch rows of [B, L, N], () for the whole tensor."""
    if isinstance(got, torch.Tensor):
        got = got.detach().float().cpu().double().numpy()
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    if not np.array_equal(np.isfinite(got), np.isfinite(ref)):
        return float("inf")
    red = tuple(a for a in range(ref.ndim) if a not in rows_axis)
    err = np.max(np.abs(got - ref), axis=red, keepdims=False)
    scale = np.max(np.abs(ref), axis=red, keepdims=False)
    rel = np.where(scale > 0, err / np.where(scale > 0, scale, 1.0), err)
    return float(np.max(rel))


# axes that index a row of each output (see normwise_rows)
ROWS = {"y": (0, 2), "du": (0, 2), "ddelta": (0, 2), "dz": (0, 2), "dB": (0,), "dC": (0,), "last_state": (),
        "dA": (), "dD": (), "ddelta_bias": ()}


def elementwise_diag(got, ref) -> dict:
    """The elementwise diagnostic |got - ref| / (|ref| + 1e-3 rms(ref)): its maximum
    and 99th percentile (reported, not gated)."""
    if isinstance(got, torch.Tensor):
        got = got.detach().float().cpu().double().numpy()
    got = np.asarray(got, np.float64).reshape(-1)
    ref = np.asarray(ref, np.float64).reshape(-1)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    e = np.abs(got - ref) / (np.abs(ref) + 1e-3 * rms + 1e-300)
    return {"max": float(np.max(e)) if e.size else 0.0, "p99": float(np.percentile(e, 99)) if e.size else 0.0}


def report(config: str, output: str, got, ref, rows_axis=None):
    """Append the achieved errors of one output to the JSON-lines file named by the
    SS_PARITY_REPORT environment variable (nothing when it is unset)."""
    path = os.environ.get("SS_PARITY_REPORT")
    if not path:
        return
    rec = {"config": config, "output": output, "normwise": normwise(got, ref),
           "normwise_rows": normwise_rows(got, ref, ROWS.get(output, ()) if rows_axis is None else rows_axis)}
    rec.update({f"elementwise_{k}": v for k, v in elementwise_diag(got, ref).items()})
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def gpu_fwd(t, softplus=True):
    return ss.ss_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], softplus)


def gpu_bwd(t, softplus=True):
    return ss.ss_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], softplus, t["dy"])


def gpu_fwd_save(t, softplus=True):
    """Forward that also stores the backward's restart states: (y, last_state, saved)."""
    return ss.ss_fwd_save(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], softplus)


def gpu_bwd_saved(t, saved, softplus=True):
    return ss.ss_bwd_saved(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], softplus,
                           t["dy"], saved)


def oracle_fwd(orc, x, softplus=True, rows=None):
    return orc.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], softplus, rows=rows)


def oracle_bwd(orc, x, softplus=True, rows=None, want_dBdC=True):
    return orc.bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], softplus, dy=x["dy"],
                   rows=rows, want_dBdC=want_dBdC)


def ref_y(y, io):
    """The oracle's y as the kernel must return it: rounded to the 16-bit I/O type."""
    if io == "bf16":
        return round_bf16(y.astype(np.float32)).astype(np.float64)
    if io == "f16":
        return y.astype(np.float16).astype(np.float64)
    return y
