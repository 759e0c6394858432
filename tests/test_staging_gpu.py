"""Tile staging on the GPU: TMA copies against per-thread asynchronous copies,
and the device status word that a kernel which gives up waiting leaves.

The scan kernels stage each tile of delta, u, z, dy, y0, B and C (and the
backward's saved states) into shared memory either with TMA boxes
(cp.async.bulk.tensor over 3-D tensor maps, completion on an mbarrier) or
with per-thread asynchronous copies.  Only where the bytes come from
differs: the arithmetic after staging is the same code, so every output must
be equal bit for bit.  Shapes cover a channel tile that runs past D (the TMA
box is zero-filled there), a ragged last time tile (zero-filled past L),
chunked sequences (the summary passes stage through TMA too), the split plan
and all three io types.

Every wait on a TMA copy has a time limit; the self-test entry point runs a
wait on a barrier nothing completes, which must leave SS_ERR_DEVICE_TIMEOUT
in the status word and leave the context usable.  No GPU fault is involved.
"""

import pytest
import torch

import mamba_selective_scan_fwd_gb300 as ss
from mamba_selective_scan_fwd_gb300.inputs import small_inputs
from gpu_util import to_device

pytestmark = pytest.mark.gpu

DT = {"f32": ss.SS_F32, "bf16": ss.SS_BF16, "f16": ss.SS_F16}


def _all_outputs(t):
    """Forward, forward with saved states, backward and backward from the saved
    states, flattened into one list of tensors."""
    args = (t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True)
    y, last = ss.ss_fwd(*args)
    y2, last2, saved = ss.ss_fwd_save(*args)
    g = ss.ss_bwd(*args, t["dy"])
    g2 = ss.ss_bwd_saved(*args, t["dy"], saved)
    out = [y, last, y2, last2]
    for grads in (g, g2):
        out += [v for _, v in sorted(grads.items()) if v is not None]
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("shape,io,gate", [
    ((2, 300, 72, 16), "bf16", True),     # channel tile past D = 72, ragged last tile
    ((1, 500, 40, 16), "bf16", False),    # no z: no z / y0 boxes
    ((1, 1000, 16, 32), "f32", True),     # N = 32, 16-channel tiles
    ((2, 777, 64, 8), "f16", True),       # 16-bit B / C rows of 8 states (one 16-byte unit)
    ((1, 4100, 8, 4), "f32", True),       # few units: the sequence is cut into chunks
    ((2, 300, 9920, 16), "bf16", True),   # split plan: 608 one-chunk units, then a chunked segment
    ((6, 320, 2048, 16), "bf16", True),   # 384 units x 3 chunks: 768 forward summaries (their own kernel)
    ((6, 320, 2048, 16), "f32", True),    # the same with f32 rows read where TMA put them
])
def test_tma_and_copies_stage_identical_tiles(shape, io, gate):
    Bsz, L, Dch, N = shape
    x = small_inputs(Bsz, L, Dch, N, io=io, seed=777 + L + Dch, has_z=gate)
    t = to_device(x, io)
    prev = ss.set_copies_only(False)
    try:
        assert ss.staging_uses_tma(Bsz, L, Dch, N, DT[io])
        with_tma = _all_outputs(t)
        ss.set_copies_only(True)
        assert not ss.staging_uses_tma(Bsz, L, Dch, N, DT[io])
        with_copies = _all_outputs(t)
    finally:
        ss.set_copies_only(prev)
    assert len(with_tma) == len(with_copies)
    for a, b in zip(with_tma, with_copies):
        assert torch.equal(a, b)
    assert ss.device_status() == ss.SS_OK


@pytest.mark.parametrize("shape,io", [((1, 64, 12, 16), "bf16"), ((1, 64, 8, 2), "bf16"), ((1, 64, 5, 16), "f32")])
def test_problems_outside_tma_rules_use_copies(shape, io):
    # D or N times the element size not a multiple of 16 bytes, or D not a multiple of 4
    assert not ss.staging_uses_tma(*shape, DT[io])


def test_wait_timeout_is_reported_and_context_survives():
    x = small_inputs(1, 200, 32, 16, io="bf16", seed=5)
    t = to_device(x, "bf16")
    args = (t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True)
    y_before, _ = ss.ss_fwd(*args)
    assert ss.device_status() == ss.SS_OK
    # a wait of 1 ms on a barrier that nothing completes
    ss.selftest_wait_timeout(1_000_000)
    assert ss.device_status() == ss.SS_ERR_DEVICE_TIMEOUT
    assert ss.device_status() == ss.SS_OK  # the read cleared it
    ss.selftest_wait_timeout(0)
    assert ss.device_status() == ss.SS_ERR_DEVICE_TIMEOUT
    # the context is still usable and computes the same result
    y_after, _ = ss.ss_fwd(*args)
    torch.cuda.synchronize()
    assert torch.equal(y_before, y_after)
    assert ss.device_status() == ss.SS_OK


def test_ex2_rate_probe():
    # MUFU ex2 results per clock per SM: a whole number of results per cycle per
    # sub-partition on any part this library builds for (GB300: 32 per SM)
    r = ss.binding.measure_ex2_rate(2048)
    assert 8.0 <= r <= 64.0
    assert abs(r - round(r / 4) * 4) < 0.5
    assert ss.device_status() == ss.SS_OK


def test_fma_rate_probe():
    # f32 FMA results per clock per SM: a whole number of warp-wide results per
    # cycle per sub-partition (GB300: 128 per SM, a packed f32x2 FMA taking two
    # cycles of the FP32 pipe)
    r = ss.binding.measure_fma_rate(2048)
    assert 64.0 <= r <= 256.0
    assert abs(r - round(r / 32) * 32) < 2.0
    assert ss.device_status() == ss.SS_OK
