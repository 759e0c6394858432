"""GPU parity when the launch plan splits the units (batch row, channel tile)
into two segments: the units that make whole rounds over the GPU's SMs run as
one chunk each, the remaining ones are cut in time, their chunk summaries
carrying the state forward and the adjoint backward.  Every output element is
compared with the oracle, on a problem whose time-cut segment holds a ragged
channel tile and a ragged last chunk, through the plain entry points and the
extended ones (h0, an incoming gradient of last_state, A_log)."""

import numpy as np
import pytest
import torch

import mamba_selective_scan_fwd_gb300 as ss
from mamba_selective_scan_fwd_gb300.inputs import small_inputs
from gpu_util import (TOL, gpu_bwd, gpu_bwd_saved, gpu_fwd, gpu_fwd_save, normwise, normwise_rows, oracle_bwd,
                      oracle_fwd, ref_y, to_device)

pytestmark = pytest.mark.gpu

# Two-warp blocks (N = 16): a round is 608 blocks.  2 x 310 = 620 units: 608
# of one chunk, then 12 (batch row 1, tiles 298..309, the last one 25 channels
# wide) cut into chunks of 128, 128 and 44 steps
SHAPE = (2, 300, 9913, 16)
GRADS = ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias")


def test_shape_is_split():
    p = ss.plan_info(*SHAPE, ss.SS_BF16)
    assert p["segments"] == [(608, 1), (12, 3)]


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_split_plan_parity(orc, io):
    x = small_inputs(*SHAPE, io=io, seed=5100)
    t = to_device(x, io)
    y, last, saved = gpu_fwd_save(t)
    g = gpu_bwd_saved(t, saved)
    torch.cuda.synchronize()
    rf = oracle_fwd(orc, x)
    rb = oracle_bwd(orc, x)
    tf, tb = TOL[io]["fwd"], TOL[io]["bwd"]
    errs = {"y": normwise(y, ref_y(rf.y, io)), "last_state": normwise(last, rf.last_state)}
    for k in GRADS:
        errs[k] = normwise(g[k], getattr(rb, k))
    bad = {k: e for k, e in errs.items() if e > (tf if k in ("y", "last_state") else tb)}
    assert not bad, (bad, errs)
    # the time-cut units alone (batch row 1, channels of tiles 298..): the
    # normwise errors above are dominated by the far larger one-chunk segment
    d0 = 298 * 32
    assert normwise(y[1, :, d0:], ref_y(rf.y, io)[1, :, d0:]) <= tf
    assert normwise(last[1, d0:], rf.last_state[1, d0:]) <= tf
    for k in ("du", "ddelta", "dz"):
        assert normwise(g[k][1, :, d0:], getattr(rb, k)[1, :, d0:]) <= tb, k
    # the plain forward and the backward that recomputes the states give the same bits
    y2, last2 = gpu_fwd(t)
    assert torch.equal(y, y2) and torch.equal(last, last2)
    g2 = gpu_bwd(t)
    for k in GRADS:
        assert torch.equal(g[k], g2[k]), k


def test_split_plan_state_parity(orc):
    Bsz, L, Dch, N = SHAPE
    x = small_inputs(*SHAPE, io="f32", seed=5200)
    rng = np.random.default_rng(5201)
    x["A_log"] = np.log(-x["A"]).astype(np.float32)
    x["h0"] = rng.normal(size=(Bsz, Dch, N)).astype(np.float32)
    x["dlast"] = rng.normal(size=(Bsz, Dch, N)).astype(np.float32)
    t = to_device({k: v for k, v in x.items() if k not in ("A_log", "h0", "dlast")}, "f32")
    for k in ("A_log", "h0", "dlast"):
        t[k] = torch.from_numpy(x[k]).cuda()
    y, last, saved = ss.ss_fwd_ex(t["u"], t["delta"], t["A_log"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                                  True, h0=t["h0"], a_is_log=True, save=True)
    g = ss.ss_bwd_ex(t["u"], t["delta"], t["A_log"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True, t["dy"],
                     h0=t["h0"], dlast_state=t["dlast"], a_is_log=True, saved=saved)
    torch.cuda.synchronize()
    rf = orc.fwd(x["u"], x["delta"], None, x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True, h0=x["h0"],
                 A_log=x["A_log"])
    rb = orc.bwd(x["u"], x["delta"], None, x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True, dy=x["dy"],
                 h0=x["h0"], dlast_state=x["dlast"], A_log=x["A_log"])
    tf, tb = TOL["f32"]["fwd"], TOL["f32"]["bwd"]
    errs = {"y": normwise(y, rf.y), "last_state": normwise(last, rf.last_state)}
    for k in GRADS + ("dh0",):
        errs[k] = normwise(g[k], getattr(rb, k))
    bad = {k: e for k, e in errs.items() if e > (tf if k in ("y", "last_state") else tb)}
    assert not bad, (bad, errs)
    d0 = 298 * 32
    assert normwise(g["dh0"][1, d0:], rb.dh0[1, d0:]) <= tb
    assert normwise(last[1, d0:], rf.last_state[1, d0:]) <= tf


# One-warp blocks (N = 8): a round is 1216 blocks.  2 x 658 = 1316 units: 1216
# of one chunk, then 100 (batch row 1, tiles 558..657) cut into 4 chunks.
SHAPE8 = (2, 512, 21056, 8)


def test_split_plan_parity_one_warp_blocks(orc):
    assert ss.plan_info(*SHAPE8, ss.SS_BF16)["segments"] == [(1216, 1), (100, 4)]
    x = small_inputs(*SHAPE8, io="bf16", seed=5300)
    t = to_device(x, "bf16")
    y, last, saved = gpu_fwd_save(t)
    g = gpu_bwd_saved(t, saved)
    torch.cuda.synchronize()
    rf = oracle_fwd(orc, x)
    rb = oracle_bwd(orc, x)
    tf, tb = TOL["bf16"]["fwd"], TOL["bf16"]["bwd"]
    errs = {"y": normwise(y, ref_y(rf.y, "bf16")), "last_state": normwise(last, rf.last_state)}
    for k in GRADS:
        errs[k] = normwise(g[k], getattr(rb, k))
    bad = {k: e for k, e in errs.items() if e > (tf if k in ("y", "last_state") else tb)}
    assert not bad, (bad, errs)
    d0 = 558 * 32
    assert normwise(y[1, :, d0:], ref_y(rf.y, "bf16")[1, :, d0:]) <= tf
    assert normwise(last[1, d0:], rf.last_state[1, d0:]) <= tf
    for k in ("du", "ddelta", "dz"):
        assert normwise(g[k][1, :, d0:], getattr(rb, k)[1, :, d0:]) <= tb, k


# 384 units (6 batch rows x 64 channel tiles) hold fewer than 8 warps per SM:
# every unit is cut into 3 chunks, and the 768 forward summaries (chunks 0, 1)
# are more blocks than one round of the main kernel, which takes the dedicated
# summary kernel
WIDE = (6, 320, 2048, 16)


def test_wide_summary_plan():
    p = ss.plan_info(*WIDE, ss.SS_BF16)
    assert p["segments"] == [(384, 3)]


@pytest.mark.parametrize("io", ["bf16", "f16", "f32"])
def test_wide_summary_parity(orc, io):
    x = small_inputs(*WIDE, io=io, seed=5300)
    t = to_device(x, io)
    y, last, saved = gpu_fwd_save(t)
    g = gpu_bwd_saved(t, saved)
    torch.cuda.synchronize()
    rows = np.random.default_rng(5301).choice(WIDE[0] * WIDE[2], 96, replace=False)
    rows[0] = WIDE[0] * WIDE[2] - 1
    rf = oracle_fwd(orc, x, rows=rows)
    rb = oracle_bwd(orc, x, rows=rows, want_dBdC=False)
    bi = torch.as_tensor(rows // WIDE[2], device=y.device)
    di = torch.as_tensor(rows % WIDE[2], device=y.device)
    tf, tb = TOL[io]["fwd"], TOL[io]["bwd"]
    # sampled rows [n_rows, L], each bounded on its own scale
    assert normwise_rows(y[bi, :, di].float().cpu().numpy(), ref_y(rf.y, io), (0,)) <= tf
    assert normwise(last[bi, di].cpu().numpy(), rf.last_state) <= tf
    for k in ("du", "ddelta", "dz"):
        assert normwise_rows(g[k][bi, :, di].cpu().numpy(), getattr(rb, k), (0,)) <= tb, k
    # the plain forward gives the same bits as the saving one
    y2, last2 = gpu_fwd(t)
    assert torch.equal(y, y2) and torch.equal(last, last2)
