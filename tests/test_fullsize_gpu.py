"""Parity at the full workload sizes, in the launch configuration the bench
times (the forward that saves the backward's restart states, then the
backward that reads them).  The CUDA path runs the whole problem; the oracle
recomputes sampled outputs one row at a time:

* y, last_state, du, ddelta, dz on sampled (b, d) rows;
* dA, dD, ddelta_bias for sampled channels (every batch row of them);
* dB, dC for one batch entry (every channel of it), which is the sum the
  kernel reduces across the full channel dimension.

Plus properties that hold at any size: ddelta_bias = sum_{b,t} ddelta and
dD = sum_{b,t} dy silu(z) u, bit-identical repeated runs, and results
bit-identical to the entry points that recompute the states.
"""

import numpy as np
import pytest
import torch

from mamba_selective_scan_fwd_gb300.inputs import WORKLOADS, make_inputs
from gpu_util import (TOL, gpu_bwd, gpu_bwd_saved, gpu_fwd, gpu_fwd_save, normwise, normwise_rows, oracle_bwd,
                      oracle_fwd, ref_y, report, to_device)

pytestmark = pytest.mark.gpu


def _rows(w, n, rng):
    b = rng.integers(0, w.Bsz, size=n)
    d = rng.integers(0, w.Dch, size=n)
    d[0], b[0] = w.Dch - 1, w.Bsz - 1  # the last channel of the last batch (ragged-tile edge)
    return b * w.Dch + d


@pytest.mark.parametrize("wi", [1, 2, 3, 4], ids=[WORKLOADS[i].name for i in (1, 2, 3, 4)])
def test_fullsize_sampled(orc, wi):
    w = WORKLOADS[wi]
    x = make_inputs(w)
    t = to_device(x, w.io)
    y, last, saved = gpu_fwd_save(t, w.softplus)
    g = gpu_bwd_saved(t, saved, w.softplus) if w.backward else None
    torch.cuda.synchronize()
    tf, tb = TOL[w.io]["fwd"], TOL[w.io]["bwd"]
    rng = np.random.default_rng(wi)
    rows = _rows(w, 24, rng)
    bb, dd = rows // w.Dch, rows % w.Dch
    rf = oracle_fwd(orc, x, w.softplus, rows=rows)
    bi, di = torch.as_tensor(bb, device=y.device), torch.as_tensor(dd, device=y.device)
    y_rows = y[bi, :, di].float().cpu().numpy()
    # sampled rows [n_rows, L]: each row bounded on its own scale (axis 0 indexes the rows)
    assert normwise_rows(y_rows, ref_y(rf.y, w.io), (0,)) <= tf
    assert normwise(last[bi, di].cpu().numpy(), rf.last_state) <= tf
    report(w.name, "y", y_rows, ref_y(rf.y, w.io), (0,))
    report(w.name, "last_state", last[bi, di].cpu().numpy(), rf.last_state)
    # forward bit-identical on a second run, and to the forward that saves nothing
    y2, last2, saved2 = gpu_fwd_save(t, w.softplus)
    assert torch.equal(y, y2) and torch.equal(last, last2) and torch.equal(saved, saved2)
    y3, last3 = gpu_fwd(t, w.softplus)
    assert torch.equal(y, y3) and torch.equal(last, last3)
    del y2, last2, saved2, y3, last3
    if not w.backward:
        return
    rb = oracle_bwd(orc, x, w.softplus, rows=rows, want_dBdC=False)
    for k in ("du", "ddelta", "dz"):
        got_k = g[k][bi, :, di].cpu().numpy()
        assert normwise_rows(got_k, getattr(rb, k), (0,)) <= tb, k
        report(w.name, k, got_k, getattr(rb, k), (0,))
    # parameter gradients of sampled channels: all batch rows of those channels
    chans = np.unique(np.concatenate([dd[:4], [0, w.Dch - 1]]))
    prow = (np.arange(w.Bsz)[:, None] * w.Dch + chans[None, :]).reshape(-1)
    rp = oracle_bwd(orc, x, w.softplus, rows=prow, want_dBdC=False)
    dA = rp.dA_rows.reshape(w.Bsz, len(chans), w.N).sum(axis=0)
    dD = rp.dD_rows.reshape(w.Bsz, len(chans)).sum(axis=0)
    db = rp.dbias_rows.reshape(w.Bsz, len(chans)).sum(axis=0)
    ci = torch.as_tensor(chans, device=y.device)
    assert normwise(g["dA"][ci].cpu().numpy(), dA) <= tb
    assert normwise(g["dD"][ci].cpu().numpy(), dD) <= tb
    assert normwise(g["ddelta_bias"][ci].cpu().numpy(), db) <= tb
    for k, ref in (("dA", dA), ("dD", dD), ("ddelta_bias", db)):
        report(w.name, k, g[k][ci].cpu().numpy(), ref)
    # dB, dC of one batch entry: every channel contributes
    b0 = w.Bsz - 1
    crow = b0 * w.Dch + np.arange(w.Dch)
    rc = oracle_bwd(orc, x, w.softplus, rows=crow, want_dBdC=True)
    assert normwise(g["dB"][b0].cpu().numpy(), rc.dB[b0]) <= tb
    assert normwise(g["dC"][b0].cpu().numpy(), rc.dC[b0]) <= tb
    report(w.name, "dB", g["dB"][b0].cpu().numpy(), rc.dB[b0], ())
    report(w.name, "dC", g["dC"][b0].cpu().numpy(), rc.dC[b0], ())
    # identities at full size (computed in f64 from the kernel's own outputs)
    dl = g["ddelta"].double()
    assert normwise(g["ddelta_bias"].cpu().numpy(), dl.sum(dim=(0, 1)).cpu().numpy()) <= 1e-5
    gate = t["dy"].double() * torch.nn.functional.silu(t["z"].double())
    assert normwise(g["dD"].cpu().numpy(), (gate * t["u"].double()).sum(dim=(0, 1)).cpu().numpy()) <= 1e-5
    # backward bit-identical on a second run, and to the backward that recomputes the states
    for g2 in (gpu_bwd_saved(t, saved, w.softplus), gpu_bwd(t, w.softplus)):
        for k, v in g.items():
            if v is not None:
                assert torch.equal(v, g2[k]), k
        del g2


def test_tiny_workload_full_parity(orc):
    """The tiny f32 workload, every output element compared."""
    w = WORKLOADS[0]
    x = make_inputs(w)
    t = to_device(x, w.io)
    y, last = gpu_fwd(t, w.softplus)
    g = gpu_bwd(t, w.softplus)
    torch.cuda.synchronize()
    rf = oracle_fwd(orc, x, w.softplus)
    rb = oracle_bwd(orc, x, w.softplus)
    assert normwise(y, rf.y) <= 1e-5 and normwise(last, rf.last_state) <= 1e-5
    for k in ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias"):
        assert normwise(g[k], getattr(rb, k)) <= 1e-4, k
