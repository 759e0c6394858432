"""Seeded random problems against the oracle: sizes, state size, io type,
optional terms and softplus drawn at random, so that the launch plan meets
shapes the hand-picked cases do not (ragged tiles and chunks of every kind,
uniform chunking, split plans).  Every output element is compared; the
saved-state pair must give the same bits as the recomputing pair.  The same
draws drive the extended entry points (initial state, incoming gradient of
last_state, A_log) and the single decoding step."""

import numpy as np
import pytest
import torch

import mamba_selective_scan_fwd_gb300 as ss
from mamba_selective_scan_fwd_gb300.inputs import small_inputs
from gpu_util import (TOL, gpu_bwd, gpu_bwd_saved, gpu_fwd, gpu_fwd_save, normwise, oracle_bwd, oracle_fwd, ref_y,
                      to_device)

pytestmark = pytest.mark.gpu

GRADS = ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias")


def draw(i):
    rng = np.random.default_rng(7000 + i)
    N = int(rng.choice([1, 2, 4, 8, 16, 32]))
    io = str(rng.choice(["f32", "bf16", "f16"]))
    if i % 8 == 7:
        # batch x channels past one round of blocks: a split plan when the tail is small
        tile = 32 if N >= 2 else 64
        rb = 608 if N >= 16 else 1216
        Bsz = int(rng.integers(1, 3))
        units = rb + int(rng.integers(1, 160))
        Dch = -(-units // Bsz) * tile - int(rng.integers(0, tile))
        L = int(rng.integers(130, 400))
    else:
        Bsz = int(rng.integers(1, 4))
        Dch = int(rng.integers(1, 300))
        L = int(rng.integers(1, 700))
    terms = dict(has_D=bool(rng.integers(0, 2)), has_z=bool(rng.integers(0, 2)), has_bias=bool(rng.integers(0, 2)))
    softplus = bool(rng.integers(0, 4))  # mostly on
    return (Bsz, L, Dch, N), io, terms, softplus


CASES = list(range(32))


@pytest.mark.parametrize("i", CASES)
def test_random_problem(orc, i):
    shape, io, terms, softplus = draw(i)
    x = small_inputs(*shape, io=io, seed=7100 + i, **terms)
    if not softplus:
        # delta + bias used as is: keep it a decay (halving keeps io-rounded values exact)
        x["delta"] = np.abs(x["delta"]) * np.float32(0.5)
        if x["delta_bias"] is not None:
            x["delta_bias"] = (np.abs(x["delta_bias"]) * np.float32(0.02)).astype(np.float32)
    t = to_device(x, io)
    y, last, saved = gpu_fwd_save(t, softplus)
    g = gpu_bwd_saved(t, saved, softplus)
    torch.cuda.synchronize()
    rf = oracle_fwd(orc, x, softplus)
    rb = oracle_bwd(orc, x, softplus)
    tf, tb = TOL[io]["fwd"], TOL[io]["bwd"]
    errs = {"y": normwise(y, ref_y(rf.y, io)), "last_state": normwise(last, rf.last_state)}
    for k in GRADS:
        ref = getattr(rb, k)
        if ref is None:
            assert g[k] is None, k
        else:
            errs[k] = normwise(g[k], ref)
    bad = {k: e for k, e in errs.items() if e > (tf if k in ("y", "last_state") else tb)}
    assert not bad, (shape, io, terms, softplus, ss.plan_info(*shape, 0)["segments"], bad, errs)
    y2, last2 = gpu_fwd(t, softplus)
    assert torch.equal(y, y2) and torch.equal(last, last2)
    g2 = gpu_bwd(t, softplus)
    for k in GRADS:
        if g[k] is not None:
            assert torch.equal(g[k], g2[k]), k


STATE_GRADS = GRADS + ("dh0",)


@pytest.mark.parametrize("i", list(range(12)))
def test_random_problem_with_state(orc, i):
    """ss_fwd_ex / ss_bwd_ex on random problems: an initial state, an incoming
    gradient of last_state and A given as A_log, all terms drawn at random."""
    (Bsz, L, Dch, N), io, terms, softplus = draw(100 + i)
    x = small_inputs(Bsz, L, Dch, N, io=io, seed=7300 + i, **terms)
    if not softplus:
        x["delta"] = np.abs(x["delta"]) * np.float32(0.5)
        if x["delta_bias"] is not None:
            x["delta_bias"] = (np.abs(x["delta_bias"]) * np.float32(0.02)).astype(np.float32)
    rng = np.random.default_rng(7400 + i)
    A_log = np.log(-x["A"]).astype(np.float32)
    h0 = rng.normal(size=(Bsz, Dch, N)).astype(np.float32)
    dlast = rng.normal(size=(Bsz, Dch, N)).astype(np.float32)
    t = to_device(x, io)
    A_d, h0_d, dl_d = (torch.from_numpy(v).cuda() for v in (A_log, h0, dlast))
    y, last, saved = ss.ss_fwd_ex(t["u"], t["delta"], A_d, t["B"], t["C"], t["D"], t["z"], t["delta_bias"], softplus,
                                  h0=h0_d, a_is_log=True, save=True)
    g = ss.ss_bwd_ex(t["u"], t["delta"], A_d, t["B"], t["C"], t["D"], t["z"], t["delta_bias"], softplus, t["dy"],
                     h0=h0_d, dlast_state=dl_d, a_is_log=True, saved=saved)
    torch.cuda.synchronize()
    rf = orc.fwd(x["u"], x["delta"], None, x["B"], x["C"], x["D"], x["z"], x["delta_bias"], softplus, h0=h0,
                 A_log=A_log)
    rb = orc.bwd(x["u"], x["delta"], None, x["B"], x["C"], x["D"], x["z"], x["delta_bias"], softplus, dy=x["dy"],
                 h0=h0, dlast_state=dlast, A_log=A_log)
    tf, tb = TOL[io]["fwd"], TOL[io]["bwd"]
    errs = {"y": normwise(y, ref_y(rf.y, io)), "last_state": normwise(last, rf.last_state)}
    for k in STATE_GRADS:
        ref = getattr(rb, k)
        if ref is None:
            assert g[k] is None, k
        else:
            errs[k] = normwise(g[k], ref)
    bad = {k: e for k, e in errs.items() if e > (tf if k in ("y", "last_state") else tb)}
    assert not bad, ((Bsz, L, Dch, N), io, terms, softplus, bad, errs)


@pytest.mark.parametrize("i", list(range(12)))
def test_random_decode_step(orc, i):
    """ss_decode_step on random sizes, io types and terms: one step from a
    random state against the oracle's one-step forward from that state."""
    rng = np.random.default_rng(7500 + i)
    N = int(rng.choice([1, 2, 4, 8, 16, 32]))
    io = str(rng.choice(["f32", "bf16", "f16"]))
    Bsz, Dch = int(rng.integers(1, 70)), int(rng.integers(1, 400))
    terms = dict(has_D=bool(rng.integers(0, 2)), has_z=bool(rng.integers(0, 2)), has_bias=bool(rng.integers(0, 2)))
    a_is_log = bool(rng.integers(0, 2))
    x = small_inputs(Bsz, 1, Dch, N, io=io, seed=7600 + i, **terms)
    state0 = rng.normal(size=(Bsz, Dch, N)).astype(np.float32)
    A_in = np.log(-x["A"]).astype(np.float32) if a_is_log else x["A"]
    t = to_device(x, io)
    state = torch.from_numpy(state0).cuda()
    z = None if t["z"] is None else t["z"][:, 0]
    y = ss.ss_decode_step(t["u"][:, 0], t["delta"][:, 0], torch.from_numpy(A_in).cuda(), t["B"][:, 0], t["C"][:, 0],
                          t["D"], z, t["delta_bias"], True, state, a_is_log=a_is_log)
    torch.cuda.synchronize()
    r = orc.fwd(x["u"], x["delta"], None if a_is_log else x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                True, h0=state0, A_log=A_in if a_is_log else None)
    tol = TOL[io]["fwd"]
    assert normwise(y, ref_y(r.y, io)[:, 0]) <= tol, ((Bsz, Dch, N), io, terms, a_is_log)
    assert normwise(state, r.last_state) <= tol, ((Bsz, Dch, N), io, terms, a_is_log)
