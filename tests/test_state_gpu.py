"""GPU parity of the extended entry points (ss_fwd_ex / ss_bwd_ex) with the
oracle: an initial state h0, an incoming gradient of last_state, the gradient
dh0, and A given as A_log.  Element by element through the C ABI, on seeded
inputs spanning several blocks, ragged channel tiles and time chunks."""

import numpy as np
import pytest
import torch

import mamba_selective_scan_fwd_gb300 as ss
from mamba_selective_scan_fwd_gb300.inputs import small_inputs
from gpu_util import TOL, normwise, ref_y, to_device

pytestmark = pytest.mark.gpu

SHAPES = [
    (2, 19, 40, 16),    # ragged channel tile, ragged sub-chunk
    (1, 300, 3, 16),    # several time chunks (carries through the chunk summaries)
    (2, 257, 70, 32),   # N = 32, ragged chunk
    (3, 100, 130, 8),   # one-warp blocks
    (1, 33, 5, 1),      # N = 1
    (1, 1000, 2, 16),   # many chunks
]
GRADS = ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias", "dh0")


def make(shape, io, seed):
    Bsz, L, Dch, N = shape
    x = small_inputs(Bsz, L, Dch, N, io=io, seed=seed)
    rng = np.random.default_rng(seed + 7)
    x["A_log"] = np.log(-x["A"]).astype(np.float32)  # A = -exp(A_log) reproduces A = -(n+1) up to rounding
    x["h0"] = rng.normal(size=(Bsz, Dch, N)).astype(np.float32)
    x["dlast"] = rng.normal(size=(Bsz, Dch, N)).astype(np.float32)
    return x


def dev(x, io):
    t = to_device({k: v for k, v in x.items() if k not in ("A_log", "h0", "dlast")}, io)
    for k in ("A_log", "h0", "dlast"):
        t[k] = torch.from_numpy(x[k]).cuda()
    return t


def run_gpu(t, saved_path=True):
    y, last, saved = ss.ss_fwd_ex(t["u"], t["delta"], t["A_log"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                                  True, h0=t["h0"], a_is_log=True, save=saved_path)
    g = ss.ss_bwd_ex(t["u"], t["delta"], t["A_log"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True, t["dy"],
                     h0=t["h0"], dlast_state=t["dlast"], a_is_log=True, saved=saved)
    return y, last, g


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}L{s[1]}D{s[2]}N{s[3]}" for s in SHAPES])
def test_state_and_alog_parity(orc, shape, io):
    x = make(shape, io, 3000 + SHAPES.index(shape))
    t = dev(x, io)
    y, last, g = run_gpu(t)
    torch.cuda.synchronize()
    rf = orc.fwd(x["u"], x["delta"], None, x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True, h0=x["h0"],
                 A_log=x["A_log"])
    rb = orc.bwd(x["u"], x["delta"], None, x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True, dy=x["dy"],
                 h0=x["h0"], dlast_state=x["dlast"], A_log=x["A_log"])
    tf, tb = TOL[io]["fwd"], TOL[io]["bwd"]
    errs = {"y": normwise(y, ref_y(rf.y, io)), "last_state": normwise(last, rf.last_state)}
    for k in GRADS:
        errs[k] = normwise(g[k], getattr(rb, k))
    bad = {k: e for k, e in errs.items() if e > (tf if k in ("y", "last_state") else tb)}
    assert not bad, (bad, errs)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_state_saved_path_bit_identical(io):
    """The backward from saved states equals the recomputing backward bit for bit, h0 included."""
    x = make((2, 300, 70, 16), io, 3100)
    t = dev(x, io)
    _, _, g1 = run_gpu(t, saved_path=True)
    _, _, g0 = run_gpu(t, saved_path=False)
    torch.cuda.synchronize()
    for k in GRADS:
        assert torch.equal(g0[k], g1[k]), k


def test_defaults_match_plain_entry_points():
    """ss_fwd_ex / ss_bwd_ex with no h0, no dlast and plain A are the plain calls, bit for bit."""
    x = small_inputs(2, 150, 40, 16, io="bf16", seed=3200)
    t = to_device(x, "bf16")
    args = (t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True)
    y0, l0 = ss.ss_fwd(*args)
    y1, l1, _ = ss.ss_fwd_ex(*args)
    g0 = ss.ss_bwd(*args, t["dy"])
    g1 = ss.ss_bwd_ex(*args, t["dy"])
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(l0, l1)
    for k in ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias"):
        assert torch.equal(g0[k], g1[k]), k
    assert g1["dh0"] is None


def test_split_sequence_on_gpu():
    """Two calls chained through last_state -> h0 and dh0 -> dlast_state reproduce the
    single call over the whole sequence (to f32 tolerance: the two cut the time axis
    into different chunks)."""
    Bsz, L, Dch, N, L1 = 2, 600, 40, 16, 250
    x = make((Bsz, L, Dch, N), "f32", 3300)
    t = dev(x, "f32")
    seq = ("u", "delta", "B", "C", "z", "dy")
    part = lambda lo, hi: {k: (v[:, lo:hi].contiguous() if k in seq else v) for k, v in t.items()}  # noqa: E731
    t1, t2 = part(0, L1), part(L1, L)
    yf, lf, gf = run_gpu(t)
    y1, l1, s1 = ss.ss_fwd_ex(t1["u"], t1["delta"], t1["A_log"], t1["B"], t1["C"], t1["D"], t1["z"],
                              t1["delta_bias"], True, h0=t1["h0"], a_is_log=True, save=True)
    y2, l2, s2 = ss.ss_fwd_ex(t2["u"], t2["delta"], t2["A_log"], t2["B"], t2["C"], t2["D"], t2["z"],
                              t2["delta_bias"], True, h0=l1, a_is_log=True, save=True)
    g2 = ss.ss_bwd_ex(t2["u"], t2["delta"], t2["A_log"], t2["B"], t2["C"], t2["D"], t2["z"], t2["delta_bias"],
                      True, t2["dy"], h0=l1, dlast_state=t["dlast"], a_is_log=True, saved=s2)
    g1 = ss.ss_bwd_ex(t1["u"], t1["delta"], t1["A_log"], t1["B"], t1["C"], t1["D"], t1["z"], t1["delta_bias"],
                      True, t1["dy"], h0=t1["h0"], dlast_state=g2["dh0"], a_is_log=True, saved=s1)
    torch.cuda.synchronize()
    tol = TOL["f32"]
    assert normwise(torch.cat([y1, y2], 1), yf.cpu().double().numpy()) <= tol["fwd"]
    assert normwise(l2, lf.cpu().double().numpy()) <= tol["fwd"]
    for k in ("du", "ddelta", "dz", "dB", "dC"):
        assert normwise(torch.cat([g1[k], g2[k]], 1), gf[k].cpu().double().numpy()) <= tol["bwd"], k
    for k in ("dA", "dD", "ddelta_bias"):
        assert normwise(g1[k] + g2[k], gf[k].cpu().double().numpy()) <= tol["bwd"], k
    assert normwise(g1["dh0"], gf["dh0"].cpu().double().numpy()) <= tol["bwd"]


def test_empty_sequence_passes_state_through():
    """L = 0: last_state is a copy of h0 and dh0 a copy of dlast_state."""
    Bsz, Dch, N = 2, 5, 4
    u = torch.zeros((Bsz, 0, Dch), device="cuda")
    A = -torch.ones((Dch, N), device="cuda")
    Bm = torch.zeros((Bsz, 0, N), device="cuda")
    h0 = torch.randn((Bsz, Dch, N), device="cuda")
    dl = torch.randn((Bsz, Dch, N), device="cuda")
    _, last, _ = ss.ss_fwd_ex(u, u, A, Bm, Bm, None, None, None, True, h0=h0)
    g = ss.ss_bwd_ex(u, u, A, Bm, Bm, None, None, None, True, u, h0=h0, dlast_state=dl)
    torch.cuda.synchronize()
    assert torch.equal(last, h0) and torch.equal(g["dh0"], dl)
    assert torch.count_nonzero(g["dA"]) == 0
