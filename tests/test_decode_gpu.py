"""GPU parity of the single-step decoding entry point (ss_decode_step)
with the oracle's forward over one step from the given state, and with the
sequence forward it continues."""

import numpy as np
import pytest
import torch

import mamba_selective_scan_fwd_gb300 as ss
from mamba_selective_scan_fwd_gb300.inputs import small_inputs
from gpu_util import TOL, normwise, ref_y, to_device

pytestmark = pytest.mark.gpu

# N = 16 with at least 256 channels runs the channel-major kernel (blocks of 256
# channels x 16 batch rows): (8, 1536, 16) and (37, 300, 16), the latter with a
# ragged channel block and a ragged block of rows
SHAPES = [(3, 70, 16), (2, 5, 32), (4, 33, 8), (1, 9, 4), (2, 7, 2), (3, 11, 1), (8, 1536, 16), (37, 300, 16)]


@pytest.mark.parametrize("a_is_log", [False, True])
@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}D{s[1]}N{s[2]}" for s in SHAPES])
def test_decode_step_parity(orc, shape, io, a_is_log):
    Bsz, Dch, N = shape
    x = small_inputs(Bsz, 1, Dch, N, io=io, seed=4000 + SHAPES.index(shape))
    rng = np.random.default_rng(4100 + SHAPES.index(shape))
    state0 = rng.normal(size=(Bsz, Dch, N)).astype(np.float32)
    A_in = np.log(-x["A"]).astype(np.float32) if a_is_log else x["A"]
    t = to_device(x, io)
    A_dev = torch.from_numpy(A_in).cuda()
    state = torch.from_numpy(state0).cuda()
    y = ss.ss_decode_step(t["u"][:, 0], t["delta"][:, 0], A_dev, t["B"][:, 0], t["C"][:, 0], t["D"], t["z"][:, 0],
                          t["delta_bias"], True, state, a_is_log=a_is_log)
    torch.cuda.synchronize()
    r = orc.fwd(x["u"], x["delta"], None if a_is_log else x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                True, h0=state0, A_log=A_in if a_is_log else None)
    tol = TOL[io]["fwd"]
    assert normwise(y, ref_y(r.y, io)[:, 0]) <= tol
    assert normwise(state, r.last_state) <= tol


@pytest.mark.parametrize("Dch", [40, 272])
def test_decode_steps_continue_a_sequence(Dch):
    """k decoding steps from h0 give the forward of the k-step sequence from h0
    (both decode kernels: 40 channels row-major, 272 channel-major)."""
    Bsz, L, N = 2, 12, 16
    x = small_inputs(Bsz, L, Dch, N, io="f32", seed=4200)
    t = to_device(x, "f32")
    h0 = torch.randn((Bsz, Dch, N), device="cuda")
    y_seq, last, _ = ss.ss_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True,
                                  h0=h0)
    state = h0.clone()
    ys = []
    for i in range(L):
        ys.append(ss.ss_decode_step(t["u"][:, i].contiguous(), t["delta"][:, i].contiguous(), t["A"],
                                    t["B"][:, i].contiguous(), t["C"][:, i].contiguous(), t["D"],
                                    t["z"][:, i].contiguous(), t["delta_bias"], True, state))
    torch.cuda.synchronize()
    assert normwise(torch.stack(ys, 1), y_seq.double().cpu().numpy()) <= TOL["f32"]["fwd"]
    assert normwise(state, last.double().cpu().numpy()) <= TOL["f32"]["fwd"]


def test_decode_empty_batch_is_a_no_op():
    u = torch.zeros((0, 8), device="cuda")
    A = -torch.ones((8, 4), device="cuda")
    Bm = torch.zeros((0, 4), device="cuda")
    state = torch.zeros((0, 8, 4), device="cuda")
    y = ss.ss_decode_step(u, u, A, Bm, Bm, None, None, None, True, state)
    torch.cuda.synchronize()
    assert y.shape == (0, 8)
