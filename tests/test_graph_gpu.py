"""The training pair (ss_fwd_save + ss_bwd_saved) recorded once in a CUDA
graph and replayed: the library allocates nothing and never synchronises
inside a call, so the recorded kernels replay on new input values and give
the eager calls' results bit for bit."""

import pytest
import torch

import mamba_selective_scan_fwd_gb300 as ss
from mamba_selective_scan_fwd_gb300 import binding
from mamba_selective_scan_fwd_gb300.inputs import small_inputs
from gpu_util import to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(2, 300, 70, 16), (1, 2000, 8, 16)], ids=["one-chunk", "chunked"])
def test_training_pair_replays_from_a_cuda_graph(shape):
    Bsz, L, Dch, N = shape
    io = "bf16"
    t = to_device(small_inputs(Bsz, L, Dch, N, io=io, seed=5000), io)
    dt = binding.dtype_id(t["u"])
    dev = t["u"].device
    y = torch.empty_like(t["u"])
    last = torch.empty((Bsz, Dch, N), dtype=torch.float32, device=dev)
    saved = torch.empty(ss.saved_bytes(Bsz, L, Dch, N, dt), dtype=torch.uint8, device=dev)
    wsf = torch.empty(max(256, ss.fwd_workspace_bytes(Bsz, L, Dch, N, dt)), dtype=torch.uint8, device=dev)
    wsb = torch.empty(ss.bwd_saved_workspace_bytes(Bsz, L, Dch, N, dt), dtype=torch.uint8, device=dev)
    out = {k: torch.empty(v, dtype=torch.float32, device=dev) for k, v in
           {"du": (Bsz, L, Dch), "ddelta": (Bsz, L, Dch), "dA": (Dch, N), "dB": (Bsz, L, N), "dC": (Bsz, L, N),
            "dD": (Dch,), "dz": (Bsz, L, Dch), "ddelta_bias": (Dch,)}.items()}
    args = (t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True)

    def step():
        ss.ss_fwd_save(*args, y=y, last_state=last, saved=saved, workspace=wsf)
        ss.ss_bwd_saved(*args, t["dy"], saved, out=out, workspace=wsb)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # eager warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    # new input values in the same buffers, then: replay vs eager
    fresh = to_device(small_inputs(Bsz, L, Dch, N, io=io, seed=5001), io)
    for k in ("u", "delta", "B", "C", "z", "dy", "A", "D", "delta_bias"):
        t[k].copy_(fresh[k])
    graph.replay()
    torch.cuda.synchronize()
    got = {"y": y.clone(), "last": last.clone(), **{k: v.clone() for k, v in out.items()}}
    step()
    torch.cuda.synchronize()
    want = {"y": y, "last": last, **out}
    for k in got:
        assert torch.equal(got[k], want[k]), k
