"""ss_fwd_noalloc: the forward for callers that cannot allocate device memory.

Callers such as code replayed from a captured CUDA graph, or a runtime whose
allocator must not be bypassed, cannot hand the library a freshly allocated
workspace.  ss_fwd_noalloc keeps the forward's chunk-carry scratch in a fixed
device array owned by the library instead.  These tests call it through the
C ABI on problems that are cut into many time chunks (so the scratch is
really used, up to exactly its 2 MiB limit), twice in a row with a
different chunked problem run through the same scratch in between, and
require each result to equal, bit for bit, the regular ss_fwd given a
caller-allocated workspace (same plan, same kernels: only the scratch's
address differs, so any read of summaries the call did not write shows).  A
problem that needs more scratch than the array holds must be rejected.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""

import ctypes

import pytest
import torch

import mamba_selective_scan_fwd_gb300 as ss
from mamba_selective_scan_fwd_gb300 import binding
from mamba_selective_scan_fwd_gb300.inputs import small_inputs
from gpu_util import IO_DTYPE, to_device

pytestmark = pytest.mark.gpu


def _noalloc_raw(t, y, last, io):
    """One call of ss_fwd_noalloc through the C ABI with raw device pointers."""
    Bsz, L, Dch = t["u"].shape
    N = t["A"].shape[1]
    p = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())  # noqa: E731
    return ss.lib().ss_fwd_noalloc(p(t["u"]), p(t["delta"]), p(t["A"]), p(t["B"]), p(t["C"]), p(t["D"]), p(t["z"]),
                                   p(t["delta_bias"]), 1, p(y), p(last), Bsz, L, Dch, N,
                                   binding.SS_BF16 if io == "bf16" else binding.SS_F32, binding.stream_handle())


@pytest.mark.parametrize("shape,io", [
    ((1, 1000, 2, 16), "f32"),     # 8 time chunks, small scratch use
    ((1, 32768, 64, 16), "bf16"),  # 256 time chunks: the summaries fill half the 2 MiB scratch
    ((2, 777, 5, 32), "f32"),      # N = 32 over four lanes, ragged last chunk
    ((2, 300, 9913, 16), "bf16"),  # split plan: 608 one-chunk units, then 12 cut into 3 chunks
])
def test_noalloc_matches_regular_forward_twice(shape, io):
    Bsz, L, Dch, N = shape
    need = ss.fwd_workspace_bytes(Bsz, L, Dch, N, binding.SS_BF16 if io == "bf16" else binding.SS_F32)
    assert 0 < need <= binding.FWD_NOALLOC_MAX_SCRATCH_BYTES
    if L == 32768:
        assert need > binding.FWD_NOALLOC_MAX_SCRATCH_BYTES // 2
    x = small_inputs(Bsz, L, Dch, N, io=io, seed=4242 + L)
    t = to_device(x, io)
    y_ref, last_ref = ss.ss_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True)
    # another chunked problem, run through the same scratch between the two calls
    xo = small_inputs(1, 3000, 40, 16, io="f32", seed=99)
    to = to_device(xo, "f32")
    assert ss.fwd_workspace_bytes(1, 3000, 40, 16, binding.SS_F32) > 0
    yo = torch.empty((1, 3000, 40), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(2):
        y = torch.full((Bsz, L, Dch), float("nan"), dtype=IO_DTYPE[io], device="cuda")
        last = torch.full((Bsz, Dch, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc_raw(t, y, last, io) == 0
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref) and torch.equal(last, last_ref)
        assert _noalloc_raw(to, yo, None, "f32") == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 16000 channels x 2 chunks x 16 states of (P, H) summaries need about 4 MB > 2 MiB
    need = ss.fwd_workspace_bytes(1, 256, 16000, 16, binding.SS_F32)
    assert need > binding.FWD_NOALLOC_MAX_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the call is rejected before any launch
    rc = ss.lib().ss_fwd_noalloc(fake, fake, fake, fake, fake, None, None, None, 1, fake, None, 1, 256, 16000, 16,
                                 binding.SS_F32, None)
    assert rc == 3  # SS_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(ss.SSError):
        u = torch.zeros((1, 256, 16000), device="cuda")
        A = -torch.ones((16000, 16), device="cuda")
        Bm = torch.zeros((1, 256, 16), device="cuda")
        binding.ss_fwd_noalloc(u, u, A, Bm, Bm, None, None, None, True, torch.empty_like(u))
