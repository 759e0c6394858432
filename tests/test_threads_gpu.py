"""Calls from several host threads at once.

Each call's state lives in its arguments and its workspace, so training
pairs (ss_fwd_save + ss_bwd_saved) issued from four host threads on four
streams give the same bits as the same pair run alone.  The measurement
hook's event list belongs to the host thread that set it: another thread's
calls record nothing into it.
"""

import threading

import pytest
import torch

import mamba_selective_scan_fwd_gb300 as ss
from mamba_selective_scan_fwd_gb300 import binding
from mamba_selective_scan_fwd_gb300.inputs import small_inputs
from gpu_util import gpu_fwd, gpu_bwd_saved, gpu_fwd_save, to_device

pytestmark = pytest.mark.gpu

GRADS = ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias")


def _run_threads(fn, n):
    errors, threads = [], []

    def wrap(i):
        try:
            fn(i)
        except BaseException as e:  # reported to the test thread below
            errors.append(e)

    for i in range(n):
        threads.append(threading.Thread(target=wrap, args=(i,)))
        threads[-1].start()
    for th in threads:
        th.join()
    if errors:
        raise errors[0]


def test_concurrent_host_threads_match_sequential():
    # chunked in time (summaries and their workspaces), ragged last channel tile
    x = small_inputs(2, 700, 200, 16, io="bf16", seed=8100)
    t = to_device(x, "bf16")
    y_ref, last_ref, saved_ref = gpu_fwd_save(t)
    g_ref = gpu_bwd_saved(t, saved_ref)
    torch.cuda.synchronize()
    out = [None] * 4

    def work(i):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for _ in range(3):
                y, last, saved = gpu_fwd_save(t)
                g = gpu_bwd_saved(t, saved)
        s.synchronize()
        out[i] = (y, last, g)

    _run_threads(work, 4)
    for y, last, g in out:
        assert torch.equal(y, y_ref) and torch.equal(last, last_ref)
        for k in GRADS:
            assert torch.equal(g[k], g_ref[k]), k


def test_profile_events_are_per_host_thread():
    x = small_inputs(2, 300, 200, 16, io="bf16", seed=8200)
    t = to_device(x, "bf16")
    nf = ss.plan_info(2, 300, 200, 16, ss.SS_BF16)["fwd_kernels"]
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(nf + 1)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    before = evs[0].elapsed_time(evs[-1])
    binding.profile_events(evs)
    try:
        def work(i):
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                gpu_fwd(t)
            s.synchronize()

        _run_threads(work, 1)
        torch.cuda.synchronize()
        # not re-recorded by the other thread's call: the same timestamps
        assert evs[0].elapsed_time(evs[-1]) == before
        # this thread's call records them around its kernels
        gpu_fwd(t)
        torch.cuda.synchronize()
        assert evs[0].elapsed_time(evs[-1]) != before
        assert all(evs[j].elapsed_time(evs[j + 1]) >= 0.0 for j in range(nf))
    finally:
        binding.profile_events([])
