"""C-ABI checks that need no GPU: the library loads, exports every function
include/ss.h declares, and rejects bad arguments before touching CUDA.

Every call below fails validation, which happens before the first CUDA
runtime call, so these run on a machine without a GPU.
"""

import os
import re

import pytest

import mamba_selective_scan_fwd_gb300 as ss
from mamba_selective_scan_fwd_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

OK, INVALID, UNSUPPORTED, WS_SMALL = 0, 1, 2, 3
FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call here fails validation first


def declared_functions():
    names = set()
    for h in os.listdir(INCLUDE):
        if h.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
            names.update(re.findall(r"\b(ss_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_matches_binding_exports():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = ss.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.ss_abi_version() == binding.ABI_VERSION == 7


def test_status_strings():
    for code in range(7):
        assert len(ss.status_string(code)) >= 2
    assert "unknown" in ss.status_string(99)


def test_selftest_wait_limit_checked_before_any_launch():
    # the limit is validated before the first CUDA call
    assert ss.lib().ss_selftest_wait_timeout(-1, None) == INVALID
    assert ss.lib().ss_selftest_wait_timeout(2_000_000_001, None) == INVALID


def test_copies_only_switch_round_trips():
    prev = ss.set_copies_only(True)
    try:
        assert ss.set_copies_only(True) is True
        assert ss.set_copies_only(False) is True
        assert ss.set_copies_only(False) is False
    finally:
        ss.set_copies_only(prev)


def test_workspace_queries_are_pure_and_sized():
    a = ss.bwd_workspace_bytes(4, 4096, 5120, 16, ss.SS_BF16)
    assert a == ss.bwd_workspace_bytes(4, 4096, 5120, 16, ss.SS_BF16) > 0
    assert ss.fwd_workspace_bytes(4, 4096, 4864, 16, ss.SS_BF16) == 0  # 4 whole rounds of units: one chunk each
    # 640 units: the 32 past 4 whole rounds are cut in time and carry chunk summaries
    assert 0 < ss.fwd_workspace_bytes(4, 4096, 5120, 16, ss.SS_BF16) <= 2 << 20
    assert ss.fwd_workspace_bytes(1, 131072, 1024, 16, ss.SS_BF16) > 0  # long sequence: chunk carries
    assert ss.fwd_workspace_bytes(1, 8, 8, 3, ss.SS_F32) == 0  # unsupported N
    assert ss.bwd_workspace_bytes(0, 8, 8, 4, ss.SS_F32) == 0
    assert ss.fwd_workspace_bytes(1, 8, 8, 4, ss.SS_F16) == 0


def _fwd(**kw):
    a = dict(u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, softplus=1, y=FAKE, last=None,
             Bsz=2, L=16, Dch=8, N=4, dtype=0, ws=None, wsb=0, stream=None)
    a.update(kw)
    return ss.lib().ss_fwd(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"], a["softplus"], a["y"],
                           a["last"], a["Bsz"], a["L"], a["Dch"], a["N"], a["dtype"], a["ws"], a["wsb"], a["stream"])


def _bwd(**kw):
    a = dict(u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, softplus=1, dy=FAKE, du=FAKE,
             dd=FAKE, dA=FAKE, dB=FAKE, dC=FAKE, dD=None, dz=None, dbias=None, Bsz=2, L=16, Dch=8, N=4, dtype=0,
             ws=None, wsb=0, stream=None)
    a.update(kw)
    return ss.lib().ss_bwd(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"], a["softplus"],
                           a["dy"], a["du"], a["dd"], a["dA"], a["dB"], a["dC"], a["dD"], a["dz"], a["dbias"], a["Bsz"],
                           a["L"], a["Dch"], a["N"], a["dtype"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(Bsz=-1), INVALID), (dict(L=-3), INVALID), (dict(Dch=-1), INVALID), (dict(N=-1), INVALID),
    (dict(dtype=3), UNSUPPORTED), (dict(dtype=7), UNSUPPORTED), (dict(N=3), UNSUPPORTED), (dict(N=0), UNSUPPORTED),
    (dict(N=64), UNSUPPORTED), (dict(u=None), INVALID), (dict(delta=None), INVALID), (dict(A=None), INVALID),
    (dict(B=None), INVALID), (dict(C=None), INVALID), (dict(y=None), INVALID),
    (dict(u=FAKE + 4), UNSUPPORTED), (dict(B=FAKE + 2), UNSUPPORTED), (dict(D=FAKE + 8), UNSUPPORTED),
    (dict(last=FAKE + 12), UNSUPPORTED),
    (dict(Bsz=1, L=131072, Dch=1024, N=16, dtype=2), WS_SMALL),
])
def test_fwd_rejects(kw, code):
    assert _fwd(**kw) == code


def _fwd_save(**kw):
    a = dict(u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, softplus=1, y=FAKE, last=None,
             saved=FAKE, savedb=1 << 30, Bsz=2, L=16, Dch=8, N=4, dtype=0, ws=None, wsb=0, stream=None)
    a.update(kw)
    return ss.lib().ss_fwd_save(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"], a["softplus"],
                                a["y"], a["last"], a["saved"], a["savedb"], a["Bsz"], a["L"], a["Dch"], a["N"],
                                a["dtype"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(Bsz=-1), INVALID), (dict(dtype=3), UNSUPPORTED), (dict(N=3), UNSUPPORTED), (dict(y=None), INVALID),
    (dict(saved=None), WS_SMALL), (dict(saved=FAKE + 8), UNSUPPORTED), (dict(savedb=0), WS_SMALL),
])
def test_fwd_save_rejects(kw, code):
    assert _fwd_save(**kw) == code


def test_saved_sizes():
    # one f32 state of N per (b, d) row every 8 steps of L rounded up to 32, however the plan cuts time,
    # then (at a 256-byte boundary) the forward's pre-gate readout y0, f32 [B, L, D]
    def up(x):
        return -(-x // 256) * 256

    assert ss.saved_bytes(4, 4096, 5120, 16, ss.SS_BF16) == up(4 * 5120 * (4096 // 8) * 16 * 4) + 4 * 4096 * 5120 * 4
    assert ss.saved_bytes(1, 131072, 1024, 16, ss.SS_BF16) == up(1024 * (131072 // 8) * 16 * 4) + 131072 * 1024 * 4
    assert ss.saved_bytes(1, 300, 3, 16, ss.SS_F32) == up(32 * (320 // 8) * 16 * 4) + 300 * 3 * 4
    # channels are stored in whole tiles (64 for N = 4, so 8 channels take a tile): 2 x 64 x 4 slots x 4 states
    assert ss.saved_bytes(2, 16, 8, 4, ss.SS_F32) == up(2 * 64 * (32 // 8) * 4 * 4) + 2 * 16 * 8 * 4
    # 16-channel tiles for N = 32
    assert ss.saved_bytes(1, 64, 20, 32, ss.SS_F32) == up(32 * (64 // 8) * 32 * 4) + 64 * 20 * 4
    assert ss.saved_bytes(0, 16, 8, 4, ss.SS_F32) == 0
    assert _fwd_save(savedb=ss.saved_bytes(2, 16, 8, 4, 0) - 1) == WS_SMALL
    # the saved-state backward needs no room for the states
    full = ss.bwd_workspace_bytes(4, 4096, 5120, 16, ss.SS_BF16)
    part = ss.bwd_saved_workspace_bytes(4, 4096, 5120, 16, ss.SS_BF16)
    assert 0 < part <= full - ss.saved_bytes(4, 4096, 5120, 16, ss.SS_BF16)


def test_plan_info_counts():
    # 640 units over 152 SMs: 608 one-chunk units, the last 32 cut into 19 chunks
    p = ss.plan_info(4, 4096, 5120, 16, ss.SS_BF16)
    assert p == {"chunks": 19, "fwd_kernels": 3, "bwd_kernels": 9, "bwd_saved_kernels": 6,
                 "segments": [(608, 1), (32, 19)]}
    # 608 units: a whole number of rounds, no split
    p = ss.plan_info(4, 4096, 4864, 16, ss.SS_BF16)
    assert p == {"chunks": 1, "fwd_kernels": 1, "bwd_kernels": 4, "bwd_saved_kernels": 3, "segments": [(608, 1)]}
    q = ss.plan_info(1, 131072, 1024, 16, ss.SS_BF16)
    assert q["chunks"] > 1 and q["fwd_kernels"] == 2 and q["bwd_kernels"] == 7 and q["bwd_saved_kernels"] == 5
    assert q["segments"] == [(32, q["chunks"])]
    e = ss.plan_info(0, 16, 8, 4, 0)
    assert e["fwd_kernels"] == 0 and e["segments"] == []


def test_fwd_workspace_too_small_reports_before_launch():
    need = ss.fwd_workspace_bytes(1, 131072, 1024, 16, 2)
    assert need > 0
    assert _fwd(Bsz=1, L=131072, Dch=1024, N=16, dtype=2, ws=FAKE, wsb=need - 256) == WS_SMALL


@pytest.mark.parametrize("kw,code", [
    (dict(Bsz=-1), INVALID), (dict(dtype=3), UNSUPPORTED), (dict(N=5), UNSUPPORTED),
    (dict(D=FAKE), INVALID), (dict(dD=FAKE), INVALID),            # D <-> dD presence must match
    (dict(z=FAKE), INVALID), (dict(dz=FAKE), INVALID),            # z <-> dz
    (dict(bias=FAKE), INVALID), (dict(dbias=FAKE), INVALID),      # delta_bias <-> ddelta_bias
    (dict(dy=None), INVALID), (dict(du=None), INVALID), (dict(dd=None), INVALID), (dict(dA=None), INVALID),
    (dict(dB=None), INVALID), (dict(dC=None), INVALID),
    (dict(dB=FAKE + 4), UNSUPPORTED), (dict(dy=FAKE + 2), UNSUPPORTED),
    (dict(), WS_SMALL),                                            # no workspace given
])
def test_bwd_rejects(kw, code):
    assert _bwd(**kw) == code


def _bwd_saved(**kw):
    a = dict(u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, softplus=1, dy=FAKE, saved=FAKE,
             savedb=1 << 30, du=FAKE, dd=FAKE, dA=FAKE, dB=FAKE, dC=FAKE, dD=None, dz=None, dbias=None, Bsz=2, L=16,
             Dch=8, N=4, dtype=0, ws=FAKE, wsb=1 << 30, stream=None)
    a.update(kw)
    return ss.lib().ss_bwd_saved(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"],
                                 a["softplus"], a["dy"], a["saved"], a["savedb"], a["du"], a["dd"], a["dA"], a["dB"],
                                 a["dC"], a["dD"], a["dz"], a["dbias"], a["Bsz"], a["L"], a["Dch"], a["N"], a["dtype"],
                                 a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(Bsz=-1), INVALID), (dict(N=5), UNSUPPORTED), (dict(D=FAKE), INVALID), (dict(du=None), INVALID),
    (dict(saved=None), WS_SMALL), (dict(savedb=16), WS_SMALL), (dict(saved=FAKE + 4), UNSUPPORTED),
    (dict(ws=None), WS_SMALL), (dict(wsb=16), WS_SMALL),
])
def test_bwd_saved_rejects(kw, code):
    assert _bwd_saved(**kw) == code


def test_bwd_workspace_one_byte_short():
    need = ss.bwd_workspace_bytes(2, 16, 8, 4, 0)
    assert _bwd(ws=FAKE, wsb=need - 1) == WS_SMALL


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        binding.lib()


def test_product_does_not_import_oracle():
    """The CUDA path's sources never reference the oracle."""
    pkg = os.path.join(ROOT, "mamba_selective_scan_fwd_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "ss_oracle" not in text, f


def test_profile_events_validation():
    import ctypes

    lib = ss.lib()
    one = (ctypes.c_void_p * 1)(None)
    assert lib.ss_profile_events(one, -1) == INVALID
    assert lib.ss_profile_events(one, 17) == INVALID
    assert lib.ss_profile_events(None, 2) == INVALID
    assert lib.ss_profile_events(one, 1) == INVALID  # a NULL handle
    assert lib.ss_profile_events(None, 0) == OK      # switched off


def test_descriptor_layouts_match_the_header(tmp_path):
    """The ctypes descriptors have the size and field offsets of the C structs."""
    import ctypes
    import subprocess

    fields_f = [f for f, _ in binding.FwdDesc._fields_]
    fields_b = [f for f, _ in binding.BwdDesc._fields_]
    src = ['#include <stdio.h>', '#include <stddef.h>', '#include "ss.h"', "int main(void) {",
           'printf("%zu %zu\\n", sizeof(ss_fwd_desc), sizeof(ss_bwd_desc));']
    src += [f'printf("%zu\\n", offsetof(ss_fwd_desc, {f}));' for f in fields_f]
    src += [f'printf("%zu\\n", offsetof(ss_bwd_desc, {f}));' for f in fields_b]
    src += ["return 0; }"]
    c = tmp_path / "layout.c"
    c.write_text("\n".join(src))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", INCLUDE, "-o", str(exe), str(c)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    sizes, offs = [int(v) for v in out[:2]], [int(v) for v in out[2:]]
    assert sizes == [ctypes.sizeof(binding.FwdDesc), ctypes.sizeof(binding.BwdDesc)]
    want = [getattr(binding.FwdDesc, f).offset for f in fields_f] + [getattr(binding.BwdDesc, f).offset for f in fields_b]
    assert offs == want


def test_ex_entry_points_validate_before_cuda():
    import ctypes

    lib = ss.lib()
    assert lib.ss_fwd_ex(None, None) == INVALID
    assert lib.ss_bwd_ex(None, None) == INVALID
    d = binding.BwdDesc()
    for f in ("u", "delta", "A", "B", "C", "dy", "du", "ddelta", "dA", "dB", "dC", "h0", "workspace"):
        setattr(d, f, FAKE)
    d.workspace_bytes = 1 << 40
    d.Bsz, d.L, d.Dch, d.N, d.dtype, d.softplus = 1, 8, 8, 4, 0, 1
    assert lib.ss_bwd_ex(ctypes.byref(d), None) == INVALID  # h0 given without dh0
    d.h0, d.dh0 = None, FAKE
    assert lib.ss_bwd_ex(ctypes.byref(d), None) == INVALID  # dh0 without h0
    f = binding.FwdDesc()
    for k in ("u", "delta", "A", "B", "C", "y"):
        setattr(f, k, FAKE)
    f.h0 = FAKE + 4  # misaligned
    f.Bsz, f.L, f.Dch, f.N, f.dtype = 1, 8, 8, 4, 0
    assert lib.ss_fwd_ex(ctypes.byref(f), None) == UNSUPPORTED


def test_source_digest_sees_code_not_comments():
    from mamba_selective_scan_fwd_gb300 import build

    a = 'int f(int x) { return x + 1; }  // add one\n/* block\n comment */\nconst char* s = "a // b";\n'
    b = 'int f(int x)\n{\n    return x + 1;\n}\nconst char* s = "a // b";  // kept: it is a string\n'
    assert build._code(a) == build._code(b)
    assert build._code(a) != build._code(a.replace("x + 1", "x + 2"))
    assert '"a // b"' in build._code(a)


def test_binding_checks_before_any_launch():
    """The Python wrappers refuse malformed tensors before calling the library:
    a transposed (non-contiguous) u, a B of another dtype, y = None for the
    entry point that allocates nothing, and tensors that are not on a GPU."""
    import torch

    from mamba_selective_scan_fwd_gb300 import binding

    Bsz, L, Dch, N = 1, 8, 4, 4
    u = torch.zeros((Bsz, L, Dch))
    A = -torch.ones((Dch, N))
    Bm = torch.zeros((Bsz, L, N))
    y = torch.zeros((Bsz, L, Dch))
    ut = torch.zeros((Bsz, Dch, L)).transpose(1, 2)
    with pytest.raises(ValueError, match="contiguous"):
        binding.ss_fwd_noalloc(ut, u, A, Bm, Bm, None, None, None, True, y)
    with pytest.raises(TypeError, match="dtype"):
        binding.ss_fwd_noalloc(u, u, A, Bm.to(torch.float64), Bm, None, None, None, True, y)
    with pytest.raises(ValueError, match="allocates nothing"):
        binding.ss_fwd_noalloc(u, u, A, Bm, Bm, None, None, None, True, None)
    with pytest.raises(ValueError, match="shape"):
        binding.ss_fwd_noalloc(u, u, A, Bm, Bm, None, None, None, True, torch.zeros((Bsz, L, Dch + 1)))
    with pytest.raises(ValueError, match="CUDA"):
        binding.ss_fwd_noalloc(u, u, A, Bm, Bm, None, None, None, True, y)
    with pytest.raises(ValueError, match="CUDA"):
        binding.ss_fwd(u, u, A, Bm, Bm)


def test_rate_probes_check_arguments_before_any_launch():
    import ctypes

    out = ctypes.c_double()
    assert ss.lib().ss_measure_ex2_rate(0, ctypes.byref(out)) == INVALID
    assert ss.lib().ss_measure_ex2_rate(1 << 21, ctypes.byref(out)) == INVALID
    assert ss.lib().ss_measure_ex2_rate(16, None) == INVALID
    assert ss.lib().ss_measure_fma_rate(0, ctypes.byref(out)) == INVALID
    assert ss.lib().ss_measure_fma_rate(1 << 21, ctypes.byref(out)) == INVALID
    assert ss.lib().ss_measure_fma_rate(16, None) == INVALID
