"""Thin ctypes binding over ``libss.so`` (C ABI in include/ss.h).

Argument marshalling only: every step of the scan runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors used as device buffers; the current
torch stream is passed through.  There is no fallback: if the library is
missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libss.so")

SS_F32, SS_F16, SS_BF16 = 0, 1, 2
SS_OK = 0
SS_ERR_DEVICE_TIMEOUT = 5
SS_ERR_STAGING_FALLBACK = 6
STATUS_NAMES = {0: "SS_OK", 1: "SS_ERR_INVALID_PROBLEM", 2: "SS_ERR_UNSUPPORTED", 3: "SS_ERR_WORKSPACE_TOO_SMALL",
                4: "SS_ERR_CUDA", 5: "SS_ERR_DEVICE_TIMEOUT",
                6: "SS_ERR_STAGING_FALLBACK"}

# Every function include/ss.h declares.
EXPORTS = ["ss_fwd", "ss_bwd", "ss_fwd_workspace_bytes", "ss_bwd_workspace_bytes", "ss_plan_info",
           "ss_status_string", "ss_abi_version", "ss_fwd_noalloc", "ss_saved_bytes", "ss_fwd_save",
           "ss_bwd_saved_workspace_bytes", "ss_bwd_saved", "ss_profile_events", "ss_fwd_ex", "ss_bwd_ex",
           "ss_decode_step", "ss_plan_segments", "ss_device_status", "ss_selftest_wait_timeout",
           "ss_set_copies_only", "ss_staging_uses_tma", "ss_measure_ex2_rate",
           "ss_measure_fma_rate"]
ABI_VERSION = 7

# Size of the library-owned scratch behind ss_fwd_noalloc (SS_FWD_NOALLOC_MAX_SCRATCH_BYTES).
FWD_NOALLOC_MAX_SCRATCH_BYTES = 2 << 20


class SSError(RuntimeError):
    def __init__(self, fn, status, text):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}: {text}")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_I32 = ctypes.c_int32


class FwdDesc(ctypes.Structure):
    """ss_fwd_desc of include/ss.h (same field order and types)."""
    _fields_ = [(n, _P) for n in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias", "h0", "y", "last_state",
                                  "saved")] + [
        ("saved_bytes", _SZ), ("workspace", _P), ("workspace_bytes", _SZ),
        ("Bsz", _I64), ("L", _I64), ("Dch", _I64), ("N", _I64),
        ("dtype", _I32), ("softplus", _I32), ("a_is_log", _I32), ("reserved", _I32)]


class BwdDesc(ctypes.Structure):
    """ss_bwd_desc of include/ss.h (same field order and types)."""
    _fields_ = [(n, _P) for n in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias", "h0", "dy", "dlast_state",
                                  "saved")] + [("saved_bytes", _SZ)] + [
        (n, _P) for n in ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias", "dh0", "workspace")] + [
        ("workspace_bytes", _SZ), ("Bsz", _I64), ("L", _I64), ("Dch", _I64), ("N", _I64),
        ("dtype", _I32), ("softplus", _I32), ("a_is_log", _I32), ("reserved", _I32)]


def lib() -> ctypes.CDLL:
    """Load libss.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with mamba_selective_scan_fwd_gb300.build.build() "
                          "(the selective scan has no non-CUDA implementation)")
    L = ctypes.CDLL(LIB_PATH)
    L.ss_fwd.restype = ctypes.c_int
    L.ss_fwd.argtypes = [_P] * 8 + [ctypes.c_int, _P, _P] + [_I64] * 4 + [ctypes.c_int, _P, _SZ, _P]
    L.ss_bwd.restype = ctypes.c_int
    L.ss_bwd.argtypes = [_P] * 8 + [ctypes.c_int] + [_P] * 9 + [_I64] * 4 + [ctypes.c_int, _P, _SZ, _P]
    L.ss_fwd_save.restype = ctypes.c_int
    L.ss_fwd_save.argtypes = [_P] * 8 + [ctypes.c_int, _P, _P, _P, _SZ] + [_I64] * 4 + [ctypes.c_int, _P, _SZ, _P]
    L.ss_bwd_saved.restype = ctypes.c_int
    L.ss_bwd_saved.argtypes = ([_P] * 8 + [ctypes.c_int, _P, _P, _SZ] + [_P] * 8 + [_I64] * 4 +
                               [ctypes.c_int, _P, _SZ, _P])
    for fn in ("ss_fwd_workspace_bytes", "ss_bwd_workspace_bytes", "ss_saved_bytes", "ss_bwd_saved_workspace_bytes"):
        getattr(L, fn).restype = _SZ
        getattr(L, fn).argtypes = [_I64] * 4 + [ctypes.c_int]
    L.ss_plan_info.restype = ctypes.c_int
    L.ss_plan_info.argtypes = [_I64] * 4 + [ctypes.c_int, _P, _P, _P, _P]
    L.ss_plan_segments.restype = ctypes.c_int
    L.ss_plan_segments.argtypes = [_I64] * 4 + [ctypes.c_int, _P, _P, _P]
    L.ss_profile_events.restype = ctypes.c_int
    L.ss_profile_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
    L.ss_status_string.restype = ctypes.c_char_p
    L.ss_status_string.argtypes = [ctypes.c_int]
    L.ss_abi_version.restype = ctypes.c_int
    L.ss_abi_version.argtypes = []
    L.ss_fwd_noalloc.restype = ctypes.c_int
    L.ss_fwd_noalloc.argtypes = [_P] * 8 + [ctypes.c_int, _P, _P] + [_I64] * 4 + [ctypes.c_int, _P]
    L.ss_fwd_ex.restype = ctypes.c_int
    L.ss_fwd_ex.argtypes = [ctypes.POINTER(FwdDesc), _P]
    L.ss_bwd_ex.restype = ctypes.c_int
    L.ss_bwd_ex.argtypes = [ctypes.POINTER(BwdDesc), _P]
    L.ss_device_status.restype = ctypes.c_int
    L.ss_device_status.argtypes = [_P]
    L.ss_selftest_wait_timeout.restype = ctypes.c_int
    L.ss_selftest_wait_timeout.argtypes = [_I64, _P]
    L.ss_set_copies_only.restype = ctypes.c_int
    L.ss_set_copies_only.argtypes = [ctypes.c_int]
    L.ss_measure_ex2_rate.restype = ctypes.c_int
    L.ss_measure_ex2_rate.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
    L.ss_measure_fma_rate.restype = ctypes.c_int
    L.ss_measure_fma_rate.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
    L.ss_staging_uses_tma.restype = ctypes.c_int
    L.ss_staging_uses_tma.argtypes = [_I64] * 4 + [ctypes.c_int]
    L.ss_decode_step.restype = ctypes.c_int
    L.ss_decode_step.argtypes = [_P] * 8 + [ctypes.c_int, ctypes.c_int, _P, _P] + [_I64] * 3 + [ctypes.c_int, _P]
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().ss_status_string(int(status)).decode()


def _check(fn, rc):
    if rc != SS_OK:
        raise SSError(fn, rc, status_string(rc))


def dtype_id(t) -> int:
    import torch

    if t.dtype == torch.float32:
        return SS_F32
    if t.dtype == torch.bfloat16:
        return SS_BF16
    if t.dtype == torch.float16:
        return SS_F16
    raise TypeError(f"unsupported io dtype {t.dtype}")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def stream_handle(stream=None, device=None):
    """The CUDA stream handle of ``stream``, or of the current stream of ``device``
    (the current device when None)."""
    import torch

    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


class _on_device:
    """Run a library call with the tensors' GPU as the current device: the library
    launches on the current device and reads its per-device state there, so the
    tensors, the stream and the current device must agree.  A caller's stream on
    another device is refused."""

    def __init__(self, t, stream):
        import torch

        if t.device.type != "cuda":
            raise ValueError(f"tensors must be CUDA tensors, got {t.device}")
        if stream is not None and stream.device != t.device:
            raise ValueError(f"stream is on {stream.device}, the tensors on {t.device}")
        self._ctx = torch.cuda.device(t.device)

    def __enter__(self):
        self._ctx.__enter__()
        return self

    def __exit__(self, *exc):
        return self._ctx.__exit__(*exc)


def _require(t, name, shape, dtype, device):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype} != {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def fwd_workspace_bytes(Bsz, L, Dch, N, dtype) -> int:
    return int(lib().ss_fwd_workspace_bytes(Bsz, L, Dch, N, dtype))


def bwd_workspace_bytes(Bsz, L, Dch, N, dtype) -> int:
    return int(lib().ss_bwd_workspace_bytes(Bsz, L, Dch, N, dtype))


def saved_bytes(Bsz, L, Dch, N, dtype) -> int:
    """Bytes of the saved-state buffer ss_fwd_save writes and ss_bwd_saved reads."""
    return int(lib().ss_saved_bytes(Bsz, L, Dch, N, dtype))


def bwd_saved_workspace_bytes(Bsz, L, Dch, N, dtype) -> int:
    return int(lib().ss_bwd_saved_workspace_bytes(Bsz, L, Dch, N, dtype))


def plan_info(Bsz, L, Dch, N, dtype) -> dict:
    """Launch plan of these sizes: the largest chunk count, kernels per call, and the
    segments as (units, chunks) pairs (kernel order: summary passes, then each segment's main pass)."""
    k = ctypes.c_int64()
    nf = ctypes.c_int()
    nb = ctypes.c_int()
    ns = ctypes.c_int()
    _check("ss_plan_info", lib().ss_plan_info(Bsz, L, Dch, N, dtype, ctypes.byref(k), ctypes.byref(nf),
                                              ctypes.byref(nb), ctypes.byref(ns)))
    ns2 = ctypes.c_int(0)
    units, chunks = (ctypes.c_int64 * 2)(), (ctypes.c_int64 * 2)()
    _check("ss_plan_segments", lib().ss_plan_segments(Bsz, L, Dch, N, dtype, ctypes.byref(ns2), units, chunks))
    return {"chunks": k.value, "fwd_kernels": nf.value, "bwd_kernels": nb.value, "bwd_saved_kernels": ns.value,
            "segments": [(units[i], chunks[i]) for i in range(ns2.value)]}


def profile_events(events):
    """Make the following entry-point calls record ``events`` (torch.cuda.Event
    objects with timing enabled, already recorded once so that they exist)
    around their kernels: events[0] before the first, events[i] after the
    i-th.  An empty list switches the recording off."""
    handles = (ctypes.c_void_p * max(1, len(events)))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check("ss_profile_events", lib().ss_profile_events(handles, len(events)))


def device_status(stream=None, device=None) -> int:
    """Wait for ``stream`` (default: the current stream of ``device``), then read and
    clear the library's device status word: SS_OK; SS_ERR_DEVICE_TIMEOUT when a
    kernel gave up waiting for its tile copies since the last read;
    SS_ERR_STAGING_FALLBACK when a kernel staged its tiles without TMA."""
    import torch

    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        rc = lib().ss_device_status(stream_handle(stream, dev))
    if rc not in (SS_OK, SS_ERR_DEVICE_TIMEOUT, SS_ERR_STAGING_FALLBACK):
        _check("ss_device_status", rc)
    return rc


def selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Launch one block whose wait on a barrier nothing completes runs out after
    limit_ns; it records the failure in the device status word."""
    _check("ss_selftest_wait_timeout", lib().ss_selftest_wait_timeout(int(limit_ns), stream_handle(stream)))


def set_copies_only(enable: bool) -> bool:
    """Stage every tile with per-thread asynchronous copies instead of TMA (for the
    following calls of the process); returns the previous setting."""
    return bool(lib().ss_set_copies_only(1 if enable else 0))


def measure_ex2_rate(iters: int = 4096) -> float:
    """MUFU ex2 results per clock cycle per SM on the current device (median over SMs)."""
    r = ctypes.c_double()
    _check("ss_measure_ex2_rate", lib().ss_measure_ex2_rate(int(iters), ctypes.byref(r)))
    return r.value


def measure_fma_rate(iters: int = 4096) -> float:
    """f32 FMA results (packed f32x2 issue) per clock cycle per SM on the current device (median over SMs)."""
    r = ctypes.c_double()
    _check("ss_measure_fma_rate", lib().ss_measure_fma_rate(int(iters), ctypes.byref(r)))
    return r.value


def staging_uses_tma(Bsz, L, Dch, N, dtype) -> bool:
    """Whether the scan kernels of a problem of these sizes stage their tiles with TMA."""
    return bool(lib().ss_staging_uses_tma(Bsz, L, Dch, N, dtype))


def _workspace(nbytes, device, workspace):
    import torch

    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    size = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return workspace, size


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def _fwd_prepare(u, delta, A, B, C, D, z, delta_bias, y, last_state, return_last_state, allocate=True):
    """Check the forward's tensors (shapes, dtypes, contiguity, one device) and, when
    ``allocate``, create y and last_state that are not given."""
    import torch

    Bsz, L, Dch = u.shape
    N = A.shape[1]
    dev = u.device
    io = u.dtype
    _require(u, "u", (Bsz, L, Dch), io, dev)
    _require(delta, "delta", (Bsz, L, Dch), io, dev)
    _require(A, "A", (Dch, N), torch.float32, dev)
    _require(B, "B", (Bsz, L, N), io, dev)
    _require(C, "C", (Bsz, L, N), io, dev)
    if D is not None:
        _require(D, "D", (Dch,), torch.float32, dev)
    if z is not None:
        _require(z, "z", (Bsz, L, Dch), io, dev)
    if delta_bias is not None:
        _require(delta_bias, "delta_bias", (Dch,), torch.float32, dev)
    if y is None:
        if not allocate:
            raise ValueError("y must be given (this entry point allocates nothing)")
        y = torch.empty((Bsz, L, Dch), dtype=io, device=dev)
    _require(y, "y", (Bsz, L, Dch), io, dev)
    if last_state is None and return_last_state and allocate:
        last_state = torch.empty((Bsz, Dch, N), dtype=torch.float32, device=dev)
    if last_state is not None:
        _require(last_state, "last_state", (Bsz, Dch, N), torch.float32, dev)
    return (Bsz, L, Dch, N), y, last_state


def ss_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, y=None, last_state=None,
           return_last_state=True, workspace=None, stream=None):
    """Forward selective scan.  Returns (y, last_state or None)."""
    (Bsz, L, Dch, N), y, last_state = _fwd_prepare(u, delta, A, B, C, D, z, delta_bias, y, last_state,
                                                   return_last_state)
    dt = dtype_id(u)
    with _on_device(u, stream):
        workspace, wsb = _workspace(fwd_workspace_bytes(Bsz, L, Dch, N, dt), u.device, workspace)
        rc = lib().ss_fwd(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias), int(bool(softplus)),
                          _p(y), _p(last_state), Bsz, L, Dch, N, dt, _p(workspace), wsb, stream_handle(stream, u.device))
    _check("ss_fwd", rc)
    return y, last_state


def ss_fwd_save(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, y=None, last_state=None,
                saved=None, return_last_state=True, workspace=None, stream=None):
    """Forward that also fills ``saved`` (uint8 device buffer of saved_bytes(...)
    bytes, allocated when None) with the states ss_bwd_saved restarts from.
    Returns (y, last_state or None, saved)."""
    import torch

    (Bsz, L, Dch, N), y, last_state = _fwd_prepare(u, delta, A, B, C, D, z, delta_bias, y, last_state,
                                                   return_last_state)
    dt = dtype_id(u)
    with _on_device(u, stream):
        if saved is None:
            saved = torch.empty(max(saved_bytes(Bsz, L, Dch, N, dt), 16), dtype=torch.uint8, device=u.device)
        workspace, wsb = _workspace(fwd_workspace_bytes(Bsz, L, Dch, N, dt), u.device, workspace)
        rc = lib().ss_fwd_save(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias),
                               int(bool(softplus)), _p(y), _p(last_state), _p(saved), _nbytes(saved), Bsz, L, Dch, N,
                               dt, _p(workspace), wsb, stream_handle(stream, u.device))
    _check("ss_fwd_save", rc)
    return y, last_state, saved


def ss_fwd_noalloc(u, delta, A, B, C, D, z, delta_bias, softplus, y, last_state=None, stream=None):
    """Forward selective scan that allocates nothing, for callers that cannot
    allocate device memory at the call site: y (and last_state, if given) must
    be preallocated, and the chunk-carry scratch is the library's own fixed
    device array instead of a workspace.  The tensors are checked like ss_fwd's
    (and y=None is refused rather than allocated).  Raises SSError when the
    problem needs more scratch than that array holds."""
    (Bsz, L, Dch, N), y, last_state = _fwd_prepare(u, delta, A, B, C, D, z, delta_bias, y, last_state,
                                                   False, allocate=False)
    dt = dtype_id(u)
    with _on_device(u, stream):
        rc = lib().ss_fwd_noalloc(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias),
                                  int(bool(softplus)), _p(y), _p(last_state), Bsz, L, Dch, N, dt,
                                  stream_handle(stream, u.device))
    _check("ss_fwd_noalloc", rc)
    return y, last_state


GRAD_SHAPES = ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias")


def _bwd_prepare(u, delta, A, B, C, D, z, delta_bias, dy, out):
    import torch

    Bsz, L, Dch = u.shape
    N = A.shape[1]
    dev = u.device
    io = u.dtype
    for name, t, shape, dtype in (("u", u, (Bsz, L, Dch), io), ("delta", delta, (Bsz, L, Dch), io),
                                  ("A", A, (Dch, N), torch.float32), ("B", B, (Bsz, L, N), io),
                                  ("C", C, (Bsz, L, N), io), ("dy", dy, (Bsz, L, Dch), io)):
        _require(t, name, shape, dtype, dev)
    if D is not None:
        _require(D, "D", (Dch,), torch.float32, dev)
    if z is not None:
        _require(z, "z", (Bsz, L, Dch), io, dev)
    if delta_bias is not None:
        _require(delta_bias, "delta_bias", (Dch,), torch.float32, dev)
    f32 = torch.float32
    shapes = {"du": (Bsz, L, Dch), "ddelta": (Bsz, L, Dch), "dA": (Dch, N), "dB": (Bsz, L, N), "dC": (Bsz, L, N),
              "dD": (Dch,), "dz": (Bsz, L, Dch), "ddelta_bias": (Dch,)}
    present = {"dD": D is not None, "dz": z is not None, "ddelta_bias": delta_bias is not None}
    out = dict(out or {})
    for k, shp in shapes.items():
        if not present.get(k, True):
            out[k] = None
            continue
        if out.get(k) is None:
            out[k] = torch.empty(shp, dtype=f32, device=dev)
        _require(out[k], k, shp, f32, dev)
    return (Bsz, L, Dch, N), out


def _grad_ptrs(out):
    return [_p(out[k]) for k in GRAD_SHAPES]


def ss_bwd(u, delta, A, B, C, D, z, delta_bias, softplus, dy, out=None, workspace=None, stream=None):
    """Backward selective scan.  Returns a dict du, ddelta, dA, dB, dC, dD, dz,
    ddelta_bias (f32; the optional ones are None when their input is None)."""
    (Bsz, L, Dch, N), out = _bwd_prepare(u, delta, A, B, C, D, z, delta_bias, dy, out)
    dt = dtype_id(u)
    with _on_device(u, stream):
        workspace, wsb = _workspace(bwd_workspace_bytes(Bsz, L, Dch, N, dt), u.device, workspace)
        rc = lib().ss_bwd(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias), int(bool(softplus)),
                          _p(dy), *_grad_ptrs(out), Bsz, L, Dch, N, dt, _p(workspace), wsb,
                          stream_handle(stream, u.device))
    _check("ss_bwd", rc)
    return out


def ss_bwd_saved(u, delta, A, B, C, D, z, delta_bias, softplus, dy, saved, out=None, workspace=None, stream=None):
    """ss_bwd reading the states ss_fwd_save stored in ``saved`` for the same inputs."""
    (Bsz, L, Dch, N), out = _bwd_prepare(u, delta, A, B, C, D, z, delta_bias, dy, out)
    dt = dtype_id(u)
    with _on_device(u, stream):
        workspace, wsb = _workspace(bwd_saved_workspace_bytes(Bsz, L, Dch, N, dt), u.device, workspace)
        rc = lib().ss_bwd_saved(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias),
                                int(bool(softplus)), _p(dy), _p(saved), _nbytes(saved), *_grad_ptrs(out), Bsz, L, Dch,
                                N, dt, _p(workspace), wsb, stream_handle(stream, u.device))
    _check("ss_bwd_saved", rc)
    return out


def _state_arg(t, name, shape, dev):
    import torch

    if t is not None:
        _require(t, name, shape, torch.float32, dev)
    return t


def ss_fwd_ex(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None, a_is_log=False,
              y=None, last_state=None, return_last_state=True, saved=None, save=False, workspace=None, stream=None):
    """Extended forward (ss_fwd_ex): an initial state ``h0`` [Bsz, Dch, N] f32
    and/or ``A`` given as A_log (``a_is_log``; the scan uses -exp(A_log)).
    With ``save`` (or a ``saved`` buffer) the restart states for ss_bwd_ex are
    kept.  Returns (y, last_state or None, saved or None)."""
    import torch

    (Bsz, L, Dch, N), y, last_state = _fwd_prepare(u, delta, A, B, C, D, z, delta_bias, y, last_state,
                                                   return_last_state)
    _state_arg(h0, "h0", (Bsz, Dch, N), u.device)
    dt = dtype_id(u)
    if saved is None and save:
        saved = torch.empty(max(saved_bytes(Bsz, L, Dch, N, dt), 16), dtype=torch.uint8, device=u.device)
    workspace, wsb = _workspace(fwd_workspace_bytes(Bsz, L, Dch, N, dt), u.device, workspace)
    d = FwdDesc()
    for k, t in (("u", u), ("delta", delta), ("A", A), ("B", B), ("C", C), ("D", D), ("z", z),
                 ("delta_bias", delta_bias), ("h0", h0), ("y", y), ("last_state", last_state), ("saved", saved),
                 ("workspace", workspace)):
        setattr(d, k, None if t is None else t.data_ptr())
    d.saved_bytes, d.workspace_bytes = _nbytes(saved), wsb
    d.Bsz, d.L, d.Dch, d.N = Bsz, L, Dch, N
    d.dtype, d.softplus, d.a_is_log, d.reserved = dt, int(bool(softplus)), int(bool(a_is_log)), 0
    with _on_device(u, stream):
        rc = lib().ss_fwd_ex(ctypes.byref(d), stream_handle(stream, u.device))
    _check("ss_fwd_ex", rc)
    return y, last_state, saved


def ss_bwd_ex(u, delta, A, B, C, D, z, delta_bias, softplus, dy, h0=None, dlast_state=None, a_is_log=False,
              saved=None, out=None, workspace=None, stream=None):
    """Extended backward (ss_bwd_ex) of sum(dy * y) + sum(dlast_state * last_state).
    Returns the ss_bwd dict plus ``dh0`` (present iff h0 is given); with
    ``a_is_log`` dA is the gradient of A_log.  ``saved``: the buffer ss_fwd_ex
    filled for the same inputs (None: the states are recomputed)."""
    import torch

    (Bsz, L, Dch, N), out = _bwd_prepare(u, delta, A, B, C, D, z, delta_bias, dy, out)
    dev = u.device
    _state_arg(h0, "h0", (Bsz, Dch, N), dev)
    _state_arg(dlast_state, "dlast_state", (Bsz, Dch, N), dev)
    if h0 is None:
        out["dh0"] = None
    else:
        if out.get("dh0") is None:
            out["dh0"] = torch.empty((Bsz, Dch, N), dtype=torch.float32, device=dev)
        _require(out["dh0"], "dh0", (Bsz, Dch, N), torch.float32, dev)
    dt = dtype_id(u)
    need = (bwd_saved_workspace_bytes if saved is not None else bwd_workspace_bytes)(Bsz, L, Dch, N, dt)
    workspace, wsb = _workspace(need, dev, workspace)
    d = BwdDesc()
    for k, t in (("u", u), ("delta", delta), ("A", A), ("B", B), ("C", C), ("D", D), ("z", z),
                 ("delta_bias", delta_bias), ("h0", h0), ("dy", dy), ("dlast_state", dlast_state), ("saved", saved),
                 ("workspace", workspace)):
        setattr(d, k, None if t is None else t.data_ptr())
    for k in GRAD_SHAPES + ("dh0",):
        setattr(d, k, None if out[k] is None else out[k].data_ptr())
    d.saved_bytes, d.workspace_bytes = _nbytes(saved), wsb
    d.Bsz, d.L, d.Dch, d.N = Bsz, L, Dch, N
    d.dtype, d.softplus, d.a_is_log, d.reserved = dt, int(bool(softplus)), int(bool(a_is_log)), 0
    with _on_device(u, stream):
        rc = lib().ss_bwd_ex(ctypes.byref(d), stream_handle(stream, dev))
    _check("ss_bwd_ex", rc)
    return out


def ss_decode_step(u, delta, A, B, C, D, z, delta_bias, softplus, state, y=None, a_is_log=False, stream=None):
    """One decoding step in place on ``state`` [Bsz, Dch, N] f32: u, delta, z
    [Bsz, Dch] and B, C [Bsz, N] of the new token (io dtype).  Returns y [Bsz, Dch]."""
    import torch

    Bsz, Dch = u.shape
    N = A.shape[1]
    dev, io = u.device, u.dtype
    for name, t, shape in (("u", u, (Bsz, Dch)), ("delta", delta, (Bsz, Dch)), ("B", B, (Bsz, N)),
                           ("C", C, (Bsz, N))):
        _require(t, name, shape, io, dev)
    _require(A, "A", (Dch, N), torch.float32, dev)
    _require(state, "state", (Bsz, Dch, N), torch.float32, dev)
    if z is not None:
        _require(z, "z", (Bsz, Dch), io, dev)
    for name, t in (("D", D), ("delta_bias", delta_bias)):
        if t is not None:
            _require(t, name, (Dch,), torch.float32, dev)
    if y is None:
        y = torch.empty((Bsz, Dch), dtype=io, device=dev)
    _require(y, "y", (Bsz, Dch), io, dev)
    with _on_device(u, stream):
        rc = lib().ss_decode_step(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias),
                                  int(bool(softplus)), int(bool(a_is_log)), _p(state), _p(y), Bsz, Dch, N,
                                  dtype_id(u), stream_handle(stream, dev))
    _check("ss_decode_step", rc)
    return y
