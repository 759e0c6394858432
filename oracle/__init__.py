"""CPU oracle for the Mamba-1 selective scan -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports it, and it imports nothing from the product.

The arithmetic lives in ``ss_oracle.c`` (plain C, f64, sequential per row);
this module builds it with gcc and marshals numpy arrays into it.  The one
step done here is the A_log parameterisation (mamba-rs ``gpu/backward.rs``
trains A through A_log): A = -exp(A_log) elementwise in f64 before the scan,
and dA_log = dA * A (the chain rule of that map) after it.

Functions follow baracuda-kernels ``selective_scan.rs`` (module doc,
"Algorithm summary": the forward definition; "Shape contract": the layouts)
and the chain rule of that definition for the backward, structured as in
mamba-rs ``gpu/backward.rs`` (B2 gating backward, B3 SSM BPTT with local
gradients then reductions, B4 softplus backward on the raw delta).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "ss_oracle.c")
LIB = os.path.join(_HERE, "libss_oracle.so")

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-Wall", "-Wextra", "-shared", "-fPIC"]


def build(src: str = SRC, out: str = LIB, extra: tuple = ()) -> str:
    """Compile the oracle with gcc (no FMA contraction, IEEE semantics)."""
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src) and not extra:
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, *extra, "-o", tmp, src, "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


@dataclass
class FwdResult:
    y: np.ndarray          # [n_rows, L]  (or [Bsz, L, Dch] when all rows)
    y0: np.ndarray         # pre-gate output, same shape as y
    last_state: np.ndarray  # [n_rows, N] (or [Bsz, Dch, N])


def a_from_log(A_log):
    """A = -exp(A_log), elementwise in f64."""
    return -np.exp(np.asarray(A_log, np.float64))


def dA_log_rows(dA_rows, A_rows):
    """Chain rule of A = -exp(A_log): dA_log = dA * dA/dA_log = dA * A, per row's (d, n)."""
    return dA_rows * A_rows


@dataclass
class BwdResult:
    du: np.ndarray
    ddelta: np.ndarray
    dz: np.ndarray | None
    dA: np.ndarray | None        # [Dch, N] (all rows) -- per-row contributions in dA_rows
    dD: np.ndarray | None
    ddelta_bias: np.ndarray | None
    dB: np.ndarray | None        # [Bsz, L, N]
    dC: np.ndarray | None
    dA_rows: np.ndarray = None   # [n_rows, N]
    dD_rows: np.ndarray = None   # [n_rows]
    dbias_rows: np.ndarray = None
    dh0: np.ndarray | None = None  # [n_rows, N] (or [Bsz, Dch, N]); only when h0 or dlast_state is given


class Oracle:
    """Handle on one compiled copy of the oracle library."""

    def __init__(self, path: str | None = None):
        self.path = path or build()
        self.lib = ctypes.CDLL(self.path)
        self.lib.ss_oracle_fwd.restype = ctypes.c_int
        self.lib.ss_oracle_fwd.argtypes = ([_P] * 8 + [ctypes.c_int] + [_I64] * 4 + [_P, _I64] + [_P] * 3
                                           + [ctypes.c_int, _P])
        self.lib.ss_oracle_bwd.restype = ctypes.c_int
        self.lib.ss_oracle_bwd.argtypes = ([_P] * 8 + [ctypes.c_int, _P] + [_I64] * 4 + [_P, _I64] + [_P] * 8
                                           + [ctypes.c_int, _P, _P, _P])

    @staticmethod
    def _rows(rows, Bsz, Dch):
        if rows is None:
            return None, Bsz * Dch
        r = np.ascontiguousarray(rows, dtype=np.int64)
        return r, r.size

    def fwd(self, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, rows=None,
            nthreads=None, h0=None, A_log=None) -> FwdResult:
        """Forward.  rows=None: every row, outputs shaped like the tensors
        (y [Bsz, L, Dch], last_state [Bsz, Dch, N]); otherwise row ids b*Dch+d and
        outputs [n_rows, L] / [n_rows, N].  h0 [Bsz, Dch, N]: the state before
        t = 0 (None: zero).  A_log given instead of A: A = -exp(A_log)."""
        if A_log is not None:
            A = a_from_log(A_log)
        u, delta, A, B, C, D, z, bias, h0 = map(_f64, (u, delta, A, B, C, D, z, delta_bias, h0))
        Bsz, L, Dch = u.shape
        N = A.shape[1]
        r, n_rows = self._rows(rows, Bsz, Dch)
        y = np.zeros((n_rows, L), np.float64)
        y0 = np.zeros((n_rows, L), np.float64)
        last = np.zeros((n_rows, N), np.float64)
        rc = self.lib.ss_oracle_fwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(bias),
                                    int(bool(softplus)), Bsz, L, Dch, N, _ptr(r), n_rows, _ptr(y), _ptr(y0),
                                    _ptr(last), nthreads or default_threads(), _ptr(h0))
        if rc != 0:
            raise RuntimeError(f"ss_oracle_fwd failed with code {rc}")
        if rows is None:
            y = y.reshape(Bsz, Dch, L).transpose(0, 2, 1).copy()
            y0 = y0.reshape(Bsz, Dch, L).transpose(0, 2, 1).copy()
            last = last.reshape(Bsz, Dch, N)
        return FwdResult(y, y0, last)

    def bwd(self, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, dy=None, rows=None,
            want_dBdC=True, nthreads=None, h0=None, dlast_state=None, A_log=None) -> BwdResult:
        """Backward of sum(dy * y) + sum(dlast_state * last_state).  rows=None:
        every row; dA/dD/ddelta_bias are then summed over batch in order
        b = 0..Bsz-1, and du/ddelta/dz are shaped [Bsz, L, Dch].  With a row
        list, per-row outputs are [n_rows, L] and dB/dC hold the sum over the
        listed rows only.  h0 / dlast_state [Bsz, Dch, N] (None: zero); dh0 is
        returned when either is given.  A_log given instead of A: the scan uses
        A = -exp(A_log) and dA (and dA_rows) hold the gradient of A_log."""
        A_used = a_from_log(A_log) if A_log is not None else A
        u, delta, A, B, C, D, z, bias, dy, h0, dlast = map(
            _f64, (u, delta, A_used, B, C, D, z, delta_bias, dy, h0, dlast_state))
        Bsz, L, Dch = u.shape
        N = A.shape[1]
        r, n_rows = self._rows(rows, Bsz, Dch)
        du = np.zeros((n_rows, L), np.float64)
        dd = np.zeros((n_rows, L), np.float64)
        dz = np.zeros((n_rows, L), np.float64) if z is not None else None
        dA_rows = np.zeros((n_rows, N), np.float64)
        dD_rows = np.zeros(n_rows, np.float64)
        db_rows = np.zeros(n_rows, np.float64)
        dB = np.zeros((Bsz, L, N), np.float64) if want_dBdC else None
        dC = np.zeros((Bsz, L, N), np.float64) if want_dBdC else None
        want_dh0 = h0 is not None or dlast is not None
        dh0 = np.zeros((n_rows, N), np.float64) if want_dh0 else None
        rc = self.lib.ss_oracle_bwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(bias),
                                    int(bool(softplus)), _ptr(dy), Bsz, L, Dch, N, _ptr(r), n_rows, _ptr(du),
                                    _ptr(dd), _ptr(dz), _ptr(dA_rows), _ptr(dD_rows), _ptr(db_rows), _ptr(dB),
                                    _ptr(dC), nthreads or default_threads(), _ptr(h0), _ptr(dlast), _ptr(dh0))
        if rc != 0:
            raise RuntimeError(f"ss_oracle_bwd failed with code {rc}")
        if A_log is not None:  # chain rule of A = -exp(A_log), per row's (d, n)
            d_of_row = (r if r is not None else np.arange(Bsz * Dch)) % Dch
            dA_rows = dA_log_rows(dA_rows, A[d_of_row])
        res = BwdResult(du, dd, dz, None, None, None, dB, dC, dA_rows, dD_rows, db_rows, dh0)
        if rows is None:
            res.du = du.reshape(Bsz, Dch, L).transpose(0, 2, 1).copy()
            res.ddelta = dd.reshape(Bsz, Dch, L).transpose(0, 2, 1).copy()
            if dz is not None:
                res.dz = dz.reshape(Bsz, Dch, L).transpose(0, 2, 1).copy()
            dA = np.zeros((Dch, N), np.float64)
            dDv = np.zeros(Dch, np.float64)
            dbv = np.zeros(Dch, np.float64)
            rA = dA_rows.reshape(Bsz, Dch, N)
            rD = dD_rows.reshape(Bsz, Dch)
            rb = db_rows.reshape(Bsz, Dch)
            for b in range(Bsz):  # fixed order over batch
                dA += rA[b]
                dDv += rD[b]
                dbv += rb[b]
            res.dA = dA
            res.dD = dDv if D is not None else None
            res.ddelta_bias = dbv if bias is not None else None
            if dh0 is not None:
                res.dh0 = dh0.reshape(Bsz, Dch, N)
        return res


_default = None


def get() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
