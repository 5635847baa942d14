"""fp64 CPU oracle for the Interleaved Head Attention forward pass.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline call it; the product (the CUDA library and its binding) never does.
It shares no code with the CUDA path.  The arithmetic lives in iha_oracle.c;
this module compiles it with gcc and marshals NumPy float64 arrays.

Pinned by tests/test_oracle_pins.py against the pages' worked examples
("注意力机制" eqs. (5.13)-(5.17), (5.23), exercise 5.3), the MHA inclusion
and repeated-token closed forms of "Interleaved Head Attention" Theorem 2,
and invariants (row sums, stacking order, prefix isolation, window limits,
linearity in R and alpha_V).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "iha_oracle.c")
_LIB = os.path.join(_HERE, "libiha_oracle.so")
_lock = threading.Lock()

ERRORS = {0: "ok", -1: "invalid argument", -2: "empty allowed set",
          -3: "non-finite score", -4: "row sum != 1", -5: "out of memory"}


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle C source into a shared library (portable C11, -O2)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _dp(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)) if a is not None else None


def _i64p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)) if a is not None else None


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def default_threads() -> int:
    return os.cpu_count() or 1


class Oracle:
    """The oracle's entry points bound to one compiled copy of iha_oracle.c."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_longlong)
        lib.iha_oracle_forward.argtypes = [dp] * 8 + [ctypes.c_int] * 8 + [i64p, ctypes.c_int, dp, dp, ctypes.c_int]
        lib.iha_oracle_forward.restype = ctypes.c_int
        lib.iha_oracle_forward_from_projections.argtypes = [dp] * 7 + [ctypes.c_int] * 8 + [i64p, ctypes.c_int, dp, dp, ctypes.c_int]
        lib.iha_oracle_forward_from_projections.restype = ctypes.c_int
        lib.iha_oracle_mha.argtypes = [dp] * 4 + [ctypes.c_int] * 6 + [i64p, ctypes.c_int, dp, ctypes.c_int]
        lib.iha_oracle_mha.restype = ctypes.c_int
        lib.iha_oracle_softmax_read.argtypes = [dp, ctypes.POINTER(ctypes.c_ubyte), ctypes.c_int, dp,
                                                ctypes.c_int, dp, dp]
        lib.iha_oracle_softmax_read.restype = ctypes.c_int
        lib.iha_oracle_param_count.argtypes = [ctypes.c_int] * 4
        lib.iha_oracle_param_count.restype = ctypes.c_longlong
        self.lib = lib

    def forward(self, X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, *, H, d, P,
                mask_mode=0, window=0, stack_order=0, rows=None, with_weights=False,
                nthreads=None, projection="c"):
        """IHA forward (Algorithm 1) in float64.

        X [B, N, H*d]; W_s [H*d, H*d]; alpha_s [H, H, P]; R [H, H*P].
        rows: optional flat (b*N + t) output rows (ascending within each b);
        default every row.  Returns out [B, N, H*d] or [len(rows), H*d]; with
        with_weights=True also the attention weights [B, H, P*N, P*N] in
        stacked order (stack_order 0: row j*N + t; 1: row t*P + j).
        projection: "c" computes the per-head projections X W^(m) with the C
        loop; "numpy" takes them from a float64 library matmul (X @ W_s) and
        runs every later step in C -- the same arithmetic, faster on large X.
        """
        X = _f64(X)
        B, N, D = X.shape
        if D != H * d:
            raise ValueError("X's last dimension must equal H*d")
        args = [_f64(a) for a in (W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R)]
        for w in args[:3]:
            if w.shape != (D, H * d):
                raise ValueError("W must be [H*d, H*d]")
        for a in args[3:6]:
            if a.shape != (H, H, P):
                raise ValueError("alpha must be [H, H, P]")
        if args[6].shape != (H, H * P):
            raise ValueError("R must be [H, H*P]")
        sel = None
        if rows is not None:
            sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
            out = np.zeros((len(sel), D), dtype=np.float64)
        else:
            out = np.zeros((B, N, D), dtype=np.float64)
        wts = np.zeros((B, H, P * N, P * N), dtype=np.float64) if with_weights else None
        common = (B, N, H, d, P, mask_mode, window, stack_order,
                  _i64p(sel), len(sel) if sel is not None else 0, _dp(out), _dp(wts),
                  nthreads or default_threads())
        if projection == "c":
            rc = self.lib.iha_oracle_forward(_dp(X), *[_dp(a) for a in args], *common)
        elif projection == "numpy":
            XW = [np.ascontiguousarray(np.matmul(X, w)) for w in args[:3]]
            rc = self.lib.iha_oracle_forward_from_projections(*[_dp(a) for a in XW],
                                                              *[_dp(a) for a in args[3:]], *common)
        else:
            raise ValueError("projection must be 'c' or 'numpy'")
        if rc != 0:
            raise RuntimeError(f"iha_oracle_forward failed: {ERRORS.get(rc, rc)}")
        return (out, wts) if with_weights else out

    def mha(self, X, W_Q, W_K, W_V, *, H, d, mask_mode=0, window=0, rows=None, nthreads=None):
        """Plain multi-head attention (Definition 1) in float64, its own loop."""
        X = _f64(X)
        B, N, D = X.shape
        W = [_f64(w) for w in (W_Q, W_K, W_V)]
        sel = None
        if rows is not None:
            sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
            out = np.zeros((len(sel), D), dtype=np.float64)
        else:
            out = np.zeros((B, N, D), dtype=np.float64)
        rc = self.lib.iha_oracle_mha(_dp(X), *[_dp(w) for w in W], B, N, H, d, mask_mode, window,
                                     _i64p(sel), len(sel) if sel is not None else 0, _dp(out),
                                     nthreads or default_threads())
        if rc != 0:
            raise RuntimeError(f"iha_oracle_mha failed: {ERRORS.get(rc, rc)}")
        return out

    def softmax_read(self, u, allowed, V):
        """Softmax on an allowed set for one query row: u [S] scores,
        allowed [S] bools, V [S, dv] -> (weights [S], output [dv])."""
        u = _f64(u)
        V = _f64(V)
        al = np.ascontiguousarray(np.asarray(allowed, dtype=np.uint8))
        S, dv = V.shape
        a = np.zeros(S, dtype=np.float64)
        o = np.zeros(dv, dtype=np.float64)
        rc = self.lib.iha_oracle_softmax_read(_dp(u), al.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)),
                                              S, _dp(V), dv, _dp(a), _dp(o))
        if rc != 0:
            raise RuntimeError(f"iha_oracle_softmax_read failed: {ERRORS.get(rc, rc)}")
        return a, o

    def param_count(self, D, H, d, P) -> int:
        """Element count of the module's parameters as the oracle consumes them."""
        return int(self.lib.iha_oracle_param_count(D, H, d, P))


_default = None


def get() -> Oracle:
    """The oracle compiled from iha_oracle.c (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def forward(*a, **k):
    return get().forward(*a, **k)


def mha(*a, **k):
    return get().mha(*a, **k)


def softmax_read(*a, **k):
    return get().softmax_read(*a, **k)


def param_count(*a, **k):
    return get().param_count(*a, **k)
