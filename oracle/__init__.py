"""ctypes front-end of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may use it; the product path never does.  It
imports nothing from the CUDA package.

The oracle follows the forward formula and the backward formulas of the
Ascend pages "aclnnFlashAttentionUnpaddingScoreGrad" (function description)
and "aclnnFlashAttentionUnpaddingScoreGradV5" (sink / dSink); the C source
states every formula and reading it implements.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, OpenMP over independent units)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        os.makedirs(_LIB_DIR, exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64),
        ("cu_q", ctypes.POINTER(ctypes.c_int64)),
        ("cu_kv", ctypes.POINTER(ctypes.c_int64)),
        ("Nq", ctypes.c_int64), ("Nkv", ctypes.c_int64), ("D", ctypes.c_int64),
        ("scale", ctypes.c_double), ("keep_prob", ctypes.c_double),
        ("pre_tokens", ctypes.c_int64), ("next_tokens", ctypes.c_int64),
        ("sparse_mode", ctypes.c_int64),
        ("drop_mask", ctypes.POINTER(ctypes.c_uint8)),
        ("sink", ctypes.POINTER(ctypes.c_double)),
        ("h_lo", ctypes.c_int64), ("h_hi", ctypes.c_int64),
        ("row_lo", ctypes.POINTER(ctypes.c_int64)),
        ("atten_mask", ctypes.POINTER(ctypes.c_uint8)),
        ("mask_rows", ctypes.c_int64), ("mask_cols", ctypes.c_int64),
        ("prefix", ctypes.POINTER(ctypes.c_int64)),
        ("pse", ctypes.POINTER(ctypes.c_double)),
        ("pse_batch", ctypes.c_int64), ("pse_cols", ctypes.c_int64), ("pse_type", ctypes.c_int64),
        ("Dv", ctypes.c_int64),
    ]


_lib = None


def bind(path: str):
    """Load an oracle shared library and declare its signatures."""
    cdll = ctypes.CDLL(path)
    P = ctypes.POINTER
    dp = P(ctypes.c_double)
    cdll.ora_fwd.argtypes = [P(_Problem), dp, dp, dp, dp, dp, dp]
    cdll.ora_fwd.restype = ctypes.c_int
    cdll.ora_grad.argtypes = [P(_Problem), dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp]
    cdll.ora_grad.restype = ctypes.c_int
    cdll.ora_keep.argtypes = [ctypes.c_int64] * 7
    cdll.ora_keep.restype = ctypes.c_int
    cdll.ora_keep_bit.argtypes = [P(ctypes.c_uint8), ctypes.c_int64]
    cdll.ora_keep_bit.restype = ctypes.c_int
    cdll.ora_mask_base.argtypes = [P(_Problem), ctypes.c_int64]
    cdll.ora_mask_base.restype = ctypes.c_int64
    cdll.ora_keep_at.argtypes = [P(_Problem)] + [ctypes.c_int64] * 5
    cdll.ora_keep_at.restype = ctypes.c_int
    cdll.ora_pse_at.argtypes = [P(_Problem)] + [ctypes.c_int64] * 5
    cdll.ora_pse_at.restype = ctypes.c_double
    return cdll


def lib():
    global _lib
    if _lib is None:
        _lib = bind(build())
    return _lib


def use_library(cdll):
    """Swap the library the wrappers call (tests plant mistakes in copies);
    returns the previous one."""
    global _lib
    prev = _lib
    _lib = cdll
    return prev


def _dptr(a: Optional[np.ndarray]):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


class Problem:
    """Problem description (shapes, scalars, optional sink and dropout bits).

    ``heads`` = (h_lo, h_hi) restricts the computation to those query heads;
    ``row_lo`` (one int per sequence) skips query rows i < row_lo[b].
    ``atten_mask`` is the [S1Max, S2Max] attention-mask matrix (nonzero masks)
    for sparseMode 0 / 1; ``prefix`` the per-sequence prefix N for mode 6.
    ``dv`` is the head dim of value, dy, the output and dV (default ``d``;
    the pages allow qD == kD >= vD).
    """

    def __init__(self, cu_q: Sequence[int], cu_kv: Sequence[int], nq: int, nkv: int, d: int,
                 scale: float, keep_prob: float = 1.0, pre_tokens: int = 2147483647,
                 next_tokens: int = 2147483647, sparse_mode: int = 0,
                 drop_mask: Optional[np.ndarray] = None, sink: Optional[np.ndarray] = None,
                 heads: Optional[Sequence[int]] = None, row_lo: Optional[Sequence[int]] = None,
                 atten_mask: Optional[np.ndarray] = None, prefix: Optional[Sequence[int]] = None,
                 pse: Optional[np.ndarray] = None, pse_type: int = 1, dv: Optional[int] = None):
        self.cu_q = np.ascontiguousarray(cu_q, dtype=np.int64)
        self.cu_kv = np.ascontiguousarray(cu_kv, dtype=np.int64)
        self.nq, self.nkv, self.d = int(nq), int(nkv), int(d)
        self.dv = self.d if dv is None else int(dv)
        assert self.nq % self.nkv == 0
        if not 1 <= self.dv <= self.d:
            raise ValueError("value head dim must be in [1, D] (qD == kD >= vD)")
        self.drop_mask = None if drop_mask is None else np.ascontiguousarray(drop_mask, dtype=np.uint8)
        self.sink = None if sink is None else np.ascontiguousarray(sink, dtype=np.float64)
        self.row_lo = None if row_lo is None else np.ascontiguousarray(row_lo, dtype=np.int64)
        self.atten_mask = None if atten_mask is None else np.ascontiguousarray(atten_mask, dtype=np.uint8)
        self.prefix = None if prefix is None else np.ascontiguousarray(prefix, dtype=np.int64)
        self.pse = None if pse is None else np.ascontiguousarray(pse, dtype=np.float64)
        nb = len(cu_q) - 1
        if self.pse is not None and pse_type in (2, 3):
            # slopes: [B, N] or [N] (one set for every sequence)
            if self.pse.ndim == 1:
                self.pse = self.pse[None, :]
            if self.pse.ndim != 2 or self.pse.shape[0] not in (1, nb) or self.pse.shape[1] != nq:
                raise ValueError("pseType 2 / 3 take slopes of shape [B, Nq] or [Nq]")
        elif self.pse is not None:
            if self.pse.ndim != 4 or self.pse.shape[0] not in (1, nb) or self.pse.shape[1] != nq or \
                    self.pse.shape[2] != 1024:
                raise ValueError("pse is [B or 1, Nq, 1024, S]")
            skv_max = int(np.max(np.diff(np.asarray(cu_kv)))) if nb else 0
            if self.pse.shape[3] < skv_max:
                raise ValueError("pse must cover the longest key sequence")
        if sparse_mode == 1 and self.atten_mask is None:
            raise ValueError("sparseMode 1 needs the attention-mask matrix")
        if sparse_mode == 6 and (self.prefix is None or self.prefix.size != len(cu_q) - 1):
            raise ValueError("sparseMode 6 needs one prefix value per sequence")
        if self.atten_mask is not None:
            if self.atten_mask.ndim != 2:
                raise ValueError("the attention-mask matrix is two-dimensional")
            sq_max = int(np.max(np.diff(np.asarray(cu_q)))) if len(cu_q) > 1 else 0
            skv_max = int(np.max(np.diff(np.asarray(cu_kv)))) if len(cu_kv) > 1 else 0
            if self.atten_mask.shape[0] < sq_max or self.atten_mask.shape[1] < skv_max:
                raise ValueError("the attention-mask matrix must cover the longest sequences")
        h_lo, h_hi = (0, self.nq) if heads is None else heads
        self._c = _Problem(
            len(self.cu_q) - 1,
            self.cu_q.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            self.cu_kv.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            self.nq, self.nkv, self.d, float(scale), float(keep_prob), int(pre_tokens),
            int(next_tokens), int(sparse_mode),
            ctypes.POINTER(ctypes.c_uint8)() if self.drop_mask is None
            else self.drop_mask.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
            _dptr(self.sink), int(h_lo), int(h_hi),
            ctypes.POINTER(ctypes.c_int64)() if self.row_lo is None
            else self.row_lo.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            ctypes.POINTER(ctypes.c_uint8)() if self.atten_mask is None
            else self.atten_mask.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
            0 if self.atten_mask is None else self.atten_mask.shape[0],
            0 if self.atten_mask is None else self.atten_mask.shape[1],
            ctypes.POINTER(ctypes.c_int64)() if self.prefix is None
            else self.prefix.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            ctypes.POINTER(ctypes.c_double)() if self.pse is None
            else self.pse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            0 if self.pse is None else self.pse.shape[0],
            0 if self.pse is None or self.pse.ndim != 4 else self.pse.shape[3],
            int(pse_type), self.dv)

    @property
    def tq(self) -> int:
        return int(self.cu_q[-1])

    @property
    def tkv(self) -> int:
        return int(self.cu_kv[-1])

    def mask_bits(self) -> int:
        sq = np.diff(self.cu_q)
        skv = np.diff(self.cu_kv)
        return int(np.sum(self.nq * sq * skv))

    def mask_base(self, b: int) -> int:
        return int(lib().ora_mask_base(ctypes.byref(self._c), b))


def problem_from_workload(wl, drop_mask=None, sink=None, **kw) -> Problem:
    """Problem for a ``workloads.Workload`` (the sink is passed as fp64)."""
    kw.setdefault("dv", getattr(wl, "dv", None))
    return Problem(wl.cu_q, wl.cu_kv, wl.nq, wl.nkv, wl.d, wl.scale, wl.keep_prob,
                   wl.pre_tokens, wl.next_tokens, wl.sparse_mode, drop_mask,
                   None if sink is None else np.asarray(sink, dtype=np.float64), **kw)


def pse_at(p: Problem, b: int, h: int, i: int, j: int) -> float:
    """The oracle's pse value of (sequence b, head h, row i, column j)."""
    sq = int(p.cu_q[b + 1] - p.cu_q[b])
    return float(lib().ora_pse_at(ctypes.byref(p._c), b, h, sq, i, j))


def keep_at(p: Problem, b: int, i: int, j: int) -> bool:
    """The oracle's keep rule for (sequence b, row i, column j), mask and prefix included."""
    sq = int(p.cu_q[b + 1] - p.cu_q[b])
    skv = int(p.cu_kv[b + 1] - p.cu_kv[b])
    return bool(lib().ora_keep_at(ctypes.byref(p._c), b, sq, skv, i, j))


def keep(mode: int, pre: int, nxt: int, sq: int, skv: int, i: int, j: int) -> bool:
    return bool(lib().ora_keep(mode, pre, nxt, sq, skv, i, j))


def keep_bit(mask: np.ndarray, index: int) -> int:
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    return int(lib().ora_keep_bit(m.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), index))


def _check_shapes(p: Problem, **arrays):
    want = {"q": (p.tq, p.nq, p.d), "k": (p.tkv, p.nkv, p.d), "v": (p.tkv, p.nkv, p.dv),
            "dy": (p.tq, p.nq, p.dv), "out": (p.tq, p.nq, p.dv), "smax": (p.tq, p.nq), "ssum": (p.tq, p.nq)}
    for name, a in arrays.items():
        if a.shape != want[name]:
            raise ValueError(f"{name} has shape {a.shape}, the problem needs {want[name]}")


def fwd(p: Problem, q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """fp64 forward: returns (out [Tq,Nq,Dv], smax [Tq,Nq], ssum [Tq,Nq])."""
    q, k, v = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v))
    _check_shapes(p, q=q, k=k, v=v)
    out = np.zeros((p.tq, p.nq, p.dv))
    smax = np.full((p.tq, p.nq), np.nan)
    ssum = np.full((p.tq, p.nq), np.nan)
    rc = lib().ora_fwd(ctypes.byref(p._c), _dptr(q), _dptr(k), _dptr(v), _dptr(out),
                       _dptr(smax), _dptr(ssum))
    if rc:
        raise MemoryError("oracle forward failed")
    return out, smax, ssum


def grad(p: Problem, q, k, v, dy, out, smax, ssum, want_ds: bool = False):
    """fp64 gradient: returns (dq, dk, dv, dsink[, ds_dense])."""
    q, k, v, dy, out, smax, ssum = (np.ascontiguousarray(x, dtype=np.float64)
                                    for x in (q, k, v, dy, out, smax, ssum))
    _check_shapes(p, q=q, k=k, v=v, dy=dy, out=out, smax=smax, ssum=ssum)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dsink = np.zeros(p.nq)
    ds = np.zeros(p.mask_bits()) if want_ds else None
    rc = lib().ora_grad(ctypes.byref(p._c), _dptr(q), _dptr(k), _dptr(v), _dptr(dy), _dptr(out),
                        _dptr(smax), _dptr(ssum), _dptr(dq), _dptr(dk), _dptr(dv), _dptr(dsink),
                        _dptr(ds))
    if rc:
        raise MemoryError("oracle gradient failed")
    return (dq, dk, dv, dsink, ds) if want_ds else (dq, dk, dv, dsink)


def fwd_grad(p: Problem, q, k, v, dy):
    """End-to-end oracle: its own forward, then the gradient."""
    out, smax, ssum = fwd(p, q, k, v)
    return (out, smax, ssum) + grad(p, q, k, v, dy, out, smax, ssum)
