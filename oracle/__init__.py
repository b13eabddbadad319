"""Plain CPU oracle for the TBE hot path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library itself never does, and
the two share no code: the oracle is ``tbe_oracle.c``, built with gcc into
``liboracle_tbe.so`` and called through ctypes on numpy arrays.

Every function here is a thin marshalling wrapper; the arithmetic and its
citations are in ``tbe_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tbe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_tbe.so")
_lib = None

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, f32, f64, u16 = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                   ctypes.c_double, ctypes.c_uint16)
        L.tbe_oracle_forward.restype = i64
        L.tbe_oracle_forward.argtypes = [i32, i64, P, i32, P, P, P, P, i64, P, P, P, i64, P, P, P]
        L.tbe_oracle_preprocess.restype = i64
        L.tbe_oracle_preprocess.argtypes = [i32, i64, P, P, P, P, i64, P, P, P, P, P, P]
        L.tbe_oracle_backward_adagrad.restype = i64
        L.tbe_oracle_backward_adagrad.argtypes = [i32, i64, P, i32, P, P, P, P, P, i64, P, P, P,
                                                  f32, f32, P, P, P]
        L.tbe_oracle_rows_update.restype = i64
        L.tbe_oracle_rows_update.argtypes = [i32, i64, P, i32, P, P, P, i64, P, P, P, f32, f32, P,
                                             i64, P, i64, P, P, P, P]
        L.tbe_oracle_histogram.restype = i64
        L.tbe_oracle_histogram.argtypes = [i32, i64, P, i32, P, P, P, i64, P]
        L.tbe_oracle_offsets_check.restype = i32
        L.tbe_oracle_offsets_check.argtypes = [i64, P, i64, P, P, P]
        for n in ("tbe_oracle_to_half", "tbe_oracle_to_bf16"):
            getattr(L, n).restype = u16
            getattr(L, n).argtypes = [f64]
        for n in ("tbe_oracle_from_half", "tbe_oracle_from_bf16"):
            getattr(L, n).restype = f64
            getattr(L, n).argtypes = [u16]
        _lib = L
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


class _Problem:
    """The batch and table description of a workload as the C oracle takes
    it; the widened arrays are held here while a call reads them."""

    def __init__(self, wl):
        self.T, self.NB, self.N = wl.T, wl.NB, wl.N
        self.Dmax = wl.Dmax
        self.layout = np.array([[L["wbyte"], L["out_off"], L["stride"], L["bag_off"], L["B"], L["D"],
                                 DTYPE_CODE[L["dtype"]]] for L in wl.layout()], np.int64)
        self.to = np.ascontiguousarray(wl.table_offset, dtype=np.int64)
        self.idx = _c(wl.indices, np.int64)
        self.off = _c(wl.offsets, np.int64)
        self.psw = _c(wl.per_sample_weights, np.float32)
        self.wt = _c(wl.weighted_tables, np.uint8)


def _wbytes(W: np.ndarray, wl) -> np.ndarray:
    """Weights as raw storage: a float32 array for f32 tables, uint16 bit
    patterns for f16/bf16 tables, or a byte buffer laid out as wl.layout()
    says (required for tables of different D or dtype)."""
    if W.dtype == np.uint8:
        return np.ascontiguousarray(W)
    assert wl.table_dims is None and wl.table_dtypes is None, \
        "tables of different shapes pass their weights as bytes"
    if wl.dtype == "f32":
        return np.ascontiguousarray(W, dtype=np.float32)
    assert W.dtype == np.uint16, "f16/bf16 weights are passed as uint16 bit patterns"
    return np.ascontiguousarray(W)


def forward(wl, W: np.ndarray, bags: Optional[np.ndarray] = None, want_abs: bool = False):
    """Pooled forward.  Returns (out, abs_sum|None, oob, bad_bags).

    ``W`` is the flat [rows_total, D] table store (float32, or uint16 bits for
    f16/bf16; a byte buffer for tables of different shapes).  out is
    [B, T*D] ([out_size] for tables of different shapes); with ``bags``
    (CSR bag ids) it is [len(bags), Dmax].
    """
    L = lib()
    pr = _Problem(wl)
    W = _wbytes(W, wl)
    if bags is None:
        out = np.zeros(wl.out_size if wl.mixed else (wl.B, wl.T * wl.D), dtype=np.float32)
        nb = 0
    else:
        bags = np.ascontiguousarray(bags, dtype=np.int64)
        out = np.zeros((len(bags), pr.Dmax), dtype=np.float32)
        nb = len(bags)
    ab = np.zeros(out.shape, dtype=np.float64) if want_abs else None
    bad = ctypes.c_int64(0)
    oob = L.tbe_oracle_forward(pr.T, pr.NB, _p(pr.layout), pr.Dmax, _p(W), _p(pr.to), _p(pr.idx),
                               _p(pr.off), pr.N, _p(pr.psw), _p(pr.wt), _p(bags), nb, _p(out),
                               _p(ab), ctypes.addressof(bad))
    return out, ab, int(oob), int(bad.value)


def preprocess(wl):
    """Batch inversion.  Returns dict of sorted_keys, sorted_pos, unique_keys,
    run_len, seg_off (int64) and num_unique, n_valid."""
    L = lib()
    pr = _Problem(wl)
    N = wl.N
    sk = np.zeros(max(N, 1), np.int64)
    sp = np.zeros(max(N, 1), np.int64)
    uk = np.zeros(max(N, 1), np.int64)
    rl = np.zeros(max(N, 1), np.int64)
    so = np.zeros(N + 1, np.int64)
    nv = ctypes.c_int64(0)
    U = L.tbe_oracle_preprocess(pr.T, pr.NB, _p(pr.layout), _p(pr.to), _p(pr.idx), _p(pr.off), N,
                                _p(sk), _p(sp), _p(uk), _p(rl), _p(so), ctypes.addressof(nv))
    nv = int(nv.value)
    return dict(sorted_keys=sk[:nv], sorted_pos=sp[:nv], unique_keys=uk[:U], run_len=rl[:U],
                seg_off=so[:U + 1], num_unique=int(U), n_valid=nv)


def num_runs(wl) -> int:
    """Number of runs (unique touched rows) of the batch inversion."""
    L = lib()
    pr = _Problem(wl)
    return int(L.tbe_oracle_preprocess(pr.T, pr.NB, _p(pr.layout), _p(pr.to), _p(pr.idx), _p(pr.off),
                                       pr.N, None, None, None, None, None, None))


def backward_adagrad(wl, W: np.ndarray, momentum: np.ndarray, grad_out: np.ndarray,
                     want_row_grad: bool = False, want_update_count: bool = False,
                     want_runs: bool = False):
    """Backward + exact rowwise Adagrad, in place on copies.

    Returns (W_new, momentum_new, U, row_grad|None, update_count|None);
    row_grad is dense [rows_total, Dmax] (small problems only).  With
    ``want_runs`` a sixth item is a dict of per-run arrays in ascending key
    order: keys [U], grad [U, Dmax] (the row gradient), abs [U, Dmax] (the
    sum of its terms' magnitudes) and count [U] (lookups of the run).
    """
    L = lib()
    pr = _Problem(wl)
    W = _wbytes(W, wl).copy()
    m = np.ascontiguousarray(momentum, dtype=np.float32).copy()
    go = np.ascontiguousarray(grad_out, dtype=np.float32)
    runs = None
    rg = ra = None
    if want_row_grad or want_runs:
        pre = preprocess(wl)
        U0 = pre["num_unique"]
        rg = np.zeros((max(U0, 1), pr.Dmax), np.float64)
        ra = np.zeros((max(U0, 1), pr.Dmax), np.float64)
        runs = dict(keys=pre["unique_keys"], grad=rg[:U0], abs=ra[:U0], count=pre["run_len"])
    uc = np.zeros(wl.rows_total, np.int32) if want_update_count else None
    U = L.tbe_oracle_backward_adagrad(pr.T, pr.NB, _p(pr.layout), pr.Dmax, _p(W), _p(m), _p(pr.to),
                                      _p(pr.idx), _p(pr.off), pr.N, _p(pr.psw), _p(pr.wt), _p(go),
                                      float(wl.lr), float(wl.eps), _p(rg), _p(ra), _p(uc))
    dense = None
    if want_row_grad:
        dense = np.zeros((wl.rows_total, pr.Dmax), np.float64)
        dense[runs["keys"]] = runs["grad"]
    if want_runs:
        return W, m, int(U), dense, uc, runs
    return W, m, int(U), dense, uc


def rows_update(wl, rows: np.ndarray, W_rows: np.ndarray, mom_rows: np.ndarray,
                grad_out: np.ndarray, want_row_abs: bool = False):
    """Sampled-row backward: rows (sorted distinct linearised keys) with their
    pre-update W rows ([k, D] float32, or uint16 bits; uniform tables) and
    momentum.  Returns (W_rows_new, mom_new, row_grad, counts, n_valid), plus
    row_abs as a sixth item when ``want_row_abs``."""
    L = lib()
    assert not wl.mixed
    pr = _Problem(wl)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    assert np.all(np.diff(rows) > 0)
    k = len(rows)
    Wr = _wbytes(W_rows, wl).copy()
    row_bytes = wl.D * (4 if wl.dtype == "f32" else 2)
    mr = np.ascontiguousarray(mom_rows, dtype=np.float32).copy()
    rg = np.zeros((k, wl.D), np.float64)
    ra = np.zeros((k, wl.D), np.float64) if want_row_abs else None
    cnt = np.zeros(k, np.int64)
    go = np.ascontiguousarray(grad_out, dtype=np.float32)
    nv = L.tbe_oracle_rows_update(pr.T, pr.NB, _p(pr.layout), pr.Dmax, _p(pr.to), _p(pr.idx),
                                  _p(pr.off), pr.N, _p(pr.psw), _p(pr.wt), _p(go), float(wl.lr),
                                  float(wl.eps), _p(rows), k, _p(Wr), row_bytes, _p(mr), _p(rg),
                                  _p(ra), _p(cnt))
    if want_row_abs:
        return Wr, mr, rg, cnt, int(nv), ra
    return Wr, mr, rg, cnt, int(nv)


def histogram(wl, Emax: int = 64) -> np.ndarray:
    """Per-bag row counts, int32 [T, B, Emax] (uniform tables)."""
    L = lib()
    pr = _Problem(wl)
    c = np.zeros((wl.T, wl.B, Emax), np.int32)
    L.tbe_oracle_histogram(pr.T, pr.NB, _p(pr.layout), Emax, _p(pr.to), _p(pr.idx), _p(pr.off), pr.N,
                           _p(c))
    return c


def offsets_check(wl):
    """(malformed, bad_bags, decreasing, span) of the batch's offsets: bags
    not 0 <= start <= end <= N, whether any bag has end < start, whether
    offsets[0] != 0 or offsets[NB] != N."""
    L = lib()
    bad = ctypes.c_int64(0)
    dec = ctypes.c_int32(0)
    sp = ctypes.c_int32(0)
    off = _c(wl.offsets, np.int64)
    m = L.tbe_oracle_offsets_check(wl.NB, _p(off), wl.N, ctypes.addressof(bad), ctypes.addressof(dec),
                                   ctypes.addressof(sp))
    return bool(m), int(bad.value), bool(dec.value), bool(sp.value)


def to_half_bits(x: float) -> int:
    return int(lib().tbe_oracle_to_half(float(x)))


def to_bf16_bits(x: float) -> int:
    return int(lib().tbe_oracle_to_bf16(float(x)))


def from_half_bits(h: int) -> float:
    return float(lib().tbe_oracle_from_half(int(h)))


def from_bf16_bits(h: int) -> float:
    return float(lib().tbe_oracle_from_bf16(int(h)))
