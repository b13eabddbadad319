"""Seeded synthetic TBE workloads.

This module only draws random inputs: table sizes, KeyedJagged CSR
``offsets``/``indices``, per-sample weights, initial weights and upstream
gradients.  It holds none of the method's arithmetic, so both the CPU oracle
(``oracle/``) and the CUDA library are fed from here without sharing code.

Shapes follow the pages' statement of the problem (FBTriton TBE redesign,
accesspath.com, "Backward kernels" / notation: T tables, E rows, D dim,
L pooling factor, B bags) and the KJT layout of the TorchEasyRec analysis
(39.107.221.112 article 1724244, section 1 "KeyedJaggedTensor": all ids of
all features concatenated, one length per sample per feature, key-major).

Index distributions:
  * ``uniform``          rows drawn uniformly from [0, E_t)
  * ``zipf(alpha)``      bounded Zipf  P(k) ~ k^-alpha,       k = 1..E_t
  * ``zm(alpha, q)``     Zipf-Mandelbrot P(k) ~ (k+q)^-alpha, k = 1..E_t
Ranks map to rows through a seeded per-table permutation, so hot rows are
scattered over the table instead of sitting at rows 0..k.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

DTYPES = ("f32", "f16", "bf16")
DTYPE_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


@dataclasses.dataclass
class Workload:
    name: str
    T: int
    B: int
    D: int
    dtype: str
    table_rows: np.ndarray            # int64 [T]
    offsets: np.ndarray               # int32 [T*B+1], CSR, bag (t,b) at t*B+b
    indices: np.ndarray               # int32 [N]
    per_sample_weights: Optional[np.ndarray]   # float32 [N] or None
    weighted_tables: Optional[np.ndarray]      # uint8 [T] or None (all weighted)
    lr: float = 0.01
    eps: float = 1e-8
    w_init: float = 0.01
    seed: int = 0
    desc: str = ""
    # Tables of different shapes in one batch (None: every table has D,
    # dtype and B above).  table_dims / table_dtypes give each table its own
    # row length and weight type; table_B its own number of bags (variable
    # batch size per table).
    table_dims: Optional[np.ndarray] = None
    table_dtypes: Optional[Sequence[str]] = None
    table_B: Optional[np.ndarray] = None

    @property
    def N(self) -> int:
        return int(self.indices.shape[0])

    @property
    def mixed(self) -> bool:
        return self.table_dims is not None or self.table_dtypes is not None or self.table_B is not None

    @property
    def vbe(self) -> bool:
        return self.table_B is not None

    def Dt(self, t: int) -> int:
        return int(self.table_dims[t]) if self.table_dims is not None else self.D

    def dtype_t(self, t: int) -> str:
        return self.table_dtypes[t] if self.table_dtypes is not None else self.dtype

    def Bt(self, t: int) -> int:
        return int(self.table_B[t]) if self.table_B is not None else self.B

    @property
    def NB(self) -> int:
        return int(sum(self.Bt(t) for t in range(self.T)))

    @property
    def Dmax(self) -> int:
        return max(self.Dt(t) for t in range(self.T))

    def layout(self) -> list:
        """Where each table's data lives: per table a dict of
          wbyte    first byte of its rows in the weight buffer (16-byte aligned)
          out_off  index in out / grad_out of its bag 0's first element
          stride   elements from one bag's row to the next in out / grad_out
          bag_off  CSR bag index of its bag 0
          B, D, dtype
        Without VBE, bag rows are rows of a [B, sum D_t] matrix (table t at
        columns sum_{t'<t} D_t'); with VBE, each table's bag rows are packed
        one after another, table after table."""
        lay, wb, bag, col, voff = [], 0, 0, 0, 0
        width = sum(self.Dt(t) for t in range(self.T))
        for t in range(self.T):
            D, dt, B = self.Dt(t), self.dtype_t(t), self.Bt(t)
            if self.vbe:
                out_off, stride = voff, D
                voff += B * D
            else:
                out_off, stride = col, width
                col += D
            lay.append(dict(wbyte=wb, out_off=out_off, stride=stride, bag_off=bag, B=B, D=D, dtype=dt))
            wb += self._table_bytes(t)
            bag += B
        return lay

    def _table_bytes(self, t: int) -> int:
        # one [rows_total, D] array when every table has the same D and dtype;
        # tables of different shapes each start on a 16-byte boundary
        nbytes = int(self.table_rows[t]) * self.Dt(t) * DTYPE_BYTES[self.dtype_t(t)]
        if self.table_dims is None and self.table_dtypes is None:
            return nbytes
        return (nbytes + 15) // 16 * 16

    @property
    def weight_bytes(self) -> int:
        return self.layout()[-1]["wbyte"] + self._table_bytes(self.T - 1)

    @property
    def out_size(self) -> int:
        """Elements of out / grad_out."""
        if self.vbe:
            return int(sum(self.Bt(t) * self.Dt(t) for t in range(self.T)))
        return self.B * int(sum(self.Dt(t) for t in range(self.T)))

    @property
    def table_offset(self) -> np.ndarray:
        off = np.zeros(self.T + 1, dtype=np.int64)
        np.cumsum(self.table_rows, out=off[1:])
        return off

    @property
    def rows_total(self) -> int:
        return int(self.table_rows.sum())

    def torch_dtype(self):
        import torch
        return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[self.dtype]

    def weights(self, device: str = "cpu"):
        """Initial weights ~ U(-w_init, w_init), flat [rows_total, D] in the stored dtype.

        On the CPU the draw is numpy float32 rounded to the stored dtype by
        torch; on a CUDA device it is torch's device generator (used for
        tables too large to draw on the host).  The two draws differ; a test
        feeds one draw to both sides.
        """
        import torch
        rows, D = self.rows_total, self.D
        if device == "cpu":
            rng = np.random.default_rng(self.seed + 101)
            v = rng.uniform(-self.w_init, self.w_init, size=(rows, D)).astype(np.float32)
            return torch.from_numpy(v).to(self.torch_dtype())
        g = torch.Generator(device=device)
        g.manual_seed(self.seed + 101)
        w = torch.empty((rows, D), dtype=self.torch_dtype(), device=device)
        w.uniform_(-self.w_init, self.w_init, generator=g)
        return w

    def weights_mixed(self) -> np.ndarray:
        """Initial weights of tables of different shapes: one byte buffer laid
        out as layout() says, each table's rows ~ U(-w_init, w_init) in its
        own dtype (float32 rounded to it by torch)."""
        import torch
        rng = np.random.default_rng(self.seed + 101)
        buf = np.zeros(self.weight_bytes, np.uint8)
        for t, L in enumerate(self.layout()):
            v = rng.uniform(-self.w_init, self.w_init,
                            size=(int(self.table_rows[t]), L["D"])).astype(np.float32)
            if L["dtype"] == "f32":
                raw = v.view(np.uint8).reshape(-1)
            else:
                tdt = torch.float16 if L["dtype"] == "f16" else torch.bfloat16
                raw = torch.from_numpy(v).to(tdt).view(torch.int16).numpy().view(np.uint8).reshape(-1)
            buf[L["wbyte"]:L["wbyte"] + raw.size] = raw
        return buf

    def grad_out(self) -> np.ndarray:
        """Upstream gradient of the pooled output ~ N(0, 1): float32 [B, T*D]
        (flat [out_size] for tables of different shapes)."""
        rng = np.random.default_rng(self.seed + 202)
        if self.mixed:
            return rng.standard_normal(size=self.out_size, dtype=np.float32)
        return rng.standard_normal(size=(self.B, self.T * self.D), dtype=np.float32)

    def momentum(self) -> np.ndarray:
        """Rowwise Adagrad state, float32 [rows_total], initialised to 0."""
        return np.zeros(self.rows_total, dtype=np.float32)

    def bag_lengths(self) -> np.ndarray:
        return np.diff(self.offsets.astype(np.int64))


# --------------------------------------------------------------------------
# samplers

def _rank_cdf(E: int, dist: tuple) -> Optional[np.ndarray]:
    kind = dist[0]
    if kind == "uniform":
        return None
    k = np.arange(1, E + 1, dtype=np.float64)
    if kind == "zipf":
        p = k ** (-float(dist[1]))
    elif kind == "zm":
        p = (k + float(dist[2])) ** (-float(dist[1]))
    else:
        raise ValueError(f"unknown index distribution {dist!r}")
    c = np.cumsum(p)
    return c / c[-1]


def _draw_rows(rng: np.random.Generator, E: int, n: int, dist: tuple,
               cdf_cache: dict) -> np.ndarray:
    if dist[0] == "uniform":
        return rng.integers(0, E, size=n, dtype=np.int64)
    key = (E, dist)
    if key not in cdf_cache:
        cdf_cache[key] = _rank_cdf(E, dist)
    cdf = cdf_cache[key]
    u = rng.random(n)
    ranks = np.searchsorted(cdf, u, side="right")
    np.minimum(ranks, E - 1, out=ranks)
    perm = rng.permutation(E)
    return perm[ranks]


def _draw_lengths(rng: np.random.Generator, B: int, spec: tuple) -> np.ndarray:
    kind = spec[0]
    if kind == "fixed":
        return np.full(B, int(spec[1]), dtype=np.int64)
    if kind == "poisson":
        lam = float(spec[1])
        lo, hi = (int(spec[2]), int(spec[3])) if len(spec) > 2 else (0, None)
        x = rng.poisson(lam, size=B).astype(np.int64)
        return np.clip(x, lo, hi) if hi is not None else np.maximum(x, lo)
    if kind == "uniform":
        return rng.integers(int(spec[1]), int(spec[2]) + 1, size=B, dtype=np.int64)
    raise ValueError(f"unknown length spec {spec!r}")


def make_workload(name: str, T: int, table_rows: Sequence[int], D: int, dtype: str,
                  B: int, lengths: tuple, dist, seed: int = 0,
                  weighted: Optional[Sequence[bool]] = None, lr: float = 0.01,
                  eps: float = 1e-8, w_init: float = 0.01, oob_frac: float = 0.0,
                  desc: str = "", table_dims: Optional[Sequence[int]] = None,
                  table_dtypes: Optional[Sequence[str]] = None,
                  table_B: Optional[Sequence[int]] = None) -> Workload:
    """Draw one workload.

    ``dist`` is one tuple for all tables or a list of T tuples.  ``weighted``
    (length T) turns on per-sample weights ~U(0,1) for the tables marked True;
    weights are drawn for every lookup and ignored on unweighted tables.
    ``oob_frac`` replaces that fraction of indices with out-of-range values
    (negative or >= E_t), for bounds-check tests.
    """
    assert dtype in DTYPES
    table_rows = np.asarray(table_rows, dtype=np.int64)
    assert table_rows.shape == (T,)
    dists = list(dist) if isinstance(dist, list) else [dist] * T
    rng = np.random.default_rng(seed)
    Bt = [int(x) for x in table_B] if table_B is not None else [B] * T
    lens = np.concatenate([_draw_lengths(rng, Bt[t], lengths) for t in range(T)])
    bag0 = np.concatenate([[0], np.cumsum(Bt)])          # first bag of each table
    offsets = np.zeros(int(bag0[-1]) + 1, dtype=np.int64)
    np.cumsum(lens, out=offsets[1:])
    N = int(offsets[-1])
    if N >= 2**31:
        raise ValueError("workload needs more than 2^31 lookups")
    indices = np.empty(N, dtype=np.int32)
    cdf_cache: dict = {}
    for t in range(T):
        a, b = int(offsets[bag0[t]]), int(offsets[bag0[t + 1]])
        indices[a:b] = _draw_rows(rng, int(table_rows[t]), b - a, dists[t], cdf_cache)
    if oob_frac > 0 and N > 0:
        k = max(1, int(N * oob_frac))
        where = rng.choice(N, size=k, replace=False)
        bad = rng.integers(0, 2, size=k)
        bag = np.searchsorted(offsets, where, side="right") - 1
        tab = np.searchsorted(bag0, bag, side="right") - 1
        big = table_rows[tab] + rng.integers(0, 1000, size=k)
        indices[where] = np.where(bad == 0, -1 - rng.integers(0, 1000, size=k), big).astype(np.int32)
    psw = wt = None
    if weighted is not None and any(weighted):
        psw = rng.uniform(0.0, 1.0, size=N).astype(np.float32)
        wt = np.asarray([1 if w else 0 for w in weighted], dtype=np.uint8)
    return Workload(name=name, T=T, B=B, D=D, dtype=dtype, table_rows=table_rows,
                    offsets=offsets.astype(np.int32), indices=indices,
                    per_sample_weights=psw, weighted_tables=wt, lr=lr, eps=eps,
                    w_init=w_init, seed=seed, desc=desc,
                    table_dims=None if table_dims is None else np.asarray(table_dims, np.int64),
                    table_dtypes=None if table_dtypes is None else list(table_dtypes),
                    table_B=None if table_B is None else np.asarray(table_B, np.int64))


# --------------------------------------------------------------------------
# the five named workloads

# 13 extra demo tables, log-spaced over [10K, 200K] rows (fixed list)
DEMO_EXTRA_ROWS = [int(round(x)) for x in np.geomspace(10_000, 200_000, 13)]
DEMO_ROWS = [1_141_730, 846_812, 461_498] + DEMO_EXTRA_ROWS

# Zipf-Mandelbrot parameters fitted so that T=32 tables of 2M rows with
# B=131072 bags of Poisson(20) lookups give ~3.0M unique (table,row) pairs and
# a hottest row of ~125K lookups (expected values; the realised ones are
# reported by the tests and the bench).
LARGE_ZM_ALPHA = 1.404
LARGE_ZM_Q = 7.32


def tiny(seed: int = 0) -> Workload:
    return make_workload("tiny", T=2, table_rows=[1000, 1000], D=64, dtype="f32", B=256,
                         lengths=("fixed", 8), dist=("uniform",), seed=seed,
                         desc="T=2 E=1000 D=64 f32 B=256 L=8 uniform")


def demo(seed: int = 1, B: int = 4096) -> Workload:
    return make_workload("demo", T=16, table_rows=DEMO_ROWS, D=16, dtype="f32", B=B,
                         lengths=("poisson", 3.0, 0, 50), dist=("zipf", 1.0), seed=seed,
                         desc=f"T=16 E=demo-list D=16 f32 B={B} L~Poisson(3)[0,50] zipf(1.0)")


def mid(seed: int = 2, B: int = 16384, E: int = 1_000_000) -> Workload:
    return make_workload("mid", T=32, table_rows=[E] * 32, D=128, dtype="f16", B=B,
                         lengths=("uniform", 16, 48), dist=("zipf", 1.05), seed=seed,
                         weighted=[t < 16 for t in range(32)],
                         desc=f"T=32 E={E} D=128 f16 B={B} L~U[16,48] zipf(1.05) psw on t<16")


def large(seed: int = 3, B: int = 131_072, E: int = 2_000_000) -> Workload:
    return make_workload("large", T=32, table_rows=[E] * 32, D=128, dtype="bf16", B=B,
                         lengths=("poisson", 20.0), dist=("zm", LARGE_ZM_ALPHA, LARGE_ZM_Q),
                         seed=seed,
                         desc=f"T=32 E={E} D=128 bf16 B={B} L~Poisson(20) "
                              f"zipf-mandelbrot({LARGE_ZM_ALPHA},{LARGE_ZM_Q})")


def hist(seed: int = 4, B: int = 65_536, T: int = 64) -> Workload:
    return make_workload("hist", T=T, table_rows=[64] * T, D=128, dtype="f16", B=B,
                         lengths=("fixed", 64), dist=("uniform",), seed=seed,
                         desc=f"T={T} E=64 D=128 f16 B={B} L=64 uniform")


PRESETS = {"tiny": tiny, "demo": demo, "mid": mid, "large": large, "hist": hist}


def expected_zm_stats(E: int, n: int, alpha: float, q: float) -> tuple:
    """Expected unique rows and hottest-row count for n draws of ZM(alpha,q) on E rows."""
    k = np.arange(1, E + 1, dtype=np.float64)
    p = (k + q) ** (-alpha)
    p /= p.sum()
    uniq = float(np.sum(-np.expm1(n * np.log1p(-p))))
    return uniq, float(n * p[0])
