"""Thin Python binding of the TBE C ABI (include/tbe.h).

Argument marshalling only: every step of forward, batch inversion and
backward runs in libtbe_gb300.so's CUDA kernels.  Torch provides the device
memory, the stream and the host pinned buffers.  There is no fallback: if
the shared library is missing this module raises on load.

The entry points keep the C names (tbe_forward, tbe_preprocess,
tbe_backward_rowwise_adagrad, tbe_query_sizes, tbe_meta_bind).  ``TBE`` is a
convenience owner of the per-problem device buffers (meta, workspace,
status words) that calls them in the usual training order.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtbe_gb300.so")

F32, F16, BF16 = 0, 1, 2
INDEX_I32, INDEX_I64 = 0, 1
LONG_AUTO, LONG_TWO_KERNEL, LONG_FUSED = 0, 1, 2
HIST_AUTO, HIST_OFF, HIST_FORCE = 0, 1, 2
STATUS_WORDS = 4
(FLAG_BAD_OFFSETS, FLAG_FP16_OVERFLOW, FLAG_SORT_TIMEOUT, FLAG_HIST_COUNT, FLAG_MMA_TIMEOUT,
 FLAG_COPY_TIMEOUT) = (0x1, 0x2, 0x4, 0x8, 0x10, 0x20)

_TORCH_DTYPE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}

EXPORTED = ("tbe_config_default", "tbe_query_sizes", "tbe_meta_bind", "tbe_forward",
            "tbe_preprocess", "tbe_backward_rowwise_adagrad", "tbe_select_path",
            "tbe_status_string", "tbe_status_str", "tbe_version", "tbe_preprocess_static",
            "tbe_workspace_bytes", "tbe_meta_bytes", "tbe_selftest_workspace_bytes",
            "tbe_selftest_wait_limit")
SELFTEST_SORT_LOOKBACK, SELFTEST_COPY_WAIT = 0, 1
STATIC_SCRATCH_MAX_N = 1 << 22


class TbeError(RuntimeError):
    pass


P = ctypes.c_void_p
i32, i64 = ctypes.c_int32, ctypes.c_int64


class tbe_config(ctypes.Structure):
    _fields_ = [("sl_threshold", i32), ("chunk", i32), ("long_run_mode", i32), ("hist_mode", i32),
                ("kernel_events", P), ("kernel_names", P), ("n_kernel_events", i32),
                ("kernel_events_used", P), ("key_bytes", i32)]


class tbe_tables(ctypes.Structure):
    _fields_ = [("weights", P), ("table_offset", P), ("table_offset_host", P), ("T", i32),
                ("D", i32), ("dtype", i32), ("layout", P), ("layout_host", P)]


class tbe_batch(ctypes.Structure):
    _fields_ = [("indices", P), ("offsets", P), ("N", i64), ("B", i64),
                ("per_sample_weights", P), ("weighted_tables", P), ("index_type", i32),
                ("bag_layout", P), ("bag_layout_host", P), ("out_size", i64)]


# tbe_table_layout and tbe_bag_layout records, as numpy structured dtypes
TABLE_LAYOUT = np.dtype([("weights_byte_offset", np.int64), ("D", np.int32), ("dtype", np.int32)])
BAG_LAYOUT = np.dtype([("bag_offset", np.int64), ("B", np.int64), ("out_offset", np.int64),
                       ("out_stride", np.int64)])
DTYPE_NAMES = {"f32": F32, "f16": F16, "bf16": BF16}


def _records(host: np.ndarray, device) -> tuple:
    """A host array of records and its device copy (raw bytes)."""
    host = np.ascontiguousarray(host)
    dev = torch.from_numpy(host.view(np.uint8).copy()).to(device)
    return host, dev


class tbe_meta(ctypes.Structure):
    _fields_ = [("bound_N", i64), ("bound_B", i64), ("bound_T", i32), ("path", i32),
                ("payload_is_pos", i32), ("key_bits", i32), ("rows_total", i64),
                ("key_bytes", i32), ("index_type", i32),
                ("sorted_keys", P), ("sorted_vals", P), ("keys_a", P), ("vals_a", P),
                ("keys_b", P), ("vals_b", P), ("bag_of", P), ("unique_keys", P), ("seg_off", P),
                ("counters", P), ("long_run", P), ("long_chunk_base", P), ("chunk_order", P),
                ("arrive", P), ("chunk_desc", P), ("hist", P), ("bytes", ctypes.c_size_t)]


_lib = None


def lib():
    """Load libtbe_gb300.so (built by __graft_entry__.build() or build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        L.tbe_config_default.restype = None
        L.tbe_config_default.argtypes = [P]
        L.tbe_query_sizes.restype = i32
        L.tbe_query_sizes.argtypes = [P, P, P, P, P]
        L.tbe_meta_bind.restype = i32
        L.tbe_meta_bind.argtypes = [P, P, ctypes.c_size_t, P, P, P]
        L.tbe_forward.restype = i32
        L.tbe_forward.argtypes = [P, P, P, P, P, ctypes.c_size_t, P, P, P]
        L.tbe_preprocess.restype = i32
        L.tbe_preprocess.argtypes = [P, P, P, P, ctypes.c_size_t, P, P, P]
        L.tbe_backward_rowwise_adagrad.restype = i32
        L.tbe_backward_rowwise_adagrad.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_float,
                                                   P, ctypes.c_size_t, P, P, P]
        L.tbe_preprocess_static.restype = i32
        L.tbe_preprocess_static.argtypes = [P, P, P, P, P, P]
        L.tbe_select_path.restype = i32
        L.tbe_select_path.argtypes = [P, P, P]
        L.tbe_status_string.restype = ctypes.c_char_p
        L.tbe_status_string.argtypes = [i32]
        L.tbe_version.restype = i32
        L.tbe_version.argtypes = []
        L.tbe_status_str.restype = ctypes.c_char_p
        L.tbe_status_str.argtypes = [i32]
        L.tbe_workspace_bytes.restype = ctypes.c_size_t
        L.tbe_meta_bytes.restype = ctypes.c_size_t
        L.tbe_selftest_workspace_bytes.restype = ctypes.c_size_t
        L.tbe_selftest_workspace_bytes.argtypes = []
        L.tbe_selftest_wait_limit.restype = i32
        L.tbe_selftest_wait_limit.argtypes = [i32, P, ctypes.c_size_t, P, P]
        _lib = L
    return _lib


def _check(st: int):
    if st != 0:
        raise TbeError(f"tbe status {st}: {lib().tbe_status_string(st).decode()}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def config(sl_threshold: int = 256, chunk: int = 256, long_run_mode: int = LONG_AUTO,
           hist_mode: int = HIST_AUTO, key_bytes: int = 0) -> tbe_config:
    c = tbe_config()
    lib().tbe_config_default(ctypes.byref(c))
    c.sl_threshold, c.chunk, c.long_run_mode, c.hist_mode = sl_threshold, chunk, long_run_mode, hist_mode
    c.key_bytes = key_bytes
    return c


class Tables:
    """T embedding tables on the device.

    Uniform: weights [rows_total, D] of one dtype, tables back to back.
    With ``layout`` (one dict per table with keys wbyte, D, dtype -- dtype
    'f32', 'f16' or 'bf16'): weights is a byte buffer and table t's rows of
    D_t elements of its dtype start at byte wbyte."""

    def __init__(self, weights: torch.Tensor, table_offset: Sequence[int], layout=None):
        assert weights.is_cuda and weights.is_contiguous()
        self.weights = weights
        self.table_offset_host = np.ascontiguousarray(np.asarray(table_offset, dtype=np.int64))
        self.table_offset = torch.from_numpy(self.table_offset_host).to(weights.device)
        self.T = len(self.table_offset_host) - 1
        self.layout_host = self.layout_dev = None
        if layout is None:
            assert weights.dim() == 2
            self.D = weights.shape[1]
            dt = _TORCH_DTYPE[weights.dtype]
            lay = lay_h = None
        else:
            rec = np.zeros(self.T, TABLE_LAYOUT)
            for t, L in enumerate(layout):
                rec[t] = (L["wbyte"], L["D"], DTYPE_NAMES[L["dtype"]])
            self.layout_host, self.layout_dev = _records(rec, weights.device)
            self.D = int(rec["D"].max())
            dt = F32
            lay, lay_h = self.layout_dev.data_ptr(), self.layout_host.ctypes.data
        self.c = tbe_tables(weights.data_ptr(), self.table_offset.data_ptr(),
                            self.table_offset_host.ctypes.data, self.T, self.D, dt, lay, lay_h)

    def refresh(self):
        self.c.weights = self.weights.data_ptr()


class Batch:
    """One KeyedJagged CSR batch on the device: indices and offsets both int32
    or both int64.

    With ``bag_layout`` (one dict per table with keys bag_off, B, out_off,
    stride) each table has its own number of bags and its bags' output rows
    lie at out[out_off + b*stride] of a flat out of ``out_size`` floats (B is
    then ignored); required for tables with a layout."""

    def __init__(self, indices: torch.Tensor, offsets: torch.Tensor, B: int,
                 per_sample_weights: Optional[torch.Tensor] = None,
                 weighted_tables: Optional[torch.Tensor] = None, bag_layout=None,
                 out_size: int = 0):
        assert indices.dtype == offsets.dtype and indices.dtype in (torch.int32, torch.int64)
        self.indices, self.offsets, self.B = indices, offsets, int(B)
        self.per_sample_weights, self.weighted_tables = per_sample_weights, weighted_tables
        self.N = int(indices.numel())
        itype = INDEX_I64 if indices.dtype == torch.int64 else INDEX_I32
        self.bag_layout_host = self.bag_layout_dev = None
        self.out_size = int(out_size)
        bl = bl_h = None
        if bag_layout is not None:
            rec = np.zeros(len(bag_layout), BAG_LAYOUT)
            for t, L in enumerate(bag_layout):
                rec[t] = (L["bag_off"], L["B"], L["out_off"], L["stride"])
            self.bag_layout_host, self.bag_layout_dev = _records(rec, indices.device)
            bl, bl_h = self.bag_layout_dev.data_ptr(), self.bag_layout_host.ctypes.data
        self.c = tbe_batch(_ptr(indices), _ptr(offsets), self.N, self.B, _ptr(per_sample_weights),
                           _ptr(weighted_tables), itype, bl, bl_h, self.out_size)


def tbe_query_sizes(tables: Tables, batch: Batch, cfg: Optional[tbe_config] = None):
    mb, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib().tbe_query_sizes(ctypes.byref(tables.c), ctypes.byref(batch.c),
                                 ctypes.byref(cfg) if cfg else None, ctypes.byref(mb),
                                 ctypes.byref(wb)))
    return int(mb.value), int(wb.value)


def tbe_select_path(tables: Tables, batch: Batch, cfg: Optional[tbe_config] = None) -> int:
    return int(lib().tbe_select_path(ctypes.byref(tables.c), ctypes.byref(batch.c),
                                     ctypes.byref(cfg) if cfg else None))


class Meta:
    """A bound tbe_meta and the device buffer it points into."""

    def __init__(self, buf: torch.Tensor, c: tbe_meta):
        self.buf, self.c = buf, c


def tbe_meta_bind(tables: Tables, batch: Batch, cfg: Optional[tbe_config] = None,
                  buf: Optional[torch.Tensor] = None) -> Meta:
    mb, _ = tbe_query_sizes(tables, batch, cfg)
    if buf is None:
        buf = torch.empty(max(mb, 256), dtype=torch.uint8, device=tables.weights.device)
    m = tbe_meta()
    _check(lib().tbe_meta_bind(ctypes.byref(m), buf.data_ptr(), buf.numel(), ctypes.byref(tables.c),
                               ctypes.byref(batch.c), ctypes.byref(cfg) if cfg else None))
    return Meta(buf, m)


def tbe_forward(tables: Tables, batch: Batch, out: torch.Tensor, meta: Optional[Meta],
                workspace: Optional[torch.Tensor], dev_status: torch.Tensor,
                cfg: Optional[tbe_config] = None, stream=None):
    _check(lib().tbe_forward(ctypes.byref(tables.c), ctypes.byref(batch.c), out.data_ptr(),
                             ctypes.byref(meta.c) if meta is not None else None,
                             _ptr(workspace), workspace.numel() if workspace is not None else 0,
                             dev_status.data_ptr(), ctypes.byref(cfg) if cfg else None,
                             _stream(stream)))


def tbe_preprocess(tables: Tables, batch: Batch, meta: Meta, workspace: torch.Tensor,
                   dev_status: torch.Tensor, cfg: Optional[tbe_config] = None, stream=None):
    _check(lib().tbe_preprocess(ctypes.byref(tables.c), ctypes.byref(batch.c), ctypes.byref(meta.c),
                                workspace.data_ptr(), workspace.numel(), dev_status.data_ptr(),
                                ctypes.byref(cfg) if cfg else None, _stream(stream)))


def tbe_preprocess_static(tables: Tables, batch: Batch, meta: Meta, dev_status: torch.Tensor,
                          cfg: Optional[tbe_config] = None, stream=None):
    """Batch inversion without a workspace, for callers that cannot allocate
    device memory at this point (see include/tbe.h); at most 2^22 lookups."""
    _check(lib().tbe_preprocess_static(ctypes.byref(tables.c), ctypes.byref(batch.c),
                                       ctypes.byref(meta.c), dev_status.data_ptr(),
                                       ctypes.byref(cfg) if cfg else None, _stream(stream)))


def tbe_backward_rowwise_adagrad(tables: Tables, batch: Batch, momentum: torch.Tensor,
                                 grad_out: torch.Tensor, meta: Meta, lr: float, eps: float,
                                 workspace: torch.Tensor, dev_status: torch.Tensor,
                                 cfg: Optional[tbe_config] = None, stream=None):
    _check(lib().tbe_backward_rowwise_adagrad(
        ctypes.byref(tables.c), ctypes.byref(batch.c), momentum.data_ptr(), grad_out.data_ptr(),
        ctypes.byref(meta.c), float(lr), float(eps), workspace.data_ptr(), workspace.numel(),
        dev_status.data_ptr(), ctypes.byref(cfg) if cfg else None, _stream(stream)))


def tbe_selftest_wait_limit(kind: int, dev_status: torch.Tensor, stream=None):
    """Run one device wait that nothing ends (see include/tbe.h); the wait
    gives up after one second and sets its flag in dev_status[1]."""
    ws = torch.empty(int(lib().tbe_selftest_workspace_bytes()), dtype=torch.uint8,
                     device=dev_status.device)
    _check(lib().tbe_selftest_wait_limit(int(kind), ws.data_ptr(), ws.numel(), dev_status.data_ptr(),
                                         _stream(stream)))
    return ws


class TBE:
    """Owns meta, workspace and status words for one problem shape.

    ``forward(batch)`` returns the pooled output; with
    ``preprocess_in_forward`` the batch inversion runs inside it (the pages'
    optional placement), otherwise ``backward`` runs it first.
    """

    def __init__(self, tables: Tables, batch: Batch, cfg: Optional[tbe_config] = None,
                 preprocess_in_forward: bool = True):
        self.tables, self.cfg = tables, cfg
        self.preprocess_in_forward = preprocess_in_forward
        dev = tables.weights.device
        mb, wb = tbe_query_sizes(tables, batch, cfg)
        self.workspace = torch.empty(wb, dtype=torch.uint8, device=dev)
        self.meta_buf = torch.empty(max(mb, 256), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(STATUS_WORDS, dtype=torch.int32, device=dev)
        self.meta = tbe_meta_bind(tables, batch, cfg, self.meta_buf)
        self.path = self.meta.c.path

    def forward(self, batch: Batch, out: Optional[torch.Tensor] = None, stream=None):
        if out is None:
            shape = (batch.out_size,) if batch.bag_layout_host is not None else \
                (batch.B, self.tables.T * self.tables.D)
            out = torch.empty(shape, dtype=torch.float32, device=self.tables.weights.device)
        meta = self.meta if (self.preprocess_in_forward or self.path == 2) else None
        tbe_forward(self.tables, batch, out, meta, self.workspace, self.status, self.cfg, stream)
        return out

    def backward(self, batch: Batch, momentum: torch.Tensor, grad_out: torch.Tensor, lr: float,
                 eps: float, stream=None):
        if not self.preprocess_in_forward and self.path == 1:
            tbe_preprocess(self.tables, batch, self.meta, self.workspace, self.status, self.cfg,
                           stream)
        tbe_backward_rowwise_adagrad(self.tables, batch, momentum, grad_out, self.meta, lr, eps,
                                     self.workspace, self.status, self.cfg, stream)

    def counters(self):
        """(num_unique, n_valid, num_long, num_chunks) from the device (synchronises)."""
        return tuple(int(x) for x in meta_view(self.meta, "counters", 4).cpu())


def meta_view(meta: Meta, name: str, n: int, dtype=torch.int32) -> torch.Tensor:
    """Device tensor view of n elements of one meta array (a slice of meta.buf)."""
    ptr = getattr(meta.c, name)
    if not ptr:
        raise TbeError(f"meta array {name} is not bound for this path")
    off = ptr - meta.buf.data_ptr()
    esz = torch.empty(0, dtype=dtype).element_size()
    return meta.buf[off:off + n * esz].view(dtype)
