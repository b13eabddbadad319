"""C ABI checks that need no GPU: the library loads, exports every function
include/tbe.h declares, and its host-side argument checks and sizing behave
as documented.  Only host logic runs here (device pointers are fake and are
never dereferenced)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "tbe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(tbe_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    fns = header_functions()
    for name in ("tbe_forward", "tbe_preprocess", "tbe_backward_rowwise_adagrad",
                 "tbe_query_sizes", "tbe_meta_bind"):
        assert name in fns


def test_library_exports_every_declared_symbol():
    from recsys_table_embedding_gb300 import lib
    L = lib()
    for name in header_functions():
        assert hasattr(L, name), name
    assert L.tbe_version() >= 100


FAKE = 0x7f0000000000   # 256-byte aligned fake device address, never dereferenced


class Fake:
    """tables/batch structs with fake device pointers for host-only calls."""

    def __init__(self, T=2, E=1000, D=64, dtype=0, B=16, N=128, psw=False, rows=None, itype=0):
        from recsys_table_embedding_gb300 import tbe
        rows = rows if rows is not None else [E] * T
        self.to = np.zeros(len(rows) + 1, np.int64)
        self.to[1:] = np.cumsum(rows)
        self.tab = tbe.tbe_tables(FAKE, FAKE + 4096, self.to.ctypes.data, len(rows), D, dtype)
        self.bt = tbe.tbe_batch(FAKE + 8192, FAKE + 16384, N, B, FAKE + 32768 if psw else None, None,
                                itype)
        self.tbe = tbe

    def sizes(self, cfg=None):
        mb, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
        st = self.tbe.lib().tbe_query_sizes(ctypes.byref(self.tab), ctypes.byref(self.bt),
                                            ctypes.byref(cfg) if cfg else None,
                                            ctypes.byref(mb), ctypes.byref(wb))
        return st, mb.value, wb.value


def test_query_sizes_and_meta_bind_layout():
    f = Fake(N=10000, B=100)
    st, mb, wb = f.sizes()
    assert st == 0 and mb >= 6 * 4 * 10000 and wb > 0
    L0 = f.tbe.lib()
    assert L0.tbe_meta_bytes(ctypes.byref(f.tab), ctypes.byref(f.bt), None) == mb
    assert L0.tbe_workspace_bytes(ctypes.byref(f.tab), ctypes.byref(f.bt), None) == wb
    bad = Fake(D=6)
    assert L0.tbe_workspace_bytes(ctypes.byref(bad.tab), ctypes.byref(bad.bt), None) == 0
    assert L0.tbe_status_str(3) == L0.tbe_status_string(3) == b"unsupported embedding dimension"
    m = f.tbe.tbe_meta()
    L = f.tbe.lib()
    assert L.tbe_meta_bind(ctypes.byref(m), FAKE, mb - 1, ctypes.byref(f.tab), ctypes.byref(f.bt), None) == 7
    assert L.tbe_meta_bind(ctypes.byref(m), FAKE, mb, ctypes.byref(f.tab), ctypes.byref(f.bt), None) == 0
    assert m.bound_N == 10000 and m.path == 1 and m.payload_is_pos == 0
    assert m.rows_total == 2000 and m.key_bits == 11     # sentinel 2000 needs 11 bits
    ptrs = [m.keys_a, m.vals_a, m.keys_b, m.vals_b, m.unique_keys, m.seg_off, m.counters,
            m.long_run, m.long_chunk_base, m.chunk_order, m.arrive, m.chunk_desc]
    assert all(p % 256 == 0 and FAKE <= p < FAKE + mb for p in ptrs)
    assert len(set(ptrs)) == len(ptrs)
    assert m.bag_of is None and m.hist is None
    # weighted batches carry positions as the sort payload and a bag_of array
    fw = Fake(N=10000, B=100, psw=True)
    _, mbw, _ = fw.sizes()
    m2 = f.tbe.tbe_meta()
    assert L.tbe_meta_bind(ctypes.byref(m2), FAKE, mbw, ctypes.byref(fw.tab), ctypes.byref(fw.bt), None) == 0
    assert m2.payload_is_pos == 1 and m2.bag_of is not None


@pytest.mark.parametrize("kw,code", [
    (dict(D=6), 3), (dict(D=4, dtype=1), 3), (dict(D=1024, dtype=0), 3), (dict(dtype=7), 4),
    (dict(N=1 << 30), 2), (dict(rows=[2**30, 2**30]), 0), (dict(rows=[2**61, 2**61]), 6),
    (dict(rows=[5, -1]), 2), (dict(itype=2), 2), (dict(itype=1), 0),
    # grad_out [B, T*D] float32 of 64 GB or more: gradient offsets would not fit 32 bits
    (dict(T=2, B=2**27, D=128), 2), (dict(T=2, B=2**25, D=128), 0),
])
def test_host_side_argument_errors(kw, code):
    f = Fake(**kw)
    assert f.sizes()[0] == code


def test_misaligned_and_null_pointers():
    f = Fake()
    f.tab.weights = FAKE + 8
    assert f.sizes()[0] == 5
    f = Fake()
    f.tab.weights = None
    assert f.sizes()[0] == 1


def test_histogram_path_selection_follows_the_pages_conditions():
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_constants.json")))["small_table_path"]
    from recsys_table_embedding_gb300 import tbe
    L = tbe.lib()

    def path(**kw):
        f = Fake(**kw)
        return L.tbe_select_path(ctypes.byref(f.tab), ctypes.byref(f.bt), None)

    B = 32
    ok = dict(rows=[g["E_max"]] * 3, D=g["D_max"], dtype=1, B=B, N=3 * B * g["L_min"])
    assert path(**ok) == 2
    assert path(**dict(ok, D=g["D_min"])) == 2
    assert path(**dict(ok, rows=[g["E_max"] + 1, 64, 64])) == 1       # E > 64
    assert path(**dict(ok, D=256)) == 1                                 # D > 128
    assert path(**dict(ok, D=32)) == 1                                  # D < 64
    assert path(**dict(ok, dtype=2)) == 1                               # bf16
    assert path(**dict(ok, dtype=0)) == 1                               # fp32
    assert path(**dict(ok, N=3 * B * g["L_min"] - 1)) == 1              # L < 64
    assert path(**dict(ok, psw=True)) == 1                              # weighted
    cfg = tbe.config(hist_mode=tbe.HIST_OFF)
    f = Fake(**ok)
    assert L.tbe_select_path(ctypes.byref(f.tab), ctypes.byref(f.bt), ctypes.byref(cfg)) == 1


def test_status_strings():
    from recsys_table_embedding_gb300 import lib
    L = lib()
    assert L.tbe_status_string(0) == b"ok"
    assert L.tbe_status_string(7).startswith(b"workspace")


def test_key_width_follows_the_row_range():
    # decision checklist item 6: int32 keys while the linearised range (with
    # its sentinel) fits, 64-bit keys beyond; the key arrays grow to match
    from recsys_table_embedding_gb300 import tbe
    L = tbe.lib()

    def bind(rows, cfg=None, itype=0):
        f = Fake(rows=rows, N=10000, B=100, itype=itype)
        st, mb, _ = f.sizes(cfg)
        assert st == 0
        m = tbe.tbe_meta()
        assert L.tbe_meta_bind(ctypes.byref(m), FAKE, mb, ctypes.byref(f.tab), ctypes.byref(f.bt),
                               ctypes.byref(cfg) if cfg else None) == 0
        return m, mb

    m4, mb4 = bind([2**30, 2**30 - 2])               # rows_total = 2^31 - 2: sentinel fits int32
    assert m4.key_bytes == 4 and m4.key_bits == 31
    m8, mb8 = bind([2**30, 2**30 - 1])               # rows_total = 2^31 - 1
    assert m8.key_bytes == 8 and m8.key_bits == 31
    assert mb8 >= mb4 + 3 * 4 * 10000 - 3 * 256      # three key arrays twice as wide (256-B aligned)
    mf, _ = bind([100, 100], cfg=tbe.config(key_bytes=8))
    assert mf.key_bytes == 8
    m64, _ = bind([100, 100], itype=1)
    assert m64.index_type == 1 and m64.key_bytes == 4
    f = Fake(rows=[2**31])
    assert f.sizes(tbe.config(key_bytes=4))[0] == 6  # 32-bit keys cannot hold this range
    assert f.sizes(tbe.config(key_bytes=5))[0] == 2


def test_int64_index_arrays_must_be_8_byte_aligned():
    f = Fake(itype=1)
    f.bt.indices = FAKE + 8196
    assert f.sizes()[0] == 5
    f = Fake(itype=0)
    f.bt.indices = FAKE + 8196
    assert f.sizes()[0] == 0
