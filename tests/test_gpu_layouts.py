"""Tables of different row length and dtype in one call, and a different
batch size per table (VBE), against the oracle.

TorchEasyRec analysis, section 1: one fused lookup for all features of a
KeyedJagged batch, whose features have different embedding sizes; FBTriton
TBE redesign, decision checklist item 5, names variable batch size per
feature (VBE).  Each table is described by its weight byte offset, D and
dtype; each table's bags by their first CSR bag, count and output rows."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_full, run_cuda, table_out, table_storage

pytestmark = pytest.mark.gpu


def _m0(wl):
    return np.random.default_rng(11).uniform(0, 0.5, wl.rows_total).astype(np.float32)


def _mixed(vbe=False, seed=41, B=2000, weighted=True, oob=0.01, table_B=None):
    T = 5
    return workloads.make_workload(
        "mixed", T=T, table_rows=[3000, 800, 20000, 150, 5000], D=64, dtype="f32", B=B,
        lengths=("poisson", 6.0), dist=("zipf", 1.15), seed=seed, oob_frac=oob,
        weighted=[True, False, True, True, False] if weighted else None,
        table_dims=[64, 128, 16, 256, 32], table_dtypes=["f32", "bf16", "f16", "f32", "bf16"],
        table_B=(table_B or [B, 300, 4096, 1, 900]) if vbe else None)


def _step(wl, cfg=None, pif=True, W0=None):
    W0 = wl.weights_mixed() if W0 is None else W0
    G, m0 = wl.grad_out(), _m0(wl)
    res = run_cuda(wl, W0, G, m0, cfg=cfg, preprocess_in_forward=pif)
    check_full(wl, W0, G, m0, res)
    return res


@pytest.mark.parametrize("pif", [True, False])
@pytest.mark.parametrize("long_mode", [1, 2])
def test_mixed_dims_and_dtypes(pif, long_mode):
    from recsys_table_embedding_gb300 import config
    res = _step(_mixed(), cfg=config(long_run_mode=long_mode), pif=pif)
    assert res["num_long"] > 0 and res["status"][0] > 0


@pytest.mark.parametrize("pif", [True, False])
def test_vbe_mixed_shapes(pif):
    res = _step(_mixed(vbe=True), pif=pif)
    assert res["num_long"] > 0


def test_vbe_uniform_shapes():
    # one D and dtype, a different B per table: typed [rows_total, D] weights,
    # only the bags carry a layout
    wl = workloads.make_workload("vbe", T=4, table_rows=[500, 7000, 60, 3000], D=128, dtype="bf16",
                                 B=0, lengths=("poisson", 5.0), dist=("zipf", 1.2), seed=43,
                                 table_B=[4096, 17, 2500, 1], oob_frac=0.005)
    res = _step(wl, W0=wl.weights())
    assert res["status"][0] > 0


def test_vbe_empty_tables_and_weighted_streaming():
    # a table with no bags at all, unweighted and weighted tables with
    # 512-byte gradient rows (the streaming short-run kernel)
    wl = workloads.make_workload("vbe0", T=3, table_rows=[64, 4000, 900], D=128, dtype="f16", B=0,
                                 lengths=("poisson", 9.0), dist=("zipf", 1.1), seed=47,
                                 table_B=[3000, 0, 2000], weighted=[True, True, False],
                                 table_dims=[128, 64, 128], table_dtypes=["f16", "f32", "bf16"])
    _step(wl)


def test_mixed_with_int64_inputs_and_64bit_keys():
    from recsys_table_embedding_gb300 import config
    wl = _mixed(vbe=True, seed=53)
    wl.indices = wl.indices.astype(np.int64)
    wl.offsets = wl.offsets.astype(np.int64)
    res = _step(wl, cfg=config(key_bytes=8))
    assert res["key_bytes"] == 8


def test_malformed_offsets_with_vbe():
    wl = _mixed(vbe=True, seed=59, oob=0.0)
    off = wl.offsets.astype(np.int64).copy()
    off[-1] = wl.N + 9            # last bag past N
    g = int(np.flatnonzero(np.diff(off) >= 3)[10])
    off[g + 1] = off[g] - 1       # decreasing: no backward update
    wl.offsets = off.astype(np.int32)
    res = _step(wl)
    assert res["status"][1] & 0x1 and res["num_unique"] == 0


def test_each_table_equals_running_it_alone():
    # tables are independent: the mixed batch gives, bit for bit, what each
    # table gives run alone as a uniform problem through the same library
    wl = _mixed(vbe=True, seed=61)
    W0, G, m0 = wl.weights_mixed(), wl.grad_out(), _m0(wl)
    res = run_cuda(wl, W0, G, m0)
    to = wl.table_offset
    for t, L in enumerate(wl.layout()):
        g0, g1 = L["bag_off"], L["bag_off"] + L["B"]
        s0, s1 = int(wl.offsets[g0]), int(wl.offsets[g1])
        one = workloads.Workload(
            name="one", T=1, B=L["B"], D=L["D"], dtype=L["dtype"],
            table_rows=wl.table_rows[t:t + 1].copy(),
            offsets=(wl.offsets[g0:g1 + 1].astype(np.int64) - s0).astype(np.int32),
            indices=wl.indices[s0:s1].copy(),
            per_sample_weights=None if wl.per_sample_weights is None else wl.per_sample_weights[s0:s1].copy(),
            weighted_tables=None if wl.weighted_tables is None else wl.weighted_tables[t:t + 1].copy(),
            lr=wl.lr, eps=wl.eps)
        if L["B"] == 0 or one.N == 0:
            continue
        Wt = table_storage(wl, W0, t)
        Wtt = torch.from_numpy(Wt.copy())
        if L["dtype"] != "f32":
            Wtt = Wtt.view(torch.int16).view(torch.float16 if L["dtype"] == "f16" else torch.bfloat16)
        Gt = np.ascontiguousarray(table_out(wl, G, t))
        alone = run_cuda(one, Wtt, Gt, m0[to[t]:to[t + 1]].copy())
        np.testing.assert_array_equal(table_out(wl, res["out"], t), alone["out"])
        np.testing.assert_array_equal(table_storage(wl, res["W"], t), alone["W"])
        np.testing.assert_array_equal(res["mom"][to[t]:to[t + 1]], alone["mom"])
