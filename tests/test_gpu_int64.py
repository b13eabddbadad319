"""int64 indices and offsets, and 64-bit linearised keys (FBTriton TBE
redesign, decision checklist item 6: int32 keys only while the linearised
range is below 2^31; KeyedJagged batches often carry int64 indices).

  * int64 CSR inputs on the generic and histogram paths, including offsets
    with values beyond 2^31 (malformed: past N);
  * the 64-bit key path (forced through tbe_config.key_bytes = 8) on the
    parity workloads: radix sort of 64-bit keys, RLE, chunked long runs,
    weighted streaming short runs;
  * a real row range past 2^31: two tables with 2^31 + 64 and 1000 rows of
    D = 4 FP32 weights (34 GB), indices of table 0 up to 2^31 + 63, checked
    against the oracle on every touched row and every bag.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import (assert_momentum_close, assert_out_close, assert_weights_close, check_full,
                    device_batch, meta_keys, run_cuda, w_arith_bound, wbits_np, wvals_np)

pytestmark = pytest.mark.gpu


def _m0(wl):
    return np.random.default_rng(7).uniform(0, 0.5, wl.rows_total).astype(np.float32)


def _wide(wl):
    wl.indices = wl.indices.astype(np.int64)
    wl.offsets = wl.offsets.astype(np.int64)
    return wl


def _step(wl, cfg=None, pif=True):
    W0, G, m0 = wl.weights(), wl.grad_out(), _m0(wl)
    res = run_cuda(wl, W0, G, m0, cfg=cfg, preprocess_in_forward=pif)
    check_full(wl, W0, G, m0, res)
    return res


@pytest.mark.parametrize("pif", [True, False])
def test_int64_indices_generic_path(pif):
    wl = _wide(workloads.make_workload("i64", T=3, table_rows=[300, 17, 5000], D=64, dtype="bf16",
                                       B=900, lengths=("poisson", 6.0), dist=("zipf", 1.2), seed=4,
                                       weighted=[True, False, True], oob_frac=0.02))
    res = _step(wl, pif=pif)
    assert res["key_bytes"] == 4 and res["status"][0] > 0


def test_int64_offsets_beyond_2_31_are_malformed():
    wl = _wide(workloads.make_workload("i64bad", T=2, table_rows=[60, 300], D=16, dtype="f32", B=50,
                                       lengths=("poisson", 4.0), dist=("uniform",), seed=5))
    off = wl.offsets.copy()
    off[-1] = 2**33 + 5          # last bag ends far past N (and past 2^31)
    off[7] = -(2**32)            # bag 6 ends before it starts, bag 7 starts below 0
    wl.offsets = off
    assert oracle.offsets_check(wl)[0]
    res = _step(wl)
    assert res["status"][1] & 0x1 and res["num_unique"] == 0


def test_int64_indices_histogram_path():
    from recsys_table_embedding_gb300 import config
    from recsys_table_embedding_gb300.tbe import HIST_FORCE
    wl = _wide(workloads.make_workload("h64", T=3, table_rows=[64, 40, 64], D=128, dtype="f16",
                                       B=700, lengths=("poisson", 12.0), dist=("uniform",), seed=6,
                                       oob_frac=0.01))
    res = _step(wl, cfg=config(hist_mode=HIST_FORCE), pif=False)
    assert res["path"] == 2 and res["status"][0] > 0


WIDE_CASES = {
    "large_reduced": lambda: workloads.large(B=4096),
    "mid_reduced": lambda: workloads.mid(B=512),
    "weighted_streaming": lambda: workloads.make_workload(
        "mixw", T=3, table_rows=[24, 6000, 300], D=128, dtype="f16", B=4096,
        lengths=("poisson", 8.0), dist=("zipf", 1.1), seed=21, weighted=[True, True, True],
        oob_frac=0.01),
    "fp32_int64_inputs": lambda: _wide(workloads.make_workload(
        "w32", T=2, table_rows=[64, 2000], D=64, dtype="f32", B=3000, lengths=("poisson", 5.0),
        dist=("zipf", 1.3), seed=5, weighted=[True, False])),
}


@pytest.mark.parametrize("case", sorted(WIDE_CASES))
@pytest.mark.parametrize("long_mode", [1, 2])
def test_forced_64bit_keys(case, long_mode):
    from recsys_table_embedding_gb300 import config
    wl = WIDE_CASES[case]()
    res = _step(wl, cfg=config(key_bytes=8, long_run_mode=long_mode))
    assert res["key_bytes"] == 8
    if case == "large_reduced":
        assert res["num_long"] > 100


def test_64bit_keys_match_32bit_keys_bit_for_bit():
    from recsys_table_embedding_gb300 import config
    wl = workloads.large(B=2048, E=50000)
    W0, G, m0 = wl.weights(), wl.grad_out(), _m0(wl)
    a = run_cuda(wl, W0, G, m0)
    b = run_cuda(wl, W0, G, m0, cfg=config(key_bytes=8))
    assert a["key_bytes"] == 4 and b["key_bytes"] == 8
    for k in ("out", "W", "mom", "sorted_keys", "sorted_vals", "unique_keys", "seg_off"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_row_range_beyond_2_31():
    from recsys_table_embedding_gb300 import TBE, Tables
    E0, E1, D, B = 2**31 + 64, 1000, 4, 3000
    rng = np.random.default_rng(31)
    lens0 = rng.poisson(4.0, B)
    lens1 = rng.poisson(3.0, B)
    n0, n1 = int(lens0.sum()), int(lens1.sum())
    idx0 = rng.integers(0, E0, n0, dtype=np.int64)
    # a long run at the very top of the range (two 256-lookup chunks), a
    # short one just past 2^31, a long one at a small key, out-of-range values
    where = rng.permutation(n0)
    idx0[where[:400]] = E0 - 1
    idx0[where[400:430]] = 2**31 + 7
    idx0[where[430:730]] = 5
    idx0[where[730:740]] = np.array([-1, E0, 2**40, -(2**35), E0 + 1] * 2)
    idx1 = rng.integers(0, E1, n1, dtype=np.int64)
    idx1[:3] = [E1, -5, 2**33]
    offsets = np.concatenate([[0], np.cumsum(np.concatenate([lens0, lens1]))]).astype(np.int64)
    wl = workloads.Workload(name="big", T=2, B=B, D=D, dtype="f32",
                            table_rows=np.array([E0, E1], np.int64), offsets=offsets,
                            indices=np.concatenate([idx0, idx1]), per_sample_weights=None,
                            weighted_tables=None)
    dev = torch.device("cuda")
    G = wl.grad_out()
    tab = np.searchsorted(offsets, np.arange(wl.N), side="right") - 1
    t_of = tab // B
    valid = (wl.indices >= 0) & (wl.indices < wl.table_rows[t_of])
    keys = wl.table_offset[t_of] + wl.indices
    rows = np.unique(keys[valid])
    assert keys[valid & (t_of == 0)].max() == 2**31 + 63 and rows.max() > 2**31
    untouched = np.setdiff1d(rng.integers(0, wl.rows_total, 64), rows)

    def weights():
        g = torch.Generator(device=dev)
        g.manual_seed(8)
        W = torch.empty((wl.rows_total, D), dtype=torch.float32, device=dev)
        W.uniform_(-0.01, 0.01, generator=g)
        return W

    for pif in (True, False):
        W = weights()
        rows_t = torch.from_numpy(rows).to(dev)
        W_rows0 = W.index_select(0, rows_t).cpu().numpy()
        un_t = torch.from_numpy(untouched).to(dev)
        W_un0 = W.index_select(0, un_t).cpu().numpy()
        mom = torch.zeros(wl.rows_total, dtype=torch.float32, device=dev)
        tables = Tables(W, wl.table_offset)
        batch = device_batch(wl)
        tbe = TBE(tables, batch, preprocess_in_forward=pif)
        assert tbe.meta.c.key_bytes == 8 and tbe.meta.c.index_type == 1
        out = tbe.forward(batch)
        tbe.backward(batch, mom, torch.from_numpy(G).to(dev), wl.lr, wl.eps)
        torch.cuda.synchronize()
        st = tbe.status.cpu().numpy()
        assert st[0] == int((~valid).sum()) and st[1] == 0
        # batch inversion, bit-exact
        pre = oracle.preprocess(wl)
        U, nv, nlong, nchunks = tbe.counters()
        assert U == pre["num_unique"] == len(rows) and nv == pre["n_valid"]
        np.testing.assert_array_equal(meta_keys(tbe.meta, "sorted_keys", nv), pre["sorted_keys"])
        np.testing.assert_array_equal(meta_keys(tbe.meta, "unique_keys", U), pre["unique_keys"])
        assert nlong == 2 and nchunks == 2 + 2
        # forward: every bag, on a compact problem holding the touched rows
        cidx = np.where(valid, np.searchsorted(rows, keys), -1)
        sub = workloads.Workload(name="c", T=1, B=wl.NB, D=D, dtype="f32",
                                 table_rows=np.array([len(rows)]), offsets=offsets,
                                 indices=cidx, per_sample_weights=None, weighted_tables=None)
        ref, ab, _, _ = oracle.forward(sub, W_rows0, want_abs=True)
        o = out.cpu().numpy()
        dev_rows = np.concatenate([o[:, :D], o[:, D:]], axis=0)     # bag (t,b) -> row t*B+b
        assert_out_close(dev_rows, ref, ab, "f32")
        # backward: every touched row; untouched rows unchanged
        m0 = np.zeros(len(rows), np.float32)
        Wr, mr, rg, cnt, nvo, ra = oracle.rows_update(wl, rows, W_rows0, m0, G, want_row_abs=True)
        assert nvo == nv and np.all(cnt > 0)
        touched = np.ones(len(rows), bool)
        assert_momentum_close(mom.index_select(0, rows_t).cpu().numpy(), mr, m0, touched)
        arith = w_arith_bound("f32", rg, ra, cnt, m0, W_rows0.astype(np.float64), wl.lr, wl.eps)
        assert_weights_close(W.index_select(0, rows_t).cpu().numpy(), Wr, W_rows0, touched, "f32",
                             arith)
        np.testing.assert_array_equal(W.index_select(0, un_t).cpu().numpy(), W_un0)
        del W, mom, tbe, tables, out
        torch.cuda.empty_cache()
