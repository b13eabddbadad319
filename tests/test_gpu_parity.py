"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs, at sizes the oracle finishes in seconds (several tiles and
a ragged tail), for the five workload shapes and the method's edge cases."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_full, run_cuda

pytestmark = pytest.mark.gpu


def _m0(wl, seed=7, zero=False):
    if zero:
        return wl.momentum()
    return np.random.default_rng(seed).uniform(0, 0.5, wl.rows_total).astype(np.float32)


def _step(wl, cfg=None, pif=True, zero_m=False):
    from recsys_table_embedding_gb300 import config
    W0 = wl.weights()
    G = wl.grad_out()
    m0 = _m0(wl, zero=zero_m)
    res = run_cuda(wl, W0, G, m0, cfg=cfg, preprocess_in_forward=pif)
    check_full(wl, W0, G, m0, res)
    return res


def test_tiny_config():
    wl = workloads.tiny()
    res = _step(wl, zero_m=True)
    assert res["status"][1] == 0


@pytest.mark.parametrize("pif", [True, False])
def test_demo_config(pif):
    _step(workloads.demo(B=1024), pif=pif)


def test_mid_config_reduced_batch():
    # full table sizes and distribution, B reduced so the oracle runs in seconds
    _step(workloads.mid(B=512))


def test_large_config_reduced_batch():
    # B reduced 32x: hottest row ~3.9K lookups, so long runs take many chunks
    res = _step(workloads.large(B=4096))
    assert res["num_long"] > 100 and res["num_chunks"] > res["num_long"]


def test_hist_shape_generic_path():
    from recsys_table_embedding_gb300 import config
    from recsys_table_embedding_gb300.tbe import HIST_OFF
    _step(workloads.hist(B=512, T=8), cfg=config(hist_mode=HIST_OFF))


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("D", [4, 8, 16, 32, 64, 128, 256, 384, 512])
def test_dims_and_dtypes(dtype, D):
    if dtype != "f32" and D in (4, 384):
        pytest.skip("row size not supported for 2-byte weights")
    wl = workloads.make_workload("dims", T=3, table_rows=[300, 17, 1000], D=D, dtype=dtype, B=70,
                                 lengths=("poisson", 6.0), dist=("zipf", 1.2), seed=D,
                                 weighted=[True, False, True])
    _step(wl)


@pytest.mark.parametrize("sl", [255, 256, 257, 513])
def test_segment_length_boundaries(sl):
    # table 0: one row looked up exactly `sl` times; the rest spread thin
    B = 600
    rows = [50, 40]
    wl = workloads.make_workload("sl", T=2, table_rows=rows, D=32, dtype="f32", B=B,
                                 lengths=("fixed", 1), dist=("uniform",), seed=sl)
    idx = wl.indices.copy()
    idx[:B] = np.where(np.arange(B) < sl, 7, 8 + np.arange(B) % 40)
    wl.indices = idx.astype(np.int32)
    res = _step(wl)
    assert res["num_long"] == (1 if sl >= 256 else 0)
    assert res["num_chunks"] == (sl + 255) // 256 * (sl >= 256)


def test_all_lookups_one_row_and_e1_tables():
    wl = workloads.make_workload("one", T=3, table_rows=[1, 1, 5], D=64, dtype="bf16", B=900,
                                 lengths=("poisson", 3.0), dist=("uniform",), seed=3)
    res = _step(wl)
    assert res["num_unique"] <= 7


def test_out_of_range_indices_weighted_and_empty_bags():
    wl = workloads.make_workload("oob", T=4, table_rows=[100, 3, 1000, 64], D=16, dtype="f16",
                                 B=333, lengths=("poisson", 1.5), dist=("zipf", 1.1), seed=9,
                                 weighted=[True, True, False, True], oob_frac=0.08)
    assert np.any(np.diff(wl.offsets) == 0)
    res = _step(wl)
    assert res["status"][0] > 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_long_run_modes_bit_identical(dtype):
    from recsys_table_embedding_gb300 import config
    wl = workloads.make_workload("modes", T=2, table_rows=[64, 2000], D=64, dtype=dtype, B=3000,
                                 lengths=("poisson", 5.0), dist=("zipf", 1.3), seed=5,
                                 weighted=[True, False])
    W0, G, m0 = wl.weights(), wl.grad_out(), _m0(wl)
    a = run_cuda(wl, W0, G, m0, cfg=config(long_run_mode=1))
    b = run_cuda(wl, W0, G, m0, cfg=config(long_run_mode=2))
    assert a["num_long"] > 0
    np.testing.assert_array_equal(a["W"], b["W"])
    np.testing.assert_array_equal(a["mom"], b["mom"])
    check_full(wl, W0, G, m0, a)


def test_preprocess_placement_bit_identical():
    wl = workloads.large(B=1024, E=20000)
    W0, G, m0 = wl.weights(), wl.grad_out(), _m0(wl)
    a = run_cuda(wl, W0, G, m0, preprocess_in_forward=True)
    b = run_cuda(wl, W0, G, m0, preprocess_in_forward=False)
    for k in ("out", "W", "mom", "sorted_keys", "sorted_vals", "unique_keys", "seg_off"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_empty_batch():
    wl = workloads.make_workload("empty", T=2, table_rows=[10, 10], D=16, dtype="f32", B=5,
                                 lengths=("fixed", 0), dist=("uniform",), seed=0)
    assert wl.N == 0
    res = _step(wl)
    assert res["num_unique"] == 0 and np.all(res["out"] == 0)


def test_bad_offsets_flagged_and_treated_empty():
    wl = workloads.make_workload("bad", T=1, table_rows=[50], D=16, dtype="f32", B=8,
                                 lengths=("fixed", 4), dist=("uniform",), seed=1)
    off = wl.offsets.copy()
    off[3] = off[2] - 1          # bag 2 has end < start; bag 3 starts earlier
    wl.offsets = off
    from parity import device_batch
    from recsys_table_embedding_gb300 import TBE, Tables
    W = wl.weights().cuda()
    tbe = TBE(Tables(W, wl.table_offset), device_batch(wl), preprocess_in_forward=False)
    out = tbe.forward(device_batch(wl))
    torch.cuda.synchronize()
    st = tbe.status.cpu().numpy()
    assert st[1] & 0x1
    ref, _, _, bad = oracle.forward(wl, W.cpu().numpy())
    assert bad == 1
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=1e-6, atol=0)


@pytest.mark.parametrize("B", [4096, 3000])
def test_chunk_descriptors_and_window_order(B):
    # every chunk slot's descriptor against the runs of the oracle's
    # inversion; with B >= 4096 the order is a permutation of the slots whose
    # (table, 512-bag window) keys never decrease
    from recsys_table_embedding_gb300 import meta_view
    wl = workloads.large(B=B, E=20000)
    W0, G, m0 = wl.weights(), wl.grad_out(), _m0(wl)
    res = run_cuda(wl, W0, G, m0)
    check_full(wl, W0, G, m0, res)
    m = res["tbe"].meta
    nch = res["num_chunks"]
    assert nch > 0
    desc = meta_view(m, "chunk_desc", nch * 8).cpu().numpy().reshape(nch, 8).astype(np.int64)
    order = meta_view(m, "chunk_order", nch).cpu().numpy().astype(np.int64)
    seg = res["seg_off"].astype(np.int64)
    keys = res["unique_keys"].astype(np.int64)
    vals = res["sorted_vals"].astype(np.int64)
    runs = np.searchsorted(seg, desc[:, 0], side="right") - 1
    rs, re = seg[runs], seg[runs + 1]
    assert np.all(re - rs >= 256)
    assert np.all((desc[:, 0] - rs) % 256 == 0)
    np.testing.assert_array_equal(desc[:, 1], np.minimum(desc[:, 0] + 256, re))
    np.testing.assert_array_equal(desc[:, 2], keys[runs])
    np.testing.assert_array_equal(desc[:, 3], np.searchsorted(wl.table_offset, keys[runs], side="right") - 1)
    np.testing.assert_array_equal(desc[:, 6], (re - rs + 255) // 256)
    slot = np.arange(nch)
    assert np.all((desc[:, 5] <= slot) & (slot < desc[:, 5] + desc[:, 6]))
    np.testing.assert_array_equal(slot - desc[:, 5], (desc[:, 0] - rs) // 256)
    assert len(np.unique(desc[:, 4])) == res["num_long"]
    if B >= 4096:
        # key = table * windows per table + (first bag >> 9): payload = bag
        np.testing.assert_array_equal(desc[:, 7], desc[:, 3] * ((B + 511) // 512) + (vals[desc[:, 0]] >> 9))
        np.testing.assert_array_equal(np.sort(order), slot)
        assert np.all(np.diff(desc[order, 7]) >= 0)
    else:
        assert np.all(desc[:, 7] == 0)


@pytest.mark.parametrize("dtype,D", [("f16", 128), ("f32", 256)])
def test_weighted_short_runs_around_long_runs(dtype, D):
    # weighted batch with gradient rows >= 512 B: short runs take the
    # streaming kernel.  Table 0 has 24 rows, each looked up ~1300 times
    # (long runs only: whole tasks of the short-run kernel are empty), table 1
    # has 6000 rows (short runs), table 2 mixes both
    wl = workloads.make_workload("mixw", T=3, table_rows=[24, 6000, 300], D=D, dtype=dtype, B=4096,
                                 lengths=("poisson", 8.0), dist=("zipf", 1.1), seed=21,
                                 weighted=[True, True, True], oob_frac=0.01)
    res = _step(wl)
    assert res["num_long"] >= 24
    assert res["payload_is_pos"] == 1
