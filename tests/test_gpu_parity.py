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
    # full size: T=16 tables of the demo list, B=4096 (~197K lookups)
    _step(workloads.demo(), pif=pif)


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


def _malformed(pattern, dtype="f32", weighted=False):
    """A batch whose offsets break the CSR rules in one way, with junk lookups
    (in-range ones too) wherever a lookup belongs to no well-formed bag."""
    wl = workloads.make_workload("bad", T=2, table_rows=[60, 300], D=16, dtype=dtype, B=40,
                                 lengths=("poisson", 5.0), dist=("zipf", 1.1), seed=17,
                                 weighted=[True, False] if weighted else None)
    rng = np.random.default_rng(3)
    off = wl.offsets.astype(np.int64)
    idx = wl.indices
    psw = wl.per_sample_weights
    NB, N = wl.NB, wl.N

    def junk(n):
        return rng.integers(0, 60, size=n).astype(np.int32)

    if pattern == "gap_before":
        idx = np.concatenate([junk(9), idx])
        off = off + 9
        psw = None if psw is None else np.concatenate([np.ones(9, np.float32), psw])
    elif pattern == "gap_after":
        idx = np.concatenate([idx, junk(11)])
        psw = None if psw is None else np.concatenate([psw, np.ones(11, np.float32)])
    elif pattern == "start_negative":
        off = off.copy()
        off[0] = -3
    elif pattern == "end_past_n":
        off = off.copy()
        off[NB] = N + 4
    elif pattern == "end_below_start":
        off = off.copy()
        g = int(np.flatnonzero(np.diff(off) >= 3)[3])
        off[g + 1] = off[g] - 2      # bag g malformed, bag g+1 overlaps bag g-1
    wl.offsets = off.astype(np.int32)
    wl.indices = idx.astype(np.int32)
    wl.per_sample_weights = psw
    return wl


@pytest.mark.parametrize("pattern", ["gap_before", "gap_after", "start_negative", "end_past_n",
                                     "end_below_start"])
@pytest.mark.parametrize("pif", [True, False])
@pytest.mark.parametrize("dtype,weighted", [("f32", False), ("bf16", True)])
def test_malformed_offsets_forward_and_backward(pattern, pif, dtype, weighted):
    # The metadata buffer starts as zero bytes (key 0 is a real row): a
    # lookup position that no kernel rewrites would update row 0 or a row of
    # a stale run.  The step must match the oracle, which ignores lookups
    # outside well-formed bags and updates nothing when offsets decrease.
    wl = _malformed(pattern, dtype, weighted)
    assert oracle.offsets_check(wl)[0]
    W0, G, m0 = wl.weights(), wl.grad_out(), _m0(wl)
    res = run_cuda(wl, W0, G, m0, preprocess_in_forward=pif, meta_fill=0)
    check_full(wl, W0, G, m0, res)
    assert res["status"][1] & 0x1
    if pattern == "end_below_start":
        assert res["num_unique"] == 0
        np.testing.assert_array_equal(res["mom"], m0)


def test_fp32_tables_accumulate_in_fp64():
    # Decision checklist item 1: FP64 accumulation for FP32 weights.  Values
    # 1, 2^-30 and -1 sum to 2^-30 exactly in FP64; an FP32 accumulator that
    # already holds a partial of magnitude >= 1 drops the 2^-30.
    #   forward: bag (0,0) = 64 x row0 (1.0), row2 (2^-30), 64 x row3 (-1.0), row1 (0)
    #   short run: row 1 of table 0 is looked up once by bags 0..128, whose
    #              gradients are 1 (b < 64), 2^-30 (b = 64), -1 (b > 64)
    #   long run:  row 0 of table 1 is looked up once by bags 0..300 (two
    #              256-lookup chunks), gradients 1 (b < 150), 2^-30, -1 (b > 150)
    tiny = 2.0 ** -30
    D, B = 16, 301
    lists = [[] for _ in range(2 * B)]
    lists[0] = [0] * 64 + [2] + [3] * 64
    for b in range(129):
        lists[b].append(1)
    for b in range(B):
        lists[B + b].append(0)
    lens = np.array([len(x) for x in lists])
    wl = workloads.Workload(name="fp64", T=2, B=B, D=D, dtype="f32", table_rows=np.array([4, 2]),
                            offsets=np.concatenate([[0], np.cumsum(lens)]).astype(np.int32),
                            indices=np.concatenate([np.array(x, np.int32) for x in lists]),
                            per_sample_weights=None, weighted_tables=None)
    W0 = torch.zeros(6, D, dtype=torch.float32)
    W0[0], W0[1], W0[2], W0[3] = 1.0, 0.0, tiny, -1.0
    W0[4] = 0.005
    W0[5] = -0.003
    G = np.zeros((B, 2 * D), np.float32)
    G[:64, :D], G[64, :D], G[65:129, :D] = 1.0, tiny, -1.0
    G[:150, D:], G[150, D:], G[151:, D:] = 1.0, tiny, -1.0
    m0 = np.zeros(6, np.float32)
    # the test data: row gradients of both runs are 2^-30 exactly
    _, _, _, rg, _ = oracle.backward_adagrad(wl, W0.numpy(), m0, G, want_row_grad=True)
    assert np.all(rg[1] == tiny) and np.all(rg[4] == tiny)
    res = run_cuda(wl, W0, G, m0)
    assert res["num_long"] == 1
    np.testing.assert_array_equal(res["out"][0, :D], np.full(D, tiny, np.float32))
    check_full(wl, W0, G, m0, res)
    # the update the 2^-30 gradient makes is far above FP32 noise
    assert np.all(np.abs(res["W"][1]) > 1e-4) and np.all(np.abs(res["W"][4] - 0.005) > 1e-4)


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
    np.testing.assert_array_equal(desc[:, 2].astype(np.uint32) | (desc[:, 3].astype(np.int64) << 32),
                                  keys[runs])
    table = np.searchsorted(wl.table_offset, keys[runs], side="right") - 1
    np.testing.assert_array_equal(desc[:, 6], (re - rs + 255) // 256)
    slot = np.arange(nch)
    assert np.all((desc[:, 5] <= slot) & (slot < desc[:, 5] + desc[:, 6]))
    np.testing.assert_array_equal(slot - desc[:, 5], (desc[:, 0] - rs) // 256)
    assert len(np.unique(desc[:, 4])) == res["num_long"]
    if B >= 4096:
        # key = table * windows per table + (first bag >> 9): payload = bag
        np.testing.assert_array_equal(desc[:, 7], table * ((B + 511) // 512) + (vals[desc[:, 0]] >> 9))
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
