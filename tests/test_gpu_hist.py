"""GPU parity of the small-table histogram path (tensor cores, FP16 hi/lo
compensation) against the CPU oracle, plus its saved counts bit-exact.

Sizes are chosen so that the persistent forward runs several 128-bag tiles
per CTA (crossing table boundaries inside a CTA, a ragged last tile) and the
K-split backward runs many 64-bag K steps per slice (double-buffered stages,
mbarrier phases past the first, a ragged last step), up to the full
histogram workload (T=64, E=64, D=128, B=65536, L=64)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import (assert_momentum_close, assert_out_close, assert_weights_close, check_full,
                    device_batch, run_cuda, w_arith_bound, wbits_np, wvals_np)

pytestmark = pytest.mark.gpu


def _m0(wl):
    return np.random.default_rng(3).uniform(0, 0.5, wl.rows_total).astype(np.float32)


def _saved_counts(res, wl):
    from recsys_table_embedding_gb300 import meta_view
    h = meta_view(res["tbe"].meta, "hist", wl.NB * 64, torch.float16).cpu().numpy()
    return h.astype(np.int64).reshape(wl.T, wl.B, 64)


def _run(wl, cfg=None, flags=0, unaligned_indices=False):
    W0, G, m0 = wl.weights(), wl.grad_out(), _m0(wl)
    res = run_cuda(wl, W0, G, m0, cfg=cfg, preprocess_in_forward=False,
                   unaligned_indices=unaligned_indices)
    assert res["path"] == 2
    check_full(wl, W0, G, m0, res)
    np.testing.assert_array_equal(_saved_counts(res, wl), oracle.histogram(wl))
    assert res["status"][1] == flags
    return res


def _force():
    from recsys_table_embedding_gb300 import config
    from recsys_table_embedding_gb300.tbe import HIST_FORCE
    return config(hist_mode=HIST_FORCE)


def test_hist_config_reduced_batch():
    _run(workloads.hist(B=1024, T=8))


def test_hist_many_tiles_per_cta_and_k_steps_per_slice():
    # T=5, B=60000: 2345 forward tiles over <= 4 CTAs per SM (4 tiles per
    # CTA, CTAs that cross a table boundary, last tile of each table 96 bags);
    # backward slices of 16 K steps (the last one 10, its last step 32 bags)
    wl = workloads.make_workload("hmulti", T=5, table_rows=[64, 64, 50, 64, 17], D=128,
                                 dtype="f16", B=60000, lengths=("poisson", 16.0),
                                 dist=("uniform",), seed=8)
    _run(wl, cfg=_force())


def _ragged_end(wl):
    """Drop lookups from the last bag until N is not a multiple of 4."""
    while wl.N % 4 == 0:
        wl.indices = wl.indices[:-1]
        wl.offsets = wl.offsets.copy()
        wl.offsets[-1] -= 1
    assert wl.offsets[-2] < wl.offsets[-1]
    return wl


@pytest.mark.parametrize("itype", ["int32", "int64"])
@pytest.mark.parametrize("unaligned", [False, True])
def test_hist_index_types_and_alignment(itype, unaligned):
    # int32 and int64 indices and offsets, indices at a 16-byte boundary or
    # one element past it, a last bag that ends on a ragged element count
    wl = workloads.make_workload("hidx", T=3, table_rows=[64, 37, 64], D=128, dtype="f16", B=700,
                                 lengths=("poisson", 70.0), dist=("uniform",), seed=21)
    wl.indices = wl.indices.astype(itype)
    wl.offsets = wl.offsets.astype(itype)
    _run(_ragged_end(wl), cfg=_force(), unaligned_indices=unaligned)


@pytest.mark.parametrize("D", [64, 96, 128])
def test_hist_forced_shapes_ragged(D):
    wl = workloads.make_workload("hshape", T=3, table_rows=[13, 64, 40], D=D, dtype="f16", B=200,
                                 lengths=("poisson", 20.0), dist=("uniform",), seed=D)
    _run(wl, cfg=_force())


def test_hist_out_of_range_and_empty_bags():
    wl = workloads.make_workload("hoob", T=2, table_rows=[64, 30], D=128, dtype="f16", B=300,
                                 lengths=("poisson", 2.0), dist=("uniform",), seed=11, oob_frac=0.05)
    assert np.any(np.diff(wl.offsets) == 0)
    res = _run(wl, cfg=_force())
    assert res["status"][0] > 0


@pytest.mark.parametrize("pattern", ["gap_after", "end_below_start"])
def test_hist_malformed_offsets(pattern):
    wl = workloads.make_workload("hbad", T=2, table_rows=[64, 40], D=64, dtype="f16", B=300,
                                 lengths=("poisson", 6.0), dist=("uniform",), seed=13)
    off = wl.offsets.astype(np.int64)
    if pattern == "gap_after":
        wl.indices = np.concatenate([wl.indices, np.arange(7, dtype=np.int32)])
    else:
        g = int(np.flatnonzero(np.diff(off) >= 3)[5])
        off[g + 1] = off[g] - 2
        wl.offsets = off.astype(np.int32)
    res = _run(wl, cfg=_force(), flags=0x1)
    if pattern == "end_below_start":
        np.testing.assert_array_equal(res["mom"], _m0(wl))


def test_hist_count_flag():
    # one bag looks up row 5 3000 times: a count above 2048 is not exact in
    # FP16, which TBE_FLAG_HIST_COUNT reports
    lists = [[5] * 3000, [1, 2, 3], [], [7] * 10]
    wl = workloads.Workload(name="hcnt", T=1, B=4, D=64, dtype="f16", table_rows=np.array([64]),
                            offsets=np.concatenate([[0], np.cumsum([len(x) for x in lists])]).astype(np.int32),
                            indices=np.concatenate([np.array(x, np.int32) for x in lists]),
                            per_sample_weights=None, weighted_tables=None)
    W0, G, m0 = wl.weights(), wl.grad_out(), _m0(wl)
    res = run_cuda(wl, W0, G, m0, cfg=_force(), preprocess_in_forward=False)
    assert res["status"][1] == 0x8 and res["status"][0] == 0
    # the other bags are exact
    ref, ab, _, _ = oracle.forward(wl, wbits_np(W0, "f16"), want_abs=True)
    assert_out_close(res["out"][1:], ref[1:], ab[1:], "f16")


def test_hist_fp16_overflow_flag():
    # an upstream gradient beyond the FP16 range cannot be split into hi/lo
    wl = workloads.hist(B=256, T=2)
    W0, G, m0 = wl.weights(), wl.grad_out(), _m0(wl)
    G[17, 5] = 1.0e5
    res = run_cuda(wl, W0, G, m0, preprocess_in_forward=False)
    assert res["path"] == 2
    assert res["status"][1] & 0x2


def test_hist_matches_generic_path():
    from recsys_table_embedding_gb300 import config
    from recsys_table_embedding_gb300.tbe import HIST_OFF
    from parity import touched_rows
    wl = workloads.hist(B=512, T=4)
    W0, G, m0 = wl.weights(), wl.grad_out(), _m0(wl)
    a = run_cuda(wl, W0, G, m0, preprocess_in_forward=False)
    b = run_cuda(wl, W0, G, m0, cfg=config(hist_mode=HIST_OFF), preprocess_in_forward=False)
    assert a["path"] == 2 and b["path"] == 1
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(a["mom"], b["mom"], rtol=1e-4)
    assert_weights_close(a["W"], b["W"], wbits_np(W0, "f16"), touched_rows(wl), "f16")


def test_hist_full_config_sampled():
    # the full histogram workload (268M lookups): counts bit-exact everywhere,
    # 200 sampled bags of the forward and 24 sampled rows of the backward
    # recomputed by the oracle one by one
    from recsys_table_embedding_gb300 import TBE, Tables
    wl = workloads.hist()
    dev = torch.device("cuda")
    W0 = wl.weights()                       # 4096 x 128 FP16: small, drawn on the host
    G = wl.grad_out()
    m0 = _m0(wl)
    W = W0.to(dev)
    tables = Tables(W, wl.table_offset)
    batch = device_batch(wl)
    tbe = TBE(tables, batch, preprocess_in_forward=False)
    assert tbe.path == 2
    out = tbe.forward(batch)
    mom = torch.from_numpy(m0).to(dev)
    tbe.backward(batch, mom, torch.from_numpy(G).to(dev), wl.lr, wl.eps)
    torch.cuda.synchronize()
    st = tbe.status.cpu().numpy()
    assert st[0] == 0 and st[1] == 0
    from recsys_table_embedding_gb300 import meta_view
    h = meta_view(tbe.meta, "hist", wl.NB * 64, torch.float16).cpu().numpy().astype(np.int32)
    np.testing.assert_array_equal(h.reshape(wl.T, wl.B, 64), oracle.histogram(wl))
    del h
    rng = np.random.default_rng(9)
    wb = wbits_np(W0, "f16")
    bags = np.sort(rng.choice(wl.NB, 200, replace=False))
    ref, ab, _, _ = oracle.forward(wl, wb, bags=bags, want_abs=True)
    outh = out.cpu().numpy()
    dev_rows = np.stack([outh[g % wl.B, (g // wl.B) * wl.D:(g // wl.B + 1) * wl.D] for g in bags])
    assert_out_close(dev_rows, ref, ab, "f16")
    rows = np.sort(rng.choice(wl.rows_total, 24, replace=False))
    Wr, mr, rg, cnt, nv, ra = oracle.rows_update(wl, rows, wb[rows], m0[rows], G, want_row_abs=True)
    assert nv == wl.N and np.all(cnt > 0)
    touched = np.ones(len(rows), bool)
    assert_momentum_close(mom.cpu().numpy()[rows], mr, m0[rows], touched)
    arith = w_arith_bound("f16", rg, ra, cnt, m0[rows], wvals_np(wb[rows], "f16"), wl.lr, wl.eps,
                          path=2)
    assert_weights_close(wbits_np(W, "f16")[rows], Wr, wb[rows], touched, "f16", arith)
