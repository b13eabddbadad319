"""Full-size parity on the large Zipf workload, in the launch configuration
the benchmark times (T=32, E=2M, D=128, bf16, B=131072, ~84M lookups,
preprocessing in the forward, fused long-run backward).

The oracle cannot run the whole step in test time, so:
  * forward: a sample of bags recomputed by the oracle, one by one;
  * backward: a sample of rows (the hottest ones, which take the chunked
    path, and random ones from the short-run path) recomputed by the oracle
    from one scan of all lookups;
  * batch inversion: properties that hold at any size -- sorted order,
    (key, bag) multiset equal to the input's, run table consistent with the
    key counts, unique count.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import (assert_momentum_close, assert_out_close, assert_weights_close, device_batch,
                    wbits_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def large_step():
    from recsys_table_embedding_gb300 import TBE, Tables, meta_view
    wl = workloads.large()
    dev = torch.device("cuda")
    W = wl.weights(device="cuda")
    G = wl.grad_out()
    tables = Tables(W, wl.table_offset)
    batch = device_batch(wl)
    tbe = TBE(tables, batch, preprocess_in_forward=True)
    rng = np.random.default_rng(5)

    # rows to check after the backward: hottest rows + random touched rows
    keys_all = (wl.table_offset[np.repeat(np.arange(wl.T), np.diff(wl.offsets[::wl.B]))]
                + wl.indices.astype(np.int64))
    counts = np.bincount(keys_all, minlength=wl.rows_total)
    hot = np.argsort(-counts, kind="stable")[:24]
    touched = np.flatnonzero(counts)
    sample_rows = np.unique(np.concatenate([hot, rng.choice(touched, 200, replace=False),
                                            rng.choice(wl.rows_total, 20, replace=False)]))
    rows_t = torch.from_numpy(sample_rows).to(dev)
    W_rows0 = W.index_select(0, rows_t).cpu()
    m0 = torch.zeros(wl.rows_total, dtype=torch.float32, device=dev)

    # forward sample: random bags with their rows, read before the update
    bags = np.sort(rng.choice(wl.NB, 300, replace=False))
    out = tbe.forward(batch)
    torch.cuda.synchronize()
    tbe.backward(batch, m0, torch.from_numpy(G).to(dev), wl.lr, wl.eps)
    torch.cuda.synchronize()
    U, nv, nlong, nchunks = tbe.counters()
    res = dict(wl=wl, G=G, counts=counts, keys_all=keys_all, sample_rows=sample_rows,
               W_rows0=W_rows0, W_rows1=W.index_select(0, rows_t).cpu(),
               m_rows=m0.index_select(0, rows_t).cpu().numpy(), bags=bags,
               out_bags=out.cpu().numpy(), status=tbe.status.cpu().numpy(), U=U, nv=nv,
               nlong=nlong, nchunks=nchunks,
               sorted_keys=meta_view(tbe.meta, "sorted_keys", wl.N, torch.int32).cpu().numpy(),
               sorted_vals=meta_view(tbe.meta, "sorted_vals", wl.N, torch.int32).cpu().numpy(),
               unique_keys=meta_view(tbe.meta, "unique_keys", U, torch.int32).cpu().numpy(),
               seg_off=meta_view(tbe.meta, "seg_off", U + 1, torch.int32).cpu().numpy())
    # rows each sampled bag touches, for the forward check (before the update)
    need = np.unique(np.concatenate([keys_all[wl.offsets[g]:wl.offsets[g + 1]] for g in bags]))
    # W was updated by the backward: rebuild the pre-update rows from the seed
    W0 = wl.weights(device="cuda")
    res["fw_rows"] = need
    res["fw_W"] = W0.index_select(0, torch.from_numpy(need).to(dev)).cpu()
    del W0
    return res


def test_forward_sampled_bags(large_step):
    r = large_step
    wl = r["wl"]
    need, Wn = r["fw_rows"], r["fw_W"]
    # a one-table sub-problem holding just the sampled bags and their rows
    offs = [0]
    idx = []
    for g in r["bags"]:
        t = g // wl.B
        k = r["keys_all"][wl.offsets[g]:wl.offsets[g + 1]]
        idx.extend(np.searchsorted(need, k).tolist())
        offs.append(len(idx))
    sub = workloads.Workload(name="s", T=1, B=len(r["bags"]), D=wl.D, dtype=wl.dtype,
                             table_rows=np.array([len(need)]), offsets=np.array(offs, np.int32),
                             indices=np.array(idx, np.int32), per_sample_weights=None,
                             weighted_tables=None)
    ref, ab, _, _ = oracle.forward(sub, wbits_np(Wn, wl.dtype), want_abs=True)
    dev_rows = np.stack([r["out_bags"][g % wl.B, (g // wl.B) * wl.D:(g // wl.B + 1) * wl.D]
                         for g in r["bags"]])
    assert_out_close(dev_rows, ref, ab, wl.dtype)
    assert r["status"][0] == 0 and r["status"][1] == 0


def test_backward_sampled_rows(large_step):
    r = large_step
    wl = r["wl"]
    rows = r["sample_rows"]
    Wr0 = wbits_np(r["W_rows0"], wl.dtype)
    m0 = np.zeros(len(rows), np.float32)
    Wr, mr, rg, cnt, nv = oracle.rows_update(wl, rows, Wr0, m0, r["G"])
    np.testing.assert_array_equal(cnt, r["counts"][rows])
    assert nv == wl.N
    touched = cnt > 0
    assert touched.sum() > 200
    assert cnt.max() > 256 * 20            # the hottest rows went through many chunks
    assert_momentum_close(r["m_rows"], mr, m0, touched)
    assert_weights_close(wbits_np(r["W_rows1"], wl.dtype), Wr, Wr0, touched, wl.dtype)


def test_inversion_properties_full_size(large_step):
    r = large_step
    wl = r["wl"]
    sk = r["sorted_keys"].view(np.uint32).astype(np.int64)
    sv = r["sorted_vals"].view(np.uint32).astype(np.int64)
    assert r["nv"] == wl.N                                  # no out-of-range lookups
    assert np.all(np.diff(sk) >= 0)
    # (key, bag) pairs: the stable order equals the lexicographic order
    bag_b = np.repeat(np.arange(wl.NB, dtype=np.int64), np.diff(wl.offsets.astype(np.int64))) % wl.B
    ref = np.sort(r["keys_all"] * wl.B + bag_b)
    np.testing.assert_array_equal(sk * wl.B + sv, ref)
    # run table against the key counts
    nz = np.flatnonzero(r["counts"])
    assert r["U"] == len(nz)
    np.testing.assert_array_equal(r["unique_keys"].view(np.uint32).astype(np.int64), nz)
    np.testing.assert_array_equal(np.diff(r["seg_off"].astype(np.int64)), r["counts"][nz])
    rl = r["counts"][nz]
    assert r["nlong"] == int((rl >= 256).sum())
    assert r["nchunks"] == int(((rl[rl >= 256] + 255) // 256).sum())
    # the workload's statistics are the pages' (within 5%)
    assert abs(r["U"] - 3.0e6) / 3.0e6 < 0.05
    assert abs(rl.max() - 125e3) / 125e3 < 0.05
