"""Full-size parity in the launch configuration the benchmark times:

  * large Zipf workload (T=32, E=2M, D=128, bf16, B=131072, ~84M lookups,
    preprocessing in the forward), with the default two-kernel long-run mode
    (grad_accum + apply) and with the fused single-launch mode;
  * mid workload (T=32, E=1M, D=128, fp16, B=16384, ~16.8M lookups,
    per-sample weights on tables 0-15, preprocessing at the start of the
    backward).

The oracle cannot run the whole step in test time, so:
  * forward: a sample of bags recomputed by the oracle, one by one;
  * backward: a sample of rows (the hottest ones, which take the chunked
    path, and random ones from the short-run path) recomputed by the oracle
    from one scan of all lookups;
  * batch inversion: properties that hold at any size -- sorted order,
    (key, payload) multiset equal to the input's, run table equal to the key
    counts, unique count -- and, for the large workload, the pages' printed
    statistics.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import (assert_momentum_close, assert_out_close, assert_weights_close, device_batch,
                    w_arith_bound, wbits_np, wvals_np)

pytestmark = pytest.mark.gpu

CASES = {"large": (workloads.large, True), "mid": (workloads.mid, False)}


def _keys(wl):
    return (wl.table_offset[np.repeat(np.arange(wl.T), np.diff(wl.offsets[::wl.B]))]
            + wl.indices.astype(np.int64))


def _step(wl, pif, long_mode=0):
    """One full-size step; returns device W, momentum, out and the TBE."""
    from recsys_table_embedding_gb300 import TBE, Tables, config
    dev = torch.device("cuda")
    W = wl.weights(device="cuda")
    tables = Tables(W, wl.table_offset)
    batch = device_batch(wl)
    tbe = TBE(tables, batch, config(long_run_mode=long_mode), preprocess_in_forward=pif)
    mom = torch.zeros(wl.rows_total, dtype=torch.float32, device=dev)
    out = tbe.forward(batch)
    tbe.backward(batch, mom, torch.from_numpy(wl.grad_out()).to(dev), wl.lr, wl.eps)
    torch.cuda.synchronize()
    return W, mom, out, tbe


@pytest.fixture(scope="module", params=sorted(CASES))
def full_step(request):
    from recsys_table_embedding_gb300 import meta_view
    make, pif = CASES[request.param]
    wl = make()
    dev = torch.device("cuda")
    G = wl.grad_out()
    rng = np.random.default_rng(5)
    keys_all = _keys(wl)
    counts = np.bincount(keys_all, minlength=wl.rows_total)
    hot = np.argsort(-counts, kind="stable")[:24]
    touched = np.flatnonzero(counts)
    sample_rows = np.unique(np.concatenate([hot, rng.choice(touched, 200, replace=False),
                                            rng.choice(wl.rows_total, 20, replace=False)]))
    rows_t = torch.from_numpy(sample_rows).to(dev)
    bags = np.sort(rng.choice(wl.NB, 300, replace=False))
    need = np.unique(np.concatenate([keys_all[wl.offsets[g]:wl.offsets[g + 1]] for g in bags]))
    W0 = wl.weights(device="cuda")
    W_rows0 = W0.index_select(0, rows_t).cpu()
    fw_W = W0.index_select(0, torch.from_numpy(need).to(dev)).cpu()
    del W0
    W, mom, out, tbe = _step(wl, pif)
    U, nv, nlong, nchunks = tbe.counters()
    res = dict(name=request.param, wl=wl, G=G, pif=pif, counts=counts, keys_all=keys_all,
               sample_rows=sample_rows, W_rows0=W_rows0, W_rows1=W.index_select(0, rows_t).cpu(),
               m_rows=mom.index_select(0, rows_t).cpu().numpy(), bags=bags,
               out_bags=out.cpu().numpy(), status=tbe.status.cpu().numpy(), U=U, nv=nv,
               nlong=nlong, nchunks=nchunks, fw_rows=need, fw_W=fw_W,
               payload_is_pos=tbe.meta.c.payload_is_pos,
               sorted_keys=meta_view(tbe.meta, "sorted_keys", wl.N, torch.int32).cpu().numpy(),
               sorted_vals=meta_view(tbe.meta, "sorted_vals", wl.N, torch.int32).cpu().numpy(),
               unique_keys=meta_view(tbe.meta, "unique_keys", U, torch.int32).cpu().numpy(),
               seg_off=meta_view(tbe.meta, "seg_off", U + 1, torch.int32).cpu().numpy())
    del W, mom, out, tbe
    torch.cuda.empty_cache()
    return res


def test_forward_sampled_bags(full_step):
    r = full_step
    wl = r["wl"]
    need, Wn = r["fw_rows"], r["fw_W"]
    # a one-table sub-problem holding just the sampled bags and their rows
    offs, idx, psw = [0], [], []
    for g in r["bags"]:
        t = g // wl.B
        s, e = wl.offsets[g], wl.offsets[g + 1]
        idx.extend(np.searchsorted(need, r["keys_all"][s:e]).tolist())
        wtd = wl.per_sample_weights is not None and wl.weighted_tables[t]
        psw.extend(wl.per_sample_weights[s:e].tolist() if wtd else [1.0] * (e - s))
        offs.append(len(idx))
    sub = workloads.Workload(name="s", T=1, B=len(r["bags"]), D=wl.D, dtype=wl.dtype,
                             table_rows=np.array([len(need)]), offsets=np.array(offs, np.int32),
                             indices=np.array(idx, np.int32),
                             per_sample_weights=np.array(psw, np.float32), weighted_tables=None)
    ref, ab, _, _ = oracle.forward(sub, wbits_np(Wn, wl.dtype), want_abs=True)
    dev_rows = np.stack([r["out_bags"][g % wl.B, (g // wl.B) * wl.D:(g // wl.B + 1) * wl.D]
                         for g in r["bags"]])
    assert_out_close(dev_rows, ref, ab, wl.dtype)
    assert r["status"][0] == 0 and r["status"][1] == 0


def test_backward_sampled_rows(full_step):
    r = full_step
    wl = r["wl"]
    rows = r["sample_rows"]
    Wr0 = wbits_np(r["W_rows0"], wl.dtype)
    m0 = np.zeros(len(rows), np.float32)
    Wr, mr, rg, cnt, nv, ra = oracle.rows_update(wl, rows, Wr0, m0, r["G"], want_row_abs=True)
    np.testing.assert_array_equal(cnt, r["counts"][rows])
    assert nv == wl.N
    touched = cnt > 0
    assert touched.sum() > 200
    assert cnt.max() > 256 * 20            # the hottest rows went through many chunks
    assert_momentum_close(r["m_rows"], mr, m0, touched)
    arith = w_arith_bound(wl.dtype, rg[touched], ra[touched], cnt[touched], m0[touched],
                          wvals_np(Wr0[touched], wl.dtype), wl.lr, wl.eps)
    assert_weights_close(wbits_np(r["W_rows1"], wl.dtype), Wr, Wr0, touched, wl.dtype, arith)


def test_inversion_properties_full_size(full_step):
    r = full_step
    wl = r["wl"]
    sk = r["sorted_keys"].view(np.uint32).astype(np.int64)
    sv = r["sorted_vals"].view(np.uint32).astype(np.int64)
    assert r["nv"] == wl.N                                  # no out-of-range lookups
    assert np.all(np.diff(sk) >= 0)
    # (key, payload) pairs: the stable order equals the lexicographic order
    if r["payload_is_pos"]:
        ref = np.sort(r["keys_all"] * wl.N + np.arange(wl.N))
        np.testing.assert_array_equal(sk * wl.N + sv, ref)
    else:
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
    if r["name"] == "large":
        # the workload's statistics are the pages' (within 5%)
        assert abs(r["U"] - 3.0e6) / 3.0e6 < 0.05
        assert abs(rl.max() - 125e3) / 125e3 < 0.05


def test_fused_long_run_mode_full_size(full_step):
    # the fused single-launch long-run mode sums the chunk partials in the
    # same order as grad_accum + apply: bit-identical weights and momentum
    r = full_step
    if r["name"] != "large":
        pytest.skip("one workload is enough")
    wl = r["wl"]
    W, mom, _, tbe = _step(wl, r["pif"], long_mode=2)
    rows_t = torch.from_numpy(r["sample_rows"]).to("cuda")
    np.testing.assert_array_equal(wbits_np(W.index_select(0, rows_t), wl.dtype),
                                  wbits_np(r["W_rows1"], wl.dtype))
    np.testing.assert_array_equal(mom.index_select(0, rows_t).cpu().numpy(), r["m_rows"])
    assert tbe.status.cpu().numpy()[1] == 0
    del W, mom, tbe
    torch.cuda.empty_cache()
