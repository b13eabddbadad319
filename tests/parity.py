"""Shared helpers of the parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, compare with the stated tolerances.

Tolerances (the stated bars, read for the cases they leave open):
  * batch inversion (sorted keys/payloads, unique keys, segment offsets,
    counts): bit-exact.
  * forward output: |dev - ref| <= rtol * S where S = sum_p |w_p W[idx_p, d]|
    is the oracle's sum of magnitudes (S = |ref| when nothing cancels);
    rtol = 1e-4, or 1e-6 for FP32 tables.  Any summation order of the terms
    stays inside n * 2^-24 * S for FP32 accumulation.
  * momentum: |dev - ref| <= 1e-4 |ref| (all its terms are non-negative).
  * FP32 weights: |dev - ref| <= 1e-6 * max(|ref|, |W_old|), the scale of the
    operands of the final subtraction W_old - update.
  * FP16/BF16 weights: |dev - ref| <= 1 ulp of the stored type at
    max(|ref|, |W_old|).
  * rows no lookup touches: weights and momentum bit-identical to the input.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

OUT_RTOL = {"f32": 1e-6, "f16": 1e-4, "bf16": 1e-4}
MOM_RTOL = 1e-4
W32_RTOL = 1e-6


def wbits_np(W: torch.Tensor, dtype: str) -> np.ndarray:
    W = W.detach().cpu().contiguous()
    if dtype == "f32":
        return W.numpy().copy()
    return W.view(torch.int16).numpy().view(np.uint16).copy()


def wvals_np(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return bits.astype(np.float64)
    t = torch.from_numpy(bits.view(np.int16))
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16).to(torch.float64).numpy()


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the stored type at magnitude |x|."""
    mant, emin = (10, -14) if dtype == "f16" else (7, -126)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - mant).astype(np.int64))


def assert_out_close(dev: np.ndarray, ref: np.ndarray, absum: np.ndarray, dtype: str):
    rtol = OUT_RTOL[dtype]
    err = np.abs(dev.astype(np.float64) - ref.astype(np.float64))
    bound = rtol * absum + 1e-30
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"forward out: {int(bad.sum())} elements off, first at {tuple(i)}: "
                             f"dev={dev[tuple(i)]!r} ref={ref[tuple(i)]!r} bound={bound[tuple(i)]!r}")


def assert_momentum_close(dev: np.ndarray, ref: np.ndarray, m0: np.ndarray, touched: np.ndarray):
    np.testing.assert_array_equal(dev[~touched], m0[~touched], err_msg="untouched momentum changed")
    err = np.abs(dev[touched].astype(np.float64) - ref[touched].astype(np.float64))
    bound = MOM_RTOL * np.abs(ref[touched].astype(np.float64))
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0][0]
        raise AssertionError(f"momentum: {int(bad.sum())} rows off, first: dev={dev[touched][i]!r} "
                             f"ref={ref[touched][i]!r}")


def assert_weights_close(dev_bits: np.ndarray, ref_bits: np.ndarray, old_bits: np.ndarray,
                         touched: np.ndarray, dtype: str):
    np.testing.assert_array_equal(dev_bits[~touched], old_bits[~touched],
                                  err_msg="untouched weight rows changed")
    d = wvals_np(dev_bits[touched], dtype)
    r = wvals_np(ref_bits[touched], dtype)
    o = wvals_np(old_bits[touched], dtype)
    scale = np.maximum(np.abs(r), np.abs(o))
    bound = W32_RTOL * scale if dtype == "f32" else ulp(scale, dtype)
    err = np.abs(d - r)
    bad = err > bound
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"weights: {int(bad.sum())} elements off, first {i}: dev={d[i]!r} "
                             f"ref={r[i]!r} old={o[i]!r} bound={bound[i]!r}")


def touched_rows(wl) -> np.ndarray:
    tab = (np.searchsorted(wl.offsets, np.arange(wl.N), side="right") - 1) // wl.B
    ok = (wl.indices >= 0) & (wl.indices < wl.table_rows[tab])
    t = np.zeros(wl.rows_total, bool)
    t[(wl.table_offset[tab] + wl.indices)[ok]] = True
    return t


def device_batch(wl, device="cuda"):
    from recsys_table_embedding_gb300 import Batch
    idx = torch.from_numpy(wl.indices).to(device)
    off = torch.from_numpy(wl.offsets).to(device)
    psw = torch.from_numpy(wl.per_sample_weights).to(device) if wl.per_sample_weights is not None else None
    wt = torch.from_numpy(wl.weighted_tables).to(device) if wl.weighted_tables is not None else None
    return Batch(idx, off, wl.B, psw, wt)


def run_cuda(wl, W0: torch.Tensor, G: np.ndarray, m0: np.ndarray, cfg=None,
             preprocess_in_forward=True, device="cuda"):
    """One forward + backward through the C ABI.  Returns a dict of host arrays."""
    from recsys_table_embedding_gb300 import TBE, Tables, meta_view
    W = W0.to(device).contiguous()
    tables = Tables(W, wl.table_offset)
    batch = device_batch(wl, device)
    tbe = TBE(tables, batch, cfg, preprocess_in_forward=preprocess_in_forward)
    out = tbe.forward(batch)
    mom = torch.from_numpy(m0).to(device)
    Gd = torch.from_numpy(G).to(device)
    tbe.backward(batch, mom, Gd, wl.lr, wl.eps)
    torch.cuda.synchronize()
    res = dict(out=out.cpu().numpy(), W=wbits_np(W, wl.dtype), mom=mom.cpu().numpy(),
               status=tbe.status.cpu().numpy(), path=tbe.path, tbe=tbe)
    if tbe.path == 1:
        m = tbe.meta
        U, nv, nlong, nchunks = tbe.counters()
        res.update(num_unique=U, n_valid=nv, num_long=nlong, num_chunks=nchunks)
        res["sorted_keys"] = meta_view(m, "sorted_keys", wl.N, torch.int32).cpu().numpy().view(np.uint32)
        res["sorted_vals"] = meta_view(m, "sorted_vals", wl.N, torch.int32).cpu().numpy().view(np.uint32)
        res["unique_keys"] = meta_view(m, "unique_keys", U, torch.int32).cpu().numpy().view(np.uint32)
        res["seg_off"] = meta_view(m, "seg_off", U + 1, torch.int32).cpu().numpy()
        res["payload_is_pos"] = m.c.payload_is_pos
    return res


def bag_of_position(wl) -> np.ndarray:
    return np.repeat(np.arange(wl.NB, dtype=np.int64), np.diff(wl.offsets.astype(np.int64)))


def check_inversion(wl, res, pre):
    """Bit-exact comparison of the batch inversion with the oracle's."""
    nv = pre["n_valid"]
    assert res["n_valid"] == nv
    assert res["num_unique"] == pre["num_unique"]
    np.testing.assert_array_equal(res["sorted_keys"][:nv].astype(np.int64), pre["sorted_keys"])
    assert np.all(res["sorted_keys"][nv:] == wl.rows_total), "out-of-range lookups not last"
    if res["payload_is_pos"]:
        np.testing.assert_array_equal(res["sorted_vals"][:nv].astype(np.int64), pre["sorted_pos"])
    else:
        bag = bag_of_position(wl)[pre["sorted_pos"]]
        np.testing.assert_array_equal(res["sorted_vals"][:nv].astype(np.int64), bag % wl.B)
    np.testing.assert_array_equal(res["unique_keys"].astype(np.int64), pre["unique_keys"])
    np.testing.assert_array_equal(res["seg_off"].astype(np.int64), pre["seg_off"])
    rl = pre["run_len"]
    assert res["num_long"] == int((rl >= 256).sum())
    assert res["num_chunks"] == int(((rl[rl >= 256] + 255) // 256).sum())


def check_full(wl, W0: torch.Tensor, G: np.ndarray, m0: np.ndarray, res: dict, pre=None):
    """Compare a full CUDA step with the oracle: forward, inversion, backward."""
    wb = wbits_np(W0, wl.dtype)
    out, ab, oob, bad = oracle.forward(wl, wb, want_abs=True)
    assert_out_close(res["out"], out, ab, wl.dtype)
    assert int(res["status"][0]) == oob
    if res["path"] == 1:
        if pre is None:
            pre = oracle.preprocess(wl)
        check_inversion(wl, res, pre)
    Wn, mn, U, _, _ = oracle.backward_adagrad(wl, wb, m0, G)
    touched = touched_rows(wl)
    assert U == int(touched.sum())
    assert_momentum_close(res["mom"], mn, m0, touched)
    assert_weights_close(res["W"], Wn, wb, touched, wl.dtype)
