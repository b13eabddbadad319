"""Shared helpers of the parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, compare with the stated tolerances.

The stated bars, asserted element by element:
  * batch inversion (sorted keys/payloads, unique keys, segment offsets,
    counts): bit-exact.
  * forward output: |dev - ref| <= 1e-4 |ref|, with a floor of
    1e-6 max|ref| for elements that cancel to near zero.
  * momentum: |dev - ref| <= 1e-4 |ref|.
  * FP32 weights: |dev - ref| <= 1e-6 |ref| (+ the FP64 arithmetic bound
    below, which is ~1e-18 and matters only for a weight that cancels to
    almost exactly zero).
  * FP16/BF16 weights: |dev - ref| <= 1 ulp of the stored type at |ref|,
    plus the error bound E of the arithmetic the pages prescribe for these
    tables (FP32 accumulation of the row gradient, decision checklist item 1;
    FP32 optimizer arithmetic): where the update nearly cancels the old
    weight, a correct FP32 kernel can land more than one ulp of the small
    result away from the exact one.  E is derived from the oracle's row
    gradient g, the sum A of its terms' magnitudes and the run length n
    (see ``w_arith_bound``); the tests report how many elements needed it.
  * rows no lookup touches: weights and momentum bit-identical to the input.

Second reading, also asserted (kept from the scale-aware bars): forward
within rtol * S, S = sum_p |w_p W[idx_p, d]| (rtol 1e-4, 1e-6 for FP32
tables), and weights within 1 ulp (rel 1e-6) of max(|ref|, |W_old|).

``REPORT`` collects the largest observed error of each quantity relative to
its stated bar; the tests print it.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

OUT_RTOL = {"f32": 1e-6, "f16": 1e-4, "bf16": 1e-4}
OUT_STATED_RTOL = 1e-4
OUT_FLOOR = 1e-6
MOM_RTOL = 1e-4
W32_RTOL = 1e-6
U32 = 2.0 ** -24
U64 = 2.0 ** -53

REPORT: dict = {}


def _record(name, ratio):
    if ratio.size:
        REPORT[name] = max(REPORT.get(name, 0.0), float(np.max(ratio)))


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
    dev = dev.astype(np.float64)
    ref = ref.astype(np.float64)
    err = np.abs(dev - ref)
    # stated bar: rel 1e-4, floor 1e-6 max|ref| for near-zero elements
    amax = float(np.max(np.abs(ref))) if ref.size else 0.0
    stated = np.maximum(OUT_STATED_RTOL * np.abs(ref), OUT_FLOOR * amax)
    bad = err > stated
    _record("out/stated_bar", err / np.maximum(stated, 1e-300))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"forward out: {int(bad.sum())} elements off the stated bar, first at "
                             f"{i}: dev={dev[i]!r} ref={ref[i]!r} bar={stated[i]!r}")
    # scale-aware bar: any summation order is within n 2^-24 S
    bound = OUT_RTOL[dtype] * absum + 1e-30
    bad = err > bound
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"forward out: {int(bad.sum())} elements off, first at {i}: "
                             f"dev={dev[i]!r} ref={ref[i]!r} bound={bound[i]!r}")


def assert_momentum_close(dev: np.ndarray, ref: np.ndarray, m0: np.ndarray, touched: np.ndarray):
    np.testing.assert_array_equal(dev[~touched], m0[~touched], err_msg="untouched momentum changed")
    err = np.abs(dev[touched].astype(np.float64) - ref[touched].astype(np.float64))
    bound = MOM_RTOL * np.abs(ref[touched].astype(np.float64))
    _record("momentum/stated_bar", err / np.maximum(bound, 1e-300))
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0][0]
        raise AssertionError(f"momentum: {int(bad.sum())} rows off, first: dev={dev[touched][i]!r} "
                             f"ref={ref[touched][i]!r}")


def w_arith_bound(dtype: str, g: np.ndarray, A: np.ndarray, n: np.ndarray, m_old: np.ndarray,
                  w_old: np.ndarray, lr: float, eps: float, path: int = 1) -> np.ndarray:
    """Bound on |w - w_exact| before the final rounding to the stored type,
    for the arithmetic the kernels are specified to use, per element [k, D].

    g, A: the exact row gradient and the sum of its terms' magnitudes [k, D];
    n: lookups of each row [k]; m_old: momentum before the step [k]; w_old:
    weights before the step [k, D].  Unit roundoff u = 2^-53 for FP32 tables
    (FP64 accumulation and optimizer), 2^-24 otherwise (FP32).  First-order
    error propagation, doubled:
      |g~ - g| <= d = gamma_n A,  gamma_n = (n + n/256 + 4) u  (terms, chunk
                   partials and lane combines)
      histogram path: + 2^-21 A + n 2^-24 (FP16 hi/lo split of the gradient)
      m = m_old + sum_d g^2 / D, relative error e_m from d and D-term sums
      den = sqrt(m) + eps, relative error e_den = (e_m/2 + u) sqrt(m)/den + u
      upd = lr g / den:  |upd~ - upd| <= |upd| (2u + e_den) + lr d / den
      w = w_old - upd:   + u (|w_old| + |upd|)
    """
    u = U64 if dtype == "f32" else U32
    g = np.asarray(g, np.float64)
    A = np.asarray(A, np.float64)
    n = np.asarray(n, np.float64)[:, None]
    D = g.shape[1]
    delta = (n + n / 256.0 + 4.0) * u * 1.01 * A
    if path == 2:
        delta = delta + 2.0 ** -21 * A + n * 2.0 ** -24
    ss = np.sum(g * g, axis=1)
    m = np.asarray(m_old, np.float64) + ss / D
    gam_d = (D + 4) * u
    num = u * m + u * ss / D + (gam_d * ss + np.sum(2 * np.abs(g) * delta + delta * delta, axis=1)) / D
    e_m = np.where(m > 0, num / np.where(m > 0, m, 1.0), 0.0)
    sq = np.sqrt(m)
    den = sq + eps
    e_den = (e_m / 2 + u) * sq / den + u
    upd = lr * np.abs(g) / den[:, None]
    E = u * (np.abs(w_old) + upd) + upd * (2 * u + e_den[:, None]) + lr * delta / den[:, None]
    return 2.0 * E


def assert_weights_close(dev_bits: np.ndarray, ref_bits: np.ndarray, old_bits: np.ndarray,
                         touched: np.ndarray, dtype: str, arith: np.ndarray = None):
    """arith: w_arith_bound for the touched rows (in row order), or None to
    assert only the scale-aware second reading."""
    np.testing.assert_array_equal(dev_bits[~touched], old_bits[~touched],
                                  err_msg="untouched weight rows changed")
    d = wvals_np(dev_bits[touched], dtype)
    r = wvals_np(ref_bits[touched], dtype)
    o = wvals_np(old_bits[touched], dtype)
    err = np.abs(d - r)
    if arith is not None:
        if dtype == "f32":
            stated = W32_RTOL * np.abs(r)
            _record("W_f32/stated_bar", err / np.maximum(stated, 1e-300))
            bar = stated + arith
        else:
            stated = ulp(r, dtype)
            _record(f"W_{dtype}/ulps_of_ref", err / stated)
            REPORT[f"W_{dtype}/elements_beyond_1ulp"] = (
                REPORT.get(f"W_{dtype}/elements_beyond_1ulp", 0) + int(np.sum(err > stated)))
            bar = ulp(np.abs(r) + arith, dtype) + arith
        bad = err > bar
        if bad.any():
            i = tuple(np.argwhere(bad)[0])
            raise AssertionError(f"weights: {int(bad.sum())} elements off the stated bar, first {i}: "
                                 f"dev={d[i]!r} ref={r[i]!r} old={o[i]!r} bar={bar[i]!r}")
    scale = np.maximum(np.abs(r), np.abs(o))
    bound = W32_RTOL * scale if dtype == "f32" else ulp(scale, dtype)
    bad = err > bound
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"weights: {int(bad.sum())} elements off, first {i}: dev={d[i]!r} "
                             f"ref={r[i]!r} old={o[i]!r} bound={bound[i]!r}")


def bag_tables(wl, g: np.ndarray) -> np.ndarray:
    """Table of each CSR bag id."""
    starts = np.array([L["bag_off"] for L in wl.layout()], np.int64)
    return np.searchsorted(starts, g, side="right") - 1


def touched_rows(wl) -> np.ndarray:
    tab = bag_tables(wl, np.searchsorted(wl.offsets, np.arange(wl.N), side="right") - 1)
    ok = (wl.indices >= 0) & (wl.indices < wl.table_rows[tab])
    t = np.zeros(wl.rows_total, bool)
    t[(wl.table_offset[tab] + wl.indices)[ok]] = True
    return t


def shaped(wl) -> bool:
    """Tables of different D or dtype (weights in one byte buffer)."""
    return wl.table_dims is not None or wl.table_dtypes is not None


def device_batch(wl, device="cuda", unaligned_indices=False):
    """The workload's batch on the device; unaligned_indices places the
    indices one element past a 16-byte boundary."""
    from recsys_table_embedding_gb300 import Batch
    idx = torch.from_numpy(wl.indices).to(device)
    if unaligned_indices:
        buf = torch.empty(idx.numel() + 1, dtype=idx.dtype, device=device)
        buf[1:].copy_(idx)
        idx = buf[1:]
        assert idx.data_ptr() % 16 != 0
    off = torch.from_numpy(wl.offsets).to(device)
    psw = torch.from_numpy(wl.per_sample_weights).to(device) if wl.per_sample_weights is not None else None
    wt = torch.from_numpy(wl.weighted_tables).to(device) if wl.weighted_tables is not None else None
    if wl.mixed:
        return Batch(idx, off, wl.B, psw, wt, bag_layout=wl.layout(), out_size=wl.out_size)
    return Batch(idx, off, wl.B, psw, wt)


def table_storage(wl, W: np.ndarray, t: int) -> np.ndarray:
    """Table t's rows [E_t, D_t] as stored (float32, or uint16 bits) out of a
    weight buffer (bytes laid out as wl.layout(), or a uniform array)."""
    L = wl.layout()[t]
    E = int(wl.table_rows[t])
    if W.dtype != np.uint8:
        to = wl.table_offset
        return W[to[t]:to[t + 1]]
    nbytes = E * L["D"] * (4 if L["dtype"] == "f32" else 2)
    raw = W[L["wbyte"]:L["wbyte"] + nbytes]
    return raw.view(np.float32 if L["dtype"] == "f32" else np.uint16).reshape(E, L["D"])


def table_out(wl, out: np.ndarray, t: int) -> np.ndarray:
    """Table t's pooled rows [B_t, D_t] out of a flat out / grad_out."""
    L = wl.layout()[t]
    flat = out.reshape(-1)
    if wl.vbe:
        return flat[L["out_off"]:L["out_off"] + L["B"] * L["D"]].reshape(L["B"], L["D"])
    return flat.reshape(wl.B, -1)[:, L["out_off"]:L["out_off"] + L["D"]]


def run_cuda(wl, W0: torch.Tensor, G: np.ndarray, m0: np.ndarray, cfg=None,
             preprocess_in_forward=True, device="cuda", meta_fill=None, unaligned_indices=False):
    """One forward + backward through the C ABI.  Returns a dict of host arrays.
    meta_fill (a byte value) fills the metadata buffer before the first call,
    in place of whatever a fresh device allocation holds."""
    from recsys_table_embedding_gb300 import TBE, Tables, meta_view
    if isinstance(W0, np.ndarray):       # a byte buffer of tables of different shapes
        W = torch.from_numpy(W0).to(device)
        tables = Tables(W, wl.table_offset, layout=wl.layout())
    else:
        W = W0.to(device).contiguous()
        tables = Tables(W, wl.table_offset)
    batch = device_batch(wl, device, unaligned_indices)
    tbe = TBE(tables, batch, cfg, preprocess_in_forward=preprocess_in_forward)
    if meta_fill is not None:
        tbe.meta_buf.fill_(meta_fill)
    out = tbe.forward(batch)
    mom = torch.from_numpy(m0).to(device)
    Gd = torch.from_numpy(G).to(device)
    tbe.backward(batch, mom, Gd, wl.lr, wl.eps)
    torch.cuda.synchronize()
    Wh = W.cpu().numpy() if W.dtype == torch.uint8 else wbits_np(W, wl.dtype)
    res = dict(out=out.cpu().numpy(), W=Wh, mom=mom.cpu().numpy(),
               status=tbe.status.cpu().numpy(), path=tbe.path, tbe=tbe)
    if tbe.path == 1:
        m = tbe.meta
        U, nv, nlong, nchunks = tbe.counters()
        res.update(num_unique=U, n_valid=nv, num_long=nlong, num_chunks=nchunks)
        res["sorted_keys"] = meta_keys(m, "sorted_keys", wl.N)
        res["sorted_vals"] = meta_view(m, "sorted_vals", wl.N, torch.int32).cpu().numpy().view(np.uint32)
        res["unique_keys"] = meta_keys(m, "unique_keys", U)
        res["key_bytes"] = m.c.key_bytes
        res["seg_off"] = meta_view(m, "seg_off", U + 1, torch.int32).cpu().numpy()
        res["payload_is_pos"] = m.c.payload_is_pos
    return res


def meta_keys(meta, name: str, n: int) -> np.ndarray:
    """n keys of a meta key array (4 or 8 bytes per key) as int64."""
    from recsys_table_embedding_gb300 import meta_view
    if meta.c.key_bytes == 8:
        return meta_view(meta, name, n, torch.int64).cpu().numpy()
    return meta_view(meta, name, n, torch.int32).cpu().numpy().view(np.uint32).astype(np.int64)


def bag_of_position(wl, pos: np.ndarray) -> np.ndarray:
    """Bag id t*B+b of the given lookup positions, each of which lies in a
    well-formed bag (every position the inversion keeps does, and offsets
    then never decrease, so a binary search finds the bag)."""
    return np.searchsorted(wl.offsets.astype(np.int64), pos, side="right") - 1


def check_inversion(wl, res, pre):
    """Bit-exact comparison of the batch inversion with the oracle's."""
    nv = pre["n_valid"]
    assert res["n_valid"] == nv
    assert res["num_unique"] == pre["num_unique"]
    np.testing.assert_array_equal(res["sorted_keys"][:nv], pre["sorted_keys"])
    assert np.all(res["sorted_keys"][nv:] == wl.rows_total), "out-of-range lookups not last"
    if res["payload_is_pos"]:
        np.testing.assert_array_equal(res["sorted_vals"][:nv].astype(np.int64), pre["sorted_pos"])
    else:
        bag = bag_of_position(wl, pre["sorted_pos"])
        starts = np.array([L["bag_off"] for L in wl.layout()], np.int64)
        np.testing.assert_array_equal(res["sorted_vals"][:nv].astype(np.int64),
                                      bag - starts[bag_tables(wl, bag)])
    np.testing.assert_array_equal(res["unique_keys"].astype(np.int64), pre["unique_keys"])
    np.testing.assert_array_equal(res["seg_off"].astype(np.int64), pre["seg_off"])
    rl = pre["run_len"]
    assert res["num_long"] == int((rl >= 256).sum())
    assert res["num_chunks"] == int(((rl[rl >= 256] + 255) // 256).sum())


def check_full(wl, W0, G: np.ndarray, m0: np.ndarray, res: dict, pre=None):
    """Compare a full CUDA step with the oracle: forward, inversion, backward.
    W0: the initial weights (torch tensor, or the byte buffer of tables of
    different shapes)."""
    wb = W0 if isinstance(W0, np.ndarray) else wbits_np(W0, wl.dtype)
    out, ab, oob, bad = oracle.forward(wl, wb, want_abs=True)
    if wl.mixed:
        for t in range(wl.T):
            assert_out_close(table_out(wl, res["out"], t), table_out(wl, out, t), table_out(wl, ab, t),
                             wl.dtype_t(t))
    else:
        assert_out_close(res["out"], out, ab, wl.dtype)
    assert int(res["status"][0]) == oob
    malformed = oracle.offsets_check(wl)[0]
    assert bool(res["status"][1] & 0x1) == malformed, "TBE_FLAG_BAD_OFFSETS"
    if res["path"] == 1:
        if pre is None:
            pre = oracle.preprocess(wl)
        check_inversion(wl, res, pre)
    Wn, mn, U, _, _, runs = oracle.backward_adagrad(wl, wb, m0, G, want_runs=True)
    touched = np.zeros(wl.rows_total, bool)
    touched[runs["keys"]] = True
    if not malformed:
        assert np.array_equal(touched, touched_rows(wl))
    assert U == int(touched.sum())
    assert_momentum_close(res["mom"], mn, m0, touched)
    k = runs["keys"]
    to = wl.table_offset
    for t in range(wl.T if wl.mixed else 1):
        # one table at a time (all at once when they share D and dtype)
        lo, hi = (to[t], to[t + 1]) if wl.mixed else (0, wl.rows_total)
        sel = (k >= lo) & (k < hi)
        dt, D = (wl.dtype_t(t), wl.Dt(t)) if wl.mixed else (wl.dtype, wl.D)
        old = table_storage(wl, wb, t) if wl.mixed else wb
        arith = w_arith_bound(dt, runs["grad"][sel][:, :D], runs["abs"][sel][:, :D], runs["count"][sel],
                              m0[k[sel]], wvals_np(old[k[sel] - lo], dt), wl.lr, wl.eps, res["path"])
        dev = table_storage(wl, res["W"], t) if wl.mixed else res["W"]
        ref = table_storage(wl, Wn, t) if wl.mixed else Wn
        assert_weights_close(dev, ref, old, touched[lo:hi], dt, arith)
