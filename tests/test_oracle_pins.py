"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks one oracle function against something fixed independently:
a brute-force dense formulation, a different library routine, a closed form,
an invariant of the method, or a value printed on the pages.  A plausible
mistake in the oracle (a dropped term, a wrong sign or index, a transposed
operand, an unstable sort, a double update) fails at least one of them.
"""
import collections
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


def small(dtype="f32", weighted=False, oob=0.0, seed=5, D=8, B=37, lengths=("poisson", 4.0),
          dist=("zipf", 1.1), rows=(13, 29, 7)):
    T = len(rows)
    return workloads.make_workload("pin", T=T, table_rows=list(rows), D=D, dtype=dtype, B=B,
                                   lengths=lengths, dist=dist, seed=seed,
                                   weighted=[t % 2 == 0 for t in range(T)] if weighted else None,
                                   oob_frac=oob)


def wbits(wl, W):
    """torch weights -> oracle storage (float32 or uint16 bit patterns)"""
    if wl.dtype == "f32":
        return W.numpy()
    return W.view(torch.int16).numpy().view(np.uint16)


def wvalues(wl, W):
    return W.to(torch.float64).numpy()


def dense_A(wl, t):
    """A_t[b, e] = sum_p w_p [idx_p == e] over in-range lookups of bag (t, b)."""
    E = int(wl.table_rows[t])
    A = np.zeros((wl.B, E), np.float64)
    for b in range(wl.B):
        g = t * wl.B + b
        for p in range(wl.offsets[g], wl.offsets[g + 1]):
            e = int(wl.indices[p])
            if 0 <= e < E:
                w = 1.0
                if wl.per_sample_weights is not None and wl.weighted_tables[t]:
                    w = float(wl.per_sample_weights[p])
                A[b, e] += w
    return A


# ---------------------------------------------------------------- conversions

def test_half_conversion_matches_numpy():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 4000),
        np.array([0.0, -0.0, 65504, 65519.99, 65520, 1e9, -1e9, 2**-24, 2**-25, 2**-25 * 1.5,
                  6.1e-5, 5.96e-8, np.inf, -np.inf], np.float32)])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.to_half_bits(float(v)) for v in x], np.uint16)
    np.testing.assert_array_equal(got, ref)
    # single rounding from double: 1 + 2^-11 + 2^-40 lies just above the tie
    # between 1 and 1 + 2^-10, so it rounds up (a detour through float32
    # would land on the tie and round to even, down to 1.0)
    assert oracle.to_half_bits(1 + 2**-11 + 2**-40) == 0x3C01
    assert oracle.to_half_bits(1 + 2**-11) == 0x3C00          # tie -> even
    assert oracle.to_half_bits(1 + 3 * 2**-11) == 0x3C02      # tie -> even (up)
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    for b, v in zip(bits[:3000], vals[:3000]):
        o = oracle.from_half_bits(int(b))
        assert (math.isnan(o) and math.isnan(v)) or o == v


def test_bf16_conversion_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 4000),
        np.array([0.0, -0.0, 3.3895314e38, 3.4e38, 1e-38, 1e-40, 1e-45, np.inf, -np.inf],
                 np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.to_bf16_bits(float(v)) for v in x], np.uint16)
    np.testing.assert_array_equal(got, ref)
    assert oracle.to_bf16_bits(1 + 2**-8) == 0x3F80          # tie -> even (down)
    assert oracle.to_bf16_bits(1 + 3 * 2**-8) == 0x3F82      # tie -> even (up)
    assert oracle.to_bf16_bits(1 + 2**-8 + 2**-30) == 0x3F81  # above the tie
    bits = np.arange(0, 65536, 11, dtype=np.uint16)
    vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b, v in zip(bits, vals):
        o = oracle.from_bf16_bits(int(b))
        assert (math.isnan(o) and math.isnan(v)) or o == v


# ---------------------------------------------------------------- forward

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("weighted", [False, True])
def test_forward_equals_dense_onehot_matmul(dtype, weighted):
    wl = small(dtype=dtype, weighted=weighted, oob=0.05)
    W = wl.weights()
    out, ab, oob, bad = oracle.forward(wl, wbits(wl, W), want_abs=True)
    Wv = wvalues(wl, W)
    to = wl.table_offset
    for t in range(wl.T):
        A = dense_A(wl, t)
        ref = A @ Wv[to[t]:to[t + 1]]
        got = out[:, t * wl.D:(t + 1) * wl.D]
        np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-12)
        refabs = np.abs(A) @ np.abs(Wv[to[t]:to[t + 1]])
        np.testing.assert_allclose(ab[:, t * wl.D:(t + 1) * wl.D], refabs, rtol=1e-12, atol=1e-300)
    # out-of-range count, computed with numpy
    tab = (np.searchsorted(wl.offsets, np.arange(wl.N), side="right") - 1) // wl.B
    E = wl.table_rows[tab]
    assert oob == int(np.sum((wl.indices < 0) | (wl.indices >= E)))
    assert oob > 0 and bad == 0


def test_forward_hand_example():
    # T=2 tables of E=3 rows, D=2, B=2; table 1 is weighted, table 0 is not.
    # bag (0,0) = {2, 0, 2}, bag (0,1) = {}, bag (1,0) = {1} with weight 0.5,
    # bag (1,1) = {0 with weight 2, 5 (out of range)}
    wl = workloads.Workload(
        name="hand", T=2, B=2, D=2, dtype="f32", table_rows=np.array([3, 3]),
        offsets=np.array([0, 3, 3, 4, 6], np.int32),
        indices=np.array([2, 0, 2, 1, 0, 5], np.int32),
        per_sample_weights=np.array([9, 9, 9, 0.5, 2, 9], np.float32),
        weighted_tables=np.array([0, 1], np.uint8))
    W = np.array([[1, 2], [3, 4], [5, 6],            # table 0 rows 0..2
                  [10, 20], [30, 40], [50, 60]],      # table 1 rows 0..2
                 np.float32)
    out, _, oob, _ = oracle.forward(wl, W)
    # out[b, t*D + d]: bag(0,0) = row2 + row0 + row2 = (11, 14); bag(0,1) empty
    # (table 0 ignores the weights 9); bag(1,0) = 0.5 * (30, 40) = (15, 20);
    # bag(1,1) = 2 * (10, 20) = (20, 40), idx 5 dropped and counted
    np.testing.assert_array_equal(out, np.array([[11, 14, 15, 20], [0, 0, 20, 40]], np.float32))
    assert oob == 1


def test_forward_oob_equals_forward_without_them():
    wl = small(oob=0.1, seed=9)
    W = wl.weights()
    out, _, oob, _ = oracle.forward(wl, wbits(wl, W))
    keep = []
    offs = [0]
    tab = (np.searchsorted(wl.offsets, np.arange(wl.N), side="right") - 1) // wl.B
    ok = (wl.indices >= 0) & (wl.indices < wl.table_rows[tab])
    for g in range(wl.NB):
        s, e = wl.offsets[g], wl.offsets[g + 1]
        keep.extend(wl.indices[s:e][ok[s:e]])
        offs.append(len(keep))
    wl2 = workloads.Workload(name="c", T=wl.T, B=wl.B, D=wl.D, dtype=wl.dtype,
                             table_rows=wl.table_rows, offsets=np.array(offs, np.int32),
                             indices=np.array(keep, np.int32), per_sample_weights=None,
                             weighted_tables=None)
    out2, _, oob2, _ = oracle.forward(wl2, wbits(wl, W))
    np.testing.assert_array_equal(out, out2)
    assert oob2 == 0 and oob == int((~ok).sum())


def test_forward_bag_subset_and_malformed_offsets():
    wl = small(seed=3)
    W = wbits(wl, wl.weights())
    full, _, _, _ = oracle.forward(wl, W)
    bags = np.array([0, 5, wl.B + 3, 2 * wl.B + wl.B - 1], np.int64)
    part, _, _, _ = oracle.forward(wl, W, bags=bags)
    for k, g in enumerate(bags):
        t, b = divmod(int(g), wl.B)
        np.testing.assert_array_equal(part[k], full[b, t * wl.D:(t + 1) * wl.D])
    # a bag whose end is below its start is malformed, counted and empty
    off = wl.offsets.copy()
    off[4] = off[3] - 1 if off[3] > 0 else 0
    wl.offsets = off
    if off[4] < off[3]:
        out, _, _, bad = oracle.forward(wl, W)
        assert bad == 1
        assert np.all(out[3, 0:wl.D] == 0)


def test_histogram_counts_sum_to_lookups():
    wl = workloads.hist(B=64, T=3)
    h = oracle.histogram(wl)
    assert h.shape == (3, 64, 64)
    assert int(h.sum()) == wl.N == 3 * 64 * 64
    np.testing.assert_array_equal(h.sum(axis=2), np.full((3, 64), 64))
    for t in range(3):
        for b in (0, 17, 63):
            g = t * wl.B + b
            ids = wl.indices[wl.offsets[g]:wl.offsets[g + 1]]
            np.testing.assert_array_equal(h[t, b], np.bincount(ids, minlength=64))


# ---------------------------------------------------------------- inversion

@pytest.mark.parametrize("oob", [0.0, 0.07])
def test_preprocess_against_numpy_stable_sort_and_counter(oob):
    wl = small(oob=oob, seed=11, B=101, rows=(50, 3, 1000, 1))
    pre = oracle.preprocess(wl)
    tab = (np.searchsorted(wl.offsets, np.arange(wl.N), side="right") - 1) // wl.B
    ok = (wl.indices >= 0) & (wl.indices < wl.table_rows[tab])
    keys = wl.table_offset[tab] + wl.indices
    pos = np.arange(wl.N)[ok]
    keys = keys[ok]
    order = np.argsort(keys, kind="stable")
    np.testing.assert_array_equal(pre["sorted_keys"], keys[order])
    np.testing.assert_array_equal(pre["sorted_pos"], pos[order])
    assert pre["num_unique"] == len(set(keys.tolist()))
    cnt = collections.Counter(keys.tolist())
    assert dict(zip(pre["unique_keys"].tolist(), pre["run_len"].tolist())) == dict(cnt)
    assert np.all(np.diff(pre["unique_keys"]) > 0)
    np.testing.assert_array_equal(pre["seg_off"], np.concatenate([[0], np.cumsum(pre["run_len"])]))
    assert pre["seg_off"][-1] == pre["n_valid"] == int(ok.sum())
    assert pre["run_len"].max() == max(cnt.values())


def test_preprocess_all_lookups_one_row():
    wl = workloads.make_workload("one", T=2, table_rows=[1, 1], D=4, dtype="f32", B=300,
                                 lengths=("fixed", 3), dist=("uniform",), seed=0)
    pre = oracle.preprocess(wl)
    assert pre["num_unique"] == 2
    np.testing.assert_array_equal(pre["run_len"], [900, 900])
    np.testing.assert_array_equal(pre["sorted_pos"], np.arange(1800))


# ---------------------------------------------------------------- backward

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("weighted", [False, True])
def test_row_gradient_equals_dense_At_G(dtype, weighted):
    wl = small(dtype=dtype, weighted=weighted, oob=0.03, seed=21)
    W = wl.weights()
    G = wl.grad_out()
    Wn, m, U, rg, uc = oracle.backward_adagrad(wl, wbits(wl, W), wl.momentum(), G,
                                               want_row_grad=True, want_update_count=True)
    to = wl.table_offset
    for t in range(wl.T):
        A = dense_A(wl, t)
        Gt = G[:, t * wl.D:(t + 1) * wl.D].astype(np.float64)
        ref = A.T @ Gt
        np.testing.assert_allclose(rg[to[t]:to[t + 1]], ref, rtol=1e-12, atol=1e-12)
    # mass conservation: sum over rows of g = sum over bags of (sum_p w_p) G_b
    for t in range(wl.T):
        A = dense_A(wl, t)
        lhs = rg[to[t]:to[t + 1]].sum(axis=0)
        rhs = A.sum(axis=1) @ G[:, t * wl.D:(t + 1) * wl.D].astype(np.float64)
        np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_each_touched_row_updated_once_untouched_rows_identical(dtype):
    wl = small(dtype=dtype, oob=0.05, seed=31, rows=(40, 400, 5))
    W = wbits(wl, wl.weights())
    m0 = np.random.default_rng(0).uniform(0, 1, wl.rows_total).astype(np.float32)
    Wn, m, U, rg, uc = oracle.backward_adagrad(wl, W, m0, wl.grad_out(), want_update_count=True)
    tab = (np.searchsorted(wl.offsets, np.arange(wl.N), side="right") - 1) // wl.B
    ok = (wl.indices >= 0) & (wl.indices < wl.table_rows[tab])
    touched = np.zeros(wl.rows_total, bool)
    touched[(wl.table_offset[tab] + wl.indices)[ok]] = True
    assert U == touched.sum()
    np.testing.assert_array_equal(uc, touched.astype(np.int32))
    np.testing.assert_array_equal(Wn[~touched], W[~touched])
    np.testing.assert_array_equal(m[~touched], m0[~touched])
    assert np.all(m[touched] >= m0[touched])


def _closed_form_workload(dtype, c, eps=1e-8):
    """One table of 6 rows; bag b looks up row b once (rows 4, 5 untouched);
    every upstream gradient element is c, so each touched row has g[d] = c."""
    wl = workloads.Workload(name="cf", T=1, B=4, D=8, dtype=dtype, table_rows=np.array([6]),
                            offsets=np.arange(5, dtype=np.int32),
                            indices=np.arange(4, dtype=np.int32), per_sample_weights=None,
                            weighted_tables=None, lr=0.01, eps=eps)
    G = np.full((4, 8), c, np.float32)
    return wl, G


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("c,eps", [(0.5, 1e-8), (-2.0, 1e-8), (0.5, 0.5), (-0.25, 2.0)])
def test_adagrad_closed_form_constant_gradient(dtype, c, eps):
    # momentum 0 and g[d] = c for all d:  m = c^2 after one step, and after k
    # steps m = k c^2 and w_k = w_{k-1} - lr c / (sqrt(k) |c| + eps).  With a
    # large eps (0.5 against |c| = 0.5: 1/(0.5+0.5) = 1 but 1/sqrt(0.25+0.5)
    # = 1.155) eps inside the square root, or the old momentum in the
    # denominator, moves every updated weight by far more than one unit of
    # its type.
    wl, G = _closed_form_workload(dtype, c, eps)
    W = wl.weights()
    Wb = wbits(wl, W)
    m = wl.momentum()
    w_ref = W.to(torch.float64).numpy().copy()
    for k in range(1, 4):
        Wb, m, U, _, _ = oracle.backward_adagrad(wl, Wb, m, G)
        assert U == 4
        np.testing.assert_array_equal(m[:4], np.float32(k * c * c))
        assert np.all(m[4:] == 0)
        den = math.sqrt(float(np.float32(k * c * c))) + float(np.float32(wl.eps))
        upd = w_ref[:4] - float(np.float32(wl.lr)) * c / den
        if dtype == "f32":
            exp = upd.astype(np.float32)
            np.testing.assert_array_equal(Wb[:4], exp)
        elif dtype == "f16":
            exp = upd.astype(np.float16).view(np.uint16)   # numpy double->half: single RNE rounding
            np.testing.assert_array_equal(Wb[:4], exp)
        else:
            exp = np.array([[oracle.to_bf16_bits(v) for v in row] for row in upd], np.uint16)
            np.testing.assert_array_equal(Wb[:4], exp)
            # and torch's rounding agrees wherever float32 holds upd exactly enough
            t = torch.from_numpy(upd.astype(np.float32)).to(torch.bfloat16)
            d = np.abs(t.view(torch.int16).numpy().astype(np.int32) - exp.view(np.int16).astype(np.int32))
            assert d.max() <= 1
        w_ref[:4] = (torch.from_numpy(Wb[:4].view(np.float32 if dtype == "f32" else np.int16))
                     .view(wl.torch_dtype()).to(torch.float64).numpy()) if dtype != "f32" else Wb[:4].astype(np.float64)
        # untouched rows 4, 5
        np.testing.assert_array_equal(Wb[4:], wbits(wl, W)[4:])


def test_rows_update_matches_full_backward():
    wl = small(dtype="bf16", weighted=True, oob=0.02, seed=41, rows=(60, 80, 20))
    W = wbits(wl, wl.weights())
    m0 = np.random.default_rng(1).uniform(0, 1, wl.rows_total).astype(np.float32)
    G = wl.grad_out()
    Wn, m, U, rg, _ = oracle.backward_adagrad(wl, W, m0, G, want_row_grad=True)
    rows = np.array([0, 3, 59, 60, 61, 100, 139, 150, 159], np.int64)
    Wr, mr, rgr, cnt, nv = oracle.rows_update(wl, rows, W[rows], m0[rows], G)
    np.testing.assert_array_equal(Wr, Wn[rows])
    np.testing.assert_array_equal(mr, m[rows])
    np.testing.assert_allclose(rgr, rg[rows], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- pages

def test_large_preset_matches_pages_statistics():
    """Expected statistics of the large preset against the numbers the
    pages print for their typical large case (T*B, B, total, unique, max)."""
    g = json.load(open(os.path.join(HERE, "golden", "pages_constants.json")))
    s = g["large_workload_statistics"]
    T, B, L, E = 32, 131072, 20, 2_000_000
    assert abs(T * B - s["T_times_B"]) / s["T_times_B"] < 0.01
    assert B == s["B"]
    assert abs(T * B * L - s["total_indices"]) / s["total_indices"] < 0.02
    uniq, hot = workloads.expected_zm_stats(E, B * L, workloads.LARGE_ZM_ALPHA, workloads.LARGE_ZM_Q)
    assert abs(T * uniq - s["unique_indices"]) / s["unique_indices"] < 0.05
    assert abs(hot - s["max_frequency"]) / s["max_frequency"] < 0.05


# ---------------------------------------------------------------- malformed offsets

def _sub_batch(wl, offsets, indices, psw=None):
    return workloads.Workload(name=wl.name, T=wl.T, B=wl.B, D=wl.D, dtype=wl.dtype,
                              table_rows=wl.table_rows, offsets=np.asarray(offsets, np.int64),
                              indices=np.asarray(indices, np.int32),
                              per_sample_weights=None if psw is None else np.asarray(psw, np.float32),
                              weighted_tables=wl.weighted_tables, lr=wl.lr, eps=wl.eps)


def _both_results(wl, W, m0, G):
    out, _, oob, bad = oracle.forward(wl, W)
    Wn, m, U, _, _ = oracle.backward_adagrad(wl, W, m0, G)
    return out, Wn, m, U


def _junk(rng, n, E=7):
    # in-range and out-of-range values alike: any of them counted would show
    return rng.integers(-3, E + 3, size=n).astype(np.int32)


def test_lookups_outside_every_bag_take_no_part():
    # the same bags with junk lookups before offsets[0] and after offsets[T*B]:
    # forward, weights and momentum equal those of the batch without them
    wl = small(seed=13, weighted=True, oob=0.03)
    W = wbits(wl, wl.weights())
    G = wl.grad_out()
    m0 = np.random.default_rng(2).uniform(0, 1, wl.rows_total).astype(np.float32)
    rng = np.random.default_rng(4)
    pre, post = 5, 7
    idx = np.concatenate([_junk(rng, pre), wl.indices, _junk(rng, post)])
    psw = np.concatenate([rng.uniform(0, 1, pre), wl.per_sample_weights, rng.uniform(0, 1, post)])
    gap = _sub_batch(wl, wl.offsets.astype(np.int64) + pre, idx, psw)
    a, b = _both_results(wl, W, m0, G), _both_results(gap, W, m0, G)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    assert oracle.offsets_check(gap) == (True, 0, False, True)
    assert oracle.offsets_check(wl) == (False, 0, False, False)


@pytest.mark.parametrize("where", ["first_start_negative", "last_end_past_n", "middle_end_below_start"])
def test_malformed_bag_is_empty(where):
    wl = small(seed=17, B=11, rows=(9, 40))
    W = wbits(wl, wl.weights())
    G = wl.grad_out()
    m0 = np.zeros(wl.rows_total, np.float32)
    off = wl.offsets.astype(np.int64).copy()
    NB, N = wl.NB, wl.N
    if where == "first_start_negative":
        g = 0
        off[0] = -2
        # expected: bag 0's lookups gone, everything else as before
        exp_idx = wl.indices[wl.offsets[1]:]
        exp_off = np.concatenate([[0], off[1:] - off[1]])
    elif where == "last_end_past_n":
        g = NB - 1
        off[NB] = N + 3
        exp_idx = wl.indices[:wl.offsets[NB - 1]]
        exp_off = np.concatenate([off[:NB], [off[NB - 1]]])
    else:
        g = 4
        while off[g] == off[g + 1]:
            g += 1
        # bag g ends before its start; bag g+1 starts there and so covers
        # bag g's lookups too
        off[g + 1] = off[g] - 1
        exp_idx = None
    mal = _sub_batch(wl, off, wl.indices)
    check = oracle.offsets_check(mal)
    assert check[0] and check[1] >= 1
    out, _, _, bad = oracle.forward(mal, W)
    assert bad == check[1]
    t, b = divmod(g, wl.B)
    assert np.all(out[b, t * wl.D:(t + 1) * wl.D] == 0)
    if exp_idx is not None:
        assert check[2] is False                     # offsets still non-decreasing
        exp = _sub_batch(wl, exp_off, exp_idx)
        a, c = _both_results(mal, W, m0, G), _both_results(exp, W, m0, G)
        for x, y in zip(a, c):
            np.testing.assert_array_equal(x, y)
    else:
        assert check[2] is True
        # forward: every well-formed bag pools its own range, as a batch that
        # holds a private copy of each well-formed bag's lookups does
        parts, lens = [], []
        for h in range(NB):
            s0, e0 = off[h], off[h + 1]
            ok = 0 <= s0 <= e0 <= N
            parts.append(wl.indices[s0:e0] if ok else np.zeros(0, np.int32))
            lens.append(e0 - s0 if ok else 0)
        copy = _sub_batch(wl, np.concatenate([[0], np.cumsum(lens)]), np.concatenate(parts))
        np.testing.assert_array_equal(out, oracle.forward(copy, W)[0])
        # backward: offsets that decrease leave some lookup in two bags, so
        # the batch updates nothing
        Wn, m, U, _, _ = oracle.backward_adagrad(mal, W, m0, G)
        assert U == 0
        np.testing.assert_array_equal(Wn, W)
        np.testing.assert_array_equal(m, m0)
        assert oracle.preprocess(mal)["n_valid"] == 0
        rows = np.arange(wl.rows_total)
        _, _, _, cnt, nv = oracle.rows_update(mal, rows, W, m0, G)
        assert nv == 0 and not cnt.any()


def test_offsets_check_patterns():
    wl = small(seed=19, B=6, rows=(5,))
    N = wl.N
    def chk(off):
        return oracle.offsets_check(_sub_batch(wl, off, wl.indices))
    base = wl.offsets.astype(np.int64)
    assert chk(base) == (False, 0, False, False)
    o = base.copy(); o[-1] = N - 1
    assert chk(o) == (True, 0, False, True)          # last lookup in no bag
    o = base.copy(); o[0] = 1
    assert chk(o)[0] and chk(o)[3]                   # first lookup in no bag
    o = base.copy(); o[2] = o[1] - 1
    r = chk(o)
    assert r[0] and r[1] >= 1 and r[2]               # decreasing
    o = base.copy(); o[-1] = N + 1
    assert chk(o) == (True, 1, False, True)          # last bag past N


# ---------------------------------------------------------------- tables of different shapes

def _mixed(vbe, weighted=False, seed=23):
    return workloads.make_workload(
        "mixed", T=4, table_rows=[13, 40, 7, 25], D=8, dtype="f32", B=11,
        lengths=("poisson", 4.0), dist=("zipf", 1.1), seed=seed, oob_frac=0.04,
        weighted=[True, False, True, True] if weighted else None,
        table_dims=[8, 16, 4, 12], table_dtypes=["f32", "bf16", "f32", "f16"],
        table_B=[11, 5, 17, 2] if vbe else None)


def _single_table(wl, t, W, G):
    """Table t of a multi-shape workload as a one-table uniform problem, with
    its weights and upstream gradient."""
    L = wl.layout()[t]
    g0, g1 = L["bag_off"], L["bag_off"] + L["B"]
    s0, s1 = int(wl.offsets[g0]), int(wl.offsets[g1])
    one = workloads.Workload(
        name="one", T=1, B=L["B"], D=L["D"], dtype=L["dtype"], table_rows=wl.table_rows[t:t + 1].copy(),
        offsets=(wl.offsets[g0:g1 + 1].astype(np.int64) - s0), indices=wl.indices[s0:s1].copy(),
        per_sample_weights=None if wl.per_sample_weights is None else wl.per_sample_weights[s0:s1].copy(),
        weighted_tables=None if wl.weighted_tables is None else wl.weighted_tables[t:t + 1].copy(),
        lr=wl.lr, eps=wl.eps)
    nbytes = int(wl.table_rows[t]) * L["D"] * (4 if L["dtype"] == "f32" else 2)
    raw = W[L["wbyte"]:L["wbyte"] + nbytes]
    Wt = raw.view(np.float32 if L["dtype"] == "f32" else np.uint16).reshape(-1, L["D"])
    if wl.vbe:
        Gt = G[L["out_off"]:L["out_off"] + L["B"] * L["D"]].reshape(L["B"], L["D"])
    else:
        Gt = G.reshape(wl.B, -1)[:, L["out_off"]:L["out_off"] + L["D"]]
    return one, Wt, np.ascontiguousarray(Gt)


def _table_out(wl, out, t):
    L = wl.layout()[t]
    if wl.vbe:
        return out[L["out_off"]:L["out_off"] + L["B"] * L["D"]].reshape(L["B"], L["D"])
    return out.reshape(wl.B, -1)[:, L["out_off"]:L["out_off"] + L["D"]]


@pytest.mark.parametrize("vbe", [False, True])
@pytest.mark.parametrize("weighted", [False, True])
def test_multi_shape_tables_decompose_into_single_tables(vbe, weighted):
    # tables are independent problems: a batch of tables with different D,
    # dtype (and, with VBE, B) equals each table run alone in the pinned
    # uniform oracle -- pooled rows, updated weights and momentum, bit for bit
    wl = _mixed(vbe, weighted)
    W = wl.weights_mixed()
    G = wl.grad_out()
    m0 = np.random.default_rng(3).uniform(0, 1, wl.rows_total).astype(np.float32)
    out, _, oob, _ = oracle.forward(wl, W)
    Wn, m, U, _, _ = oracle.backward_adagrad(wl, W, m0, G)
    to = wl.table_offset
    oob_sum = U_sum = 0
    for t in range(wl.T):
        one, Wt, Gt = _single_table(wl, t, W, G)
        o1, _, k1, _ = oracle.forward(one, Wt)
        np.testing.assert_array_equal(_table_out(wl, out, t), o1)
        W1, m1, U1, _, _ = oracle.backward_adagrad(one, Wt, m0[to[t]:to[t + 1]], Gt)
        _, Wnt, _ = _single_table(wl, t, Wn, G)
        np.testing.assert_array_equal(Wnt, W1)
        np.testing.assert_array_equal(m[to[t]:to[t + 1]], m1)
        oob_sum += k1
        U_sum += U1
    assert oob == oob_sum > 0 and U == U_sum


def test_vbe_forward_equals_dense_onehot_per_table():
    wl = _mixed(True, weighted=True, seed=29)
    W = wl.weights_mixed()
    out, _, _, _ = oracle.forward(wl, W)
    for t, L in enumerate(wl.layout()):
        E = int(wl.table_rows[t])
        A = np.zeros((L["B"], E))
        for b in range(L["B"]):
            g = L["bag_off"] + b
            for p in range(wl.offsets[g], wl.offsets[g + 1]):
                e = int(wl.indices[p])
                if 0 <= e < E:
                    A[b, e] += float(wl.per_sample_weights[p]) if wl.weighted_tables[t] else 1.0
        nbytes = E * L["D"] * (4 if L["dtype"] == "f32" else 2)
        raw = W[L["wbyte"]:L["wbyte"] + nbytes]
        if L["dtype"] == "f32":
            Wt = raw.view(np.float32).reshape(E, L["D"]).astype(np.float64)
        else:
            tdt = torch.float16 if L["dtype"] == "f16" else torch.bfloat16
            Wt = torch.from_numpy(raw.view(np.int16).copy()).view(tdt).to(torch.float64).numpy().reshape(E, L["D"])
        np.testing.assert_allclose(_table_out(wl, out, t), A @ Wt, rtol=1e-6, atol=1e-9)
