"""GPU parity of the small-table histogram path (tensor cores, FP16 hi/lo
compensation) against the CPU oracle, plus its saved counts bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_full, run_cuda

pytestmark = pytest.mark.gpu


def _m0(wl):
    return np.random.default_rng(3).uniform(0, 0.5, wl.rows_total).astype(np.float32)


def _saved_counts(res, wl):
    from recsys_table_embedding_gb300 import meta_view
    h = meta_view(res["tbe"].meta, "hist", wl.NB * 64, torch.float16).cpu().numpy()
    return h.astype(np.int64).reshape(wl.T, wl.B, 64)


def _run(wl, cfg=None):
    W0, G, m0 = wl.weights(), wl.grad_out(), _m0(wl)
    res = run_cuda(wl, W0, G, m0, cfg=cfg, preprocess_in_forward=False)
    assert res["path"] == 2
    check_full(wl, W0, G, m0, res)
    np.testing.assert_array_equal(_saved_counts(res, wl), oracle.histogram(wl))
    assert res["status"][1] == 0
    return res


def test_hist_config_reduced_batch():
    _run(workloads.hist(B=1024, T=8))


@pytest.mark.parametrize("D", [64, 96, 128])
def test_hist_forced_shapes_ragged(D):
    from recsys_table_embedding_gb300 import config
    from recsys_table_embedding_gb300.tbe import HIST_FORCE
    wl = workloads.make_workload("hshape", T=3, table_rows=[13, 64, 40], D=D, dtype="f16", B=200,
                                 lengths=("poisson", 20.0), dist=("uniform",), seed=D)
    _run(wl, cfg=config(hist_mode=HIST_FORCE))


def test_hist_out_of_range_and_empty_bags():
    from recsys_table_embedding_gb300 import config
    from recsys_table_embedding_gb300.tbe import HIST_FORCE
    wl = workloads.make_workload("hoob", T=2, table_rows=[64, 30], D=128, dtype="f16", B=300,
                                 lengths=("poisson", 2.0), dist=("uniform",), seed=11, oob_frac=0.05)
    assert np.any(np.diff(wl.offsets) == 0)
    res = _run(wl, cfg=config(hist_mode=HIST_FORCE))
    assert res["status"][0] > 0


def test_hist_matches_generic_path():
    from recsys_table_embedding_gb300 import config
    from recsys_table_embedding_gb300.tbe import HIST_OFF
    from parity import assert_weights_close, touched_rows, wbits_np
    wl = workloads.hist(B=512, T=4)
    W0, G, m0 = wl.weights(), wl.grad_out(), _m0(wl)
    a = run_cuda(wl, W0, G, m0, preprocess_in_forward=False)
    b = run_cuda(wl, W0, G, m0, cfg=config(hist_mode=HIST_OFF), preprocess_in_forward=False)
    assert a["path"] == 2 and b["path"] == 1
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(a["mom"], b["mom"], rtol=1e-4)
    assert_weights_close(a["W"], b["W"], wbits_np(W0, "f16"), touched_rows(wl), "f16")
