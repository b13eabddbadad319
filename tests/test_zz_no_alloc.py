"""tbe_preprocess_static: the batch inversion for callers that cannot allocate
device memory where they run it (code inside an allocator or memory-pool
callback, plug-ins handed only fixed buffers, services with a fixed device
footprint).  Its scratch is a device array inside the library, shared by all
calls, so this file checks two calls in a row -- on different batches, so the
second call starts from the first one's leftovers -- against tbe_preprocess
with a caller workspace (bit-exact: it is integer work).  Collected last on
purpose; it also passes alone in a fresh process, where its first call does
the one-time address lookup."""
import numpy as np
import pytest
import torch

import workloads
from parity import device_batch

pytestmark = pytest.mark.gpu


def _inversion(meta, wl):
    from recsys_table_embedding_gb300 import meta_view
    c = meta_view(meta, "counters", 4).cpu().numpy()
    U = int(c[0])
    out = dict(counters=c,
               sorted_keys=meta_view(meta, "sorted_keys", wl.N).cpu().numpy(),
               sorted_vals=meta_view(meta, "sorted_vals", wl.N).cpu().numpy(),
               unique_keys=meta_view(meta, "unique_keys", U).cpu().numpy(),
               seg_off=meta_view(meta, "seg_off", U + 1).cpu().numpy())
    if meta.c.bag_of:
        out["bag_of"] = meta_view(meta, "bag_of", wl.N).cpu().numpy()
    return out


def _both(wl):
    from recsys_table_embedding_gb300 import (Tables, tbe_meta_bind, tbe_preprocess,
                                              tbe_preprocess_static, tbe_query_sizes)
    W = wl.weights(device="cuda")
    tables = Tables(W, wl.table_offset)
    batch = device_batch(wl)
    _, wb = tbe_query_sizes(tables, batch)
    ws = torch.empty(wb, dtype=torch.uint8, device="cuda")
    st_ref = torch.zeros(4, dtype=torch.int32, device="cuda")
    st_new = torch.zeros(4, dtype=torch.int32, device="cuda")
    ref = tbe_meta_bind(tables, batch)
    new = tbe_meta_bind(tables, batch)
    tbe_preprocess(tables, batch, ref, ws, st_ref)
    tbe_preprocess_static(tables, batch, new, st_new)
    torch.cuda.synchronize()
    a, b = _inversion(ref, wl), _inversion(new, wl)
    assert a.keys() == b.keys()
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    np.testing.assert_array_equal(st_ref.cpu().numpy(), st_new.cpu().numpy())
    assert a["counters"][0] > 0


def test_static_preprocess_matches_workspace_preprocess_two_calls():
    # call 1: unweighted large-shaped batch (long runs, payload = bag index)
    _both(workloads.large(B=4096, E=200_000))
    # call 2: a different, weighted batch with out-of-range indices
    # (payload = position), on the scratch the first call left behind
    _both(workloads.make_workload("static2", T=5, table_rows=[1000, 30, 70000, 5, 4096], D=32,
                                  dtype="f16", B=20000, lengths=("poisson", 6.0),
                                  dist=("zipf", 1.2), seed=12, weighted=[True, False, True, True, False],
                                  oob_frac=0.01))


def test_static_preprocess_rejects_batches_over_its_limit():
    from recsys_table_embedding_gb300 import Tables, TbeError, tbe_meta_bind, tbe_preprocess_static
    from recsys_table_embedding_gb300.tbe import STATIC_SCRATCH_MAX_N
    wl = workloads.make_workload("over", T=1, table_rows=[100], D=16, dtype="f32",
                                 B=STATIC_SCRATCH_MAX_N + 1, lengths=("fixed", 1),
                                 dist=("uniform",), seed=0)
    assert wl.N == STATIC_SCRATCH_MAX_N + 1
    tables = Tables(wl.weights(device="cuda"), wl.table_offset)
    batch = device_batch(wl)
    meta = tbe_meta_bind(tables, batch)
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(TbeError, match="status 11"):
        tbe_preprocess_static(tables, batch, meta, st)
