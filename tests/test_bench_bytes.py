"""The benchmark's algorithmic-byte accounting (the roofline numerator)
against the per-step totals the scope table publishes for the large, mid and
histogram workloads: large ~71.2 GB (forward 24.0, preprocessing 2.4,
backward 44.9), mid ~15.7 GB (its unique count is an estimate there, hence
the wider bar), histogram ~6.46 GB.  The realised batches come from the
seeded generators and U from the oracle-independent numpy unique count."""
import numpy as np
import pytest

import workloads


def _stats(wl):
    tab = np.repeat(np.arange(wl.T), np.diff(wl.offsets[::wl.B].astype(np.int64)))
    ok = (wl.indices >= 0) & (wl.indices < wl.table_rows[tab])
    keys = (wl.table_offset[tab] + wl.indices)[ok]
    return {"N": wl.N, "NB": wl.NB, "U": int(np.unique(keys).size)}


@pytest.mark.parametrize("name,total,parts,rtol", [
    ("large", 71.2e9, (24.0e9, 2.4e9, 44.9e9), 0.01),
    ("mid", 15.7e9, None, 0.03),
])
def test_generic_path_bytes_match_the_published_totals(name, total, parts, rtol):
    import bench
    wl = workloads.PRESETS[name]()
    sb = bench.step_bytes(wl, _stats(wl), bench.PREPROCESS_IN_FORWARD[name])
    assert sb["total"] == pytest.approx(total, rel=rtol)
    if parts:
        for got, want in zip((sb["forward"], sb["preprocess"], sb["backward"]), parts):
            assert got == pytest.approx(want, rel=0.02)


def test_histogram_path_bytes_match_the_published_total():
    import bench
    wl = workloads.hist()
    sb = bench.step_bytes(wl, {"N": wl.N, "NB": wl.NB}, False)
    assert sb["total"] == pytest.approx(6.46e9, rel=0.01)
