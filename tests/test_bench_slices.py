"""bench.py's --requests slices (CPU only): the first requests of a workload with a
pool that still holds their pages and stays small -- exactly their pages for the
long-context workload, at most twice them elsewhere -- so that multi-metric
profiler captures hold a few GB on the device."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("name,requests", [
    ("long", 2), ("batched_bf16", 32), ("batched_f32", 16), ("ragged", 64),
    ("gqa8_bf16", 32), ("gqa4_bf16", 32), ("window_bf16", 16), ("prefill_bf16", 2),
])
def test_slice_keeps_first_requests_and_a_small_pool(name, requests):
    full = bench.make_workload(name)
    w = bench.make_workload(name, requests=requests)
    assert w.B == requests and w.name == f"{name}_first{requests}"
    assert np.array_equal(w.seq_lens, full.seq_lens[:requests])
    if full.new_tokens is not None:
        assert np.array_equal(w.new_tokens, full.new_tokens[:requests])
    kept = int(w.n_pages.sum())
    assert kept <= w.pool_pages <= min(full.pool_pages, 2 * kept)
    if name == "long":
        assert w.pool_pages == kept
    pool_bytes = w.pool_pages * w.H * w.P * w.D * 2 * w.elem_bytes
    assert pool_bytes < 2.5e9
    # the slice still reads more than L2 holds, so DRAM counters mean something
    if not name.startswith("prefill"):
        assert bench.algorithmic_bytes(w) > 2 * 129e6


def test_no_slice_without_requests():
    for name in ("long", "ragged"):
        a, b = bench.make_workload(name), bench.make_workload(name, requests=0)
        assert a.B == b.B and a.pool_pages == b.pool_pages and a.name == b.name
