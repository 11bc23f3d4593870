"""pa_decode_noalloc: the decode entry point for callers that cannot let a
library allocate device memory (an engine that budgets all HBM itself, or a
plugin host that hands a kernel only its tensors).

Its output must match pa_decode's on the same inputs, on two calls in a row
with different shapes, so that the shared scratch array's leftover contents
from the first call cannot leak into the second. The file is named to be
collected last.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import make_workload

from gpu_helpers import DeviceStep, out_f64, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _both(wl):
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        ref = out_f64(ds.decode(plan))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(ds.out, float("nan"))
    pa.pa_decode_noalloc(ds.q, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale, out,
                         wl.max_seq_len, device_error=err)
    torch.cuda.synchronize()
    return ref, out_f64(out), int(err.item())


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    first = make_workload("llama3_8b_gqa", seed=21, B=12, lengths=("loguniform", 1, 6000),
                          max_len=6144)
    second = make_workload("llama7b_mha", seed=22, B=5, Hq=8, Hkv=8,
                           lengths=("uniform", 1, 1500), max_len=1536, pool=("fixed", 1024))
    for wl in (first, second):
        ref, got, err = _both(wl)
        assert err == 0
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() <= tol(wl)


def test_noalloc_matches_at_the_largest_footprint():
    # 16 query heads per kv head at D = 128 is the largest partial footprint:
    # here even static ranges over the full grid (1025 warps) need more than
    # the fixed scratch, so the call runs on fewer blocks and must still
    # match pa_decode.
    wl = make_workload("llama3_8b_gqa", seed=23, B=4, Hq=32, Hkv=2, lengths=("fixed", 100),
                       max_len=8192)
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        ref = out_f64(ds.decode(plan, max_seq_len=8192))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(ds.out, float("nan"))
    pa.pa_decode_noalloc(ds.q, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale, out, 8192,
                         device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.abs(out_f64(out) - ref).max() <= tol(wl)


def test_noalloc_runs_without_the_dynamic_tail_when_it_does_not_fit():
    # One query head per kv unit, 32 x 32 heads and a 2048-token bound: the
    # dynamic tail pa_decode plans here needs about 19 MB of partials, more
    # than the fixed scratch, so the no-alloc call runs on static ranges
    # alone, and must still match pa_decode.
    wl = make_workload("llama7b_mha", seed=24, B=32, lengths=("uniform", 1, 200), max_len=2048,
                       pool=("fixed", 1024))
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        ref = out_f64(ds.decode(plan, max_seq_len=2048))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(ds.out, float("nan"))
    pa.pa_decode_noalloc(ds.q, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale, out, 2048,
                         device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.abs(out_f64(out) - ref).max() <= tol(wl)
