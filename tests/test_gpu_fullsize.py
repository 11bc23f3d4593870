"""GPU parity at the full workload sizes, in the benchmark's launch configuration.

The oracle computes sampled (sequence, q-head) rows one by one; every output
row must also be finite (a stray read of a NaN-poisoned slot would show)."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import make_workload
from oracle_steps import append_in_place

from gpu_helpers import DeviceStep, bits, out_f64, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("name,extra", [
    ("llama7b_mha", {}), ("llama3_8b_gqa", {}), ("long_splitk", {}), ("mixed_shared", {}),
    # 16 query heads per kv head: the two-column-tile decode (query fragments
    # reread from shared memory, five-warp blocks), long rows merged from many
    # static-range partials.
    ("llama3_405b_gqa", {}),
])
def test_full_size_sampled_rows(name, extra):
    wl = make_workload(name, **extra)
    ds = DeviceStep(wl)
    torch.cuda.synchronize()
    append_in_place(wl)
    with pa.Plan() as plan:
        ds.append()
        out = ds.decode(plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
        assert pa.pa_last_device_error(None) == 0
        # The appended slots hold exactly the new rows.
        bs = wl.block_size
        for b in range(0, wl.B, max(1, wl.B // 8)):
            pos = int(wl.cache_lens[b])
            phys = int(wl.block_tables[b, pos // bs])
            got_k = bits(ds.k_pool[phys, :, pos % bs])
            assert np.array_equal(got_k, wl.k_new[b])
    got = out_f64(out)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(7)
    idx = rng.choice(wl.B * wl.Hq, size=min(96, wl.B * wl.Hq), replace=False)
    # always include the longest sequence's first and last head
    bmax = int(np.argmax(wl.seq_lens))
    idx = np.unique(np.concatenate([idx, [bmax * wl.Hq, bmax * wl.Hq + wl.Hq - 1]]))
    pairs = np.stack([idx // wl.Hq, idx % wl.Hq], axis=1).astype(np.int32)
    ref = oracle.decode(wl.q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, wl.scale,
                        pairs=pairs)
    err = np.abs(got[pairs[:, 0], pairs[:, 1]] - ref).max()
    assert err <= tol(wl), f"{name}: max abs error {err:.3e}"
