"""GPU: one decode step (append + decode) captured in a CUDA graph after a
warm-up call, replayed twice: bit-identical to the same calls issued
directly. A warmed-up plan allocates nothing and caches its tensor maps, the
merge resets the dynamic-piece counter for the next call, and the split and
merge kernels start under programmatic dependent launch inside the graph."""

import numpy as np
import pytest
import torch

import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import make_workload

from gpu_helpers import DeviceStep, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("lens", [[200, 64, 1000, 5], [20000, 300, 17000]])  # short; dynamic tail
def test_graph_replay_matches_direct_calls(lens):
    wl = make_workload("llama3_8b_gqa", seed=21, B=len(lens), lengths=("list", lens),
                       max_len=max(lens) + 16)
    ds = DeviceStep(wl)
    out_direct = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    out_graph = torch.empty_like(out_direct)
    with pa.Plan() as plan:
        stream = torch.cuda.current_stream()

        def step(out, s):
            pa.pa_append_kv(ds.k_new, ds.v_new, ds.k_pool, ds.v_pool, ds.tables, ds.cache_lens, s)
            pa.pa_decode(ds.q, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale, out,
                         wl.max_seq_len, plan, s)

        step(out_direct, stream)        # warm-up: creates the workspace and tensor maps
        torch.cuda.synchronize()
        want = bits(out_direct).copy()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(out_graph, torch.cuda.current_stream())
        for _ in range(2):
            out_graph.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(bits(out_graph), want)
        assert plan.last_device_error() == 0
