"""GPU: one decode step (append + decode) captured in a CUDA graph after a
warm-up call, replayed twice: bit-identical to the same calls issued
directly. A warmed-up plan allocates nothing and caches its tensor maps, the
merge resets the dynamic-piece counter for the next call, and the split and
merge kernels start under programmatic dependent launch inside the graph.
Multi-query decodes on each of their kernels (split tiles, the one-tile
kernel with its key split and merge, the two-tile kernel) are captured and
replayed the same way."""

import numpy as np
import pytest
import torch

import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import make_workload

from oracle_steps import append_in_place

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


@pytest.mark.parametrize("lens,ns,kernel", [
    ([9000], [8], 0),                # the one-tile kernel, its key range split; merge kernel
    ([600, 2000, 40], [3, 4, 2], 0),  # the split decode's tiles (<= 16 columns per kv head)
    ([1500, 700], [64, 200], 2),     # the two-tile prefill kernel, pinned
], ids=["key_split", "split_tiles", "two_tile"])
def test_multi_query_graph_replay_matches_direct_calls(lens, ns, kernel):
    # pa_decode_multi on a warmed-up plan, captured and replayed twice: its
    # key-split partials and counters live in the plan's workspace, and the
    # tensor maps of the query and output arrays are encoded at capture.
    wl = make_workload("llama3_8b_gqa", seed=22, B=len(lens), lengths=("list", lens),
                       max_len=max(lens) + 16)
    append_in_place(wl)   # the new tokens are already in the pools
    ds = DeviceStep(wl)
    pa.pa_debug_set_prefill_kernel(kernel)
    try:
        _replay_multi(wl, ds, ns)
    finally:
        pa.pa_debug_set_prefill_kernel(pa.PA_PREFILL_AUTO)


def _replay_multi(wl, ds, ns):
    rng = np.random.default_rng(5)
    T = int(sum(ns))
    q = torch.from_numpy(rng.standard_normal((T, wl.Hq, wl.D)).astype(np.float32))
    q = q.to(torch.bfloat16).cuda()
    qs = torch.from_numpy(np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)).cuda()
    out_direct = torch.empty((T, wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    out_graph = torch.empty_like(out_direct)
    with pa.Plan() as plan:
        def call(out, s):
            pa.pa_decode_multi(q, qs, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale,
                               out, max(ns), wl.max_seq_len, plan, s)

        call(out_direct, torch.cuda.current_stream())
        torch.cuda.synchronize()
        want = bits(out_direct).copy()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                call(out_graph, side)
        torch.cuda.current_stream().wait_stream(side)
        for _ in range(2):
            out_graph.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(bits(out_graph), want)
        assert plan.last_device_error() == 0
