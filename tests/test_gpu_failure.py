"""GPU: every kernel's give-up path, made to run without a fault or a hang.

Every pipeline wait in the kernels is bounded; when one expires the kernel
raises PA_DEVERR_TIMEOUT, waits (bounded) for its own copies and tensor-core
products in flight, frees its tensor memory and returns. The wait-expiry
probe (pa_debug_set_wait_probe) makes each kernel's first wait use an
mbarrier that nothing completes, bounded by 20 us, so that path runs on
demand. Each test checks that the error bit reaches the host, and that the
device stays usable: the same call with the probe off matches the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import bf16_bits, make_workload
from oracle_steps import append_in_place, pools_after_append

from gpu_helpers import BF16_TOL, DeviceStep, out_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture
def probe():
    """Turns the probe on for the duration of a `with` block, always off after."""
    class Probe:
        def __enter__(self):
            pa.pa_debug_set_wait_probe(True)

        def __exit__(self, *exc):
            pa.pa_debug_set_wait_probe(False)
    yield Probe()
    pa.pa_debug_set_wait_probe(False)


def _gqa(seed, **extra):
    spec = dict(B=7, lengths=("loguniform", 1, 5000), max_len=5120)
    spec.update(extra)
    return make_workload("llama3_8b_gqa", seed=seed, **spec)


@pytest.mark.parametrize("extra", [dict(), dict(Hq=64, Hkv=4), dict(Hq=8, Hkv=8)],
                         ids=["g4", "g16", "mha"])
def test_decode_gives_up_reports_and_recovers(probe, extra):
    wl = _gqa(31, **extra)
    ds = DeviceStep(wl)
    ds.append()
    kp, vp = pools_after_append(wl)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    with pa.Plan() as plan:
        with probe:
            ds.decode(plan)
            err = plan.last_device_error()
        assert err & pa.PA_DEVERR_TIMEOUT
        out = ds.decode(plan)
        assert plan.last_device_error() == 0
    assert np.abs(out_f64(out) - ref).max() <= BF16_TOL


def test_decode_multi_gives_up_reports_and_recovers(probe):
    lens, ns = [900, 40, 3000], [4, 2, 3]
    wl = make_workload("llama3_8b_gqa", seed=32, B=3, lengths=("list", lens), max_len=3008)
    append_in_place(wl)
    rng = np.random.default_rng(2)
    q = bf16_bits(rng.standard_normal((sum(ns), wl.Hq, wl.D)).astype(np.float32))
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    ds = DeviceStep(wl)
    qd, qsd = to_dev(q, "bf16"), torch.from_numpy(qs).cuda()
    out = torch.empty((q.shape[0], wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    with pa.Plan() as plan:
        with probe:
            pa.pa_decode_multi(qd, qsd, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale,
                               out, max(ns), wl.max_seq_len, plan)
            err = plan.last_device_error()
        assert err & pa.PA_DEVERR_TIMEOUT
        pa.pa_decode_multi(qd, qsd, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale, out,
                           max(ns), wl.max_seq_len, plan)
        assert plan.last_device_error() == 0
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    assert np.abs(out_f64(out) - ref).max() <= BF16_TOL


def test_noalloc_decode_gives_up_reports_and_recovers(probe):
    wl = _gqa(33)
    ds = DeviceStep(wl)
    ds.append()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with probe:
        pa.pa_decode_noalloc(ds.q, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale, ds.out,
                             wl.max_seq_len, device_error=err)
        torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_DEVERR_TIMEOUT
    err.zero_()
    pa.pa_decode_noalloc(ds.q, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale, ds.out,
                         wl.max_seq_len, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kp, vp = pools_after_append(wl)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    assert np.abs(out_f64(ds.out) - ref).max() <= BF16_TOL


@pytest.fixture(params=[1, 2], ids=["one_tile", "two_tile"])
def prefill_kernel(request):
    """Pins the prefill call to one of the two tensor-core kernels."""
    which = {1: pa.PA_PREFILL_ONE_TILE, 2: pa.PA_PREFILL_TWO_TILE}[request.param]
    pa.pa_debug_set_prefill_kernel(which)
    try:
        yield which
    finally:
        pa.pa_debug_set_prefill_kernel(pa.PA_PREFILL_AUTO)


@pytest.mark.parametrize("lens,ns", [([700, 300, 2000], [200, 64, 256]), ([90], [1])])
def test_prefill_gives_up_reports_frees_tensor_memory_and_recovers(probe, prefill_kernel,
                                                                    lens, ns):
    wl = make_workload("llama3_8b_gqa", seed=34, B=len(lens), lengths=("list", lens),
                       max_len=max(lens) + 16)
    append_in_place(wl)
    rng = np.random.default_rng(3)
    q = bf16_bits(rng.standard_normal((sum(ns), wl.Hq, wl.D)).astype(np.float32))
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    ds = DeviceStep(wl)
    qd, qsd = to_dev(q, "bf16"), torch.from_numpy(qs).cuda()
    out = torch.empty((q.shape[0], wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with probe:
        pa.pa_prefill(qd, qsd, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale, out,
                      max(ns), wl.max_seq_len, device_error=err)
        torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_DEVERR_TIMEOUT
    # Two normal calls: a block that did not free its tensor memory would
    # leave the next block on that SM unable to allocate all 512 columns.
    for _ in range(2):
        err.zero_()
        pa.pa_prefill(qd, qsd, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale, out,
                      max(ns), wl.max_seq_len, device_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    assert np.abs(out_f64(out) - ref).max() <= BF16_TOL


def test_page_scores_give_up_report_and_recover(probe):
    wl = _gqa(35, lengths=("list", [16, 160, 4096, 33, 1000, 5, 2048]), max_len=4096)
    append_in_place(wl)
    ds = DeviceStep(wl)
    B, MB = wl.block_tables.shape
    scores = torch.empty((B, MB), dtype=torch.float32, device="cuda")
    victims = torch.empty(B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with probe:
        pa.pa_page_scores(ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.max_seq_len, scores,
                          victims, err)
        torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_DEVERR_TIMEOUT
    err.zero_()
    pa.pa_page_scores(ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.max_seq_len, scores,
                      victims, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_s, ref_v = oracle.page_scores(wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens)
    got = scores.cpu().numpy().astype(np.float64)
    for b in range(B):
        nb = -(-int(wl.seq_lens[b]) // wl.block_size)
        np.testing.assert_allclose(got[b, :nb], ref_s[b, :nb], rtol=1e-4)


def test_fused_merge_gives_up_reports_and_recovers(probe):
    # With the fused merge a warp that gave up leaves its segments' counters
    # short; the last warp to leave clears them, so the next call is exact.
    wl = _gqa(36)
    ds = DeviceStep(wl)
    ds.append()
    kp, vp = pools_after_append(wl)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    with pa.Plan() as plan:
        ds.decode(plan)
        plan.set_merge(pa.PA_MERGE_FUSED)
        plan.set_schedule(150, 1)
        with probe:
            ds.decode(plan)
            err = plan.last_device_error()
        assert err & pa.PA_DEVERR_TIMEOUT
        for _ in range(2):
            out = ds.decode(plan)
            assert plan.last_device_error() == 0
            assert np.abs(out_f64(out) - ref).max() <= BF16_TOL


def test_fused_append_decode_gives_up_reports_and_recovers(probe):
    # A warp that gives up may have appended some rows already; the next
    # call writes the same rows to the same slots, so it is exact.
    wl = _gqa(37)
    ds = DeviceStep(wl)
    kp, vp = pools_after_append(wl)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)

    def call(plan):
        pa.pa_append_decode(ds.q, ds.k_new, ds.v_new, ds.k_pool, ds.v_pool, ds.tables,
                            ds.seq_lens, wl.scale, ds.out, wl.max_seq_len, plan)
        return plan.last_device_error()

    with pa.Plan() as plan:
        call(plan)
        with probe:
            err = call(plan)
        assert err & pa.PA_DEVERR_TIMEOUT
        assert call(plan) == 0
    assert np.abs(out_f64(ds.out) - ref).max() <= BF16_TOL
    assert np.array_equal(ds.k_pool.view(torch.int16).cpu().numpy().view(np.uint16), kp)
