"""pa_decode_noalloc: the decode entry point for callers that cannot let a
library allocate device memory (an engine that budgets all HBM itself, or a
plugin host that hands a kernel only its tensors).

Every case compares the call's output with the fp64 oracle on the same
inputs, at the bf16 tolerance of the other decode tests: two calls in a row
with different shapes (so that the shared scratch array's leftover contents
from the first call cannot leak into the second), a call whose dynamic tail
does not fit the scratch (static ranges only) and one whose static ranges do
not fit either (a reduced grid). One more case checks the point of the entry
point: after a warm-up call, a call of a new size changes neither the
device's free memory nor torch's allocated memory. The file is named to be
collected last.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import make_workload
from oracle_steps import pools_after_append

from gpu_helpers import DeviceStep, out_f64, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _reference(wl):
    kp, vp = pools_after_append(wl)
    return oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)


def _noalloc(ds, wl, max_seq_len=None):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(ds.out, float("nan"))
    pa.pa_decode_noalloc(ds.q, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale, out,
                         max_seq_len or wl.max_seq_len, device_error=err)
    torch.cuda.synchronize()
    return out_f64(out), int(err.item())


def _check_against_oracle(wl, max_seq_len=None):
    ds = DeviceStep(wl)
    ds.append()
    got, err = _noalloc(ds, wl, max_seq_len)
    assert err == 0
    assert np.isfinite(got).all()
    e = np.abs(got - _reference(wl)).max()
    assert e <= tol(wl), f"max abs error {e:.3e}"


def test_noalloc_matches_oracle_on_two_calls_in_a_row():
    first = make_workload("llama3_8b_gqa", seed=21, B=12, lengths=("loguniform", 1, 6000),
                          max_len=6144)
    second = make_workload("llama7b_mha", seed=22, B=5, Hq=8, Hkv=8,
                           lengths=("uniform", 1, 1500), max_len=1536, pool=("fixed", 1024))
    for wl in (first, second):
        _check_against_oracle(wl)


def test_noalloc_matches_oracle_at_the_largest_footprint():
    # 16 query heads per kv head at D = 128 is the largest partial footprint:
    # here even static ranges over the full grid (1025 warps) need more than
    # the fixed scratch, so the call runs on fewer blocks.
    wl = make_workload("llama3_8b_gqa", seed=23, B=4, Hq=32, Hkv=2, lengths=("fixed", 100),
                       max_len=8192)
    _check_against_oracle(wl, max_seq_len=8192)


def test_noalloc_matches_oracle_without_the_dynamic_tail():
    # One query head per kv unit, 32 x 32 heads and a 2048-token bound: the
    # dynamic tail pa_decode plans here needs about 19 MB of partials, more
    # than the fixed scratch, so the call runs on static ranges alone.
    wl = make_workload("llama7b_mha", seed=24, B=32, lengths=("uniform", 1, 200), max_len=2048,
                       pool=("fixed", 1024))
    _check_against_oracle(wl, max_seq_len=2048)


def test_noalloc_takes_no_device_memory_after_a_warm_up_call():
    # Warm up with both kinds of launch this test makes (a dynamic tail and
    # static ranges only), so that every kernel they use is loaded; then a
    # call of a new, larger size must leave the device's free memory and
    # torch's allocations exactly as they were.
    warm_tail = make_workload("llama3_8b_gqa", seed=25, B=3, lengths=("fixed", 300), max_len=32768)
    warm_static = make_workload("llama3_8b_gqa", seed=26, B=3, lengths=("fixed", 300), max_len=512)
    new = make_workload("llama3_8b_gqa", seed=27, B=40, lengths=("loguniform", 1, 3000),
                        max_len=32768)
    steps = [DeviceStep(w) for w in (warm_tail, warm_static, new)]
    outs = [torch.full_like(ds.out, float("nan")) for ds in steps]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for ds in steps:
        ds.append()

    def call(i, wl):
        ds = steps[i]
        pa.pa_decode_noalloc(ds.q, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale,
                             outs[i], wl.max_blocks * wl.block_size, device_error=err)

    call(0, warm_tail)
    call(1, warm_static)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    torch_before = torch.cuda.memory_allocated()
    call(2, new)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert torch.cuda.memory_allocated() == torch_before
    assert int(err.item()) == 0
    got = out_f64(outs[2])
    assert np.abs(got - _reference(new)).max() <= tol(new)


@pytest.mark.parametrize("B,Hq,Hkv,D", [(8192, 16, 1, 128), (4096, 32, 2, 128),
                                        (8192, 8, 1, 64), (2048, 64, 4, 128)])
def test_noalloc_never_runs_out_of_scratch_within_the_limits(B, Hq, Hkv, D):
    # The largest batches the call takes, with 16 or 8 query heads per kv head
    # and a 2048-block table bound (32768 tokens): the planned partials far
    # exceed the scratch, yet a smaller grid is planned instead of
    # PA_ERR_WORKSPACE; sampled rows match the oracle.
    wl = make_workload("llama3_8b_gqa", seed=28, B=B, Hq=Hq, Hkv=Hkv, D=D,
                       lengths=("uniform", 1, 40), max_len=64, max_blocks=2048,
                       pool=("factor", 1.05))
    ds = DeviceStep(wl)
    ds.append()
    got, err = _noalloc(ds, wl, max_seq_len=wl.max_blocks * wl.block_size)
    assert err == 0
    kp, vp = pools_after_append(wl)
    rng = np.random.default_rng(B + Hq)
    idx = rng.choice(B * Hq, size=64, replace=False)
    pairs = np.stack([idx // Hq, idx % Hq], axis=1).astype(np.int32)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale, pairs=pairs)
    assert np.abs(got[pairs[:, 0], pairs[:, 1]] - ref).max() <= tol(wl)
