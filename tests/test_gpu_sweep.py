"""GPU: a seeded random sweep of shapes through every attention entry point,
against the fp64 oracle.

Each case draws a head dimension (64 or 128), a block size (16 or 32), a kv
head count and a group size (1 to 16 query heads per kv head, including ones
that do not divide 128), a batch of 1 to 24 sequences and their lengths: some
on the edges of a page (1, bs - 1, bs, bs + 1, 2 bs), the rest log-uniform up
to a few thousand tokens. It then runs one append + decode step (as two
calls and as one pa_append_decode call), a
multi-query decode with 1 to 6 queries per sequence (on the split tiles up to
16 (query, head) columns per kv head, on the prefill kernel above, or refused
where that kernel does not serve the shape), and, where the shape allows, a
prefill of up to 48 queries per sequence. The hand-picked cases of the other
files cover each feature on purpose; this file covers their combinations.
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

N_CASES = 160


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _draw(i):
    rng = np.random.default_rng(7000 + i)
    D = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32]))
    g = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    Hkv = int(rng.choice([1, 2, 3, 4, 8]))
    while g * Hkv > 128:
        Hkv //= 2
    B = int(rng.integers(1, 25))
    top = int(rng.choice([64, 600, 3000]))
    lens = []
    for _ in range(B):
        if rng.random() < 0.3:
            lens.append(int(rng.choice([1, bs - 1, bs, bs + 1, 2 * bs])))
        else:
            lens.append(int(np.clip(np.floor(np.exp(rng.uniform(0, np.log(top)))), 1, top)))
    return rng, dict(D=D, bs=bs, g=g, Hkv=Hkv, Hq=g * Hkv, lens=lens)


def _workload(i, c):
    return make_workload("llama3_8b_gqa", seed=7000 + i, B=len(c["lens"]), Hq=c["Hq"],
                         Hkv=c["Hkv"], D=c["D"], block_size=c["bs"],
                         lengths=("list", c["lens"]), max_len=max(c["lens"]) + c["bs"])


def _queries(rng, wl, nmax):
    L = wl.seq_lens.astype(np.int64)
    ns = np.minimum(rng.integers(1, nmax + 1, size=wl.B), L).astype(np.int64)
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    q = bf16_bits(rng.standard_normal((int(qs[-1]), wl.Hq, wl.D)).astype(np.float32))
    return ns, qs, q


@pytest.mark.parametrize("i", range(N_CASES))
def test_decode_step_matches_oracle(i):
    _, c = _draw(i)
    wl = _workload(i, c)
    kp, vp = pools_after_append(wl)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        got = out_f64(ds.decode(plan))
        assert plan.last_device_error() == 0
    assert np.isfinite(got).all()
    e = np.abs(got - ref).max()
    assert e <= BF16_TOL, f"{c}: max abs error {e:.3e}"


@pytest.mark.parametrize("i", range(N_CASES))
def test_one_call_step_matches_oracle(i):
    # pa_append_decode on the same shapes: the pools equal oracle.append bit
    # for bit and the output matches the oracle.
    _, c = _draw(i)
    wl = _workload(i, c)
    kp, vp = pools_after_append(wl)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    ds = DeviceStep(wl)
    with pa.Plan() as plan:
        pa.pa_append_decode(ds.q, ds.k_new, ds.v_new, ds.k_pool, ds.v_pool, ds.tables,
                            ds.seq_lens, wl.scale, ds.out, wl.max_seq_len, plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    got = out_f64(ds.out)
    assert np.isfinite(got).all()
    e = np.abs(got - ref).max()
    assert e <= BF16_TOL, f"{c}: max abs error {e:.3e}"
    assert np.array_equal(ds.k_pool.view(torch.int16).cpu().numpy().view(np.uint16), kp)
    assert np.array_equal(ds.v_pool.view(torch.int16).cpu().numpy().view(np.uint16), vp)


@pytest.mark.parametrize("i", range(N_CASES))
def test_multi_query_decode_matches_oracle(i):
    rng, c = _draw(i)
    wl = _workload(i, c)
    append_in_place(wl)
    ns, qs, q = _queries(rng, wl, int(rng.integers(1, 7)))
    max_q = int(ns.max())
    ds = DeviceStep(wl)
    out = torch.full((q.shape[0], wl.Hq, wl.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    args = (to_dev(q, "bf16"), torch.from_numpy(qs).cuda(), ds.k_pool, ds.v_pool, ds.tables,
            ds.seq_lens, wl.scale, out, max_q, wl.max_seq_len)
    served = max_q * c["g"] <= 16 or (c["D"] == 128 and 128 % c["g"] == 0)
    with pa.Plan() as plan:
        if not served:
            with pytest.raises(pa.PagedAttentionError) as ex:
                pa.pa_decode_multi(*args, plan)
            assert ex.value.status == pa.PA_ERR_SHAPE
            return
        pa.pa_decode_multi(*args, plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
        path = plan.info()[0]
        assert (path == pa.PA_PATH_PREFILL) == (max_q * c["g"] > 16)
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    got = out_f64(out)
    assert np.isfinite(got).all()
    e = np.abs(got - ref).max()
    assert e <= BF16_TOL, f"{c}, max_q {max_q}: max abs error {e:.3e}"


@pytest.mark.parametrize("i", range(N_CASES))
def test_prefill_matches_oracle_where_served(i):
    rng, c = _draw(i)
    if c["D"] != 128 or 128 % c["g"] != 0:
        pytest.skip("the prefill kernel's tiles need D = 128 and a group size dividing 128")
    wl = _workload(i, c)
    append_in_place(wl)
    ns, qs, q = _queries(rng, wl, 48)
    ds = DeviceStep(wl)
    out = torch.full((q.shape[0], wl.Hq, wl.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_prefill(to_dev(q, "bf16"), torch.from_numpy(qs).cuda(), ds.k_pool, ds.v_pool, ds.tables,
                  ds.seq_lens, wl.scale, out, int(ns.max()), wl.max_seq_len, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    got = out_f64(out)
    assert np.isfinite(got).all()
    e = np.abs(got - ref).max()
    assert e <= BF16_TOL, f"{c}: max abs error {e:.3e}"


@pytest.mark.parametrize("i", range(8))
def test_long_sequences_with_the_dynamic_tail_match_oracle(i):
    # Up to 20,000 tokens in a table of 1,280 pages at block size 16: the
    # decode's dynamic tail and the many-partial merge, for random group
    # sizes and head dimensions; then a few queries per sequence.
    rng = np.random.default_rng(7500 + i)
    D = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 3, 4, 8, 16]))
    Hkv = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 5))
    lens = [int(x) for x in np.floor(np.exp(rng.uniform(np.log(2000), np.log(20000), size=B)))]
    wl = make_workload("llama3_8b_gqa", seed=7500 + i, B=B, Hq=g * Hkv, Hkv=Hkv, D=D,
                       block_size=16, lengths=("list", lens), max_len=20480)
    kp, vp = pools_after_append(wl)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        got = out_f64(ds.decode(plan))
        assert plan.last_device_error() == 0
    assert np.isfinite(got).all()
    e = np.abs(got - ref).max()
    assert e <= BF16_TOL, f"D {D} g {g} Hkv {Hkv} lens {lens}: max abs error {e:.3e}"
    # The same step as one call, on fresh pools: the dynamic tail's pieces
    # carry the appended slots too.
    ds1 = DeviceStep(wl)
    with pa.Plan() as plan:
        pa.pa_append_decode(ds1.q, ds1.k_new, ds1.v_new, ds1.k_pool, ds1.v_pool, ds1.tables,
                            ds1.seq_lens, wl.scale, ds1.out, wl.max_seq_len, plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert torch.equal(ds1.out.view(torch.int16), ds.out.view(torch.int16))
    assert torch.equal(ds1.k_pool.view(torch.int16), ds.k_pool.view(torch.int16))

    append_in_place(wl)
    ns, qs, q = _queries(rng, wl, max(1, 16 // g))
    out = torch.full((q.shape[0], wl.Hq, wl.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    with pa.Plan() as plan:
        pa.pa_decode_multi(to_dev(q, "bf16"), torch.from_numpy(qs).cuda(), ds.k_pool, ds.v_pool,
                           ds.tables, ds.seq_lens, wl.scale, out, int(ns.max()), wl.max_seq_len,
                           plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    got = out_f64(out)
    assert np.isfinite(got).all()
    e = np.abs(got - ref).max()
    assert e <= BF16_TOL, f"D {D} g {g} Hkv {Hkv} lens {lens}, multi: max abs error {e:.3e}"
