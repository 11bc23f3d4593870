"""GPU: decode attention for a few new queries per sequence (speculative
verification) on the split decode kernels, against the fp64 oracle's causal
multi-query attention: ragged query counts, GQA group sizes 1..16, both block
sizes, D = 64, sequences as short as their query count, sequences long
enough for the dynamically scheduled tail (merged across many partials),
invalid counts, one query per sequence equal to pa_decode, and the
speculative-verification workload at full size on sampled rows."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import bf16_bits, make_workload
from oracle_steps import append_in_place

from gpu_helpers import BF16_TOL, DeviceStep, out_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _case(lens, ns, Hq=32, Hkv=8, bs=16, D=128, seed=0):
    wl = make_workload("llama3_8b_gqa", seed=seed, B=len(lens), Hq=Hq, Hkv=Hkv, D=D,
                       block_size=bs, lengths=("list", lens), max_len=max(lens) + bs)
    append_in_place(wl)   # the drafted tokens are already in the pools
    rng = np.random.default_rng(seed + 1)
    q = bf16_bits(rng.standard_normal((int(sum(ns)), Hq, D)).astype(np.float32))
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    return wl, q, qs


def _run(wl, q, qs, max_q, plan=None):
    ds = DeviceStep(wl)
    out = torch.full((q.shape[0], wl.Hq, wl.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    own = plan is None
    plan = plan or pa.Plan()
    pa.pa_decode_multi(to_dev(q, "bf16"), torch.from_numpy(qs).cuda(), ds.k_pool, ds.v_pool,
                       ds.tables, ds.seq_lens, wl.scale, out, max_q, wl.max_seq_len, plan)
    torch.cuda.synchronize()
    err = plan.last_device_error()
    if own:
        plan.free()
    return out_f64(out), err


@pytest.mark.parametrize("Hq,Hkv,bs,D,lens,ns", [
    (32, 8, 16, 128, [200, 64, 1000, 5], [4, 4, 3, 1]),     # g = 4, 16 columns, ragged counts
    (64, 8, 32, 128, [513, 129], [2, 1]),                   # g = 8, block size 32
    (8, 8, 16, 128, [300, 40, 17], [4, 8, 2]),              # g = 1 (MHA), 8 queries
    (16, 1, 16, 128, [90, 640], [1, 1]),                    # g = 16, one query each
    (16, 4, 16, 64, [77, 300, 9], [4, 2, 4]),               # D = 64
    (32, 8, 32, 128, [3, 4, 33], [3, 4, 4]),                # as many queries as tokens
])
def test_decode_multi_matches_oracle(Hq, Hkv, bs, D, lens, ns):
    wl, q, qs = _case(lens, ns, Hq=Hq, Hkv=Hkv, bs=bs, D=D)
    got, err = _run(wl, q, qs, max(ns))
    assert err == 0
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    assert np.isfinite(got).all()
    e = np.abs(got - ref).max()
    assert e <= BF16_TOL, f"max abs error {e:.3e}"


@pytest.mark.parametrize("tail", [None, (150, 1)])
def test_long_sequences_merge_many_partials(tail):
    # Long rows are cut by many static ranges; with a forced dynamic tail of
    # one-page pieces (pa_plan_set_schedule) they are also cut into many
    # pieces and merged four warps per row.
    lens, ns = [20000, 17000, 300, 9000], [4, 2, 4, 1]
    wl, q, qs = _case(lens, ns, seed=3)
    with pa.Plan() as plan:
        if tail:
            _run(wl, q, qs, 4, plan)      # creates the plan
            plan.set_schedule(*tail)
        got, err = _run(wl, q, qs, 4, plan)
    assert err == 0
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    assert np.abs(got - ref).max() <= BF16_TOL


def test_one_query_per_sequence_equals_decode():
    lens = [200, 64, 1000, 5, 333]
    wl, q, qs = _case(lens, [1] * len(lens), seed=4)
    got, err = _run(wl, q, qs, 1)
    assert err == 0
    ds = DeviceStep(wl)
    out = torch.empty((len(lens), wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    with pa.Plan() as plan:
        pa.pa_decode(to_dev(q, "bf16"), ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale,
                     out, wl.max_seq_len, plan)
        torch.cuda.synchronize()
    assert np.abs(got - out_f64(out)).max() <= BF16_TOL


def test_invalid_query_count_gives_zero_rows_and_an_error():
    lens, ns = [100, 3, 50], [2, 4, 2]   # sequence 1 has more queries than tokens
    wl, q, qs = _case(lens, ns, seed=5)
    got, err = _run(wl, q, qs, 4)
    assert err & pa.PA_DEVERR_SEQ_LEN
    assert (got[qs[1]:qs[2]] == 0).all()
    ref = oracle.prefill(q[:2], wl.k_pool, wl.v_pool, wl.block_tables[:1], wl.seq_lens[:1],
                         qs[:2], wl.scale)
    assert np.abs(got[:2] - ref).max() <= BF16_TOL
    ref2 = oracle.prefill(q[qs[2]:qs[3]], wl.k_pool, wl.v_pool, wl.block_tables[2:3],
                          wl.seq_lens[2:3], [0, ns[2]], wl.scale)
    assert np.abs(got[qs[2]:qs[3]] - ref2).max() <= BF16_TOL


def test_more_queries_than_max_q_give_zero_rows_and_an_error():
    lens, ns = [100, 50, 70], [2, 5, 2]   # sequence 1 has more queries than max_q = 2
    wl, q, qs = _case(lens, ns, seed=6)
    got, err = _run(wl, q, qs, 2)
    assert err & pa.PA_DEVERR_SEQ_LEN
    assert (got[qs[1]:qs[2]] == 0).all()
    for b in (0, 2):
        ref = oracle.prefill(q[qs[b]:qs[b + 1]], wl.k_pool, wl.v_pool, wl.block_tables[b:b + 1],
                             wl.seq_lens[b:b + 1], [0, ns[b]], wl.scale)
        assert np.abs(got[qs[b]:qs[b + 1]] - ref).max() <= BF16_TOL


def test_speculative_workload_full_size_sampled_rows():
    wl = make_workload("spec_gqa")
    append_in_place(wl)
    ns = np.minimum(wl.seq_lens, 4).astype(np.int64)
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    T = int(qs[-1])
    q = bf16_bits(np.random.default_rng(13).standard_normal((T, wl.Hq, wl.D)).astype(np.float32))
    got, err = _run(wl, q, qs, 4)
    assert err == 0
    rows = set(np.random.default_rng(14).choice(T, size=48, replace=False).tolist())
    rows |= set(qs[:-1].tolist()) | set((qs[1:] - 1).tolist())
    worst = 0.0
    for r in sorted(rows):
        b = int(np.searchsorted(qs, r, side="right") - 1)
        i = r - int(qs[b])
        ref = oracle.prefill(q[r:r + 1], wl.k_pool, wl.v_pool, wl.block_tables[b:b + 1],
                             [int(wl.seq_lens[b] - ns[b] + i + 1)], [0, 1], wl.scale)
        assert np.isfinite(got[r]).all()
        worst = max(worst, float(np.abs(got[r] - ref[0]).max()))
    assert worst <= BF16_TOL, f"max abs error {worst:.3e}"


def test_one_plan_alternates_decode_and_multi():
    # The two calls need different workspace sizes (the multi-query tile is
    # wider); a plan serves both in turn, growing its workspace once.
    lens = [20000, 300, 17000, 64]
    wl, q1, _ = _case(lens, [1] * len(lens), seed=6)
    ns = [4, 2, 4, 3]
    q = bf16_bits(np.random.default_rng(16).standard_normal((sum(ns), wl.Hq, wl.D)).astype(np.float32))
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    ds = DeviceStep(wl)
    want_multi, _ = _run(wl, q, qs, 4)
    out1 = torch.empty((len(lens), wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    with pa.Plan() as fresh:
        pa.pa_decode(to_dev(q1, "bf16"), ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale,
                     out1, wl.max_seq_len, fresh)
        torch.cuda.synchronize()
    want_dec = out_f64(out1)
    with pa.Plan() as plan:
        for _ in range(2):
            pa.pa_decode(to_dev(q1, "bf16"), ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale,
                         out1, wl.max_seq_len, plan)
            torch.cuda.synchronize()
            assert np.array_equal(out_f64(out1), want_dec)
            got, err = _run(wl, q, qs, 4, plan=plan)
            assert err == 0 and np.array_equal(got, want_multi)


def test_launch_shape():
    # 16 columns (4 queries x 4 heads) run two blocks of five warps per SM,
    # the kernel's launch bound.
    lens, ns = [700, 300, 2000], [4, 4, 3]
    wl, q, qs = _case(lens, ns, seed=12)
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    with pa.Plan() as plan:
        got, err = _run(wl, q, qs, 4, plan)
        path, blocks, warps = plan.info()
    assert err == 0 and path == pa.PA_PATH_MMA
    assert warps == 5 * blocks
    assert np.abs(got - ref).max() <= BF16_TOL


@pytest.mark.parametrize("Hq,Hkv,lens,ns", [
    (32, 8, [700, 300, 2000], [64, 17, 5]),      # 64 queries x 4 heads: the prefill kernel's tiles
    (8, 8, [129, 40], [20, 3]),                  # g = 1, 20 queries: 20 columns
])
def test_many_queries_route_to_the_prefill_kernel(Hq, Hkv, lens, ns):
    # Above 16 (query, head) columns per kv head the call runs the tcgen05
    # prefill kernel on the same arguments and reports it; the rows are the
    # same causal attention.
    wl, q, qs = _case(lens, ns, Hq=Hq, Hkv=Hkv, seed=40)
    with pa.Plan() as plan:
        got, err = _run(wl, q, qs, max(ns), plan)
        assert plan.info()[0] == pa.PA_PATH_PREFILL
    assert err == 0
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    assert np.abs(got - ref).max() <= BF16_TOL
