"""GPU: causal paged multi-query attention (tcgen05 tensor cores) against the
fp64 oracle, within the bf16 tolerance. Query counts that do not fill a block,
partial final chunks, NaN-poisoned slots past each sequence, GQA group sizes
1..16, both block sizes, ties in the longest-first block order and batches
past the size it is applied to are covered."""

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


_rng = np.random.default_rng(5)
_MANY_LENS = [int(x) for x in _rng.integers(1, 80, size=300)]
_MANY_NS = [int(min(x, y)) for x, y in zip(_MANY_LENS, _rng.integers(1, 20, size=300))]


# Small calls choose the one-tile kernel by themselves; the tests below run
# each case on both kernels, pinned through the test hook.
KERNELS = [pa.PA_PREFILL_ONE_TILE, pa.PA_PREFILL_TWO_TILE]


@pytest.fixture(params=KERNELS, ids=["one_tile", "two_tile"])
def kernel(request):
    pa.pa_debug_set_prefill_kernel(request.param)
    try:
        yield request.param
    finally:
        pa.pa_debug_set_prefill_kernel(pa.PA_PREFILL_AUTO)


def _case(lens, ns, Hq=32, Hkv=8, bs=16, seed=0):
    wl = make_workload("llama3_8b_gqa", seed=seed, B=len(lens), Hq=Hq, Hkv=Hkv, block_size=bs,
                       lengths=("list", lens), max_len=max(lens) + bs)
    append_in_place(wl)   # every token of the chunk is already in the pools
    rng = np.random.default_rng(seed + 1)
    T = int(sum(ns))
    q = bf16_bits(rng.standard_normal((T, Hq, wl.D)).astype(np.float32))
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    return wl, q, qs


def _run(wl, q, qs, ns):
    ds = DeviceStep(wl)
    qd = to_dev(q, "bf16")
    out = torch.full((q.shape[0], wl.Hq, wl.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_prefill(qd, torch.from_numpy(qs).cuda(), ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens,
                  wl.scale, out, max(ns), wl.max_seq_len, device_error=err)
    torch.cuda.synchronize()
    return out_f64(out), int(err.item())


@pytest.mark.parametrize("Hq,Hkv,bs,lens,ns", [
    (32, 8, 16, [200, 64, 1000], [37, 64, 130]),        # g = 4: 32 queries per block
    (64, 8, 32, [513, 129], [129, 1]),                  # g = 8, block size 32
    (8, 8, 16, [300, 1], [150, 1]),                     # g = 1: 128 queries per block
    (16, 1, 16, [90, 640], [8, 40]),                    # g = 16 (MQA-like)
    (4, 2, 32, [64, 65, 66], [64, 65, 2]),              # g = 2, ragged edges
    (32, 8, 16, [50] * 20 + [120] * 20, [10] * 40),     # equal lengths: the longest-first order breaks ties
    (32, 8, 16, _MANY_LENS, _MANY_NS),                  # more sequences than are ordered by length
])
def test_prefill_matches_oracle(Hq, Hkv, bs, lens, ns, kernel):
    wl, q, qs = _case(lens, ns, Hq=Hq, Hkv=Hkv, bs=bs)
    got, err = _run(wl, q, qs, ns)
    assert err == 0
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    assert np.isfinite(got).all()
    e = np.abs(got - ref).max()
    assert e <= BF16_TOL, f"max abs error {e:.3e}"


@pytest.mark.parametrize("lens,ns", [
    ([200, 64, 1000], [37, 64, 130]),   # full and partial query tiles
    ([300, 500], [64, 128]),            # full tiles only
])
def test_float_output_rounds_to_the_bf16_output(lens, ns, kernel):
    # bf16 output of full tiles leaves through tiled tensor stores, float
    # output and partial tiles through the threads' own stores; the same
    # normalised values rounded to nearest even must agree bit for bit.
    wl, q, qs = _case(lens, ns)
    ds = DeviceStep(wl)
    qd = to_dev(q, "bf16")
    outs = {}
    for dt in (torch.bfloat16, torch.float32):
        out = torch.full((q.shape[0], wl.Hq, wl.D), float("nan"), dtype=dt, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pa.pa_prefill(qd, torch.from_numpy(qs).cuda(), ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens,
                      wl.scale, out, max(ns), wl.max_seq_len, device_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs[dt] = out
    f32 = outs[torch.float32]
    assert torch.isfinite(f32).all()
    assert torch.equal(f32.to(torch.bfloat16).view(torch.int16), outs[torch.bfloat16].view(torch.int16))
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    assert np.abs(f32.double().cpu().numpy() - ref).max() <= BF16_TOL


def test_single_query_prefill_matches_decode(kernel):
    wl, q, qs = _case([77, 300, 16], [1, 1, 1])
    got, err = _run(wl, q, qs, [1, 1, 1])
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    assert err == 0 and np.abs(got - ref).max() <= BF16_TOL


def test_prefill_bad_lengths_and_table(kernel):
    wl, q, qs = _case([100, 50], [10, 10])
    ds = DeviceStep(wl)
    qd = to_dev(q, "bf16")
    out = torch.zeros((q.shape[0], wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = ds.tables.clone()
    t[1, 0] = wl.num_blocks + 1
    pa.pa_prefill(qd, torch.from_numpy(qs).cuda(), ds.k_pool, ds.v_pool, t, ds.seq_lens, wl.scale,
                  out, 10, wl.max_seq_len, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_DEVERR_TABLE
    got = out_f64(out)
    assert (got[10:] == 0).all()
    ref = oracle.prefill(q[:10], wl.k_pool, wl.v_pool, wl.block_tables[:1], wl.seq_lens[:1],
                         qs[:2], wl.scale)
    assert np.abs(got[:10] - ref).max() <= BF16_TOL


def test_prefill_rows_past_the_query_array_are_refused(kernel):
    # q_start says 20 rows, but q and out hold 15: the second sequence's rows
    # would fall outside them, so it is refused (PA_DEVERR_SEQ_LEN, rows
    # untouched) and nothing is read or written past the arrays.
    wl, q, qs = _case([100, 50], [10, 10])
    ds = DeviceStep(wl)
    qd = to_dev(q[:15], "bf16")
    out = torch.full((15, wl.Hq, wl.D), 7.0, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_prefill(qd, torch.from_numpy(qs).cuda(), ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens,
                  wl.scale, out, 10, wl.max_seq_len, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_DEVERR_SEQ_LEN
    got = out_f64(out)
    assert (got[10:] == 7.0).all()
    ref = oracle.prefill(q[:10], wl.k_pool, wl.v_pool, wl.block_tables[:1], wl.seq_lens[:1],
                         qs[:2], wl.scale)
    assert np.abs(got[:10] - ref).max() <= BF16_TOL


def test_prefill_more_queries_than_max_q_are_refused(kernel):
    # The second sequence has 70 queries against max_q = 64: refused
    # (PA_DEVERR_SEQ_LEN, its rows untouched); the first is computed.
    wl, q, qs = _case([900, 1500], [64, 70])
    ds = DeviceStep(wl)
    out = torch.full((q.shape[0], wl.Hq, wl.D), 7.0, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_prefill(to_dev(q, "bf16"), torch.from_numpy(qs).cuda(), ds.k_pool, ds.v_pool, ds.tables,
                  ds.seq_lens, wl.scale, out, 64, wl.max_seq_len, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_DEVERR_SEQ_LEN
    got = out_f64(out)
    assert (got[qs[1]:] == 7.0).all()
    ref = oracle.prefill(q[:64], wl.k_pool, wl.v_pool, wl.block_tables[:1], wl.seq_lens[:1],
                         qs[:2], wl.scale)
    assert np.abs(got[:64] - ref).max() <= BF16_TOL


@pytest.mark.parametrize("name", ["prefill_gqa", "llama3_8b_gqa"])
def test_prefill_full_size_sampled_rows(name):
    """The benchmark's workloads at full size (the newest 256 tokens of every
    sequence are queries): sampled query rows, each checked against the
    oracle on its own (query i of sequence b sees its first L - n + i + 1
    tokens), including the first and last query row of every sequence."""
    wl = make_workload(name)
    append_in_place(wl)
    ns = np.minimum(wl.seq_lens, 256).astype(np.int64)
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    T = int(qs[-1])
    q = bf16_bits(np.random.default_rng(11).standard_normal((T, wl.Hq, wl.D)).astype(np.float32))
    got, err = _run(wl, q, qs, [int(x) for x in ns])
    assert err == 0
    rng = np.random.default_rng(12)
    rows = set(rng.choice(T, size=48, replace=False).tolist())
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
