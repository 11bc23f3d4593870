"""GPU: speculative verification of more drafted tokens than the split decode
tiles hold (pa_decode_multi above 16 (query, head) columns per kv head) on
small batches, where the one-tile tensor-core kernel splits every tile's key
range over several blocks and a second kernel merges their partials.

Against the fp64 oracle's causal multi-query attention: one to three
sequences of up to ~20k tokens with 5 to 32 queries each (one and several
splits, splits past a short sequence's end), both block sizes, float
output; a bad table entry (the poisoned partials give zero rows); a
sequence with more queries than max_q or than tokens (an error and zero
rows, on split and unsplit calls of both prefill kernels); a plain decode
on the same plan afterwards (the split decode's counters in the workspace
are left intact), and a second call giving the same bits.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import bf16_bits, make_workload
from oracle_steps import append_in_place, pools_after_append

from gpu_helpers import BF16_TOL, DeviceStep, bits, out_f64, to_dev, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _case(lens, ns, bs=16, seed=0):
    wl = make_workload("llama3_8b_gqa", seed=seed, B=len(lens), Hq=32, Hkv=8, D=128,
                       block_size=bs, lengths=("list", lens), max_len=max(lens) + bs)
    append_in_place(wl)   # the drafted tokens are already in the pools
    rng = np.random.default_rng(seed + 1)
    q = bf16_bits(rng.standard_normal((int(sum(ns)), wl.Hq, wl.D)).astype(np.float32))
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    return wl, q, qs


def _call(ds, wl, q, qs, max_q, plan, out_dtype=torch.bfloat16):
    out = torch.full((q.shape[0], wl.Hq, wl.D), float("nan"), dtype=out_dtype, device="cuda")
    pa.pa_decode_multi(to_dev(q, "bf16"), torch.from_numpy(qs).cuda(), ds.k_pool, ds.v_pool,
                       ds.tables, ds.seq_lens, wl.scale, out, max_q, wl.max_seq_len, plan)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("lens,ns,bs", [
    ([20000], [8], 16),                # one sequence: many splits
    ([20000], [32], 16),               # a whole tile of queries
    ([6000, 300, 15000], [5, 8, 7], 16),   # ragged: splits past the short sequence's end
    ([9000, 4001], [16, 6], 32),       # block size 32
    ([700], [12], 16),                 # short: a few splits of two chunks
])
def test_split_verification_matches_oracle(lens, ns, bs):
    wl, q, qs = _case(lens, ns, bs=bs)
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    ds = DeviceStep(wl)
    with pa.Plan() as plan:
        out = _call(ds, wl, q, qs, max(ns), plan)
        assert plan.last_device_error() == 0
        assert plan.info()[0] == pa.PA_PATH_PREFILL
        first = bits(out).copy()
        out2 = _call(ds, wl, q, qs, max(ns), plan)
    got = out_f64(out)
    assert np.isfinite(got).all()
    e = np.abs(got - ref).max()
    assert e <= BF16_TOL, f"max abs error {e:.3e}"
    assert np.array_equal(bits(out2), first)


def test_split_float_output_rounds_to_the_bf16_output():
    wl, q, qs = _case([12000, 5000], [8, 8])
    ds = DeviceStep(wl)
    with pa.Plan() as plan:
        o16 = _call(ds, wl, q, qs, 8, plan)
        o32 = _call(ds, wl, q, qs, 8, plan, out_dtype=torch.float32)
        assert plan.last_device_error() == 0
    assert torch.isfinite(o32).all()
    assert torch.equal(o32.to(torch.bfloat16).view(torch.int16), o16.view(torch.int16))


def test_bad_table_entry_zeroes_that_sequence_only():
    wl, q, qs = _case([9000, 9000], [8, 8])
    ref = oracle.prefill(q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens, qs, wl.scale)
    ds = DeviceStep(wl)
    bad = wl.block_tables.copy()
    bad[1, 3] = wl.num_blocks          # outside the pool, inside sequence 1's range
    ds.tables.copy_(torch.from_numpy(bad))
    with pa.Plan() as plan:
        out = _call(ds, wl, q, qs, 8, plan)
        assert plan.last_device_error() & pa.PA_DEVERR_TABLE
    got = out_f64(out)
    assert (got[qs[1]:qs[2]] == 0).all()
    assert np.abs(got[qs[0]:qs[1]] - ref[qs[0]:qs[1]]).max() <= BF16_TOL


def test_decode_on_the_same_plan_after_a_split_call():
    # The split call's partials share the plan's workspace with the split
    # decode, whose counters must still be zero for the next decode.
    wl, q, qs = _case([20000, 3000], [8, 8])
    ds = DeviceStep(wl)
    with pa.Plan() as plan:
        _call(ds, wl, q, qs, 8, plan)
        # A decode whose workspace fits in the one the split call sized, so
        # that both calls share it.
        dwl = make_workload("llama3_8b_gqa", seed=9, B=2, lengths=("loguniform", 1, 8000),
                            max_len=8016)
        kp, vp = pools_after_append(dwl)
        dref = oracle.decode(dwl.q, kp, vp, dwl.block_tables, dwl.seq_lens, dwl.scale)
        dds = DeviceStep(dwl)
        dds.append()
        for _ in range(2):
            dout = dds.decode(plan)
            torch.cuda.synchronize()
            assert plan.last_device_error() == 0
            assert np.abs(out_f64(dout) - dref).max() <= tol(dwl)


@pytest.mark.parametrize("lens,ns,max_q,bad", [
    ([9000, 6000], [8, 20], 8, 1),     # more queries than max_q (split call)
    ([9000, 10], [8, 12], 12, 1),      # more queries than tokens (split call)
    ([3000] * 39 + [20], [24] * 39 + [30], 24, 39),   # one-tile kernel, no split; n > max_q
    ([3000] * 39 + [2000], [64] * 39 + [70], 64, 39),  # two-tile kernel; n > max_q
])
def test_invalid_sequence_gets_zero_rows_and_an_error(lens, ns, max_q, bad):
    # Above 16 columns pa_decode_multi runs the prefill kernels; an invalid
    # sequence raises PA_DEVERR_SEQ_LEN and gets zero rows, as on the split
    # decode's tiles, and the split merge reads no partial for it.
    wl, q, qs = _case(lens, [min(n, l) for n, l in zip(ns, lens)])
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    rng = np.random.default_rng(7)
    q = bf16_bits(rng.standard_normal((int(qs[-1]), wl.Hq, wl.D)).astype(np.float32))
    ds = DeviceStep(wl)
    with pa.Plan() as plan:
        out = _call(ds, wl, q, qs, max_q, plan)
        assert plan.last_device_error() & pa.PA_DEVERR_SEQ_LEN
        assert plan.info()[0] == pa.PA_PATH_PREFILL
    got = out_f64(out)
    assert (got[qs[bad]:qs[bad + 1]] == 0).all()
    good = [b for b in range(len(lens)) if b != bad][:3]
    for b in good:
        ref = oracle.prefill(q[qs[b]:qs[b + 1]], wl.k_pool, wl.v_pool, wl.block_tables[b:b + 1],
                             wl.seq_lens[b:b + 1], np.array([0, ns[b]], np.int32), wl.scale)
        assert np.abs(got[qs[b]:qs[b + 1]] - ref).max() <= BF16_TOL
