"""GPU: pa_append_decode (the step's append and decode in one call) against
the fp64 oracle and against the two separate calls.

The pools after the call must equal oracle.append bit for bit (NaN payloads
included); the attention output must match the oracle within the bf16 / f32
tolerance and the separate pa_append_kv + pa_decode calls bit for bit (the
fused path runs the same tile arithmetic). Covered: the five reduced
workloads, 1 to 32 query heads per kv head (two kv units per head at 32),
both head dimensions and block sizes, lengths on page edges, a sequence long
enough for the dynamic tail, every fallback path (CUDA-core, one warp per
row, fused merge, float32 pools), bad table entries and lengths, and two
steps in a row on one plan.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import make_workload
from oracle_steps import pools_after_append

from gpu_helpers import DeviceStep, bits, out_f64, to_dev, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


CASES = {
    "tiny_worked_60": dict(name="tiny_worked_60"),
    "mha_small": dict(name="llama7b_mha", B=6, lengths=("uniform", 1, 900), max_len=1024,
                      pool=("fixed", 2048)),
    "gqa_small": dict(name="llama3_8b_gqa", B=9, lengths=("loguniform", 1, 3000), max_len=3072),
    "long_small": dict(name="long_splitk", B=2, lengths=("fixed", 6001), max_len=6016),
    "mixed_small": dict(name="mixed_shared", B=20, shared_prefix_blocks=4, max_len=512,
                        lengths=("geometric", 1 / 90, 1, 512)),
    "g32": dict(name="llama3_8b_gqa", B=5, Hq=64, Hkv=2, lengths=("loguniform", 1, 2000),
                max_len=2048),
    "d64_bs32": dict(name="llama3_8b_gqa", B=7, Hq=12, Hkv=2, D=64, block_size=32,
                     lengths=("list", [1, 31, 32, 33, 64, 65, 500]), max_len=512),
    "tail_long": dict(name="llama3_8b_gqa", B=3, lengths=("list", [17000, 3, 9000]),
                      max_len=17408),
}


def _wl(key, **extra):
    spec = dict(CASES[key])
    spec.update(extra)
    return make_workload(spec.pop("name"), **spec)


def _fused(ds, plan, out=None, max_seq_len=None):
    out = ds.out if out is None else out
    pa.pa_append_decode(ds.q, ds.k_new, ds.v_new, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens,
                        ds.wl.scale, out, max_seq_len or ds.wl.max_seq_len, plan)
    return out


def _pool_bits(t):
    return bits(t).copy()


@pytest.mark.parametrize("key", sorted(CASES))
def test_fused_step_matches_oracle_and_the_separate_calls(key):
    wl = _wl(key)
    kp, vp = pools_after_append(wl)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)

    fused = DeviceStep(wl)
    with pa.Plan() as plan:
        out = _fused(fused, plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert pa.pa_last_device_error(None) == 0
    got = out_f64(out)
    assert np.isfinite(got).all()
    e = np.abs(got - ref).max()
    assert e <= tol(wl), f"max abs error {e:.3e}"
    # The pools hold exactly the oracle's append.
    assert np.array_equal(_pool_bits(fused.k_pool), kp.view(bits(fused.k_pool).dtype))
    assert np.array_equal(_pool_bits(fused.v_pool), vp.view(bits(fused.v_pool).dtype))

    apart = DeviceStep(wl)
    apart.append()
    with pa.Plan() as plan:
        out2 = apart.decode(plan)
        torch.cuda.synchronize()
    assert np.array_equal(bits(out), bits(out2))


@pytest.mark.parametrize("path", [pa.PA_PATH_FMA, pa.PA_PATH_SIMPLE, "fused_merge"])
def test_fallback_paths_append_first_and_agree(path):
    wl = _wl("mha_small") if path == pa.PA_PATH_FMA else _wl("gqa_small")
    kp, vp = pools_after_append(wl)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    fused = DeviceStep(wl)
    apart = DeviceStep(wl)
    apart.append()
    with pa.Plan() as p1, pa.Plan() as p2:
        # A plan exists after its first call; the append is idempotent (the
        # same rows to the same slots), so the second fused call sees the
        # same pools.
        _fused(fused, p1)
        apart.decode(p2)
        for p in (p1, p2):
            if path == "fused_merge":
                p.set_merge(pa.PA_MERGE_FUSED)
            else:
                p.set_path(path)
        out = _fused(fused, p1)
        out2 = apart.decode(p2)
        assert p1.info()[0] == (pa.PA_PATH_MMA if path == "fused_merge" else path)
        torch.cuda.synchronize()
        assert p1.last_device_error() == 0
    assert np.abs(out_f64(out) - ref).max() <= tol(wl)
    assert np.array_equal(bits(out), bits(out2))
    assert np.array_equal(_pool_bits(fused.k_pool), kp.view(bits(fused.k_pool).dtype))
    assert np.array_equal(_pool_bits(fused.v_pool), vp.view(bits(fused.v_pool).dtype))


def test_bad_tail_entry_skips_the_append_and_zeroes_the_rows():
    # Sequence 1's last table entry points past the pool: its append is
    # skipped (the pools keep their bits), its rows are zeros, the others
    # are exact.
    wl = _wl("gqa_small")
    b = 1
    nb = -(-int(wl.seq_lens[b]) // wl.block_size)
    before_k, before_v = wl.k_pool.copy(), wl.v_pool.copy()
    kp, vp = pools_after_append(wl)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    ds = DeviceStep(wl)
    bad = wl.block_tables.copy()
    bad[b, nb - 1] = wl.num_blocks
    ds.tables.copy_(torch.from_numpy(bad))
    with pa.Plan() as plan:
        out = _fused(ds, plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() & pa.PA_DEVERR_TABLE
    got = out_f64(out)
    assert (got[b] == 0).all()
    others = [i for i in range(wl.B) if i != b]
    assert np.abs(got[others] - ref[others]).max() <= tol(wl)
    # Sequence b's blocks, its real tail block included, are unchanged; the
    # others got their append.
    k_after, v_after = bits(ds.k_pool), bits(ds.v_pool)
    own = wl.block_tables[b, :nb]
    assert np.array_equal(k_after[own], before_k[own])
    assert np.array_equal(v_after[own], before_v[own])
    for i in others:
        nbi = -(-int(wl.seq_lens[i]) // wl.block_size)
        blk = wl.block_tables[i, nbi - 1]
        assert np.array_equal(k_after[blk], kp[blk])


def test_bad_length_gets_no_append_and_zero_rows():
    wl = _wl("gqa_small")
    b = 2
    before_k = wl.k_pool.copy()
    ds = DeviceStep(wl)
    lens = wl.seq_lens.copy()
    lens[b] = 0
    ds.seq_lens.copy_(torch.from_numpy(lens))
    with pa.Plan() as plan:
        out = _fused(ds, plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() & pa.PA_DEVERR_SEQ_LEN
    assert (out_f64(out)[b] == 0).all()
    k_after = bits(ds.k_pool)
    nb = -(-int(wl.seq_lens[b]) // wl.block_size)
    blocks = wl.block_tables[b, :nb]
    assert np.array_equal(k_after[blocks], before_k[blocks])


def test_two_steps_in_a_row_on_one_plan():
    # Step 1 appends token L-1 and attends over L tokens; step 2 appends
    # token L with fresh rows and attends over L+1, in the same pools.
    wl = _wl("gqa_small", max_len=3100)
    rng = np.random.default_rng(5)
    ds = DeviceStep(wl)
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    with pa.Plan() as plan:
        _fused(ds, plan)
        oracle.append(wl.k_new, wl.v_new, kp, vp, wl.block_tables, wl.cache_lens)
        # Step 2: one more token per sequence (the workload's tables reach it).
        lens2 = wl.seq_lens + 1
        kn2 = (rng.standard_normal(wl.k_new.shape).astype(np.float32).view(np.uint32) >> 16
               ).astype(np.uint16)
        vn2 = (rng.standard_normal(wl.v_new.shape).astype(np.float32).view(np.uint32) >> 16
               ).astype(np.uint16)
        ok = np.array([-(-int(L) // wl.block_size) <= wl.max_blocks for L in lens2])
        assert ok.all()
        tables2 = wl.block_tables.copy()
        for i in range(wl.B):
            nb_old = -(-int(wl.seq_lens[i]) // wl.block_size)
            nb_new = -(-int(lens2[i]) // wl.block_size)
            if nb_new > nb_old:  # a fresh block for the token that opens a page
                tables2[i, nb_new - 1] = np.nonzero(wl.refcount == 0)[0][i]
        ds.tables.copy_(torch.from_numpy(tables2))
        ds.seq_lens.copy_(torch.from_numpy(lens2.astype(np.int32)))
        ds.k_new.copy_(to_dev(kn2, "bf16"))
        ds.v_new.copy_(to_dev(vn2, "bf16"))
        out = _fused(ds, plan, max_seq_len=int(lens2.max()))
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    oracle.append(kn2, vn2, kp, vp, tables2, wl.seq_lens)
    ref = oracle.decode(wl.q, kp, vp, tables2, lens2, wl.scale)
    assert np.abs(out_f64(out) - ref).max() <= tol(wl)
    assert np.array_equal(bits(ds.k_pool), kp)
    assert np.array_equal(bits(ds.v_pool), vp)
