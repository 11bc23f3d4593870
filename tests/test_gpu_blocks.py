"""GPU: batched block copies (bit-exact against the oracle) and the full
copy-on-write step -- prepare_append, pa_copy_blocks, pa_append_kv,
pa_decode -- against the oracle doing the same steps on the host."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import make_workload

from gpu_helpers import DeviceStep, bits, out_f64, to_dev, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("name,extra", [
    ("llama3_8b_gqa", dict(B=6, lengths=("uniform", 1, 500), max_len=512)),
    ("long_splitk", dict(B=2, lengths=("fixed", 300), max_len=320)),
    ("tiny_worked_60", dict()),
])
def test_copy_blocks_bit_exact(name, extra):
    wl = make_workload(name, **extra)
    ds = DeviceStep(wl)
    rng = np.random.default_rng(4)
    n = min(wl.num_blocks // 2, 200)
    perm = rng.permutation(wl.num_blocks)
    src, dst = perm[:n].astype(np.int32), perm[n:2 * n].astype(np.int32)
    pa.pa_copy_blocks(ds.k_pool, ds.v_pool, torch.from_numpy(src).cuda(),
                      torch.from_numpy(dst).cuda())
    torch.cuda.synchronize()
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.copy_blocks(kp, vp, src, dst)
    assert np.array_equal(bits(ds.k_pool), kp.view(bits(ds.k_pool).dtype))
    assert np.array_equal(bits(ds.v_pool), vp.view(bits(ds.v_pool).dtype))
    assert pa.pa_last_device_error(None) == 0


def test_copy_blocks_bad_id_is_skipped_and_reported():
    wl = make_workload("llama3_8b_gqa", B=3, lengths=("uniform", 1, 200), max_len=256)
    ds = DeviceStep(wl)
    pa.pa_last_device_error(None)
    src = np.array([0, wl.num_blocks, 2], dtype=np.int32)
    dst = np.array([3, 4, -1], dtype=np.int32)
    pa.pa_copy_blocks(ds.k_pool, ds.v_pool, torch.from_numpy(src).cuda(),
                      torch.from_numpy(dst).cuda())
    assert pa.pa_last_device_error(None) & pa.PA_DEVERR_COPY
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.copy_blocks(kp, vp, src[:1], dst[:1])
    assert np.array_equal(bits(ds.k_pool), kp)


def test_copy_on_write_step_matches_oracle():
    # Even sequences share the first 4 physical blocks and, with clip_shared off,
    # several append inside them: each such step needs a private copy first.
    lens = [10, 300, 40, 50, 64, 70, 65, 9, 33, 120]
    wl = make_workload("mixed_shared", B=len(lens), shared_prefix_blocks=4,
                       lengths=("list", lens), max_len=512, clip_shared=False)
    bs = wl.block_size
    ds = DeviceStep(wl)
    with pa.BlockManager(wl.num_blocks) as bm:
        # Mirror the generated tables in the manager: allocate exactly the blocks in
        # use (a fresh manager hands out ids in order, so take them all and release
        # the rest), then add one reference per extra table naming a block.
        all_ids = bm.alloc(wl.num_blocks)
        bm.release([i for i in all_ids if wl.refcount[i] == 0])
        for blk in np.nonzero(wl.refcount > 1)[0]:
            bm.fork([int(blk)] * (int(wl.refcount[blk]) - 1))
        tables = wl.block_tables.copy()
        src, dst = bm.prepare_append(tables, wl.cache_lens, bs)
        assert len(src) >= 3, "the workload should exercise copy on write"
        pa.pa_copy_blocks(ds.k_pool, ds.v_pool, torch.from_numpy(src).cuda(),
                          torch.from_numpy(dst).cuda())
        ds.tables.copy_(torch.from_numpy(tables))
        ds.append()
        with pa.Plan() as plan:
            out = ds.decode(plan)
            torch.cuda.synchronize()
            assert plan.last_device_error() == 0
        assert pa.pa_last_device_error(None) == 0
        # The shared blocks were never written.
        for blk in np.nonzero(wl.refcount > 1)[0]:
            assert np.array_equal(bits(ds.k_pool[int(blk)]), wl.k_pool[blk])
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.copy_blocks(kp, vp, src, dst)
    oracle.append(wl.k_new, wl.v_new, kp, vp, tables, wl.cache_lens)
    assert np.array_equal(bits(ds.k_pool), kp) and np.array_equal(bits(ds.v_pool), vp)
    ref = oracle.decode(wl.q, kp, vp, tables, wl.seq_lens, wl.scale)
    got = out_f64(out)
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= tol(wl)
