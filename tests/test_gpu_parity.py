"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Append and block-table addressing are checked bit for bit; attention within
max abs error 2e-3 (float32 output) or 1.5e-2 (bf16 output) on the same
seeded inputs. Every unused pool block and every slot past a sequence's
length holds NaN, so a stray read shows up in the output.
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

# Reduced versions of the five workloads: sizes the oracle finishes in seconds
# that still span many pages, many warps and ragged tails.
CASES = {
    "tiny_worked_60": dict(name="tiny_worked_60"),
    "mha_small": dict(name="llama7b_mha", B=6, lengths=("uniform", 1, 900), max_len=1024,
                      pool=("fixed", 2048)),
    "gqa_small": dict(name="llama3_8b_gqa", B=9, lengths=("loguniform", 1, 3000), max_len=3072),
    "long_small": dict(name="long_splitk", B=2, lengths=("fixed", 6001), max_len=6016),
    "mixed_small": dict(name="mixed_shared", B=20, shared_prefix_blocks=4, max_len=512,
                        lengths=("geometric", 1 / 90, 1, 512)),
}


def _wl(key, **extra):
    spec = dict(CASES[key])
    spec.update(extra)
    return make_workload(spec.pop("name"), **spec)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _reference(wl):
    kp, vp = pools_after_append(wl)
    return oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale), kp, vp


# ---------------------------------------------------------------- append

@pytest.mark.parametrize("key", sorted(CASES))
def test_append_is_bit_exact(key):
    wl = _wl(key)
    ds = DeviceStep(wl)
    ds.append()
    torch.cuda.synchronize()
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.append(wl.k_new, wl.v_new, kp, vp, wl.block_tables, wl.cache_lens)
    assert np.array_equal(bits(ds.k_pool), kp.view(bits(ds.k_pool).dtype))
    assert np.array_equal(bits(ds.v_pool), vp.view(bits(ds.v_pool).dtype))
    assert pa.pa_last_device_error(None) == 0


# ---------------------------------------------------------------- decode parity, every path

PATHS = {"auto": pa.PA_PATH_AUTO, "simple": pa.PA_PATH_SIMPLE, "fma": pa.PA_PATH_FMA,
         "mma": pa.PA_PATH_MMA}


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("key", sorted(CASES))
def test_decode_matches_oracle(key, path):
    wl = _wl(key)
    if wl.dtype == "f32" and path in ("fma", "mma"):
        pytest.skip("staged paths take bf16 pools")
    ref, _, _ = _reference(wl)
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        if PATHS[path] != pa.PA_PATH_AUTO:
            ds.decode(plan)          # creates the plan
            plan.set_path(PATHS[path])
        out = ds.decode(plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
        used = plan.info()[0]
    if path != "auto":
        assert used == PATHS[path]
    got = out_f64(out)
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    assert err <= tol(wl), f"{key}/{path}: max abs error {err:.3e}"


def test_auto_path_choice():
    for key, want in (("tiny_worked_60", pa.PA_PATH_SIMPLE), ("mha_small", pa.PA_PATH_MMA),
                      ("gqa_small", pa.PA_PATH_MMA), ("long_small", pa.PA_PATH_MMA)):
        wl = _wl(key)
        ds = DeviceStep(wl)
        with pa.Plan() as plan:
            ds.decode(plan)
            assert plan.info()[0] == want


@pytest.mark.parametrize("Hq,Hkv,warps_per_block", [(32, 8, 3), (64, 4, 11), (128, 8, 11), (8, 8, 3)])
def test_launch_shape(Hq, Hkv, warps_per_block):
    # Up to 8 query heads per kv head: blocks of three warps; 9-16 (two
    # n-tiles, query fragments reread from a per-warp region of shared
    # memory): one block of eleven warps per SM at D = 128.
    wl = _exact(Hq, Hkv, 128, 16, [300, 1200], seed=77)
    ref, _, _ = _reference(wl)
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        out = ds.decode(plan)
        torch.cuda.synchronize()
        _, blocks, warps = plan.info()
    assert warps == warps_per_block * blocks
    assert np.abs(out_f64(out) - ref).max() <= tol(wl)


# ---------------------------------------------------------------- invariances

@pytest.mark.parametrize("key", ["gqa_small", "mha_small", "long_small"])
def test_physical_permutation_gives_identical_bits(key):
    wl = _wl(key)
    kp, vp = pools_after_append(wl)
    ds = DeviceStep(wl)
    ds.k_pool.copy_(to_dev(kp, wl.dtype))
    ds.v_pool.copy_(to_dev(vp, wl.dtype))
    with pa.Plan() as plan:
        a = bits(ds.decode(plan).clone())
        perm = np.random.default_rng(3).permutation(wl.num_blocks)
        kp2 = np.empty_like(kp)
        vp2 = np.empty_like(vp)
        kp2[perm] = kp
        vp2[perm] = vp
        bt2 = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1)
        ds.k_pool.copy_(to_dev(kp2, wl.dtype))
        ds.v_pool.copy_(to_dev(vp2, wl.dtype))
        ds.tables.copy_(torch.from_numpy(bt2.astype(np.int32)))
        b = bits(ds.decode(plan))
    assert np.array_equal(a, b)


def test_contiguous_layout_equals_paged_layout():
    wl = _wl("gqa_small")
    kp, vp = pools_after_append(wl)
    ds = DeviceStep(wl)
    ds.k_pool.copy_(to_dev(kp, wl.dtype))
    ds.v_pool.copy_(to_dev(vp, wl.dtype))
    with pa.Plan() as plan:
        paged = bits(ds.decode(plan).clone())
        # Lay every sequence out contiguously: logical block i of sequence b at
        # physical b * max_blocks + i (an identity-like table).
        MB = wl.max_blocks
        kc = np.full((wl.B * MB,) + kp.shape[1:], 0x7FC0, dtype=kp.dtype)
        vc = np.full_like(kc, 0x7FC0)
        bt = np.full_like(wl.block_tables, -1)
        for b in range(wl.B):
            nb = -(-int(wl.seq_lens[b]) // wl.block_size)
            kc[b * MB:b * MB + nb] = kp[wl.block_tables[b, :nb]]
            vc[b * MB:b * MB + nb] = vp[wl.block_tables[b, :nb]]
            bt[b, :nb] = np.arange(b * MB, b * MB + nb)
        k2, v2 = to_dev(kc, wl.dtype), to_dev(vc, wl.dtype)
        t2 = torch.from_numpy(bt).cuda()
        out2 = torch.empty_like(ds.out)
        pa.pa_decode(ds.q, k2, v2, t2, ds.seq_lens, wl.scale, out2, wl.max_seq_len, plan)
        contiguous = bits(out2)
    assert np.array_equal(paged, contiguous)


# ---------------------------------------------------------------- shapes and edge cases

SHAPES = [
    # (Hq, Hkv, D, bs, lengths)
    (8, 4, 128, 16, [1, 15, 16, 17, 31, 32, 33]),
    (6, 2, 64, 32, [1, 31, 32, 33, 64, 65, 200]),
    (5, 1, 128, 16, [7, 300, 1]),
    (16, 1, 128, 32, [100, 1000]),
    (24, 1, 64, 16, [77, 500]),
    (32, 2, 128, 16, [1, 129, 640]),
    (2, 2, 64, 16, [3, 48, 49]),
    (4, 4, 128, 32, [1, 2, 95, 96, 97]),
]


@pytest.mark.parametrize("path", ["auto", "simple", "fma", "mma"])
@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_edge_shapes(shape, path):
    Hq, Hkv, D, bs, lens = SHAPES[shape]
    wl = _exact(Hq, Hkv, D, bs, lens, seed=600 + shape)
    ref, _, _ = _reference(wl)
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        ds.decode(plan)
        plan.set_path(PATHS[path])
        out = ds.decode(plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    err = np.abs(out_f64(out) - ref).max()
    assert err <= tol(wl), f"max abs error {err:.3e}"


def _exact(Hq, Hkv, D, bs, lens, seed, dtype="bf16"):
    """A workload with exactly the given lengths."""
    return make_workload("llama3_8b_gqa", seed=seed, B=len(lens), Hq=Hq, Hkv=Hkv, D=D,
                         block_size=bs, dtype=dtype, lengths=("list", list(lens)),
                         pool=("factor", 1.3), max_len=int(max(lens)) + bs)


def test_one_long_sequence_spans_many_warps():
    wl = _exact(32, 8, 128, 16, [40000], seed=9)
    ref, _, _ = _reference(wl)
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        out = ds.decode(plan)
        torch.cuda.synchronize()
        _, blocks, warps = plan.info()
    assert warps > 100   # the single sequence is cut across many warps and merged
    assert np.abs(out_f64(out) - ref).max() <= tol(wl)


def test_plan_reuse_across_shapes_and_streams():
    small, big = _wl("gqa_small"), _wl("long_small")
    s = torch.cuda.Stream()
    with pa.Plan() as plan:
        for wl in (small, big, small):
            ref, _, _ = _reference(wl)
            ds = DeviceStep(wl)
            with torch.cuda.stream(s):
                ds.append()
                out = ds.decode(plan)
            s.synchronize()
            assert np.abs(out_f64(out) - ref).max() <= tol(wl)


def test_max_seq_len_larger_than_needed_is_fine():
    wl = _wl("gqa_small")
    ref, _, _ = _reference(wl)
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        out = ds.decode(plan, max_seq_len=wl.max_blocks * wl.block_size)
        torch.cuda.synchronize()
    assert np.abs(out_f64(out) - ref).max() <= tol(wl)


# ---------------------------------------------------------------- device-side error reporting

@pytest.mark.parametrize("path", ["auto", "simple"])
def test_bad_table_entry_sets_error_and_zeroes_rows(path):
    wl = _wl("gqa_small")
    ref, _, _ = _reference(wl)
    ds = DeviceStep(wl)
    ds.append()
    bad_b = int(np.argmax(wl.seq_lens))
    t = ds.tables.clone()
    t[bad_b, 1] = wl.num_blocks + 5       # outside the pool
    ds.tables = t
    with pa.Plan() as plan:
        ds.decode(plan)
        plan.set_path(PATHS[path])
        plan.last_device_error()
        out = ds.decode(plan)
        err = plan.last_device_error()
    assert err & pa.PA_DEVERR_TABLE
    got = out_f64(out)
    assert (got[bad_b] == 0).all()
    keep = [b for b in range(wl.B) if b != bad_b]
    assert np.abs(got[keep] - ref[keep]).max() <= tol(wl)


@pytest.mark.parametrize("path", ["auto", "simple"])
def test_bad_seq_len_sets_error_and_zeroes_rows(path):
    wl = _wl("gqa_small")
    ref, _, _ = _reference(wl)
    ds = DeviceStep(wl)
    ds.append()
    sl = ds.seq_lens.clone()
    sl[0] = 0
    sl[1] = wl.max_seq_len + 1            # beyond the declared bound
    ds.seq_lens = sl
    with pa.Plan() as plan:
        ds.decode(plan)
        plan.set_path(PATHS[path])
        plan.last_device_error()
        out = ds.decode(plan)
        err = plan.last_device_error()
    assert err & pa.PA_DEVERR_SEQ_LEN
    got = out_f64(out)
    assert (got[:2] == 0).all()
    assert np.abs(got[2:] - ref[2:]).max() <= tol(wl)


def test_bad_cache_len_skips_the_append():
    wl = _wl("gqa_small")
    ds = DeviceStep(wl)
    pa.pa_last_device_error(None)
    cl = ds.cache_lens.clone()
    cl[0] = -1
    cl[1] = wl.max_blocks * wl.block_size
    ds.cache_lens = cl
    before_k = bits(ds.k_pool)
    ds.append()
    assert pa.pa_last_device_error(None) & pa.PA_DEVERR_CACHE_LEN
    kp = wl.k_pool.copy()
    vp = wl.v_pool.copy()
    keep = np.arange(2, wl.B)
    oracle.append(wl.k_new[keep], wl.v_new[keep], kp, vp, wl.block_tables[keep],
                  wl.cache_lens[keep])
    assert np.array_equal(bits(ds.k_pool), kp)
    assert not np.array_equal(before_k, kp) or wl.B <= 2


def test_python_binding_raises_on_bad_arguments():
    wl = _wl("gqa_small")
    ds = DeviceStep(wl)
    with pa.Plan() as plan:
        with pytest.raises(pa.PagedAttentionError) as ei:
            pa.pa_decode(ds.q, ds.k_pool, ds.v_pool, ds.tables, ds.seq_lens, wl.scale, ds.out, 0,
                         plan)
        assert ei.value.status == pa.PA_ERR_SHAPE


# ---------------------------------------------------------------- fused merge

@pytest.mark.parametrize("key", ["gqa_small", "mha_small", "long_small", "mixed_small"])
def test_fused_merge_matches_oracle(key):
    # The warp that writes a segment's last partial folds them: no merge
    # kernel. Two calls in a row (the segment counters must come back to
    # zero), with the automatic tail and with a forced tail of one-page
    # pieces (many partials per segment).
    wl = _wl(key)
    ref, _, _ = _reference(wl)
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        ds.decode(plan)
        plan.set_merge(pa.PA_MERGE_FUSED)
        for tail in (None, (150, 1), (0, 1)):
            if tail:
                plan.set_schedule(*tail)
            for _ in range(2):
                out = ds.decode(plan)
                torch.cuda.synchronize()
                assert plan.last_device_error() == 0
                err = np.abs(out_f64(out) - ref).max()
                assert err <= tol(wl), f"{key}/{tail}: max abs error {err:.3e}"


def test_fused_merge_after_other_calls_on_the_same_plan():
    # A workspace whose end held another call's partials: the fused call must
    # clear its counters first. Shapes alternate between a long batch (large
    # workspace) and a short one, with and without the fused merge.
    big, small = _wl("long_small"), _wl("gqa_small")
    refs = {id(w): _reference(w)[0] for w in (big, small)}
    steps = {id(w): DeviceStep(w) for w in (big, small)}
    for ds in steps.values():
        ds.append()
    with pa.Plan() as plan:
        for wl, mode in ((big, pa.PA_MERGE_KERNEL), (small, pa.PA_MERGE_FUSED),
                         (big, pa.PA_MERGE_KERNEL), (big, pa.PA_MERGE_FUSED),
                         (small, pa.PA_MERGE_KERNEL), (small, pa.PA_MERGE_FUSED)):
            ds = steps[id(wl)]
            ds.decode(plan)
            plan.set_merge(mode)
            plan.set_schedule(150, 1)
            out = ds.decode(plan)
            torch.cuda.synchronize()
            assert plan.last_device_error() == 0
            assert np.abs(out_f64(out) - refs[id(wl)]).max() <= tol(wl)


def test_fused_merge_bad_inputs_give_zero_rows():
    wl = _wl("gqa_small")
    ref, _, _ = _reference(wl)
    ds = DeviceStep(wl)
    ds.append()
    bad_b = int(np.argmax(wl.seq_lens))
    t = ds.tables.clone()
    t[bad_b, 1] = wl.num_blocks + 5
    sl = ds.seq_lens.clone()
    sl[0 if bad_b else 1] = 0
    zero_b = 0 if bad_b else 1
    ds.tables, ds.seq_lens = t, sl
    with pa.Plan() as plan:
        ds.decode(plan)
        plan.set_merge(pa.PA_MERGE_FUSED)
        plan.set_schedule(150, 1)
        plan.last_device_error()
        for _ in range(2):
            out = ds.decode(plan)
            err = plan.last_device_error()
            assert err & pa.PA_DEVERR_TABLE and err & pa.PA_DEVERR_SEQ_LEN
            got = out_f64(out)
            assert (got[bad_b] == 0).all() and (got[zero_b] == 0).all()
            keep = [b for b in range(wl.B) if b not in (bad_b, zero_b)]
            assert np.abs(got[keep] - ref[keep]).max() <= tol(wl)


def test_fused_merge_refuses_shapes_it_does_not_serve():
    # 16 query heads per kv head run two n-tiles: no fused merge.
    wl = _exact(32, 2, 128, 16, [100, 300], seed=78)
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        ds.decode(plan)
        plan.set_merge(pa.PA_MERGE_FUSED)
        with pytest.raises(pa.PagedAttentionError) as ei:
            ds.decode(plan)
        assert ei.value.status == pa.PA_ERR_SHAPE
