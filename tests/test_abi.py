"""The C-ABI library builds for sm_103a, loads, exports every declared symbol,
and rejects bad arguments on the host before touching a GPU (no GPU needed)."""

import ctypes

import numpy as np
import pytest

import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pa.lib()


def test_exports_every_declared_function(lib):
    names = pa.declared_functions()
    assert {"pa_append_kv", "pa_decode", "pa_free", "pa_status_str",
            "pa_last_device_error"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libpa.so does not export {n}"


def test_status_strings(lib):
    for s in range(0, 9):
        assert pa.pa_status_str(s) and pa.pa_status_str(s) != "unknown status"
    assert pa.pa_status_str(99) == "unknown status"


ALIGNED = 0x10000  # a fake, 16-byte aligned device address: never dereferenced


def _decode(lib, **kw):
    args = dict(q=ALIGNED, k=ALIGNED, v=ALIGNED, bt=ALIGNED, mb=4, sl=ALIGNED, B=2, Hq=8, Hkv=2,
                D=128, bs=16, NB=64, maxlen=64, scale=0.1, kvdt=pa.PA_BF16, out=ALIGNED,
                odt=pa.PA_BF16, plan=True)
    args.update(kw)
    plan = ctypes.c_void_p(None)
    pp = ctypes.byref(plan) if args["plan"] else None
    st = lib.pa_decode(args["q"], args["k"], args["v"], args["bt"], args["mb"], args["sl"],
                       args["B"], args["Hq"], args["Hkv"], args["D"], args["bs"], args["NB"],
                       args["maxlen"], args["scale"], args["kvdt"], args["out"], args["odt"], pp,
                       None)
    assert plan.value is None, "an argument error must not create a plan"
    return st


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), pa.PA_ERR_NULL),
    (dict(k=None), pa.PA_ERR_NULL),
    (dict(bt=None), pa.PA_ERR_NULL),
    (dict(sl=None), pa.PA_ERR_NULL),
    (dict(out=None), pa.PA_ERR_NULL),
    (dict(plan=False), pa.PA_ERR_NULL),
    (dict(kvdt=7), pa.PA_ERR_DTYPE),
    (dict(odt=-1), pa.PA_ERR_DTYPE),
    (dict(bs=8), pa.PA_ERR_BLOCK_SIZE),
    (dict(bs=64), pa.PA_ERR_BLOCK_SIZE),
    (dict(D=96), pa.PA_ERR_SHAPE),
    (dict(Hq=6, Hkv=4), pa.PA_ERR_SHAPE),
    (dict(Hkv=0), pa.PA_ERR_SHAPE),
    (dict(B=-1), pa.PA_ERR_SHAPE),
    (dict(NB=0), pa.PA_ERR_SHAPE),
    (dict(mb=0), pa.PA_ERR_SHAPE),
    (dict(maxlen=0), pa.PA_ERR_SHAPE),
    (dict(scale=float("nan")), pa.PA_ERR_SHAPE),
    (dict(B=100000), pa.PA_ERR_SHAPE),
    (dict(B=8192, Hq=131080, Hkv=8), pa.PA_ERR_SHAPE),   # more than 2^30 output rows
    (dict(q=ALIGNED + 8), pa.PA_ERR_ALIGN),
    (dict(out=ALIGNED + 2), pa.PA_ERR_ALIGN),
    (dict(v=ALIGNED + 4), pa.PA_ERR_ALIGN),
    # float32 pools run on the unsplit kernel, bounded in length
    (dict(kvdt=pa.PA_F32, odt=pa.PA_F32, maxlen=pa.PA_SIMPLE_MAX_SEQ_LEN + 1, mb=1024),
     pa.PA_ERR_SHAPE),
    (dict(kvdt=pa.PA_F32, odt=pa.PA_F32, maxlen=131072, mb=8192), pa.PA_ERR_SHAPE),
])
def test_decode_rejects_bad_arguments_on_host(lib, kw, status):
    assert _decode(lib, **kw) == status


def test_decode_late_shape_errors_create_no_plan(lib):
    # Rejected from the sizes alone, before any CUDA call: the page count
    # over all (sequence, kv head) units overflows 32 bits.
    assert _decode(lib, B=8192, Hq=64, Hkv=64, mb=65536, maxlen=1 << 20) == pa.PA_ERR_SHAPE


def _append_decode(lib, **kw):
    args = dict(q=ALIGNED, kn=ALIGNED, vn=ALIGNED, k=ALIGNED, v=ALIGNED, bt=ALIGNED, mb=4,
                sl=ALIGNED, B=2, Hq=8, Hkv=2, D=128, bs=16, NB=64, maxlen=64, scale=0.1,
                kvdt=pa.PA_BF16, out=ALIGNED, odt=pa.PA_BF16)
    args.update(kw)
    plan = ctypes.c_void_p(None)
    st = lib.pa_append_decode(args["q"], args["kn"], args["vn"], args["k"], args["v"], args["bt"],
                              args["mb"], args["sl"], args["B"], args["Hq"], args["Hkv"],
                              args["D"], args["bs"], args["NB"], args["maxlen"], args["scale"],
                              args["kvdt"], args["out"], args["odt"], ctypes.byref(plan), None)
    assert plan.value is None, "an argument error must not create a plan"
    return st


@pytest.mark.parametrize("kw,status", [
    (dict(kn=None), pa.PA_ERR_NULL),
    (dict(vn=None), pa.PA_ERR_NULL),
    (dict(q=None), pa.PA_ERR_NULL),
    (dict(kn=ALIGNED + 8), pa.PA_ERR_ALIGN),
    (dict(vn=ALIGNED + 4), pa.PA_ERR_ALIGN),
    (dict(D=96), pa.PA_ERR_SHAPE),
    (dict(bs=8), pa.PA_ERR_BLOCK_SIZE),
    (dict(kvdt=7), pa.PA_ERR_DTYPE),
    (dict(kvdt=pa.PA_F32, odt=pa.PA_F32, maxlen=pa.PA_SIMPLE_MAX_SEQ_LEN + 1, mb=1024),
     pa.PA_ERR_SHAPE),
])
def test_append_decode_rejects_bad_arguments_on_host(lib, kw, status):
    # Every argument error returns before anything launches: the append is
    # never run ahead of a decode that would be refused.
    assert _append_decode(lib, **kw) == status


def test_append_decode_empty_batch_is_a_no_op(lib):
    assert _append_decode(lib, B=0) == pa.PA_OK


def test_library_reads_no_environment_variables(lib):
    # Launch shapes come from the arguments and explicit plan setters only:
    # the library's code names no environment variable.
    import glob
    import os
    for src in glob.glob(os.path.join(os.path.dirname(pa.__file__), "csrc", "*")):
        with open(src) as f:
            assert "getenv" not in f.read(), src


def test_decode_empty_batch_is_a_no_op(lib):
    assert _decode(lib, B=0) == pa.PA_OK


def _decode_multi(lib, **kw):
    args = dict(q=ALIGNED, qs=ALIGNED, T=8, maxq=4, k=ALIGNED, v=ALIGNED, bt=ALIGNED, mb=4,
                sl=ALIGNED, B=2, Hq=8, Hkv=2, D=128, bs=16, NB=64, maxlen=64, scale=0.1,
                kvdt=pa.PA_BF16, out=ALIGNED, odt=pa.PA_BF16)
    args.update(kw)
    plan = ctypes.c_void_p(None)
    st = lib.pa_decode_multi(args["q"], args["qs"], args["T"], args["maxq"], args["k"], args["v"],
                             args["bt"], args["mb"], args["sl"], args["B"], args["Hq"], args["Hkv"],
                             args["D"], args["bs"], args["NB"], args["maxlen"], args["scale"],
                             args["kvdt"], args["out"], args["odt"], ctypes.byref(plan), None)
    assert plan.value is None, "an argument error must not create a plan"
    return st


@pytest.mark.parametrize("kw,status", [
    (dict(qs=None), pa.PA_ERR_NULL),
    (dict(q=None), pa.PA_ERR_NULL),
    (dict(kvdt=pa.PA_F32), pa.PA_ERR_DTYPE),       # tensor-core tiles take bf16 pools
    # More than 16 (query, head) columns run on the prefill kernel's 128-row
    # tiles, which need D = 128 and a group size dividing 128.
    (dict(maxq=5, D=64), pa.PA_ERR_SHAPE),
    (dict(maxq=6, Hq=24, Hkv=8), pa.PA_ERR_SHAPE),     # 18 columns, g = 3
    (dict(maxq=5, mb=16385), pa.PA_ERR_SHAPE),
    (dict(maxq=20, Hq=70000, Hkv=70000), pa.PA_ERR_SHAPE),   # kv heads past the grid limit
    (dict(T=1 << 25, Hq=64, Hkv=8), pa.PA_ERR_SHAPE),        # more than 2^30 output rows
    (dict(maxq=0), pa.PA_ERR_SHAPE),
    (dict(T=-1), pa.PA_ERR_SHAPE),
    (dict(q=ALIGNED + 8), pa.PA_ERR_ALIGN),
])
def test_decode_multi_rejects_bad_arguments_on_host(lib, kw, status):
    assert _decode_multi(lib, **kw) == status


def test_decode_multi_without_queries_is_a_no_op(lib):
    assert _decode_multi(lib, T=0) == pa.PA_OK
    assert _decode_multi(lib, B=0) == pa.PA_OK


def _append(lib, **kw):
    args = dict(kn=ALIGNED, vn=ALIGNED, k=ALIGNED, v=ALIGNED, bt=ALIGNED, mb=4, cl=ALIGNED, B=2,
                Hkv=2, D=128, bs=16, NB=64, dt=pa.PA_BF16)
    args.update(kw)
    return lib.pa_append_kv(args["kn"], args["vn"], args["k"], args["v"], args["bt"], args["mb"],
                            args["cl"], args["B"], args["Hkv"], args["D"], args["bs"], args["NB"],
                            args["dt"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(kn=None), pa.PA_ERR_NULL),
    (dict(cl=None), pa.PA_ERR_NULL),
    (dict(dt=3), pa.PA_ERR_DTYPE),
    (dict(bs=48), pa.PA_ERR_BLOCK_SIZE),
    (dict(D=32), pa.PA_ERR_SHAPE),
    (dict(Hkv=0), pa.PA_ERR_SHAPE),
    (dict(NB=0), pa.PA_ERR_SHAPE),
    (dict(k=ALIGNED + 2), pa.PA_ERR_ALIGN),
])
def test_append_rejects_bad_arguments_on_host(lib, kw, status):
    assert _append(lib, **kw) == status


def test_append_empty_batch_is_a_no_op(lib):
    assert _append(lib, B=0) == pa.PA_OK


def test_plan_calls_reject_null(lib):
    assert lib.pa_free(None) == pa.PA_OK
    assert lib.pa_plan_set_path(None, 0) == pa.PA_ERR_NULL
    assert lib.pa_plan_info(None, None, None, None) == pa.PA_ERR_NULL
    assert lib.pa_plan_set_split_events(None, None, None) == pa.PA_ERR_NULL
    assert lib.pa_plan_set_schedule(None, 150, 16) == pa.PA_ERR_NULL
    assert lib.pa_plan_set_merge(None, pa.PA_MERGE_FUSED) == pa.PA_ERR_NULL


def test_wait_probe_switch_is_host_only(lib):
    # Switching the test hook touches no device; it is read at launch time.
    assert lib.pa_debug_set_wait_probe(1) == pa.PA_OK
    assert lib.pa_debug_set_wait_probe(0) == pa.PA_OK
    assert lib.pa_last_device_error(None, None) == pa.PA_ERR_NULL


def test_prefill_kernel_pin_is_host_only_and_checked(lib):
    # The prefill-kernel pin is a host setting read at launch time; values
    # other than the three named ones are refused and leave it unchanged.
    for which in (pa.PA_PREFILL_ONE_TILE, pa.PA_PREFILL_TWO_TILE, pa.PA_PREFILL_AUTO):
        assert lib.pa_debug_set_prefill_kernel(which) == pa.PA_OK
    for bad in (-1, 3, 1 << 20):
        assert lib.pa_debug_set_prefill_kernel(bad) == pa.PA_ERR_SHAPE
    with pytest.raises(RuntimeError):
        pa.pa_debug_set_prefill_kernel(7)
    assert lib.pa_debug_set_prefill_kernel(pa.PA_PREFILL_AUTO) == pa.PA_OK


def test_binding_byte_counter_matches_oracle():
    import numpy as np
    import oracle
    rng = np.random.default_rng(0)
    for bs in (16, 32):
        lens = rng.integers(1, 5000, size=17)
        for Hq, Hkv, D, e, eo in ((32, 8, 128, 2, 2), (4, 4, 64, 4, 4), (64, 8, 128, 2, 4)):
            assert pa.decode_bytes(lens, Hq, Hkv, D, bs, e, eo) == \
                oracle.decode_bytes(lens, Hq, Hkv, D, bs, e, eo)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(pa, "_lib", None)
    monkeypatch.setattr(pa, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        pa.lib()


def _host_tensors(B=2, Hq=8, Hkv=2, D=128, bs=16, NB=16, MB=4):
    import torch
    bf = torch.bfloat16
    return dict(q=torch.zeros(B, Hq, D, dtype=bf), k=torch.zeros(NB, Hkv, bs, D, dtype=bf),
                v=torch.zeros(NB, Hkv, bs, D, dtype=bf),
                bt=torch.zeros(B, MB, dtype=torch.int32), sl=torch.ones(B, dtype=torch.int32),
                qs=torch.arange(B + 1, dtype=torch.int32), out=torch.zeros(B, Hq, D, dtype=bf),
                kn=torch.zeros(B, Hkv, D, dtype=bf), sc=torch.zeros(B, MB),
                vic=torch.zeros(B, dtype=torch.int32))


def test_binding_rejects_host_tensors():
    # A host pointer must never reach a kernel: every entry point refuses
    # tensors that are not CUDA memory before it calls the library.
    t = _host_tensors()
    plan = pa.Plan()
    calls = [
        lambda: pa.pa_decode(t["q"], t["k"], t["v"], t["bt"], t["sl"], 0.1, t["out"], 64, plan),
        lambda: pa.pa_decode_multi(t["q"], t["qs"], t["k"], t["v"], t["bt"], t["sl"], 0.1,
                                   t["out"], 1, 64, plan),
        lambda: pa.pa_decode_noalloc(t["q"], t["k"], t["v"], t["bt"], t["sl"], 0.1, t["out"], 64),
        lambda: pa.pa_append_kv(t["kn"], t["kn"], t["k"], t["v"], t["bt"], t["sl"]),
        lambda: pa.pa_prefill(t["q"], t["qs"], t["k"], t["v"], t["bt"], t["sl"], 0.1, t["out"],
                              1, 64),
        lambda: pa.pa_page_scores(t["k"], t["v"], t["bt"], t["sl"], 64, t["sc"], t["vic"]),
        lambda: pa.pa_copy_blocks(t["k"], t["v"], t["vic"], t["vic"]),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA device"):
            call()
    assert plan.handle.value is None


# Host-side argument errors of the other entry points: a status before any
# CUDA call, so these run without a GPU.

def _prefill(lib, **kw):
    args = dict(q=ALIGNED, qs=ALIGNED, T=8, k=ALIGNED, v=ALIGNED, bt=ALIGNED, mb=4, sl=ALIGNED,
                B=2, Hq=8, Hkv=2, D=128, bs=16, NB=64, maxq=4, maxlen=64, scale=0.1,
                kvdt=pa.PA_BF16, out=ALIGNED, odt=pa.PA_BF16)
    args.update(kw)
    return lib.pa_prefill(args["q"], args["qs"], args["T"], args["k"], args["v"], args["bt"],
                          args["mb"], args["sl"], args["B"], args["Hq"], args["Hkv"], args["D"],
                          args["bs"],
                          args["NB"], args["maxq"], args["maxlen"], args["scale"], args["kvdt"],
                          args["out"], args["odt"], None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(qs=None), pa.PA_ERR_NULL),
    (dict(out=None), pa.PA_ERR_NULL),
    (dict(kvdt=pa.PA_F32), pa.PA_ERR_DTYPE),      # tensor-core tiles take bf16 pools
    (dict(bs=8), pa.PA_ERR_BLOCK_SIZE),
    (dict(D=64), pa.PA_ERR_SHAPE),                # the tcgen05 tiles are built for D = 128
    (dict(Hq=24, Hkv=8), pa.PA_ERR_SHAPE),        # g = 3 does not divide the 128-row tile
    (dict(maxq=0), pa.PA_ERR_SHAPE),
    (dict(T=-1), pa.PA_ERR_SHAPE),
    (dict(scale=float("inf")), pa.PA_ERR_SHAPE),
    (dict(B=70000), pa.PA_ERR_SHAPE),             # sequences past the grid limit
    (dict(Hq=70000, Hkv=70000), pa.PA_ERR_SHAPE), # kv heads past the grid limit
    (dict(k=ALIGNED + 4), pa.PA_ERR_ALIGN),
])
def test_prefill_rejects_bad_arguments_on_host(lib, kw, status):
    assert _prefill(lib, **kw) == status


def test_prefill_empty_batch_is_a_no_op(lib):
    assert _prefill(lib, B=0) == pa.PA_OK
    assert _prefill(lib, T=0) == pa.PA_OK


def _scores(lib, **kw):
    args = dict(k=ALIGNED, v=ALIGNED, bt=ALIGNED, mb=4, sl=ALIGNED, B=2, Hkv=2, D=128, bs=16,
                NB=64, maxlen=64, dt=pa.PA_BF16, sc=ALIGNED, vic=ALIGNED)
    args.update(kw)
    return lib.pa_page_scores(args["k"], args["v"], args["bt"], args["mb"], args["sl"], args["B"],
                              args["Hkv"], args["D"], args["bs"], args["NB"], args["maxlen"],
                              args["dt"], args["sc"], args["vic"], None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(vic=None), pa.PA_ERR_NULL),
    (dict(sc=None), pa.PA_ERR_NULL),
    (dict(dt=5), pa.PA_ERR_DTYPE),
    (dict(bs=64), pa.PA_ERR_BLOCK_SIZE),
    (dict(D=96), pa.PA_ERR_SHAPE),
    (dict(B=9000), pa.PA_ERR_SHAPE),
    (dict(v=ALIGNED + 8), pa.PA_ERR_ALIGN),
])
def test_page_scores_reject_bad_arguments_on_host(lib, kw, status):
    assert _scores(lib, **kw) == status


def test_page_scores_empty_batch_is_a_no_op(lib):
    assert _scores(lib, B=0) == pa.PA_OK


def _copies(lib, **kw):
    args = dict(k=ALIGNED, v=ALIGNED, src=ALIGNED, dst=ALIGNED, n=3, Hkv=2, D=128, bs=16, NB=64,
                dt=pa.PA_BF16)
    args.update(kw)
    return lib.pa_copy_blocks(args["k"], args["v"], args["src"], args["dst"], args["n"],
                              args["Hkv"], args["D"], args["bs"], args["NB"], args["dt"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(src=None), pa.PA_ERR_NULL),
    (dict(k=None), pa.PA_ERR_NULL),
    (dict(dt=2), pa.PA_ERR_DTYPE),
    (dict(bs=24), pa.PA_ERR_BLOCK_SIZE),
    (dict(n=-1), pa.PA_ERR_SHAPE),
    (dict(NB=0), pa.PA_ERR_SHAPE),
    (dict(v=ALIGNED + 2), pa.PA_ERR_ALIGN),
])
def test_copy_blocks_reject_bad_arguments_on_host(lib, kw, status):
    assert _copies(lib, **kw) == status


def test_copy_blocks_without_pairs_is_a_no_op(lib):
    assert _copies(lib, n=0, src=None, dst=None) == pa.PA_OK


def _noalloc(lib, **kw):
    args = dict(q=ALIGNED, k=ALIGNED, v=ALIGNED, bt=ALIGNED, mb=4, sl=ALIGNED, B=2, Hq=8, Hkv=2,
                D=128, bs=16, NB=64, maxlen=64, scale=0.1, kvdt=pa.PA_BF16, out=ALIGNED,
                odt=pa.PA_BF16)
    args.update(kw)
    return lib.pa_decode_noalloc(args["q"], args["k"], args["v"], args["bt"], args["mb"],
                                 args["sl"], args["B"], args["Hq"], args["Hkv"], args["D"],
                                 args["bs"], args["NB"], args["maxlen"], args["scale"],
                                 args["kvdt"], args["out"], args["odt"], None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), pa.PA_ERR_NULL),
    (dict(kvdt=pa.PA_F32), pa.PA_ERR_DTYPE),      # the split kernels take bf16 pools
    (dict(bs=8), pa.PA_ERR_BLOCK_SIZE),
    (dict(Hq=6, Hkv=4), pa.PA_ERR_SHAPE),
    (dict(B=8193), pa.PA_ERR_SHAPE),
    (dict(B=8192, Hq=64, Hkv=64, mb=65536, maxlen=1 << 20), pa.PA_ERR_SHAPE),  # pages over 32 bits
    (dict(B=8192, Hq=131080, Hkv=8), pa.PA_ERR_SHAPE),   # more than 2^30 output rows
    (dict(out=ALIGNED + 2), pa.PA_ERR_ALIGN),
])
def test_noalloc_rejects_bad_arguments_on_host(lib, kw, status):
    assert _noalloc(lib, **kw) == status


def test_noalloc_empty_batch_is_a_no_op(lib):
    assert _noalloc(lib, B=0) == pa.PA_OK


@pytest.mark.parametrize("name", ["llama7b_mha", "llama3_8b_gqa", "mixed_shared", "spec_gqa",
                                  "llama3_405b_gqa", "prefill_gqa"])
def test_workload_lengths_are_the_lengths_make_workload_draws(name):
    # The read-ceiling row sizes its buffer from these lengths without the pools.
    from paged_kv_cache_202_gb300.workloads import make_workload, workload_lengths
    wl = make_workload(name, B=6, max_len=4096, lengths=("uniform", 100, 4000))
    np.testing.assert_array_equal(
        workload_lengths(name, B=6, max_len=4096, lengths=("uniform", 100, 4000)), wl.seq_lens)
    wl = make_workload(name, seed=5, B=3, max_len=2048, lengths=("loguniform", 20, 2000))
    np.testing.assert_array_equal(
        workload_lengths(name, seed=5, B=3, max_len=2048, lengths=("loguniform", 20, 2000)),
        wl.seq_lens)
