"""GPU: no kernel writes outside the arrays it is given.

With the sanitizer unavailable, out-of-bounds writes are caught with guard
canaries: every array a call may write (outputs, and the pools for the calls
that write them) is a view carved out of a larger device buffer whose bytes
before and after the view hold a seeded random pattern; after the call every
guard byte must be unchanged. The arrays a call only reads must come back
bit-identical too. Each case also checks the written values against the
oracle, so that a kernel that wrote nothing cannot pass. Shapes are small and
ragged: partial last blocks, one-token sequences, both block sizes, D = 64
and 128, group sizes 1 to 16.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import bf16_bits, make_workload
from oracle_steps import pools_after_append

from gpu_helpers import BF16_TOL, bits, out_f64

pytestmark = pytest.mark.gpu

GUARD = 4096  # guard bytes before and after each view (a multiple of 256: views stay aligned)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


class Guarded:
    """A device tensor view inside a buffer with random guard bytes on both sides."""

    def __init__(self, host: np.ndarray, torch_dtype: torch.dtype, seed: int):
        host = np.ascontiguousarray(host)
        self.nbytes = host.nbytes
        rng = np.random.default_rng(seed)
        self.before = rng.integers(0, 256, GUARD, dtype=np.uint8)
        self.after = rng.integers(0, 256, GUARD, dtype=np.uint8)
        buf = np.concatenate([self.before, host.view(np.uint8).reshape(-1), self.after])
        self.buf = torch.from_numpy(buf).cuda()
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(torch_dtype).view(host.shape)

    def guards_intact(self) -> bool:
        b = self.buf.cpu().numpy()
        return np.array_equal(b[:GUARD], self.before) and \
            np.array_equal(b[GUARD + self.nbytes:], self.after)

    def inner_bytes(self) -> np.ndarray:
        return self.buf[GUARD:GUARD + self.nbytes].cpu().numpy()


def _t_dtype(wl):
    return torch.bfloat16 if wl.dtype == "bf16" else torch.float32


def _host(a, wl):
    return a.view(np.int16) if wl.dtype == "bf16" else a


class GuardedStep:
    """Every array of one append + decode step in guarded buffers."""

    def __init__(self, wl, seed=0):
        dt = _t_dtype(wl)
        self.wl = wl
        self.q = Guarded(_host(wl.q, wl), dt, seed + 1)
        self.k_pool = Guarded(_host(wl.k_pool, wl), dt, seed + 2)
        self.v_pool = Guarded(_host(wl.v_pool, wl), dt, seed + 3)
        self.k_new = Guarded(_host(wl.k_new, wl), dt, seed + 4)
        self.v_new = Guarded(_host(wl.v_new, wl), dt, seed + 5)
        self.tables = Guarded(wl.block_tables, torch.int32, seed + 6)
        self.seq_lens = Guarded(wl.seq_lens, torch.int32, seed + 7)
        self.cache_lens = Guarded(wl.cache_lens, torch.int32, seed + 8)
        nan = np.full((wl.B, wl.Hq, wl.D), np.nan, dtype=np.float32)
        self.out = Guarded(_host(bf16_bits(nan), wl) if wl.dtype == "bf16" else nan, dt, seed + 9)
        self.read_only = [self.q, self.k_new, self.v_new, self.tables, self.seq_lens,
                          self.cache_lens]
        self.snapshot = [g.inner_bytes() for g in self.read_only]

    def all_guards_intact(self):
        return all(g.guards_intact() for g in (*self.read_only, self.k_pool, self.v_pool,
                                               self.out))

    def inputs_unchanged(self):
        return all(np.array_equal(g.inner_bytes(), s) for g, s in zip(self.read_only,
                                                                       self.snapshot))


SHAPES = [  # (name, overrides)
    ("llama3_8b_gqa", dict(B=5, lengths=("list", [1, 15, 17, 33, 700]), max_len=704)),
    ("llama7b_mha", dict(B=4, Hq=8, Hkv=8, lengths=("list", [2, 16, 31, 200]), max_len=208,
                         pool=("fixed", 64))),
    ("long_splitk", dict(B=2, lengths=("list", [31, 1000]), max_len=1024)),
    ("llama3_8b_gqa", dict(B=3, Hq=16, Hkv=1, D=64, lengths=("list", [5, 64, 65]), max_len=80)),
    ("llama3_405b_gqa", dict(B=3, lengths=("list", [47, 300, 1]), max_len=320)),
    ("tiny_worked_60", dict()),
]


@pytest.mark.parametrize("case", range(len(SHAPES)))
def test_append_and_decode_write_only_their_arrays(case):
    name, extra = SHAPES[case]
    wl = make_workload(name, seed=900 + case, **extra)
    gs = GuardedStep(wl, seed=case * 10)
    pa.pa_append_kv(gs.k_new.t, gs.v_new.t, gs.k_pool.t, gs.v_pool.t, gs.tables.t,
                    gs.cache_lens.t)
    with pa.Plan() as plan:
        pa.pa_decode(gs.q.t, gs.k_pool.t, gs.v_pool.t, gs.tables.t, gs.seq_lens.t, wl.scale,
                     gs.out.t, wl.max_seq_len, plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert pa.pa_last_device_error(None) == 0
    assert gs.all_guards_intact()
    assert gs.inputs_unchanged()
    kp, vp = pools_after_append(wl)
    assert np.array_equal(bits(gs.k_pool.t), kp.view(bits(gs.k_pool.t).dtype))
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    tol = BF16_TOL if wl.dtype == "bf16" else 2e-3
    assert np.abs(out_f64(gs.out.t) - ref).max() <= tol


@pytest.mark.parametrize("case", range(len(SHAPES)))
def test_fused_append_decode_writes_only_its_arrays(case):
    # The fused call writes the pools (one slot per sequence and kv head) and
    # the output; every guard byte and every input must survive.
    name, extra = SHAPES[case]
    wl = make_workload(name, seed=900 + case, **extra)
    gs = GuardedStep(wl, seed=case * 10 + 5)
    with pa.Plan() as plan:
        pa.pa_append_decode(gs.q.t, gs.k_new.t, gs.v_new.t, gs.k_pool.t, gs.v_pool.t,
                            gs.tables.t, gs.seq_lens.t, wl.scale, gs.out.t, wl.max_seq_len, plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert pa.pa_last_device_error(None) == 0
    assert gs.all_guards_intact()
    assert gs.inputs_unchanged()
    kp, vp = pools_after_append(wl)
    assert np.array_equal(bits(gs.k_pool.t), kp.view(bits(gs.k_pool.t).dtype))
    assert np.array_equal(bits(gs.v_pool.t), vp.view(bits(gs.v_pool.t).dtype))
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    tol = BF16_TOL if wl.dtype == "bf16" else 2e-3
    assert np.abs(out_f64(gs.out.t) - ref).max() <= tol


@pytest.mark.parametrize("case", [0, 1, 2])
def test_noalloc_decode_writes_only_its_output(case):
    name, extra = SHAPES[case]
    wl = make_workload(name, seed=950 + case, **extra)
    kp, vp = pools_after_append(wl)
    wl.k_pool, wl.v_pool = kp, vp
    gs = GuardedStep(wl, seed=case * 10 + 5)
    pools = [gs.k_pool.inner_bytes(), gs.v_pool.inner_bytes()]
    err = Guarded(np.zeros(1, dtype=np.int32), torch.int32, 77)
    pa.pa_decode_noalloc(gs.q.t, gs.k_pool.t, gs.v_pool.t, gs.tables.t, gs.seq_lens.t, wl.scale,
                         gs.out.t, wl.max_seq_len, device_error=err.t)
    torch.cuda.synchronize()
    assert int(err.t.item()) == 0 and err.guards_intact()
    assert gs.all_guards_intact() and gs.inputs_unchanged()
    assert np.array_equal(gs.k_pool.inner_bytes(), pools[0])
    assert np.array_equal(gs.v_pool.inner_bytes(), pools[1])
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    assert np.abs(out_f64(gs.out.t) - ref).max() <= BF16_TOL


@pytest.mark.parametrize("multi", [False, True], ids=["prefill", "decode_multi"])
@pytest.mark.parametrize("Hq,Hkv,bs,lens,ns", [
    (32, 8, 16, [40, 300, 7], [3, 4, 1]),
    (16, 16, 32, [1, 90, 33], [1, 1, 1]),
    (16, 1, 16, [130, 17], [1, 1]),
])
def test_multi_query_calls_write_only_their_output(multi, Hq, Hkv, bs, lens, ns):
    _multi_query_guarded(multi, Hq, Hkv, bs, lens, ns)


# Both tensor-core prefill kernels, pinned through the test hook: whole query
# tiles (the output leaves by tiled bulk tensor stores) and ragged tiles.
@pytest.mark.parametrize("kernel", [1, 2], ids=["one_tile", "two_tile"])
@pytest.mark.parametrize("lens,ns", [
    ([700, 2000], [64, 128]),      # whole tiles of 32 queries x 4 heads
    ([900, 1500, 260], [40, 77, 5]),   # ragged tiles
    ([6000], [32]),                # one whole tile over a long key range
])
def test_tensor_core_prefill_writes_only_its_output(kernel, lens, ns):
    which = {1: pa.PA_PREFILL_ONE_TILE, 2: pa.PA_PREFILL_TWO_TILE}[kernel]
    pa.pa_debug_set_prefill_kernel(which)
    try:
        _multi_query_guarded(False, 32, 8, 16, lens, ns)
    finally:
        pa.pa_debug_set_prefill_kernel(pa.PA_PREFILL_AUTO)


@pytest.mark.parametrize("lens,ns", [([12000], [8]), ([5000, 300], [12, 9])])
def test_split_verification_writes_only_its_output(lens, ns):
    # More than 16 (query, head) columns per kv head on a small batch: the
    # key split's partials go to the plan's workspace and a merge kernel
    # writes the output.
    _multi_query_guarded(True, 32, 8, 16, lens, ns)


def _multi_query_guarded(multi, Hq, Hkv, bs, lens, ns):
    wl = make_workload("llama3_8b_gqa", seed=sum(lens), B=len(lens), Hq=Hq, Hkv=Hkv,
                       block_size=bs, lengths=("list", lens), max_len=max(lens) + bs)
    kp, vp = pools_after_append(wl)
    wl.k_pool, wl.v_pool = kp, vp
    rng = np.random.default_rng(len(lens))
    T = int(sum(ns))
    qh = bf16_bits(rng.standard_normal((T, Hq, wl.D)).astype(np.float32))
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    wl.q = qh
    gs = GuardedStep(wl, seed=3)
    out = Guarded(bf16_bits(np.full((T, Hq, wl.D), np.nan, dtype=np.float32)).view(np.int16),
                  torch.bfloat16, 31)
    q_start = Guarded(qs, torch.int32, 32)
    pools = [gs.k_pool.inner_bytes(), gs.v_pool.inner_bytes()]
    if multi:
        with pa.Plan() as plan:
            pa.pa_decode_multi(gs.q.t, q_start.t, gs.k_pool.t, gs.v_pool.t, gs.tables.t,
                               gs.seq_lens.t, wl.scale, out.t, max(ns), wl.max_seq_len, plan)
            torch.cuda.synchronize()
            assert plan.last_device_error() == 0
    else:
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pa.pa_prefill(gs.q.t, q_start.t, gs.k_pool.t, gs.v_pool.t, gs.tables.t, gs.seq_lens.t,
                      wl.scale, out.t, max(ns), wl.max_seq_len, device_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
    assert out.guards_intact() and q_start.guards_intact()
    assert gs.all_guards_intact() and gs.inputs_unchanged()
    assert np.array_equal(gs.k_pool.inner_bytes(), pools[0])
    assert np.array_equal(gs.v_pool.inner_bytes(), pools[1])
    ref = oracle.prefill(qh, kp, vp, wl.block_tables, wl.seq_lens, qs, wl.scale)
    assert np.abs(out_f64(out.t) - ref).max() <= BF16_TOL


@pytest.mark.parametrize("name,extra", [
    ("llama3_8b_gqa", dict(B=6, lengths=("list", [16, 17, 1, 64, 300, 48]), max_len=320)),
    ("long_splitk", dict(B=2, lengths=("list", [64, 95]), max_len=96)),
])
def test_page_scores_write_only_their_outputs(name, extra):
    wl = make_workload(name, seed=71, **extra)
    kp, vp = pools_after_append(wl)
    wl.k_pool, wl.v_pool = kp, vp
    gs = GuardedStep(wl, seed=40)
    B, MB = wl.block_tables.shape
    scores = Guarded(np.full((B, MB), -7.0, dtype=np.float32), torch.float32, 41)
    victims = Guarded(np.full(B, -9, dtype=np.int32), torch.int32, 42)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_page_scores(gs.k_pool.t, gs.v_pool.t, gs.tables.t, gs.seq_lens.t, wl.max_seq_len,
                      scores.t, victims.t, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert scores.guards_intact() and victims.guards_intact()
    assert gs.all_guards_intact() and gs.inputs_unchanged()
    ref_s, ref_v = oracle.page_scores(kp, vp, wl.block_tables, wl.seq_lens)
    got = scores.t.cpu().numpy().astype(np.float64)
    for b in range(B):
        nb = -(-int(wl.seq_lens[b]) // wl.block_size)
        np.testing.assert_allclose(got[b, :nb], ref_s[b, :nb], rtol=1e-4)
        assert (got[b, nb:] == -7.0).all()


def test_block_copies_write_only_their_destinations():
    wl = make_workload("llama3_8b_gqa", seed=72, B=4, lengths=("uniform", 1, 300), max_len=320)
    gs = GuardedStep(wl, seed=50)
    rng = np.random.default_rng(6)
    perm = rng.permutation(wl.num_blocks)
    n = min(20, wl.num_blocks // 2)
    src_h, dst_h = perm[:n].astype(np.int32), perm[n:2 * n].astype(np.int32)
    src, dst = Guarded(src_h, torch.int32, 51), Guarded(dst_h, torch.int32, 52)
    pa.pa_copy_blocks(gs.k_pool.t, gs.v_pool.t, src.t, dst.t)
    torch.cuda.synchronize()
    assert pa.pa_last_device_error(None) == 0
    assert src.guards_intact() and dst.guards_intact()
    assert gs.all_guards_intact()
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.copy_blocks(kp, vp, src_h, dst_h)
    assert np.array_equal(bits(gs.k_pool.t), kp)
    assert np.array_equal(bits(gs.v_pool.t), vp)
