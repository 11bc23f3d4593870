"""GPU: decodes whose merge takes 8, 16 or 32 warps per row, against the oracle.

The plan gives the merge kernel more warps per output row the more partials
a kv unit has (one or a few long sequences split over many warps). These
shapes put ~25, ~100 and ~300 partials on each kv unit, for both head
dimensions, so that every merge width folds real partials; the output must
match the fp64 oracle within the bf16 tolerance, and a second call on the
same plan must give the same bits.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import make_workload
from oracle_steps import pools_after_append

from gpu_helpers import DeviceStep, bits, out_f64, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


# (head dim, one sequence's length): ~25, ~100 and ~300 partials per kv unit
# with 8 query heads over 2 kv heads at block size 16.
SHAPES = [(D, L) for D in (64, 128) for L in (1600, 6400, 20000)]


@pytest.mark.parametrize("D,L", SHAPES)
def test_long_single_sequence_matches_oracle(D, L):
    wl = make_workload("llama3_8b_gqa", seed=31, B=1, Hq=8, Hkv=2, D=D,
                       lengths=("fixed", L), max_len=L, pool=("factor", 1.0))
    kp, vp = pools_after_append(wl)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        out = ds.decode(plan)
        torch.cuda.synchronize()
        first = bits(out).copy()
        out2 = ds.decode(plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    got = out_f64(out2)
    assert np.isfinite(got).all()
    e = np.abs(got - ref).max()
    assert e <= tol(wl), f"max abs error {e:.3e}"
    assert np.array_equal(bits(out2), first)


def test_two_long_sequences_of_different_lengths_match_oracle():
    # Rows of two segments whose partial counts differ by a factor of three.
    wl = make_workload("llama3_8b_gqa", seed=32, B=2, Hq=8, Hkv=2,
                       lengths=("list", [15000, 5000]), max_len=15008, pool=("factor", 1.0))
    kp, vp = pools_after_append(wl)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    ds = DeviceStep(wl)
    ds.append()
    with pa.Plan() as plan:
        out = ds.decode(plan)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    e = np.abs(out_f64(out) - ref).max()
    assert e <= tol(wl), f"max abs error {e:.3e}"
