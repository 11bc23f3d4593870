"""GPU: PagedEviction page scores against the oracle.

Scores are fp32 on the GPU and fp64 in the oracle: compared within a relative
1e-4. The victim is an argmin over those scores: where the oracle says -1 the
GPU must too; otherwise the GPU's page must be a valid minimum of the oracle's
scores (within the same tolerance), since near-ties may fall either way.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300.workloads import make_workload
from oracle_steps import append_in_place

from gpu_helpers import DeviceStep

pytestmark = pytest.mark.gpu
RTOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run(ds, wl, tables=None):
    B, MB = wl.block_tables.shape
    scores = torch.full((B, MB), -7.0, dtype=torch.float32, device="cuda")
    victims = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_page_scores(ds.k_pool, ds.v_pool, ds.tables if tables is None else tables, ds.seq_lens,
                      wl.max_seq_len, scores, victims, err)
    torch.cuda.synchronize()
    return scores.cpu().numpy().astype(np.float64), victims.cpu().numpy(), int(err.item())


def _check(wl, got_s, got_v, ref_s, ref_v):
    for b in range(wl.B):
        nb = -(-int(wl.seq_lens[b]) // wl.block_size)
        np.testing.assert_allclose(got_s[b, :nb], ref_s[b, :nb], rtol=RTOL)
        assert (got_s[b, nb:] == -7.0).all(), "entries past the sequence must stay untouched"
        if ref_v[b] < 0:
            assert got_v[b] == -1
        else:
            assert 0 <= got_v[b] < nb
            assert ref_s[b, got_v[b]] <= ref_s[b, :nb].min() * (1 + 2 * RTOL)


CASES = [
    ("llama3_8b_gqa", dict(B=12, lengths=("list", [16, 32, 48, 64, 17, 1, 160, 320, 335, 512,
                                                    1024, 999]), max_len=1024)),
    ("long_splitk", dict(B=3, lengths=("list", [32, 64, 300]), max_len=320)),
    ("llama7b_mha", dict(B=5, Hq=4, Hkv=4, D=128, lengths=("list", [128, 16, 31, 256, 80]),
                         max_len=256, pool=("fixed", 256))),
    ("tiny_worked_60", dict()),
    ("mixed_shared", dict(B=16, shared_prefix_blocks=3, max_len=256,
                          lengths=("geometric", 1 / 60, 1, 256))),
]


@pytest.mark.parametrize("name,extra", CASES)
def test_page_scores_match_oracle(name, extra):
    wl = make_workload(name, **extra)
    ds = DeviceStep(wl)
    ds.append()
    append_in_place(wl)
    got_s, got_v, err = _run(ds, wl)
    assert err == 0
    ref_s, ref_v = oracle.page_scores(wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens)
    _check(wl, got_s, got_v, ref_s, ref_v)


def test_page_scores_full_size():
    wl = make_workload("llama3_8b_gqa")
    ds = DeviceStep(wl)
    ds.append()
    append_in_place(wl)
    got_s, got_v, err = _run(ds, wl)
    assert err == 0
    ref_s, ref_v = oracle.page_scores(wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens)
    _check(wl, got_s, got_v, ref_s, ref_v)


def test_bad_table_entry_gives_nan_and_no_victim():
    wl = make_workload("llama3_8b_gqa", B=3, lengths=("list", [64, 64, 48]), max_len=64)
    ds = DeviceStep(wl)
    ds.append()
    append_in_place(wl)
    t = ds.tables.clone()
    t[1, 2] = wl.num_blocks
    got_s, got_v, err = _run(ds, wl, tables=t)
    assert err & pa.PA_DEVERR_TABLE
    assert np.isnan(got_s[1, 2]) and got_v[1] == -1
    ref_s, ref_v = oracle.page_scores(wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens)
    np.testing.assert_allclose(got_s[0, :4], ref_s[0, :4], rtol=RTOL)
    assert got_v[0] == ref_v[0] or ref_s[0, got_v[0]] <= ref_s[0, :4].min() * (1 + 2 * RTOL)
