"""Pins for the oracle's PagedEviction page scores (no GPU).

Pith review of arXiv 2509.04377, "Core claim" / "What carries the argument":
token importance S = ||V||_2 / ||K||_2, page importance = the mean of S over
the page's tokens, and when the newest page has just filled (L % B == 0) the
lowest-scoring page is evicted.
"""

import math

import numpy as np
import pytest

import oracle
from paged_kv_cache_202_gb300.workloads import bf16_bits, make_workload
from oracle_steps import pools_after_append


def _pool(NB, Hkv, bs, D, seed=0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    v = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    return k, v


def test_constant_tokens_give_the_norm_ratio():
    NB, Hkv, bs, D = 3, 2, 4, 8
    k = np.full((NB, Hkv, bs, D), 0.5, dtype=np.float32)
    v = np.full((NB, Hkv, bs, D), -2.0, dtype=np.float32)
    scores, victims = oracle.page_scores(k, v, [[2, 0]], [8])
    assert scores[0, 0] == 4.0 and scores[0, 1] == 4.0
    assert victims[0] == 0          # tie: the lowest logical page


def test_scaling_v_and_k():
    k, v = _pool(5, 2, 16, 8)
    tables = [[4, 1, 3], [0, 2, -1]]
    lens = [40, 32]
    s, _ = oracle.page_scores(k, v, tables, lens)
    s2, _ = oracle.page_scores(k, v * np.float32(2), tables, lens)
    s3, _ = oracle.page_scores(k * np.float32(4), v, tables, lens)
    m = ~np.isnan(s)
    assert np.array_equal(s2[m], 2 * s[m])
    assert np.array_equal(s3[m], s[m] / 4)


def test_brute_force_tiny():
    rng = np.random.default_rng(3)
    NB, Hkv, bs, D = 6, 2, 4, 3
    k, v = _pool(NB, Hkv, bs, D, seed=5)
    tables = np.array([[5, 2, 0], [1, 3, -1]], dtype=np.int32)
    lens = [11, 8]
    s, victims = oracle.page_scores(k, v, tables, lens)
    for b, L in enumerate(lens):
        nb = -(-L // bs)
        for p in range(nb):
            phys = int(tables[b][p])
            toks = []
            for slot in range(min(bs, L - p * bs)):
                kk = math.fsum(float(x) ** 2 for x in k[phys, :, slot, :].ravel())
                vv = math.fsum(float(x) ** 2 for x in v[phys, :, slot, :].ravel())
                toks.append(math.sqrt(vv) / math.sqrt(kk))
            assert s[b, p] == pytest.approx(math.fsum(toks) / len(toks), rel=1e-14)
    assert victims[0] == -1                        # 11 % 4 != 0: no eviction this step
    assert victims[1] == int(np.argmin(s[1, :2]))  # both pages full


def test_tail_slots_and_unused_blocks_are_not_read():
    wl = make_workload("llama3_8b_gqa", B=4, lengths=("list", [17, 32, 5, 48]), max_len=64)
    kp, vp = pools_after_append(wl)
    s, victims = oracle.page_scores(kp, vp, wl.block_tables, wl.seq_lens)
    for b in range(wl.B):
        nb = -(-int(wl.seq_lens[b]) // 16)
        assert np.isfinite(s[b, :nb]).all()
    assert victims.tolist()[0] == -1 and victims.tolist()[2] == -1
    assert victims[1] in (0, 1) and victims[3] in (0, 1, 2)


def test_physical_permutation_invariance():
    wl = make_workload("mixed_shared", B=8, shared_prefix_blocks=2, max_len=128,
                       lengths=("geometric", 1 / 40, 1, 128))
    kp, vp = pools_after_append(wl)
    s, vic = oracle.page_scores(kp, vp, wl.block_tables, wl.seq_lens)
    perm = np.random.default_rng(1).permutation(wl.num_blocks)
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp
    bt2 = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1)
    s2, vic2 = oracle.page_scores(kp2, vp2, bt2, wl.seq_lens)
    assert np.array_equal(s, s2, equal_nan=True) and np.array_equal(vic, vic2)


def test_zero_key_scores_infinity_and_is_never_the_victim():
    k, v = _pool(3, 1, 4, 4)
    k[1] = 0.0
    s, victims = oracle.page_scores(k, v, [[1, 2]], [8])
    assert s[0, 0] == math.inf and victims[0] == 1


def test_bf16_storage():
    k, v = _pool(4, 2, 16, 8, seed=9)
    kb, vb = bf16_bits(k), bf16_bits(v)
    s, _ = oracle.page_scores(kb, vb, [[3, 0]], [32])
    kf = (kb.astype(np.uint32) << 16).view(np.float32)
    vf = (vb.astype(np.uint32) << 16).view(np.float32)
    s2, _ = oracle.page_scores(kf, vf, [[3, 0]], [32])
    assert np.array_equal(s, s2)


def test_table_entries_must_name_a_block_of_the_pool():
    # The last block of the pool is scored; an entry equal to NB is refused.
    NB, Hkv, bs, D = 3, 2, 4, 8
    k, v = _pool(NB, Hkv, bs, D, seed=4)
    scores, _ = oracle.page_scores(k, v, [[NB - 1]], [bs])
    assert np.isfinite(scores[0, 0])
    with pytest.raises(ValueError):
        oracle.page_scores(k, v, [[NB]], [bs])
