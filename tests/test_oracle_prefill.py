"""Pins for the oracle's causal paged multi-query attention (no GPU).

"FlashAttention vs PagedAttention", "How prefill and decode change the
diagnosis": prefill processes many positions at once, decode one; query i of
the n newest tokens sits at position L - n + i and sees the tokens up to it.
"""

import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from paged_kv_cache_202_gb300.workloads import bits_to_f32, make_workload
from oracle_steps import pools_after_append


def _wl(lens, **kw):
    return make_workload("llama3_8b_gqa", seed=31, B=len(lens), lengths=("list", lens),
                         max_len=max(lens) + 16, **kw)


def _qs(ns):
    return np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)


def _queries(wl, ns, seed=0):
    rng = np.random.default_rng(seed)
    from paged_kv_cache_202_gb300.workloads import bf16_bits
    return bf16_bits(rng.standard_normal((int(sum(ns)), wl.Hq, wl.D)).astype(np.float32))


def test_single_query_equals_decode():
    wl = _wl([40, 17, 64, 1])
    kp, vp = pools_after_append(wl)
    out = oracle.prefill(wl.q, kp, vp, wl.block_tables, wl.seq_lens, _qs([1, 1, 1, 1]), wl.scale)
    ref = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    assert np.array_equal(out, ref)


def test_matches_scipy_with_causal_mask():
    lens, ns = [70, 33, 128], [9, 33, 16]
    wl = _wl(lens)
    kp, vp = pools_after_append(wl)
    q = _queries(wl, ns)
    out = oracle.prefill(q, kp, vp, wl.block_tables, wl.seq_lens, _qs(ns), wl.scale)
    g = wl.Hq // wl.Hkv
    qf = bits_to_f32(q).astype(np.float64)
    row = 0
    for b, (L, n) in enumerate(zip(lens, ns)):
        nb = -(-L // 16)
        blocks = wl.block_tables[b, :nb]
        K = bits_to_f32(np.swapaxes(kp[blocks], 0, 1).reshape(wl.Hkv, nb * 16, wl.D)[:, :L]).astype(np.float64)
        V = bits_to_f32(np.swapaxes(vp[blocks], 0, 1).reshape(wl.Hkv, nb * 16, wl.D)[:, :L]).astype(np.float64)
        pos = L - n + np.arange(n)
        mask = np.arange(L)[None, :] > pos[:, None]
        for h in range(wl.Hq):
            s = qf[row:row + n, h] @ K[h // g].T * np.float64(np.float32(wl.scale))
            s[mask] = -np.inf
            np.testing.assert_allclose(out[row:row + n, h], softmax(s, axis=1) @ V[h // g],
                                       rtol=1e-12, atol=1e-13)
        row += n


def test_future_tokens_are_not_read():
    lens, ns = [50], [20]
    wl = _wl(lens)
    kp, vp = pools_after_append(wl)
    q = _queries(wl, ns)
    a = oracle.prefill(q, kp, vp, wl.block_tables, wl.seq_lens, _qs(ns), wl.scale)
    # Query 0 sits at position 30: poison tokens 31..49 and its row must not move.
    kp2, vp2 = kp.copy(), vp.copy()
    for t in range(31, 50):
        phys = wl.block_tables[0, t // 16]
        kp2[phys, :, t % 16] = 0x7FC0
        vp2[phys, :, t % 16] = 0x7FC0
    b = oracle.prefill(q[:1], kp2, vp2, wl.block_tables, [31], _qs([1]), wl.scale)
    assert np.array_equal(a[0], b[0])


def test_brute_force_tiny():
    rng = np.random.default_rng(2)
    bs, NB, Hkv, g, D = 2, 6, 1, 2, 3
    kp = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    vp = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    tables = np.array([[4, 0, 2]], dtype=np.int32)
    L, n = 5, 3
    q = rng.standard_normal((n, Hkv * g, D)).astype(np.float32)
    out = oracle.prefill(q, kp, vp, tables, [L], _qs([n]), 0.9)
    for i in range(n):
        pos = L - n + i
        for h in range(Hkv * g):
            keys = [kp[tables[0][t // bs], 0, t % bs] for t in range(pos + 1)]
            vals = [vp[tables[0][t // bs], 0, t % bs] for t in range(pos + 1)]
            s = [float(np.float32(0.9)) * math.fsum(float(a) * float(c) for a, c in zip(q[i, h], k))
                 for k in keys]
            e = [math.exp(x) for x in s]
            ref = [math.fsum(e[t] * float(vals[t][d]) for t in range(len(e))) / math.fsum(e)
                   for d in range(D)]
            np.testing.assert_allclose(out[i, h], ref, rtol=1e-13, atol=1e-15)


def test_rejects_more_queries_than_tokens():
    wl = _wl([8])
    kp, vp = pools_after_append(wl)
    with pytest.raises(ValueError):
        oracle.prefill(_queries(wl, [9]), kp, vp, wl.block_tables, wl.seq_lens, _qs([9]), wl.scale)
