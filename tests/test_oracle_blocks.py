"""Pins for the oracle's batched block copy (no GPU).

"PagedAttention: The Cache Was Storing Nothing" §2.3: a shared block is
copied before a sequence writes it (copy on write). A copy is exact: every
kv head and slot of the destination block takes the source block's bits.
The batch form copies pairs whose destinations are distinct and are not
sources, so the pairs are independent; checked against numpy's block-wise
assignment, on payloads that include NaN bit patterns.
"""

import numpy as np

import oracle


def _pools(NB, Hkv, bs, D, dtype, seed):
    rng = np.random.default_rng(seed)
    if dtype == "bf16":
        k = rng.integers(-32768, 32768, size=(NB, Hkv, bs, D), dtype=np.int64).astype(np.int16)
        v = rng.integers(-32768, 32768, size=(NB, Hkv, bs, D), dtype=np.int64).astype(np.int16)
        k.reshape(-1)[:7] = np.int16(0x7FC1)  # quiet-NaN bf16 patterns
    else:
        k = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
        v = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
        k.view(np.uint32).reshape(-1)[:5] = 0x7FC00123  # NaN payloads
    return k, v


def _pairs(NB, n, seed):
    ids = np.random.default_rng(seed).permutation(NB)
    return ids[:n].astype(np.int32), ids[n:2 * n].astype(np.int32)  # disjoint sources and destinations


def test_copies_match_numpy_block_assignment():
    for dtype, bs in (("bf16", 16), ("f32", 32), ("bf16", 32)):
        k, v = _pools(40, 3, bs, 64, dtype, seed=1)
        src, dst = _pairs(40, 9, seed=2)
        k0, v0 = k.copy(), v.copy()
        oracle.copy_blocks(k, v, src, dst)
        want_k, want_v = k0.copy(), v0.copy()
        want_k[dst] = k0[src]
        want_v[dst] = v0[src]
        assert k.tobytes() == want_k.tobytes() and v.tobytes() == want_v.tobytes()


def test_untouched_blocks_keep_their_bits():
    k, v = _pools(32, 2, 16, 128, "bf16", seed=3)
    src, dst = _pairs(32, 5, seed=4)
    k0, v0 = k.copy(), v.copy()
    oracle.copy_blocks(k, v, src, dst)
    rest = np.setdiff1d(np.arange(32), dst)
    assert k[rest].tobytes() == k0[rest].tobytes() and v[rest].tobytes() == v0[rest].tobytes()


def test_no_pairs_is_a_no_op():
    k, v = _pools(8, 1, 16, 64, "f32", seed=5)
    k0, v0 = k.copy(), v.copy()
    oracle.copy_blocks(k, v, np.zeros(0, np.int32), np.zeros(0, np.int32))
    assert k.tobytes() == k0.tobytes() and v.tobytes() == v0.tobytes()


def test_ids_must_name_a_block_of_the_pool():
    # Ids run 0 .. NB-1: the last block copies; an id equal to NB is refused.
    import pytest
    NB = 6
    k, v = _pools(NB, 2, 16, 8, "f32", seed=9)
    kr, vr = k.copy(), v.copy()
    oracle.copy_blocks(k, v, np.array([NB - 1], np.int32), np.array([0], np.int32))
    assert np.array_equal(k[0], kr[NB - 1]) and np.array_equal(v[0], vr[NB - 1])
    for src, dst in ((NB, 0), (0, NB)):
        with pytest.raises(ValueError):
            oracle.copy_blocks(k.copy(), v.copy(), np.array([src], np.int32),
                               np.array([dst], np.int32))
