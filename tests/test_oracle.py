"""Pins for the fp64 oracle, checked against what the pages and mathematics fix.

None of these needs a GPU. Each test ties the oracle to something other than
itself: numbers the pages print (``tests/golden``), the library routine
``scipy.special.softmax`` on contiguous K/V, closed forms, invariances the
pages state, and brute force on tiny inputs in pure Python.
"""

import json
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from paged_kv_cache_202_gb300.workloads import bf16_bits, bits_to_f32, make_workload
from oracle_steps import pools_after_append


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- block and byte arithmetic

def test_block_rounding_200_tokens(golden_dir):
    g = _golden(golden_dir, "block_arithmetic.json")["rounding_200"]
    nb = oracle.num_blocks(g["tokens"], g["block_size"])
    assert nb == g["blocks"]
    assert nb * g["block_size"] == g["slots"]
    assert round(100.0 * g["tokens"] / (nb * g["block_size"]), 1) == g["utilisation_pct_1dp"]


def test_three_request_printout(golden_dir):
    g = _golden(golden_dir, "block_arithmetic.json")["three_requests"]
    bs = g["block_size"]
    rounded = [oracle.num_blocks(L, bs) * bs for L in g["lengths"]]
    assert rounded == g["rounded_slots"]
    paged = sum(rounded)
    used = sum(g["lengths"])
    fixed = len(g["lengths"]) * g["reserved_per_request"]
    mib = lambda tokens: f"{tokens * g['kv_bytes_per_token'] / 2**20:.2f}"
    assert (paged, used, fixed) == (g["paged_slots"], g["used_slots"], g["fixed_slots"])
    assert (mib(paged), mib(used), mib(fixed)) == (g["paged_mib"], g["used_mib"], g["fixed_mib"])
    assert paged - used == g["unused_paged_slots"]


def test_worked_example_block_count(golden_dir):
    g = _golden(golden_dir, "block_arithmetic.json")["worked_60"]
    nb = oracle.num_blocks(g["tokens"], g["block_size"])
    assert nb == g["blocks"] == len(g["table"])
    assert g["tokens"] - (nb - 1) * g["block_size"] == g["last_block_tokens"]
    assert oracle.num_blocks(64, 16) == 4 and oracle.num_blocks(65, 16) == 5
    assert oracle.num_blocks(1, 32) == 1 and oracle.num_blocks(0, 16) == 0


def test_kv_bytes_per_token(golden_dir):
    g = _golden(golden_dir, "kv_bytes.json")
    c = g["llama7b_layer_2048"]
    per_tok = oracle.kv_elems_per_token(c["kv_heads"], c["head_dim"], c["layers"])
    assert per_tok * c["tokens"] * c["elem_bytes"] == c["bytes"]
    for key in ("llama3_70b_gqa_per_layer", "llama3_70b_mha_per_layer",
                "deepseek_v2_full_kv_per_layer"):
        c = g[key]
        assert oracle.kv_elems_per_token(c["kv_heads"], c["head_dim"], c["layers"]) == c["elems"]
    c = g["deepseek_v2_full_kv_per_layer"]
    assert round(c["elems"] / c["latent_elems"]) == c["ratio_rounded"]
    c = g["llama3_70b_per_token_kib"]
    bytes_tok = oracle.kv_elems_per_token(c["kv_heads"], c["head_dim"], c["layers"]) * c["elem_bytes"]
    assert bytes_tok == c["kib"] * 1024
    full = oracle.kv_elems_per_token(c["kv_heads"] * c["without_grouping_factor"], c["head_dim"],
                                     c["layers"])
    assert full == c["without_grouping_factor"] * bytes_tok // c["elem_bytes"]


def test_decode_bytes_counts_kv_table_q_lens_out(golden_dir):
    c = _golden(golden_dir, "kv_bytes.json")["llama7b_layer_2048"]
    # One 2048-token sequence, MHA with LLaMA-7B's 32 heads of 128: the KV part is
    # the page's 33,554,432 bytes; the rest is 128 table entries, q, length, output.
    n = oracle.decode_bytes([2048], 32, 32, 128, 16, 2, 2)
    assert n - c["bytes"] == 128 * 4 + 32 * 128 * 2 + 4 + 32 * 128 * 2
    # A partly filled last block counts its table entry but not its pad slots.
    assert oracle.decode_bytes([17], 1, 1, 64, 16, 4, 4) - oracle.decode_bytes([16], 1, 1, 64, 16, 4, 4) \
        == 2 * 64 * 4 + 4


def test_decode_bytes_equal_the_arrays_a_decode_touches():
    # bf16 pools and an f32 output, so the query and output element sizes
    # differ: the counter must equal the bytes of the K and V rows the decode
    # attends, the table entries of its attended blocks, and the q, length
    # and output arrays as allocated.
    wl = _small("gqa_bf16")
    out = np.zeros((wl.B, wl.Hq, wl.D), dtype=np.float32)
    lens = [int(x) for x in wl.seq_lens]
    kv = 2 * sum(lens) * wl.Hkv * wl.k_pool[0, 0, 0].nbytes
    table = sum(-(-L // wl.block_size) for L in lens) * wl.block_tables.itemsize
    want = kv + table + wl.q.nbytes + wl.seq_lens.nbytes + out.nbytes
    got = oracle.decode_bytes(wl.seq_lens, wl.Hq, wl.Hkv, wl.D, wl.block_size,
                              wl.k_pool.itemsize, out.itemsize)
    assert got == want


# ---------------------------------------------------------------- the worked 60-token request

def _worked_problem(golden_dir, seed=7):
    g = _golden(golden_dir, "worked_example_60.json")
    rng = np.random.default_rng(seed)
    L, bs, NB, D = g["tokens"], g["block_size"], g["num_blocks"], 64
    q = rng.standard_normal((1, 1, D), dtype=np.float32)
    Kc = rng.standard_normal((L, D), dtype=np.float32)
    Vc = rng.standard_normal((L, D), dtype=np.float32)
    kpool = np.full((NB, 1, bs, D), np.nan, dtype=np.float32)
    vpool = np.full((NB, 1, bs, D), np.nan, dtype=np.float32)
    # Logical block i holds tokens [16 i, 16 i + 16) and lives at physical table[i].
    for i, phys in enumerate(g["table"]):
        n = min(bs, L - i * bs)
        kpool[phys, 0, :n] = Kc[i * bs:i * bs + n]
        vpool[phys, 0, :n] = Vc[i * bs:i * bs + n]
    table = np.asarray([g["table"]], dtype=np.int32)
    return g, q, Kc, Vc, kpool, vpool, table


def test_worked_example_addresses(golden_dir):
    g, q, Kc, Vc, kpool, vpool, table = _worked_problem(golden_dir)
    for t, phys, slot in g["token_to_physical"]:
        assert np.array_equal(kpool[phys, 0, slot], Kc[t])
    for blk in g["blocks_never_read"]:
        assert np.isnan(kpool[blk]).all()
    assert np.isnan(kpool[4, 0, g["slots_never_read_in_block_4"]]).all()


def test_worked_example_equals_contiguous_attention(golden_dir):
    g, q, Kc, Vc, kpool, vpool, table = _worked_problem(golden_dir)
    scale = 1.0 / math.sqrt(64)
    out = oracle.decode(q, kpool, vpool, table, [g["tokens"]], scale)
    assert np.isfinite(out).all(), "a NaN sentinel was read"
    w = softmax(Kc.astype(np.float64) @ q[0, 0].astype(np.float64) * np.float64(np.float32(scale)))
    ref = w @ Vc.astype(np.float64)
    np.testing.assert_allclose(out[0, 0], ref, rtol=1e-12, atol=1e-14)
    # Same values laid out contiguously (identity table): bit-identical output.
    kc = np.full((4, 1, 16, 64), np.nan, dtype=np.float32)
    vc = np.full((4, 1, 16, 64), np.nan, dtype=np.float32)
    kc.reshape(64, 64)[:60] = Kc
    vc.reshape(64, 64)[:60] = Vc
    out_c = oracle.decode(q, kc, vc, np.arange(4, dtype=np.int32)[None], [60], scale)
    assert np.array_equal(out, out_c)


# ---------------------------------------------------------------- dense equivalence, invariances

def _dense_reference(wl, kpool, vpool):
    """Gather each sequence's K/V with numpy fancy indexing, then softmax(q K^T s) V."""
    g = wl.Hq // wl.Hkv
    conv = (lambda a: a.astype(np.float64)) if wl.dtype == "f32" else \
        (lambda a: bits_to_f32(a).astype(np.float64))
    out = np.empty((wl.B, wl.Hq, wl.D))
    for b in range(wl.B):
        L = int(wl.seq_lens[b])
        nb = -(-L // wl.block_size)
        blocks = wl.block_tables[b, :nb]
        Kb = np.swapaxes(kpool[blocks], 0, 1).reshape(wl.Hkv, nb * wl.block_size, wl.D)[:, :L]
        Vb = np.swapaxes(vpool[blocks], 0, 1).reshape(wl.Hkv, nb * wl.block_size, wl.D)[:, :L]
        for h in range(wl.Hq):
            s = conv(Kb[h // g]) @ conv(wl.q[b, h]) * np.float64(np.float32(wl.scale))
            out[b, h] = softmax(s) @ conv(Vb[h // g])
    return out


SMALL = {
    "gqa_bf16": dict(name="llama3_8b_gqa", B=5, lengths=("loguniform", 1, 300), max_len=320),
    "mha_bf16": dict(name="llama7b_mha", B=3, Hq=4, Hkv=4, lengths=("uniform", 1, 70), max_len=80,
                     pool=("fixed", 64)),
    "mqa_f32": dict(name="tiny_worked_60", B=4, Hq=3, Hkv=1, lengths=("uniform", 1, 90),
                    max_len=96, pool=("fixed", 40), table=None),
    "bs32_bf16": dict(name="long_splitk", B=2, Hq=8, Hkv=2, lengths=("fixed", 77), max_len=128),
    "shared_bf16": dict(name="mixed_shared", B=6, shared_prefix_blocks=2, max_len=128,
                        lengths=("geometric", 1 / 40, 1, 128)),
}


def _small(key, seed=None):
    spec = dict(SMALL[key])
    name = spec.pop("name")
    return make_workload(name, seed=seed, **spec)


@pytest.mark.parametrize("key", sorted(SMALL))
def test_oracle_matches_dense_softmax(key):
    wl = _small(key)
    kp, vp = pools_after_append(wl)
    out = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, _dense_reference(wl, kp, vp), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("key", ["gqa_bf16", "bs32_bf16", "shared_bf16"])
def test_physical_permutation_is_bitwise_invariant(key):
    wl = _small(key)
    kp, vp = pools_after_append(wl)
    out = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    perm = np.random.default_rng(5).permutation(wl.num_blocks)
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    bt2 = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
    out2 = oracle.decode(wl.q, kp2, vp2, bt2, wl.seq_lens, wl.scale)
    assert np.array_equal(out, out2)


def test_sampled_pairs_equal_full_rows():
    wl = _small("gqa_bf16")
    kp, vp = pools_after_append(wl)
    full = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    pairs = [(4, 31), (0, 0), (2, 17)]
    some = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale, pairs=pairs)
    for i, (b, h) in enumerate(pairs):
        assert np.array_equal(some[i], full[b, h])


def test_thread_count_does_not_change_bits():
    wl = _small("gqa_bf16")
    kp, vp = pools_after_append(wl)
    a = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale, nthreads=1)
    b = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale, nthreads=5)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- softmax weights and merge

def test_weights_sum_to_one_and_match_softmax():
    wl = _small("gqa_bf16")
    kp, vp = pools_after_append(wl)
    for b, h in [(0, 3), (3, 30), (4, 8)]:
        w = oracle.weights(wl.q, kp, wl.block_tables, wl.seq_lens, wl.scale, b, h)
        assert w.shape == (wl.seq_lens[b],)
        assert (w >= 0).all()
        assert abs(math.fsum(w) - 1.0) < 1e-12


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_merge_of_random_splits_equals_one_pass(seed):
    wl = _small("bs32_bf16")
    kp, vp = pools_after_append(wl)
    full = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    rng = np.random.default_rng(seed)
    for b, h in [(0, 0), (1, 7), (1, 2)]:
        L = int(wl.seq_lens[b])
        cuts = np.sort(rng.choice(np.arange(0, L + 1), size=4, replace=True))
        bounds = [0, *cuts.tolist(), L]   # repeated cuts give empty partials
        parts = [oracle.partial(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale, b, h, lo, hi)
                 for lo, hi in zip(bounds[:-1], bounds[1:])]
        out = oracle.merge([p[0] for p in parts], [p[1] for p in parts], [p[2] for p in parts])
        np.testing.assert_allclose(out, full[b, h], rtol=1e-12, atol=1e-13)


def test_merge_with_leading_and_inner_empty_partials():
    # A partition of the tokens is still a partition when some pieces are
    # empty: two empty pieces first, one in the middle and one at the end
    # must merge to the one-pass result (an empty partial contributes
    # nothing, even before any non-empty one has been folded in).
    wl = _small("bs32_bf16")
    kp, vp = pools_after_append(wl)
    full = oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale)
    b, h = 1, 3
    L = int(wl.seq_lens[b])
    mid = L // 2
    bounds = [0, 0, 0, mid, mid, L, L]
    parts = [oracle.partial(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale, b, h, lo, hi)
             for lo, hi in zip(bounds[:-1], bounds[1:])]
    assert parts[0][0] == -math.inf and parts[0][1] == 0.0
    out = oracle.merge([p[0] for p in parts], [p[1] for p in parts], [p[2] for p in parts])
    np.testing.assert_allclose(out, full[b, h], rtol=1e-12, atol=1e-13)


def test_two_partial_merge_rule():
    # Two partials with different maxima: the rule must rescale both l and acc.
    m = [3.0, -1.5]
    l = [2.0, 5.0]
    acc = np.array([[1.0, -2.0], [4.0, 0.5]])
    out = oracle.merge(m, l, acc)
    mm = 3.0
    ll = 2.0 * math.exp(0.0) + 5.0 * math.exp(-4.5)
    ref = (acc[0] * math.exp(0.0) + acc[1] * math.exp(-4.5)) / ll
    np.testing.assert_allclose(out, ref, rtol=1e-15)
    assert mm == max(m)


# ---------------------------------------------------------------- closed forms

def _one_seq(L, D=8, Hq=1, Hkv=1, bs=16, seed=3):
    rng = np.random.default_rng(seed)
    nb = -(-L // bs)
    NB = nb + 3
    perm = rng.permutation(NB)[:nb].astype(np.int32)
    q = rng.standard_normal((1, Hq, D), dtype=np.float32)
    Kc = rng.standard_normal((Hkv, L, D), dtype=np.float32)
    Vc = rng.standard_normal((Hkv, L, D), dtype=np.float32)
    return q, Kc, Vc, perm, NB


def _pack(Kc, perm, NB, bs=16):
    Hkv, L, D = Kc.shape
    pool = np.full((NB, Hkv, bs, D), np.nan, dtype=np.float32)
    for i, phys in enumerate(perm):
        n = min(bs, L - i * bs)
        pool[phys, :, :n] = Kc[:, i * bs:i * bs + n]
    return pool


def test_single_token_returns_its_value_exactly():
    q, Kc, Vc, perm, NB = _one_seq(1)
    out = oracle.decode(q, _pack(Kc, perm, NB), _pack(Vc, perm, NB), perm[None], [1], 0.3)
    assert np.array_equal(out[0, 0], Vc[0, 0].astype(np.float64))


@pytest.mark.parametrize("how", ["zero_query", "equal_keys", "zero_scale"])
def test_uniform_weights_give_mean_of_values(how):
    L = 37
    q, Kc, Vc, perm, NB = _one_seq(L)
    scale = 0.25
    if how == "zero_query":
        q[:] = 0
    elif how == "equal_keys":
        Kc[:] = Kc[:, :1]
    else:
        scale = 0.0
    out = oracle.decode(q, _pack(Kc, perm, NB), _pack(Vc, perm, NB), perm[None], [L], scale)
    np.testing.assert_allclose(out[0, 0], Vc[0].astype(np.float64).mean(axis=0), rtol=1e-13,
                               atol=1e-14)


@pytest.mark.parametrize("L", [16, 48])
def test_sequence_that_fills_its_table(L):
    # The largest length a table allows: every entry names a full block
    # (max_blocks * block_size tokens). It must be attended like any other,
    # equal to softmax(q K^T s) V on the contiguous K and V.
    q, Kc, Vc, perm, NB = _one_seq(L)
    assert perm.size * 16 == L
    scale = 0.3
    out = oracle.decode(q, _pack(Kc, perm, NB), _pack(Vc, perm, NB), perm[None], [L], scale)
    s = (Kc[0].astype(np.float64) @ q[0, 0].astype(np.float64)) * np.float64(np.float32(scale))
    w = softmax(s)
    np.testing.assert_allclose(out[0, 0], w @ Vc[0].astype(np.float64), rtol=1e-12, atol=1e-13)


def test_one_dominant_key_selects_its_value():
    L = 40
    q, Kc, Vc, perm, NB = _one_seq(L)
    q[:] = 0
    q[0, 0, 0] = 64.0
    Kc[0, 23, 0] = 64.0
    out = oracle.decode(q, _pack(Kc, perm, NB), _pack(Vc, perm, NB), perm[None], [L], 1.0)
    np.testing.assert_allclose(out[0, 0], Vc[0, 23].astype(np.float64), rtol=0, atol=1e-12)


def test_scale_multiplies_scores():
    L = 29
    q, Kc, Vc, perm, NB = _one_seq(L)
    kp, vp = _pack(Kc, perm, NB), _pack(Vc, perm, NB)
    a = oracle.decode(q, kp, vp, perm[None], [L], 2.0)
    b = oracle.decode(q * np.float32(2.0), kp, vp, perm[None], [L], 1.0)
    assert np.array_equal(a, b)


def test_mqa_equals_mha_with_broadcast_kv():
    L, Hq = 50, 4
    q, Kc, Vc, perm, NB = _one_seq(L, Hq=Hq, Hkv=1)
    one = oracle.decode(q, _pack(Kc, perm, NB), _pack(Vc, perm, NB), perm[None], [L], 0.2)
    Kb = np.repeat(Kc, Hq, axis=0)
    Vb = np.repeat(Vc, Hq, axis=0)
    many = oracle.decode(q, _pack(Kb, perm, NB), _pack(Vb, perm, NB), perm[None], [L], 0.2)
    assert np.array_equal(one, many)


# ---------------------------------------------------------------- brute force on tiny inputs

@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    bs = 2
    Hkv = 1 + seed % 2
    g = 1 + (seed // 2) % 2
    Hq = Hkv * g
    D = 1 + seed % 4
    B = 2
    lens = rng.integers(1, 6, size=B)
    NB = 8
    tables = np.full((B, 3), -1, dtype=np.int32)
    perm = rng.permutation(NB)
    k = 0
    for b in range(B):
        for i in range(-(-int(lens[b]) // bs)):
            tables[b, i] = perm[k]
            k += 1
    kpool = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    vpool = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    scale = 0.7
    out = oracle.decode(q, kpool, vpool, tables, lens, scale)
    for b in range(B):
        for h in range(Hq):
            j = h // g
            keys, vals = [], []
            for t in range(int(lens[b])):
                phys = int(tables[b][t // bs])
                keys.append([float(x) for x in kpool[phys][j][t % bs]])
                vals.append([float(x) for x in vpool[phys][j][t % bs]])
            qq = [float(x) for x in q[b][h]]
            s = [float(np.float32(scale)) * math.fsum(a * c for a, c in zip(qq, kk)) for kk in keys]
            e = [math.exp(x) for x in s]
            z = math.fsum(e)
            ref = [math.fsum(e[t] * vals[t][d] for t in range(len(e))) / z for d in range(D)]
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- append and error paths

def test_append_writes_one_slot_bit_exactly(golden_dir):
    g, q, Kc, Vc, kpool, vpool, table = _worked_problem(golden_dir)
    k_new = np.full((1, 1, 64), np.nan, dtype=np.float32)
    k_new.view(np.uint32)[..., 0] = 0x7FC00ABC           # a NaN payload must survive
    k_new.view(np.uint32)[..., 1:] = np.arange(1, 64, dtype=np.uint32)
    v_new = np.arange(64, dtype=np.float32).reshape(1, 1, 64)
    kp, vp = kpool.copy(), vpool.copy()
    oracle.append(k_new, v_new, kp, vp, table, [59])     # token 59 -> physical 4, slot 11
    changed = np.nonzero((kp.view(np.uint32) != kpool.view(np.uint32)).any(axis=-1))
    assert [tuple(int(x) for x in c) for c in zip(*changed)] == [(4, 0, 11)]
    assert np.array_equal(kp[4, 0, 11].view(np.uint32), k_new[0, 0].view(np.uint32))
    assert np.array_equal(vp[4, 0, 11], v_new[0, 0])


def test_append_puts_each_new_token_at_its_logical_position():
    # After the append, gathering each sequence's blocks in table order and
    # reading the flattened token axis gives the new K/V row at logical
    # position cache_len ("The Cache Was Storing Nothing" §2.2: the table maps
    # logical blocks to physical ones); no other slot of either pool changes.
    wl = _small("shared_bf16")
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.append(wl.k_new, wl.v_new, kp, vp, wl.block_tables, wl.cache_lens)
    bs = wl.block_size
    for b in range(wl.B):
        nb = -(-int(wl.seq_lens[b]) // bs)
        blocks = wl.block_tables[b, :nb]
        k_tokens = kp[blocks].transpose(1, 0, 2, 3).reshape(wl.Hkv, nb * bs, wl.D)
        v_tokens = vp[blocks].transpose(1, 0, 2, 3).reshape(wl.Hkv, nb * bs, wl.D)
        pos = int(wl.cache_lens[b])
        assert np.array_equal(k_tokens[:, pos], wl.k_new[b])
        assert np.array_equal(v_tokens[:, pos], wl.v_new[b])
    # Exactly one (block, kv head, slot) row per (sequence, kv head) changes:
    # the target slot held the NaN poison, the new row is finite.
    for new, before in ((kp, wl.k_pool), (vp, wl.v_pool)):
        rows = np.nonzero((new != before).any(axis=-1))
        assert len(rows[0]) == wl.B * wl.Hkv
    # The shared prefix blocks are never the append target.
    for b in range(wl.B):
        phys = wl.block_tables[b, wl.cache_lens[b] // wl.block_size]
        assert wl.refcount[phys] == 1


def test_oracle_rejects_bad_inputs():
    q, Kc, Vc, perm, NB = _one_seq(20)
    kp, vp = _pack(Kc, perm, NB), _pack(Vc, perm, NB)
    with pytest.raises(ValueError):
        oracle.decode(q, kp, vp, perm[None], [0], 1.0)
    bad = perm.copy()
    bad[1] = NB
    with pytest.raises(ValueError):
        oracle.decode(q, kp, vp, bad[None], [20], 1.0)
    with pytest.raises(ValueError):
        oracle.decode(q, kp, vp, perm[None], [33], 1.0)   # needs a third table entry


def test_append_takes_the_last_slot_of_the_table_and_no_further():
    # Tables of two 16-token blocks hold positions 0 .. 31: position 31 is
    # slot 15 of a sequence's second block; position 32 has no block and is
    # refused (the next row of the table is another sequence's).
    rng = np.random.default_rng(5)
    NB, Hkv, bs, D = 4, 2, 16, 8
    kp = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    vp = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    kn = rng.standard_normal((2, Hkv, D)).astype(np.float32)
    vn = rng.standard_normal((2, Hkv, D)).astype(np.float32)
    table = np.array([[2, 0], [1, 3]], dtype=np.int32)
    k2, v2 = kp.copy(), vp.copy()
    oracle.append(kn, vn, k2, v2, table, [31, 0])
    assert np.array_equal(k2[0, :, 15], kn[0]) and np.array_equal(v2[0, :, 15], vn[0])
    assert np.array_equal(k2[1, :, 0], kn[1]) and np.array_equal(v2[1, :, 0], vn[1])
    k2[0, :, 15], v2[0, :, 15] = kp[0, :, 15], vp[0, :, 15]
    k2[1, :, 0], v2[1, :, 0] = kp[1, :, 0], vp[1, :, 0]
    assert np.array_equal(k2, kp) and np.array_equal(v2, vp)
    with pytest.raises(ValueError):
        oracle.append(kn, vn, kp.copy(), vp.copy(), table, [32, 0])


def test_bf16_storage_is_widened_exactly():
    x = np.array([1.0, -2.5, 3.140625, 1e-3, 65504.0], dtype=np.float32)
    bits = bf16_bits(x)
    # One token, one dimension: the output is that token's value, widened exactly.
    for v in bits:
        kp = np.full((1, 1, 16, 1), 0, dtype=np.uint16)
        vp = kp.copy()
        vp[0, 0, 0, 0] = v
        out = oracle.decode(np.zeros((1, 1, 1), dtype=np.uint16), kp, vp, [[0]], [1], 1.0)
        assert out[0, 0, 0] == float(bits_to_f32(np.array([v], dtype=np.uint16))[0])
