"""The seeded input generator's contiguous relayout (no GPU): the same step
with each sequence's blocks renumbered to lie consecutively in the pool."""

import numpy as np
import pytest

import oracle
from paged_kv_cache_202_gb300.workloads import contiguous_layout, make_workload


def _gather(pool, table, nb):
    return pool[table[:nb]]


@pytest.mark.parametrize("name,extra", [
    ("llama3_8b_gqa", dict(B=6, lengths=("loguniform", 20, 3000), max_len=3072)),
    ("llama7b_mha", dict(B=5, Hq=4, Hkv=4)),
    ("mixed_shared", dict(B=8, max_len=2048, shared_prefix_blocks=4,
                          lengths=("geometric", 1.0 / 256.0, 1, 2048))),
])
def test_contiguous_layout_keeps_every_page_and_renumbers_consecutively(name, extra):
    wl = make_workload(name, seed=21, **extra)
    cw = contiguous_layout(wl)
    bs = wl.block_size
    seen = set()
    nxt = 0
    for b in range(wl.B):
        nb = -(-int(wl.seq_lens[b]) // bs)
        # The same bits behind every logical block, NaN sentinels included.
        assert np.array_equal(_gather(cw.k_pool, cw.block_tables[b], nb).view(np.uint8),
                              _gather(wl.k_pool, wl.block_tables[b], nb).view(np.uint8))
        assert np.array_equal(_gather(cw.v_pool, cw.block_tables[b], nb).view(np.uint8),
                              _gather(wl.v_pool, wl.block_tables[b], nb).view(np.uint8))
        # Blocks first used by this sequence are the next ids in order.
        for p in cw.block_tables[b, :nb]:
            if int(p) not in seen:
                assert p == nxt
                seen.add(int(p))
                nxt += 1
        assert (cw.block_tables[b, nb:] == -1).all()
    # Reference counts follow their blocks.
    for b in range(wl.B):
        nb = -(-int(wl.seq_lens[b]) // bs)
        assert np.array_equal(cw.refcount[cw.block_tables[b, :nb]],
                              wl.refcount[wl.block_tables[b, :nb]])


def test_contiguous_layout_gives_the_oracle_identical_bits():
    wl = make_workload("llama3_8b_gqa", seed=22, B=4, lengths=("list", [2, 17, 300, 1000]),
                       max_len=1024)
    cw = contiguous_layout(wl)
    # Over the cached tokens (the pools before this step's append).
    a = oracle.decode(wl.q, wl.k_pool, wl.v_pool, wl.block_tables, wl.seq_lens - 1, wl.scale)
    c = oracle.decode(cw.q, cw.k_pool, cw.v_pool, cw.block_tables, cw.seq_lens - 1, cw.scale)
    assert np.array_equal(a.view(np.uint64), c.view(np.uint64))
