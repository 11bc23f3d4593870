"""Host block manager (pa_bm_*): free list, reference counts, copy on write.

Checked against a plain Python model of the same rules ("PagedAttention: The
Cache Was Storing Nothing" §2.2-§2.3: any free block serves any request;
several tables may name one block; a shared block is copied when a sequence
writes into it). No GPU needed.
"""

import threading

import numpy as np
import pytest

import paged_kv_cache_202_gb300 as pa
from paged_kv_cache_202_gb300 import _build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    pa.lib()


class Model:
    """Reference semantics: counts per block; free = count 0."""

    def __init__(self, n):
        self.count = [0] * n

    def alloc(self, ids):
        for i in ids:
            assert self.count[i] == 0
            self.count[i] = 1

    def fork(self, ids):
        for i in ids:
            self.count[i] += 1

    def release(self, ids):
        for i in ids:
            self.count[i] -= 1

    @property
    def num_free(self):
        return sum(c == 0 for c in self.count)


def test_alloc_release_reuse():
    with pa.BlockManager(6) as bm:
        a = bm.alloc(4)
        assert len(set(a.tolist())) == 4 and bm.num_free == 2
        assert all(bm.refcount(i) == 1 for i in a)
        bm.release(a[:2])
        assert bm.num_free == 4
        b = bm.alloc(4)
        assert set(b.tolist()) | set(a[2:].tolist()) == set(range(6))


def test_exhaustion_changes_nothing():
    with pa.BlockManager(3) as bm:
        bm.alloc(2)
        with pytest.raises(pa.PagedAttentionError) as ei:
            bm.alloc(2)
        assert ei.value.status == pa.PA_ERR_NO_BLOCKS
        assert bm.num_free == 1


def test_fork_and_release_counts():
    with pa.BlockManager(4) as bm:
        a = bm.alloc(2)
        bm.fork(a)
        bm.fork(a[:1])
        assert [bm.refcount(i) for i in a] == [3, 2]
        bm.release(a)
        assert [bm.refcount(i) for i in a] == [2, 1] and bm.num_free == 2
        bm.release([a[1]])
        assert bm.num_free == 3
        with pytest.raises(pa.PagedAttentionError):
            bm.release([a[1]])             # not held any more
        with pytest.raises(pa.PagedAttentionError):
            bm.release([a[0], a[0], a[0]])  # held twice only
        assert bm.refcount(a[0]) == 2
        with pytest.raises(pa.PagedAttentionError):
            bm.fork([a[1]])                 # a free block cannot be forked
        with pytest.raises(pa.PagedAttentionError):
            bm.refcount(99)


def test_random_operations_match_the_model():
    rng = np.random.default_rng(0)
    n = 64
    model = Model(n)
    with pa.BlockManager(n) as bm:
        held = []
        for _ in range(2000):
            op = rng.integers(0, 3)
            if op == 0:
                k = int(rng.integers(0, 6))
                if k <= model.num_free:
                    ids = bm.alloc(k).tolist()
                    model.alloc(ids)
                    held += ids
                else:
                    with pytest.raises(pa.PagedAttentionError):
                        bm.alloc(k)
            elif op == 1 and held:
                ids = [held[i] for i in rng.integers(0, len(held), size=3)]
                bm.fork(ids)
                model.fork(ids)
                held += ids
            elif held:
                idx = sorted(set(rng.integers(0, len(held), size=3).tolist()), reverse=True)
                ids = [held.pop(i) for i in idx]
                bm.release(ids)
                model.release(ids)
            assert bm.num_free == model.num_free
        for i in range(n):
            assert bm.refcount(i) == model.count[i]


def test_prepare_append_private_missing_and_shared():
    bs = 16
    with pa.BlockManager(16) as bm:
        prefix = bm.alloc(2)
        bm.fork(prefix)
        bm.fork(prefix)          # three tables share the prefix
        own = bm.alloc(1)
        tables = np.full((4, 4), -1, dtype=np.int32)
        tables[0, :2] = prefix           # writes at 20: block 1 of the prefix, shared
        tables[1, :2] = prefix           # writes at 31: same shared block
        tables[2, :2] = prefix           # writes at 32: logical block 2, missing
        tables[3, 0] = own[0]            # writes at 5: private block
        before = tables.copy()
        src, dst = bm.prepare_append(tables, [20, 31, 32, 5], bs)
        # Sequence 0 and 1 both write shared block prefix[1] (count 3): both copy,
        # and the block keeps the third table's reference.
        assert src.tolist() == [prefix[1], prefix[1]]
        assert tables[0, 1] == dst[0] and tables[1, 1] == dst[1]
        assert len(set(dst.tolist()) | set(prefix.tolist()) | {int(own[0])}) == 5
        assert bm.refcount(prefix[1]) == 1 and bm.refcount(prefix[0]) == 3
        assert tables[2, 2] >= 0 and bm.refcount(int(tables[2, 2])) == 1
        assert tables[3, 0] == own[0]
        unchanged = np.ones_like(tables, dtype=bool)
        unchanged[0, 1] = unchanged[1, 1] = unchanged[2, 2] = False
        assert np.array_equal(tables[unchanged], before[unchanged])


def test_prepare_append_last_sharer_keeps_the_block():
    with pa.BlockManager(8) as bm:
        blk = bm.alloc(1)
        bm.fork(blk)             # two tables, one block
        tables = np.array([[blk[0], -1], [blk[0], -1]], dtype=np.int32)
        src, dst = bm.prepare_append(tables, [3, 4], 16)
        assert src.tolist() == [blk[0]] and tables[1, 0] == blk[0] and tables[0, 0] == dst[0]
        assert bm.refcount(blk[0]) == 1


def test_prepare_append_failure_changes_nothing():
    with pa.BlockManager(3) as bm:
        blk = bm.alloc(2)
        bm.fork(blk)
        tables = np.array([[blk[0], -1], [blk[1], -1], [blk[0], -1]], dtype=np.int32)
        # needs 2 copies + 1 new block (position 16 -> logical 1, missing) but 1 block is free
        before = tables.copy()
        free = bm.num_free
        with pytest.raises(pa.PagedAttentionError) as ei:
            bm.prepare_append(tables, [3, 4, 16], 16)
        assert ei.value.status == pa.PA_ERR_NO_BLOCKS
        assert np.array_equal(tables, before) and bm.num_free == free
        assert bm.refcount(blk[0]) == 2
        with pytest.raises(pa.PagedAttentionError) as ei:
            bm.prepare_append(tables, [3, 4, 32], 16)   # position past the table
        assert ei.value.status == pa.PA_ERR_BOUNDS


def test_concurrent_alloc_release_is_consistent():
    n = 4096
    with pa.BlockManager(n) as bm:
        errors = []

        def worker(seed):
            rng = np.random.default_rng(seed)
            mine = []
            try:
                for _ in range(300):
                    if rng.random() < 0.6:
                        mine += bm.alloc(int(rng.integers(1, 4))).tolist()
                    elif mine:
                        k = int(rng.integers(1, len(mine) + 1))
                        bm.release(mine[:k])
                        mine = mine[k:]
                bm.release(mine)
            except Exception as e:  # pragma: no cover - reported below
                errors.append(e)

        threads = [threading.Thread(target=worker, args=(s,)) for s in range(8)]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        assert not errors
        assert bm.num_free == n
        assert all(bm.refcount(i) == 0 for i in range(0, n, 97))
