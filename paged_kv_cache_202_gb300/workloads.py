"""Seeded synthetic decode workloads: block pools, block tables and lengths.

This module only draws inputs. It holds none of the attention arithmetic: it
decides sequence lengths, hands out physical blocks from a shuffled free list
(a host-side block allocator with reference counts), fills the K/V pools with
seeded normal values, and poisons every slot that a decode must not read with
NaN. The GPU benchmark and the test suite (including the oracle checks) both
take their inputs from here, so that the same bits reach both sides.

The workloads follow the shapes of the pages' long-context decode
("PagedAttention: The Cache Was Storing Nothing" §2.2 and §3.1; "39 ·
PagedAttention" §2 for the worked 60-token request):

====================  ====================================================
name                  shape
====================  ====================================================
``tiny_worked_60``    1 sequence, 60 tokens, block size 16, table [7,1,12,4]
                      into 16 blocks, 1 q head / 1 kv head, D=64, float32
``llama7b_mha``       B=32, 32 q / 32 kv heads, D=128, bf16, block 16,
                      lengths uniform in [128, 2048], 8192-block pool
``llama3_8b_gqa``     B=64, 32 q / 8 kv heads, D=128, bf16, block 16,
                      lengths log-uniform in [512, 32768], pool = 1.1 x
                      the blocks in use
``long_splitk``       B=8, 64 q / 8 kv heads, D=128, bf16, block 32, every
                      length 131072, 1% of tokens have K scaled by 8
``prefill_gqa``       B=16, 32 q / 8 kv heads, D=128, bf16, block 16, lengths
                      log-uniform in [1024, 16384]; the newest 256 tokens of
                      each sequence are queries (chunked prefill)
``mixed_shared``      B=256, 32 q / 8 kv heads, D=128, bf16, block 16,
                      lengths geometric (mean 1024) clipped to [1, 8192];
                      even sequences share the same first 64 physical blocks
``spec_gqa``          the ``llama3_8b_gqa`` batch (its own seed); the newest 4
                      tokens of each sequence are queries (speculative
                      verification of 4 drafted tokens)
``llama3_405b_gqa``   the ``llama3_8b_gqa`` recipe (its own seed) with
                      Llama-3-405B's grouping: 128 q / 8 kv heads
====================  ====================================================

Every workload is one decode step: the pools hold ``cache_len = L - 1``
tokens per sequence, ``k_new``/``v_new`` hold the step's new token, and the
step appends it at position ``cache_len`` and then attends over ``L`` tokens.
"""

from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os

import numpy as np
import torch

# numpy PCG64 seeds: 1000 + the workload's ordinal.
_ORDINAL = {"tiny_worked_60": 1, "llama7b_mha": 2, "llama3_8b_gqa": 3, "long_splitk": 4,
            "mixed_shared": 5, "prefill_gqa": 6, "spec_gqa": 7, "llama3_405b_gqa": 8}

CONFIGS = {
    "tiny_worked_60": dict(B=1, Hq=1, Hkv=1, D=64, block_size=16, dtype="f32",
                           lengths=("fixed", 60), pool=("fixed", 16), table=[[7, 1, 12, 4]],
                           max_len=64),
    "llama7b_mha": dict(B=32, Hq=32, Hkv=32, D=128, block_size=16, dtype="bf16",
                        lengths=("uniform", 128, 2048), pool=("fixed", 8192), max_len=2048),
    "llama3_8b_gqa": dict(B=64, Hq=32, Hkv=8, D=128, block_size=16, dtype="bf16",
                          lengths=("loguniform", 512, 32768), pool=("factor", 1.1),
                          max_len=32768),
    "long_splitk": dict(B=8, Hq=64, Hkv=8, D=128, block_size=32, dtype="bf16",
                        lengths=("fixed", 131072), pool=("factor", 1.0), max_len=131072,
                        k_outliers=(0.01, 8.0)),
    "prefill_gqa": dict(B=16, Hq=32, Hkv=8, D=128, block_size=16, dtype="bf16",
                        lengths=("loguniform", 1024, 16384), pool=("factor", 1.1), max_len=16384,
                        new_tokens=256),
    "mixed_shared": dict(B=256, Hq=32, Hkv=8, D=128, block_size=16, dtype="bf16",
                         lengths=("geometric", 1.0 / 1024.0, 1, 8192), pool=("factor", 1.1),
                         max_len=8192, shared_prefix_blocks=64),
    "spec_gqa": dict(B=64, Hq=32, Hkv=8, D=128, block_size=16, dtype="bf16",
                     lengths=("loguniform", 512, 32768), pool=("factor", 1.1), max_len=32768,
                     new_tokens=4),
    "llama3_405b_gqa": dict(B=64, Hq=128, Hkv=8, D=128, block_size=16, dtype="bf16",
                            lengths=("loguniform", 512, 32768), pool=("factor", 1.1),
                            max_len=32768),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest-even) and return the bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


class BlockAllocator:
    """Host-side block allocator: a shuffled free list with reference counts.

    Free blocks are handed out in the order of a seeded random permutation of
    [0, num_blocks), so a sequence's blocks land anywhere in the pool. A block
    can be shared by several tables; its reference count says by how many.
    """

    def __init__(self, num_blocks: int, rng: np.random.Generator):
        self.num_blocks = int(num_blocks)
        self._free = list(rng.permutation(self.num_blocks).astype(np.int64)[::-1])
        self.refcount = np.zeros(self.num_blocks, dtype=np.int32)

    def alloc(self, n: int) -> list[int]:
        if n > len(self._free):
            raise MemoryError(f"block pool exhausted: want {n}, have {len(self._free)}")
        out = [int(self._free.pop()) for _ in range(n)]
        self.refcount[out] += 1
        return out

    def share(self, blocks) -> list[int]:
        self.refcount[list(blocks)] += 1
        return list(blocks)

    def free(self, blocks) -> None:
        for blk in blocks:
            self.refcount[blk] -= 1
            if self.refcount[blk] == 0:
                self._free.append(int(blk))

    @property
    def num_free(self) -> int:
        return len(self._free)


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    max_blocks: int
    dtype: str                 # "f32" or "bf16"
    scale: float               # 1/sqrt(D)
    seq_lens: np.ndarray       # int32 [B], decode lengths (include the new token)
    cache_lens: np.ndarray     # int32 [B], seq_lens - 1 = append positions
    block_tables: np.ndarray   # int32 [B, max_blocks], -1 past each sequence
    q: np.ndarray              # [B, Hq, D]       float32 or uint16 (bf16 bits)
    k_pool: np.ndarray         # [NB, Hkv, bs, D] float32 or uint16
    v_pool: np.ndarray
    k_new: np.ndarray          # [B, Hkv, D]
    v_new: np.ndarray
    refcount: np.ndarray       # int32 [NB]

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.B else 1


def _draw_lengths(spec, B: int, rng: np.random.Generator) -> np.ndarray:
    kind = spec[0]
    if kind == "fixed":
        return np.full(B, spec[1], dtype=np.int64)
    if kind == "list":             # explicit lengths, one per sequence
        out = np.asarray(spec[1], dtype=np.int64)
        if out.shape != (B,):
            raise ValueError("length list does not match B")
        return out
    if kind == "uniform":          # integers, both ends included
        return rng.integers(spec[1], spec[2] + 1, size=B)
    if kind == "loguniform":       # floor(exp(U(ln lo, ln hi))), clipped
        lo, hi = spec[1], spec[2]
        u = rng.uniform(math.log(lo), math.log(hi), size=B)
        return np.clip(np.floor(np.exp(u)).astype(np.int64), lo, hi)
    if kind == "geometric":        # support >= 1, mean 1/p, clipped
        p, lo, hi = spec[1], spec[2], spec[3]
        return np.clip(rng.geometric(p, size=B).astype(np.int64), lo, hi)
    raise ValueError(kind)


_CHUNK = 1 << 24


def _normal(seq: np.random.SeedSequence, shape, dtype: str) -> np.ndarray:
    """Standard normal values, float32 or rounded to bfloat16 bits.

    The array is filled in fixed chunks of 2^24 elements; chunk c draws from
    its own PCG64 stream spawned from ``seq``, so the values do not depend on
    how many threads fill them.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32 if dtype == "f32" else np.uint16)
    nchunks = max(1, -(-n // _CHUNK))
    streams = seq.spawn(nchunks)

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        x = np.random.Generator(np.random.PCG64(streams[c])).standard_normal(hi - lo,
                                                                            dtype=np.float32)
        out[lo:hi] = x if dtype == "f32" else bf16_bits(x)

    if nchunks == 1:
        fill(0)
    else:
        with concurrent.futures.ThreadPoolExecutor(min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def _lengths(cfg: dict, rng: np.random.Generator) -> np.ndarray:
    """Sequence lengths of a recipe: the first draw from the workload's generator."""
    B, bs = cfg["B"], cfg["block_size"]
    shared = int(cfg.get("shared_prefix_blocks", 0))
    L = _draw_lengths(cfg["lengths"], B, rng) if B else np.zeros(0, dtype=np.int64)
    if shared and cfg.get("clip_shared", True):
        # Sharing sequences (even b) keep their append position past the shared
        # prefix so that the shared blocks are never written. With
        # clip_shared=False a sharing sequence may append inside the prefix;
        # its step then needs copy on write first.
        L[0::2] = np.clip(L[0::2], shared * bs + 1, cfg["max_len"])
    return L


def workload_lengths(name: str, seed: int | None = None, **overrides) -> np.ndarray:
    """The sequence lengths `make_workload` draws for the same arguments, without the pools."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    if seed is None:
        seed = 1000 + _ORDINAL[name]
    return _lengths(cfg, np.random.default_rng(seed))


def make_workload(name: str, seed: int | None = None, **overrides) -> Workload:
    """Build one seeded decode-step workload.

    ``overrides`` replace entries of the named recipe (for example a smaller
    ``B`` or ``lengths`` for a case the oracle finishes in seconds).

    Draw order from ``numpy.random.default_rng(seed)``: lengths, the free-list
    permutation, then the K outlier mask. The K pool, V pool, q, k_new and
    v_new values come from five PCG64 streams spawned from
    ``SeedSequence(seed)`` (see ``_normal``).
    """
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    if seed is None:
        seed = 1000 + _ORDINAL[name]
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, D, bs = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["block_size"]
    dtype = cfg["dtype"]
    shared = int(cfg.get("shared_prefix_blocks", 0))

    L = _lengths(cfg, rng)
    nblk = (L + bs - 1) // bs
    max_blocks = int(cfg.get("max_blocks", -(-cfg["max_len"] // bs)))
    if B and int(nblk.max()) > max_blocks:
        raise ValueError("a sequence needs more blocks than the table holds")

    # Pool size.
    private = int(nblk.sum()) - (int(np.minimum(nblk[0::2], shared).sum()) if shared else 0)
    in_use = private + shared
    pk = cfg["pool"]
    NB = int(pk[1]) if pk[0] == "fixed" else int(math.ceil(pk[1] * (in_use + (B if shared else 0))))
    NB = max(NB, in_use, 1)

    alloc = BlockAllocator(NB, rng)
    tables = np.full((B, max_blocks), -1, dtype=np.int32)
    if cfg.get("table") is not None:
        fixed = np.asarray(cfg["table"], dtype=np.int32)
        tables[:, :fixed.shape[1]] = fixed
        alloc.refcount[fixed.ravel()] += 1
    else:
        prefix = alloc.alloc(shared) if shared else []
        for b in range(B):
            if shared and b % 2 == 0:
                n_sh = min(shared, int(nblk[b]))
                blocks = alloc.share(prefix[:n_sh]) + alloc.alloc(int(nblk[b]) - n_sh)
            else:
                blocks = alloc.alloc(int(nblk[b]))
            tables[b, :len(blocks)] = blocks
        if shared:
            alloc.refcount[prefix] -= 1  # the prefix itself was counted once at alloc

    pool_shape = (NB, Hkv, bs, D)
    seqs = np.random.SeedSequence(seed).spawn(5)
    kpool = _normal(seqs[0], pool_shape, dtype)
    vpool = _normal(seqs[1], pool_shape, dtype)
    q = _normal(seqs[2], (B, Hq, D), dtype)
    k_new = _normal(seqs[3], (B, Hkv, D), dtype)
    v_new = _normal(seqs[4], (B, Hkv, D), dtype)
    nan = np.float32(np.nan) if dtype == "f32" else np.uint16(0x7FC0)

    if "k_outliers" in cfg:
        # A Bernoulli(frac) mask per (sequence, token) scales that token's keys
        # (all kv heads) in float32 before rounding to the storage type.
        frac, factor = cfg["k_outliers"]
        for b in range(B):
            toks = np.nonzero(rng.random(int(L[b])) < frac)[0]
            for t in toks:
                if t == L[b] - 1:
                    k_new[b] = _scale_stored(k_new[b], factor, dtype)
                else:
                    phys = tables[b, t // bs]
                    kpool[phys, :, t % bs, :] = _scale_stored(kpool[phys, :, t % bs, :],
                                                              factor, dtype)

    # Poison everything a decode of this step must not read: blocks no table
    # names, and every slot at or past each sequence's append position.
    used = np.zeros(NB, dtype=bool)
    for b in range(B):
        used[tables[b, :int(nblk[b])]] = True
    kpool[~used] = nan
    vpool[~used] = nan
    for b in range(B):
        c = int(L[b]) - 1
        last = int(tables[b, c // bs])
        if alloc.refcount[last] > 1:
            continue  # a shared block holds tokens other sequences still read
        kpool[last, :, c % bs:, :] = nan
        vpool[last, :, c % bs:, :] = nan

    return Workload(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=bs, num_blocks=NB,
                    max_blocks=max_blocks, dtype=dtype, scale=1.0 / math.sqrt(D),
                    seq_lens=L.astype(np.int32), cache_lens=(L - 1).astype(np.int32),
                    block_tables=tables, q=q, k_pool=kpool, v_pool=vpool, k_new=k_new,
                    v_new=v_new, refcount=alloc.refcount.copy())


def _scale_stored(x: np.ndarray, factor: float, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return (x * np.float32(factor)).astype(np.float32)
    return bf16_bits(bits_to_f32(x) * np.float32(factor))


def contiguous_layout(wl: Workload) -> Workload:
    """The same step with every sequence's blocks renumbered to lie consecutively.

    Physical ids are handed out in order of first appearance, sequence by
    sequence and logical block by logical block (a block two tables share
    keeps the place of its first use); blocks no table names come last. The
    pools are permuted to match, so every gathered page holds the same bits
    and only the addresses change: the layout of an unpaged cache, for
    comparing a paged read against a contiguous one on the same data.
    """
    NB, bs = wl.num_blocks, wl.block_size
    new_id = np.full(NB, -1, dtype=np.int64)
    nxt = 0
    for b in range(wl.B):
        nb = -(-int(wl.seq_lens[b]) // bs)
        for p in wl.block_tables[b, :nb]:
            if new_id[p] < 0:
                new_id[p] = nxt
                nxt += 1
    rest = np.nonzero(new_id < 0)[0]
    new_id[rest] = np.arange(nxt, nxt + len(rest))
    k_pool = np.empty_like(wl.k_pool)
    v_pool = np.empty_like(wl.v_pool)
    k_pool[new_id] = wl.k_pool
    v_pool[new_id] = wl.v_pool
    tables = np.where(wl.block_tables >= 0, new_id[np.maximum(wl.block_tables, 0)],
                      -1).astype(np.int32)
    refcount = np.empty_like(wl.refcount)
    refcount[new_id] = wl.refcount
    return dataclasses.replace(wl, block_tables=tables, k_pool=k_pool, v_pool=v_pool,
                               refcount=refcount)
