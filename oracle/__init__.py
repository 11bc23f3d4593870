"""fp64 CPU oracle for paged decode attention (TEST INFRASTRUCTURE ONLY).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package. The GPU library never does, and the
two share no code: this wrapper loads ``liboracle.so`` built from
``oracle.cpp`` with the host C++ compiler.

Every function states the passage it follows (page title and section):

* ``decode`` / ``weights`` -- "39 · PagedAttention" §1-§2: the new query is
  scored against every earlier key in logical order through the block table,
  one softmax turns the scores into weights summing to one, and the output is
  the weighted sum of the values. Scores are q.k times ``scale``
  ("FlashAttention vs PagedAttention": 1/sqrt(d)).
* ``partial`` / ``merge`` -- "39 · PagedAttention" §3: two partials combine as
  m = max(m1, m2), l = l1 e^(m1-m) + l2 e^(m2-m); the value sums scale alike.
* ``num_blocks`` / ``kv_elems_per_token`` / ``decode_bytes`` -- "PagedAttention:
  The Cache Was Storing Nothing" §2.1 (ceil(L / block_size) blocks per request)
  and §3 (2 x heads x head_dim x layers cached numbers per token).
* ``copy_blocks`` -- the same page, §2.3: a block shared by several tables is
  copied when one sequence diverges and writes into it (copy on write).
* ``prefill`` -- "FlashAttention vs PagedAttention", "How prefill and decode
  change the diagnosis": the newest n_b tokens of a sequence are queries at
  once; query i (position L - n_b + i) attends causally to tokens <= its
  position, each row computed as ``decode`` over that prefix.
* ``page_scores`` -- Pith review of arXiv 2509.04377 (PagedEviction), "Core
  claim" and "What carries the argument": token importance ||V||_2 / ||K||_2,
  page importance = mean over the page's tokens, and when the newest page has
  just filled (L % block_size == 0) the lowest-scoring page is evicted.
* ``append`` -- the same page, §1-§2.2: the cache grows by one token per step
  and only the last block is partly full, so the new token goes to slot
  ``cache_len % bs`` of the block the table names for ``cache_len // bs``.

Inputs are numpy arrays: float32 (dtype 0) or bfloat16 bit patterns stored as
uint16 (dtype 1); every value is widened exactly to float64 before arithmetic.
Pools are [num_blocks, Hkv, block_size, D]; tables int32 [B, max_blocks].
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with g++ if it is missing or older than its source."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
                   "-o", tmp, _SRC]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    # ORACLE_LIB names another build of oracle.cpp to load instead; the
    # mutation test points it at deliberately broken copies to show that the
    # pins catch them.
    path = os.environ.get("ORACLE_LIB") or build()
    lib = ctypes.CDLL(path)
    vp, i32p, f64p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_double)
    ci, cf, ci64 = ctypes.c_int, ctypes.c_float, ctypes.c_int64
    lib.oracle_num_blocks.argtypes = [ci64, ci64]
    lib.oracle_num_blocks.restype = ci64
    lib.oracle_kv_elems_per_token.argtypes = [ci64, ci64, ci64]
    lib.oracle_kv_elems_per_token.restype = ci64
    lib.oracle_decode_bytes.argtypes = [i32p, ci, ci, ci, ci, ci, ci, ci]
    lib.oracle_decode_bytes.restype = ci64
    lib.oracle_decode.argtypes = [vp, vp, vp, i32p, ci, i32p, ci, ci, ci, ci, ci, ci, cf, ci,
                                  f64p, i32p, ci, ci]
    lib.oracle_decode.restype = ci
    lib.oracle_weights.argtypes = [vp, vp, i32p, ci, i32p, ci, ci, ci, ci, ci, ci, cf, ci, ci, ci,
                                   f64p]
    lib.oracle_weights.restype = ci
    lib.oracle_partial.argtypes = [vp, vp, vp, i32p, ci, i32p, ci, ci, ci, ci, ci, ci, cf, ci, ci,
                                   ci, ci64, ci64, f64p, f64p, f64p]
    lib.oracle_partial.restype = ci
    lib.oracle_merge.argtypes = [ci, f64p, f64p, f64p, ci, f64p]
    lib.oracle_merge.restype = ci
    lib.oracle_append.argtypes = [vp, vp, vp, vp, i32p, ci, i32p, ci, ci, ci, ci, ci, ci]
    lib.oracle_append.restype = ci
    lib.oracle_copy_blocks.argtypes = [vp, vp, i32p, i32p, ci, ci, ci64]
    lib.oracle_copy_blocks.restype = ci
    lib.oracle_page_scores.argtypes = [vp, vp, i32p, ci, i32p, ci, ci, ci, ci, ci, ci, f64p, i32p]
    lib.oracle_page_scores.restype = ci
    lib.oracle_prefill.argtypes = [vp, vp, vp, i32p, ci, i32p, i32p, ci, ci, ci, ci, ci, ci, cf,
                                   ci, f64p, ci]
    lib.oracle_prefill.restype = ci
    _lib = lib
    return lib


_ERRORS = {-1: "bad shape or index", -2: "sequence/cache length out of range",
           -3: "block table entry outside the pool"}


def _check(rc: int) -> None:
    if rc != 0:
        raise ValueError(f"oracle: {_ERRORS.get(rc, rc)}")


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _storage(a: np.ndarray) -> tuple[np.ndarray, int]:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, 0
    if a.dtype == np.uint16:
        return a, 1
    raise TypeError("oracle: storage must be float32 or uint16 (bfloat16 bits)")


def _ptr_i32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _ptr_f64(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_blocks(L: int, block_size: int) -> int:
    return int(_load().oracle_num_blocks(int(L), int(block_size)))


def kv_elems_per_token(kv_heads: int, head_dim: int, layers: int) -> int:
    return int(_load().oracle_kv_elems_per_token(int(kv_heads), int(head_dim), int(layers)))


def decode_bytes(seq_lens, Hq: int, Hkv: int, D: int, block_size: int,
                 kv_elem_bytes: int, out_elem_bytes: int) -> int:
    sl = _i32(seq_lens)
    return int(_load().oracle_decode_bytes(_ptr_i32(sl), sl.size, Hq, Hkv, D, block_size,
                                           kv_elem_bytes, out_elem_bytes))


def _problem(q, kpool, vpool, block_tables, seq_lens):
    q, dt = _storage(q)
    kpool, dk = _storage(kpool)
    vpool, dv = _storage(vpool)
    if not (dt == dk == dv):
        raise TypeError("oracle: q, K and V must share one storage type")
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = kpool.shape
    if D2 != D or vpool.shape != kpool.shape or bt.shape[0] != B or sl.shape != (B,):
        raise ValueError("oracle: inconsistent shapes")
    return q, kpool, vpool, bt, sl, dt, (B, Hq, Hkv, D, bs, NB, bt.shape[1])


def decode(q, kpool, vpool, block_tables, seq_lens, scale: float, pairs=None,
           nthreads: int | None = None) -> np.ndarray:
    """Paged decode attention in float64.

    Returns [B, Hq, D], or [len(pairs), D] for a list of (b, h) pairs.
    """
    q, kpool, vpool, bt, sl, dt, (B, Hq, Hkv, D, bs, NB, MB) = _problem(
        q, kpool, vpool, block_tables, seq_lens)
    nthreads = nthreads or os.cpu_count() or 1
    if pairs is None:
        out = np.empty((B, Hq, D), dtype=np.float64)
        pp, npairs = None, 0
    else:
        pr = _i32(pairs).reshape(-1, 2)
        out = np.empty((pr.shape[0], D), dtype=np.float64)
        pp, npairs = _ptr_i32(pr), pr.shape[0]
    rc = _load().oracle_decode(q.ctypes.data, kpool.ctypes.data, vpool.ctypes.data,
                               _ptr_i32(bt), MB, _ptr_i32(sl), B, Hq, Hkv, D, bs, NB,
                               float(scale), dt, _ptr_f64(out), pp, npairs, int(nthreads))
    _check(rc)
    return out


def weights(q, kpool, block_tables, seq_lens, scale: float, b: int, h: int) -> np.ndarray:
    """The L normalised softmax weights of (b, h)."""
    q, kpool, _, bt, sl, dt, (B, Hq, Hkv, D, bs, NB, MB) = _problem(
        q, kpool, kpool, block_tables, seq_lens)
    w = np.empty(int(sl[b]) if 0 <= b < B else 1, dtype=np.float64)
    rc = _load().oracle_weights(q.ctypes.data, kpool.ctypes.data, _ptr_i32(bt), MB, _ptr_i32(sl),
                                B, Hq, Hkv, D, bs, NB, float(scale), dt, int(b), int(h),
                                _ptr_f64(w))
    _check(rc)
    return w


def partial(q, kpool, vpool, block_tables, seq_lens, scale: float, b: int, h: int,
            t0: int, t1: int):
    """(m, l, acc[D]) over the tokens [t0, t1) of (b, h)."""
    q, kpool, vpool, bt, sl, dt, (B, Hq, Hkv, D, bs, NB, MB) = _problem(
        q, kpool, vpool, block_tables, seq_lens)
    m = np.zeros(1, dtype=np.float64)
    l = np.zeros(1, dtype=np.float64)
    acc = np.zeros(D, dtype=np.float64)
    rc = _load().oracle_partial(q.ctypes.data, kpool.ctypes.data, vpool.ctypes.data, _ptr_i32(bt),
                                MB, _ptr_i32(sl), B, Hq, Hkv, D, bs, NB, float(scale), dt,
                                int(b), int(h), int(t0), int(t1), _ptr_f64(m), _ptr_f64(l),
                                _ptr_f64(acc))
    _check(rc)
    return float(m[0]), float(l[0]), acc


def merge(ms, ls, accs) -> np.ndarray:
    """Fold partials in order with the two-partial rule and normalise."""
    m = np.ascontiguousarray(np.asarray(ms, dtype=np.float64))
    l = np.ascontiguousarray(np.asarray(ls, dtype=np.float64))
    a = np.ascontiguousarray(np.asarray(accs, dtype=np.float64))
    n, D = a.shape
    out = np.empty(D, dtype=np.float64)
    _check(_load().oracle_merge(n, _ptr_f64(m), _ptr_f64(l), _ptr_f64(a), D, _ptr_f64(out)))
    return out


def append(k_new, v_new, kpool: np.ndarray, vpool: np.ndarray, block_tables, cache_lens) -> None:
    """Write the new K/V rows into the pools in place (raw bit copy)."""
    if kpool.dtype != vpool.dtype or kpool.dtype not in (np.float32, np.uint16):
        raise TypeError("oracle: pools must be float32 or uint16 (bfloat16 bits)")
    if not (kpool.flags.c_contiguous and vpool.flags.c_contiguous):
        raise ValueError("oracle: pools must be contiguous")
    kn = np.ascontiguousarray(k_new, dtype=kpool.dtype)
    vn = np.ascontiguousarray(v_new, dtype=kpool.dtype)
    bt = _i32(block_tables)
    cl = _i32(cache_lens)
    NB, Hkv, bs, D = kpool.shape
    B = cl.shape[0]
    if kn.shape != (B, Hkv, D) or vn.shape != (B, Hkv, D) or bt.shape[0] != B:
        raise ValueError("oracle: inconsistent shapes")
    rc = _load().oracle_append(kn.ctypes.data, vn.ctypes.data, kpool.ctypes.data,
                               vpool.ctypes.data, _ptr_i32(bt), bt.shape[1], _ptr_i32(cl), B, Hkv,
                               D, bs, NB, kpool.dtype.itemsize)
    _check(rc)


def copy_blocks(kpool: np.ndarray, vpool: np.ndarray, src, dst) -> None:
    """Copy whole blocks src[i] -> dst[i] of both pools in place, in order."""
    if kpool.dtype != vpool.dtype or kpool.shape != vpool.shape:
        raise TypeError("oracle: pools must match")
    if not (kpool.flags.c_contiguous and vpool.flags.c_contiguous):
        raise ValueError("oracle: pools must be contiguous")
    s, d = _i32(src), _i32(dst)
    if s.shape != d.shape:
        raise ValueError("oracle: src and dst differ in length")
    NB = kpool.shape[0]
    block_bytes = kpool.nbytes // NB
    _check(_load().oracle_copy_blocks(kpool.ctypes.data, vpool.ctypes.data, _ptr_i32(s),
                                      _ptr_i32(d), s.size, NB, block_bytes))


def page_scores(kpool, vpool, block_tables, seq_lens):
    """Per-page mean of ||V||/||K|| and the page to evict (or -1) per sequence.

    Returns (scores float64 [B, max_blocks] with NaN past each sequence's
    pages, victims int32 [B]).
    """
    kpool, dk = _storage(kpool)
    vpool, dv = _storage(vpool)
    if dk != dv or kpool.shape != vpool.shape:
        raise TypeError("oracle: pools must match")
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    NB, Hkv, bs, D = kpool.shape
    B, MB = bt.shape
    scores = np.full((B, MB), np.nan, dtype=np.float64)
    victims = np.empty(B, dtype=np.int32)
    _check(_load().oracle_page_scores(kpool.ctypes.data, vpool.ctypes.data, _ptr_i32(bt), MB,
                                      _ptr_i32(sl), B, Hkv, D, bs, NB, dk, _ptr_f64(scores),
                                      _ptr_i32(victims)))
    return scores, victims


def prefill(q, kpool, vpool, block_tables, seq_lens, q_start, scale: float,
            nthreads: int | None = None) -> np.ndarray:
    """Causal paged multi-query attention in float64; returns [q_start[-1], Hq, D]."""
    q, dt = _storage(q)
    kpool, dk = _storage(kpool)
    vpool, dv = _storage(vpool)
    if not (dt == dk == dv):
        raise TypeError("oracle: q, K and V must share one storage type")
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    qs = _i32(q_start)
    T, Hq, D = q.shape
    NB, Hkv, bs, D2 = kpool.shape
    B, MB = bt.shape
    if D2 != D or qs.shape != (B + 1,) or int(qs[-1]) != T or sl.shape != (B,):
        raise ValueError("oracle: inconsistent shapes")
    out = np.empty((T, Hq, D), dtype=np.float64)
    nthreads = nthreads or os.cpu_count() or 1
    _check(_load().oracle_prefill(q.ctypes.data, kpool.ctypes.data, vpool.ctypes.data,
                                  _ptr_i32(bt), MB, _ptr_i32(sl), _ptr_i32(qs), B, Hq, Hkv, D, bs,
                                  NB, float(scale), dt, _ptr_f64(out), int(nthreads)))
    return out
