"""Paged decode attention on GB300 (sm_103a): Python binding of libpa.so.

The functions here carry the C-ABI names of ``include/pa.h`` and only
marshal arguments: torch tensors give device pointers, shapes and the current
CUDA stream; every step of the computation runs in the library's kernels.
There is no fallback: if ``libpa.so`` is missing, every call raises.

Layouts (contiguous, on one CUDA device):
    q            [B, Hq, D]               bf16 or float32 (the pool dtype)
    k_pool/v_pool [num_blocks, Hkv, block_size, D]
    block_tables int32 [B, max_blocks]
    seq_lens     int32 [B]   decode lengths (include the token appended this step)
    cache_lens   int32 [B]   append positions
    out          [B, Hq, D]               bf16 or float32
"""

from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "pa.h")

PA_OK, PA_ERR_NULL, PA_ERR_SHAPE, PA_ERR_DTYPE, PA_ERR_BLOCK_SIZE = 0, 1, 2, 3, 4
PA_ERR_WORKSPACE, PA_ERR_CUDA, PA_ERR_BOUNDS, PA_ERR_ALIGN, PA_ERR_NO_BLOCKS = 5, 6, 7, 8, 9
PA_F32, PA_BF16 = 0, 1
PA_DEVERR_SEQ_LEN, PA_DEVERR_TABLE, PA_DEVERR_TIMEOUT, PA_DEVERR_CACHE_LEN = 1, 2, 4, 8
PA_DEVERR_COPY = 16
PA_PATH_AUTO, PA_PATH_SIMPLE, PA_PATH_FMA, PA_PATH_MMA, PA_PATH_PREFILL = 0, 1, 2, 3, 4
PA_MERGE_AUTO, PA_MERGE_KERNEL, PA_MERGE_FUSED = 0, 1, 2
PA_SIMPLE_MAX_SEQ_LEN = 8192   # longest max_seq_len of the unsplit kernel (float32 pools)

_lib = None


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {pa_status_str(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded ``libpa.so`` (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.pa_append_kv.argtypes = [vp, vp, vp, vp, vp, ci, vp, ci, ci, ci, ci, ci, ci, vp]
    L.pa_append_kv.restype = ci
    L.pa_decode.argtypes = [vp, vp, vp, vp, ci, vp, ci, ci, ci, ci, ci, ci, ci, cf, ci, vp, ci,
                            ctypes.POINTER(vp), vp]
    L.pa_decode.restype = ci
    L.pa_append_decode.argtypes = [vp, vp, vp, vp, vp, vp, ci, vp, ci, ci, ci, ci, ci, ci, ci, cf,
                                   ci, vp, ci, ctypes.POINTER(vp), vp]
    L.pa_append_decode.restype = ci
    L.pa_free.argtypes = [vp]
    L.pa_free.restype = ci
    L.pa_status_str.argtypes = [ci]
    L.pa_status_str.restype = ctypes.c_char_p
    L.pa_last_device_error.argtypes = [vp, ctypes.POINTER(ci)]
    L.pa_last_device_error.restype = ci
    L.pa_plan_set_path.argtypes = [vp, ci]
    L.pa_plan_set_path.restype = ci
    L.pa_debug_set_wait_probe.argtypes = [ci]
    L.pa_debug_set_wait_probe.restype = ci
    L.pa_debug_set_prefill_kernel.argtypes = [ci]
    L.pa_debug_set_prefill_kernel.restype = ci
    L.pa_plan_set_merge.argtypes = [vp, ci]
    L.pa_plan_set_merge.restype = ci
    L.pa_plan_set_schedule.argtypes = [vp, ci, ci]
    L.pa_plan_set_schedule.restype = ci
    L.pa_plan_info.argtypes = [vp, ctypes.POINTER(ci), ctypes.POINTER(ci), ctypes.POINTER(ci)]
    L.pa_plan_info.restype = ci
    L.pa_plan_set_split_events.argtypes = [vp, vp, vp]
    L.pa_plan_set_split_events.restype = ci
    L.pa_decode_noalloc.argtypes = [vp, vp, vp, vp, ci, vp, ci, ci, ci, ci, ci, ci, ci, cf, ci, vp,
                                    ci, vp, vp]
    L.pa_decode_noalloc.restype = ci
    i32p = ctypes.POINTER(ctypes.c_int32)
    L.pa_copy_blocks.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, vp]
    L.pa_copy_blocks.restype = ci
    L.pa_bm_create.argtypes = [ci, ctypes.POINTER(vp)]
    L.pa_bm_destroy.argtypes = [vp]
    L.pa_bm_alloc.argtypes = [vp, ci, i32p]
    L.pa_bm_fork.argtypes = [vp, i32p, ci]
    L.pa_bm_release.argtypes = [vp, i32p, ci]
    L.pa_bm_refcount.argtypes = [vp, ctypes.c_int32, ctypes.POINTER(ci)]
    L.pa_bm_num_free.argtypes = [vp, ctypes.POINTER(ci)]
    L.pa_bm_prepare_append.argtypes = [vp, i32p, ci, ci, i32p, ci, i32p, i32p,
                                       ctypes.POINTER(ci)]
    L.pa_prefill.argtypes = [vp, vp, ci, vp, vp, vp, ci, vp, ci, ci, ci, ci, ci, ci, ci, ci, cf, ci,
                             vp, ci, vp, vp]
    L.pa_prefill.restype = ci
    L.pa_decode_multi.argtypes = [vp, vp, ci, ci, vp, vp, vp, ci, vp, ci, ci, ci, ci, ci, ci, ci, cf,
                                  ci, vp, ci, ctypes.POINTER(vp), vp]
    L.pa_decode_multi.restype = ci
    L.pa_page_scores.argtypes = [vp, vp, vp, ci, vp, ci, ci, ci, ci, ci, ci, ci, vp, vp, vp, vp]
    L.pa_page_scores.restype = ci
    for name in ("pa_bm_create", "pa_bm_destroy", "pa_bm_alloc", "pa_bm_fork", "pa_bm_release",
                 "pa_bm_refcount", "pa_bm_num_free", "pa_bm_prepare_append"):
        getattr(L, name).restype = ci
    _lib = L
    return L


def declared_functions() -> list[str]:
    """Names of the functions that ``include/pa.h`` declares."""
    with open(HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def pa_status_str(status: int) -> str:
    return lib().pa_status_str(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedAttentionError(status, what)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.float32:
        return PA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t: torch.Tensor) -> int:
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _on_one_device(*ts) -> None:
    """Every tensor the kernels read or write is CUDA memory of one device."""
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"tensors on {dev} and {t.device}: all must be on one device")


def _expect(t: torch.Tensor, name: str, shape: tuple, dtype: torch.dtype | None = None) -> None:
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} is {t.dtype}, expected {dtype}")


def _pools(k_pool: torch.Tensor, v_pool: torch.Tensor) -> tuple[int, int, int, int]:
    if k_pool.dim() != 4:
        raise ValueError("pools are [num_blocks, Hkv, block_size, D]")
    _expect(v_pool, "v_pool", tuple(k_pool.shape), k_pool.dtype)
    return tuple(k_pool.shape)


def _error_word(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if t.dtype != torch.int32 or t.numel() < 1:
        raise TypeError("device_error must be an int32 tensor of at least one element")
    return _ptr(t)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Plan:
    """Owner of a ``pa_plan*`` (split plan + device workspace)."""

    def __init__(self):
        self.handle = ctypes.c_void_p(None)

    def free(self) -> None:
        if self.handle.value:
            _check(lib().pa_free(self.handle), "pa_free")
            self.handle = ctypes.c_void_p(None)

    def set_path(self, path: int) -> None:
        _check(lib().pa_plan_set_path(self.handle, int(path)), "pa_plan_set_path")

    def set_merge(self, mode: int) -> None:
        """PA_MERGE_AUTO, PA_MERGE_KERNEL or PA_MERGE_FUSED for later decodes."""
        _check(lib().pa_plan_set_merge(self.handle, int(mode)), "pa_plan_set_merge")

    def set_schedule(self, dyn_permille: int, dyn_pages: int = 1) -> None:
        """Force the dynamic tail (per mille of the page stream, pages per piece);
        a negative share restores the automatic choice."""
        _check(lib().pa_plan_set_schedule(self.handle, int(dyn_permille), int(dyn_pages)),
               "pa_plan_set_schedule")

    def info(self) -> tuple[int, int, int]:
        p, b, w = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        _check(lib().pa_plan_info(self.handle, ctypes.byref(p), ctypes.byref(b), ctypes.byref(w)),
               "pa_plan_info")
        return p.value, b.value, w.value

    def set_split_events(self, start, stop) -> None:
        s = ctypes.c_void_p(start.cuda_event if start is not None else None)
        e = ctypes.c_void_p(stop.cuda_event if stop is not None else None)
        _check(lib().pa_plan_set_split_events(self.handle, s, e), "pa_plan_set_split_events")

    def last_device_error(self) -> int:
        return pa_last_device_error(self)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.free()


def _check_decode(q, k_pool, v_pool, block_tables, seq_lens, out, B: int) -> None:
    """Devices, dtypes and shapes shared by the attention calls (q and out
    have the same [rows, Hq, D] shape; q has the pools' element type)."""
    _on_one_device(q, k_pool, v_pool, block_tables, seq_lens, out)
    if q.dim() != 3:
        raise ValueError("q is [rows, Hq, D]")
    if q.dtype != k_pool.dtype:
        raise TypeError(f"q is {q.dtype}, the pools are {k_pool.dtype}")
    _expect(out, "out", tuple(q.shape))
    _expect(block_tables, "block_tables", (B, block_tables.shape[-1]), torch.int32)
    _expect(seq_lens, "seq_lens", (B,), torch.int32)


def pa_append_kv(k_new: torch.Tensor, v_new: torch.Tensor, k_pool: torch.Tensor,
                 v_pool: torch.Tensor, block_tables: torch.Tensor, cache_lens: torch.Tensor,
                 stream=None) -> None:
    """Write each sequence's new K/V token into its tail block (in place)."""
    NB, Hkv, bs, D = _pools(k_pool, v_pool)
    B = cache_lens.shape[0]
    _on_one_device(k_new, v_new, k_pool, v_pool, block_tables, cache_lens)
    _expect(k_new, "k_new", (B, Hkv, D), k_pool.dtype)
    _expect(v_new, "v_new", (B, Hkv, D), k_pool.dtype)
    _expect(cache_lens, "cache_lens", (B,), torch.int32)
    _expect(block_tables, "block_tables", (B, block_tables.shape[-1]), torch.int32)
    st = lib().pa_append_kv(_ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                            _ptr(block_tables), block_tables.shape[1], _ptr(cache_lens), B, Hkv,
                            D, bs, NB, _dtype(k_pool), _stream(stream))
    _check(st, "pa_append_kv")


def pa_decode(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
              block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
              out: torch.Tensor, max_seq_len: int, plan: Plan, stream=None) -> torch.Tensor:
    """Paged decode attention into ``out``; returns ``out``."""
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = _pools(k_pool, v_pool)
    _check_decode(q, k_pool, v_pool, block_tables, seq_lens, out, B)
    st = lib().pa_decode(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                         block_tables.shape[1], _ptr(seq_lens), B, Hq, Hkv, D, bs, NB,
                         int(max_seq_len), float(scale), _dtype(k_pool), _ptr(out), _dtype(out),
                         ctypes.byref(plan.handle), _stream(stream))
    _check(st, "pa_decode")
    return out


def pa_append_decode(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                     k_pool: torch.Tensor, v_pool: torch.Tensor, block_tables: torch.Tensor,
                     seq_lens: torch.Tensor, scale: float, out: torch.Tensor, max_seq_len: int,
                     plan: Plan, stream=None) -> torch.Tensor:
    """One decode step in one call: append the new K/V token of every sequence
    at position ``seq_lens[b] - 1`` (in place), then decode into ``out``."""
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = _pools(k_pool, v_pool)
    _check_decode(q, k_pool, v_pool, block_tables, seq_lens, out, B)
    _on_one_device(q, k_new, v_new)
    _expect(k_new, "k_new", (B, Hkv, D), k_pool.dtype)
    _expect(v_new, "v_new", (B, Hkv, D), k_pool.dtype)
    st = lib().pa_append_decode(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                                _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B, Hq,
                                Hkv, D, bs, NB, int(max_seq_len), float(scale), _dtype(k_pool),
                                _ptr(out), _dtype(out), ctypes.byref(plan.handle), _stream(stream))
    _check(st, "pa_append_decode")
    return out


def pa_decode_multi(q: torch.Tensor, q_start: torch.Tensor, k_pool: torch.Tensor,
                    v_pool: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                    scale: float, out: torch.Tensor, max_q: int, max_seq_len: int, plan: Plan,
                    stream=None) -> torch.Tensor:
    """Decode attention for a few new queries per sequence into ``out``; returns ``out``.

    ``q`` and ``out`` are ``[T, Hq, D]`` with sequence b's queries (its
    newest tokens) at rows ``q_start[b] .. q_start[b+1]``; ``q_start`` is a
    device int32 tensor of B + 1 entries and ``max_q`` bounds every count.
    """
    T, Hq, D = q.shape
    NB, Hkv, bs, _ = _pools(k_pool, v_pool)
    B = seq_lens.shape[0]
    _check_decode(q, k_pool, v_pool, block_tables, seq_lens, out, B)
    _on_one_device(q, q_start)
    _expect(q_start, "q_start", (B + 1,), torch.int32)
    st = lib().pa_decode_multi(_ptr(q), _ptr(q_start), T, int(max_q), _ptr(k_pool), _ptr(v_pool),
                               _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B, Hq,
                               Hkv, D, bs, NB, int(max_seq_len), float(scale), _dtype(k_pool),
                               _ptr(out), _dtype(out), ctypes.byref(plan.handle), _stream(stream))
    _check(st, "pa_decode_multi")
    return out


def pa_decode_noalloc(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                      out: torch.Tensor, max_seq_len: int, device_error: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """``pa_decode`` without a plan: the library allocates nothing (bf16 pools).

    For callers that manage all device memory themselves. ``device_error``, if
    given, is an int32 device tensor of one element that receives error bits.
    """
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = _pools(k_pool, v_pool)
    _check_decode(q, k_pool, v_pool, block_tables, seq_lens, out, B)
    _on_one_device(q, device_error)
    err = _error_word(device_error)
    st = lib().pa_decode_noalloc(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                 block_tables.shape[1], _ptr(seq_lens), B, Hq, Hkv, D, bs, NB,
                                 int(max_seq_len), float(scale), _dtype(k_pool), _ptr(out),
                                 _dtype(out), err, _stream(stream))
    _check(st, "pa_decode_noalloc")
    return out


def pa_copy_blocks(k_pool: torch.Tensor, v_pool: torch.Tensor, copy_src: torch.Tensor,
                   copy_dst: torch.Tensor, stream=None) -> None:
    """Copy whole blocks copy_src[i] -> copy_dst[i] of both pools (int32 device tensors)."""
    NB, Hkv, bs, D = _pools(k_pool, v_pool)
    n = copy_src.numel()
    _on_one_device(k_pool, v_pool, copy_src, copy_dst)
    _expect(copy_src, "copy_src", (n,), torch.int32)
    _expect(copy_dst, "copy_dst", (n,), torch.int32)
    st = lib().pa_copy_blocks(_ptr(k_pool), _ptr(v_pool), _ptr(copy_src) if n else None,
                              _ptr(copy_dst) if n else None, n, Hkv, D, bs, NB, _dtype(k_pool),
                              _stream(stream))
    _check(st, "pa_copy_blocks")


def pa_prefill(q: torch.Tensor, q_start: torch.Tensor, k_pool: torch.Tensor,
               v_pool: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
               scale: float, out: torch.Tensor, max_q: int, max_seq_len: int,
               device_error: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Causal paged multi-query attention (bf16 pools, D = 128); returns ``out``."""
    T, Hq, D = q.shape
    NB, Hkv, bs, _ = _pools(k_pool, v_pool)
    B, MB = block_tables.shape
    _check_decode(q, k_pool, v_pool, block_tables, seq_lens, out, B)
    _on_one_device(q, q_start, device_error)
    _expect(q_start, "q_start", (B + 1,), torch.int32)
    err = _error_word(device_error)
    st = lib().pa_prefill(_ptr(q), _ptr(q_start), T, _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                          MB, _ptr(seq_lens), B, Hq, Hkv, D, bs, NB, int(max_q),
                          int(max_seq_len), float(scale), _dtype(k_pool), _ptr(out), _dtype(out),
                          err, _stream(stream))
    _check(st, "pa_prefill")
    return out


def pa_page_scores(k_pool: torch.Tensor, v_pool: torch.Tensor, block_tables: torch.Tensor,
                   seq_lens: torch.Tensor, max_seq_len: int, scores: torch.Tensor,
                   victims: torch.Tensor, device_error: torch.Tensor | None = None,
                   stream=None) -> None:
    """PagedEviction page scores (float32 [B, max_blocks]) and victims (int32 [B])."""
    NB, Hkv, bs, D = _pools(k_pool, v_pool)
    B, MB = block_tables.shape
    _on_one_device(k_pool, v_pool, block_tables, seq_lens, scores, victims, device_error)
    _expect(block_tables, "block_tables", (B, MB), torch.int32)
    _expect(seq_lens, "seq_lens", (B,), torch.int32)
    _expect(scores, "scores", (B, MB), torch.float32)
    _expect(victims, "victims", (B,), torch.int32)
    err = _error_word(device_error)
    st = lib().pa_page_scores(_ptr(k_pool), _ptr(v_pool), _ptr(block_tables), MB, _ptr(seq_lens),
                              B, Hkv, D, bs, NB, int(max_seq_len), _dtype(k_pool), _ptr(scores),
                              _ptr(victims), err, _stream(stream))
    _check(st, "pa_page_scores")


class BlockManager:
    """Host block manager (``pa_bm_*``): O(1) free list, reference counts, copy on write.

    Arrays are numpy int32 (host memory).
    """

    def __init__(self, num_blocks: int):
        import numpy as np  # noqa: F401  (arrays below)
        self.handle = ctypes.c_void_p(None)
        _check(lib().pa_bm_create(int(num_blocks), ctypes.byref(self.handle)), "pa_bm_create")

    @staticmethod
    def _i32p(a):
        return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    def close(self) -> None:
        if self.handle.value:
            lib().pa_bm_destroy(self.handle)
            self.handle = ctypes.c_void_p(None)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def alloc(self, n: int):
        import numpy as np
        ids = np.empty(max(n, 1), dtype=np.int32)
        _check(lib().pa_bm_alloc(self.handle, int(n), self._i32p(ids)), "pa_bm_alloc")
        return ids[:n]

    def fork(self, ids) -> None:
        import numpy as np
        a = np.ascontiguousarray(ids, dtype=np.int32)
        _check(lib().pa_bm_fork(self.handle, self._i32p(a), a.size), "pa_bm_fork")

    def release(self, ids) -> None:
        import numpy as np
        a = np.ascontiguousarray(ids, dtype=np.int32)
        _check(lib().pa_bm_release(self.handle, self._i32p(a), a.size), "pa_bm_release")

    def refcount(self, block: int) -> int:
        c = ctypes.c_int()
        _check(lib().pa_bm_refcount(self.handle, int(block), ctypes.byref(c)), "pa_bm_refcount")
        return c.value

    @property
    def num_free(self) -> int:
        c = ctypes.c_int()
        _check(lib().pa_bm_num_free(self.handle, ctypes.byref(c)), "pa_bm_num_free")
        return c.value

    def prepare_append(self, tables, cache_lens, block_size: int):
        """Make each append target private; tables (host int32 [B, MB]) change in place.

        Returns (copy_src, copy_dst) int32 arrays of the copy-on-write pairs.
        """
        import numpy as np
        if not (tables.dtype == np.int32 and tables.flags.c_contiguous):
            raise ValueError("tables must be a contiguous int32 array")
        cl = np.ascontiguousarray(cache_lens, dtype=np.int32)
        B, MB = tables.shape
        src = np.empty(max(B, 1), dtype=np.int32)
        dst = np.empty(max(B, 1), dtype=np.int32)
        n = ctypes.c_int(0)
        _check(lib().pa_bm_prepare_append(self.handle, self._i32p(tables), B, MB, self._i32p(cl),
                                          int(block_size), self._i32p(src), self._i32p(dst),
                                          ctypes.byref(n)), "pa_bm_prepare_append")
        return src[:n.value].copy(), dst[:n.value].copy()


def pa_debug_set_wait_probe(enable: bool) -> None:
    """Test hook: while on, each kernel's first pipeline wait expires (bounded),
    so the kernel reports PA_DEVERR_TIMEOUT and takes its give-up path."""
    _check(lib().pa_debug_set_wait_probe(1 if enable else 0), "pa_debug_set_wait_probe")


PA_PREFILL_AUTO, PA_PREFILL_ONE_TILE, PA_PREFILL_TWO_TILE = 0, 1, 2


def pa_debug_set_prefill_kernel(which: int) -> None:
    """Test hook: pin the prefill kernel (PA_PREFILL_ONE_TILE / _TWO_TILE) or
    restore the shape-based choice (PA_PREFILL_AUTO)."""
    _check(lib().pa_debug_set_prefill_kernel(int(which)), "pa_debug_set_prefill_kernel")


def pa_free(plan: Plan) -> None:
    plan.free()


def pa_last_device_error(plan: Plan | None) -> int:
    err = ctypes.c_int(0)
    h = plan.handle if plan is not None else ctypes.c_void_p(None)
    _check(lib().pa_last_device_error(h, ctypes.byref(err)), "pa_last_device_error")
    return err.value


def decode_bytes(seq_lens, Hq: int, Hkv: int, D: int, block_size: int, kv_elem_bytes: int,
                 out_elem_bytes: int) -> int:
    """Algorithmic HBM bytes of one decode call (the roofline numerator).

    Every attended K and V element once, one 4-byte table entry per attended
    block, the queries, the lengths and the output.
    """
    total = 0
    for L in (int(x) for x in seq_lens):
        total += 2 * Hkv * D * L * kv_elem_bytes + 4 * (-(-L // block_size))
    B = len(seq_lens)
    return total + B * Hq * D * kv_elem_bytes + 4 * B + B * Hq * D * out_elem_bytes


def append_bytes(B: int, Hkv: int, D: int, kv_elem_bytes: int) -> int:
    """Algorithmic bytes of one append: new K/V rows read and written, lengths, table entries."""
    return 2 * (2 * B * Hkv * D * kv_elem_bytes) + 4 * B + 4 * B
