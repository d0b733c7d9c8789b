"""ctypes binding of libpagedgqa.so, one Python function per C entry point.

Argument marshalling only: shapes are read off the torch tensors, pointers
and the current CUDA stream are passed through, return codes become
exceptions.  Every step of the computation runs in the library's kernels;
there is no other code path.  If the library is not built, every call raises
``LibraryNotBuilt``.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedgqa.so")

PA_OK = 0
PA_ERR_NULL = -1
PA_ERR_SHAPE = -2
PA_ERR_ALIGN = -3
PA_ERR_WORKSPACE = -4
PA_ERR_CUDA = -5
PA_ERR_OPTION = -6
PA_ERR_SCRATCH_LIMIT = -7
PA_ERR_STATE = -8
PA_ERR_NO_BLOCKS = -9

PA_MAX_QUERY_TOKENS = 4096
PA_MAX_BATCH = 8192  # include/pagedgqa.h: sequences per call
PA_STATIC_SCRATCH_BYTES = 8 << 20  # include/pagedgqa.h: pa_decode_noalloc scratch

PA_BM_FREE_BLOCKS = 0
PA_BM_REF_COUNT = 1
PA_BM_SEQ_BLOCKS = 2

PA_STATUS_BAD_BLOCK = 0x1
PA_STATUS_BAD_SEQLEN = 0x2
PA_STATUS_TIMEOUT = 0x4
PA_STATUS_NO_SLOT = 0x8

PA_F16 = 0
PA_BF16 = 1

PA_COMPUTE_AUTO = 0
PA_COMPUTE_SIMT = 1
PA_COMPUTE_MMA = 2
PA_COMPUTE_TC = 3
_COMPUTE = {"auto": PA_COMPUTE_AUTO, "simt": PA_COMPUTE_SIMT, "mma": PA_COMPUTE_MMA,
            "tc": PA_COMPUTE_TC}

# Every symbol include/pagedgqa.h declares.
EXPORTS = ("pa_workspace_size", "pa_decode", "pa_decode_split", "pa_decode_merge",
           "pa_cache_append", "pa_read_status", "pa_status_string", "pa_plan_pieces",
           "pa_plan_merge", "pa_version", "pa_decode_noalloc", "pa_decode_append",
           "pa_bm_create", "pa_bm_destroy", "pa_bm_allocate", "pa_bm_free_sequence",
           "pa_bm_share_prefix", "pa_bm_copy_on_write", "pa_bm_reserve_slot",
           "pa_bm_block_table", "pa_bm_query", "pa_copy_blocks", "pa_decode_multi",
           "pa_workspace_size_multi", "pa_decode_host", "pa_workspace_size_host",
           "pa_decode_multi_host", "pa_workspace_size_multi_host", "pa_decode_host_async",
           "pa_workspace_size_host_async", "pa_decode_multi_host_async",
           "pa_workspace_size_multi_host_async", "pa_launch_plan")


class LibraryNotBuilt(RuntimeError):
    pass


class PagedGQAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (code {code})")


class pa_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("dtype", ctypes.c_int32)]


PA_PHASE_BOTH = 0
PA_PHASE_SPLIT = 1
PA_PHASE_MERGE = 2


class pa_options(ctypes.Structure):
    _fields_ = [("partition_tokens", ctypes.c_int32), ("compute", ctypes.c_int32),
                ("num_ctas", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("phase", ctypes.c_int32), ("wait_limit_us", ctypes.c_int32),
                ("stall_test", ctypes.c_int32)]


def options(partition_tokens: int = 0, compute: str = "auto", num_ctas: int = 0,
            stages: int = 0, phase: int = PA_PHASE_BOTH, wait_limit_us: int = 0,
            stall_test: int = 0) -> pa_options:
    return pa_options(int(partition_tokens), _COMPUTE[compute] if isinstance(compute, str)
                      else int(compute), int(num_ctas), int(stages), int(phase),
                      int(wait_limit_us), int(stall_test))


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded library (raises LibraryNotBuilt if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise LibraryNotBuilt(
                f"{LIB_PATH} is missing: build it with "
                "`python -m paged_gqa_decode_pa_gb300.build` (or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        SP = ctypes.POINTER(pa_shape)
        OP = ctypes.POINTER(pa_options)
        i32 = ctypes.c_int32
        L.pa_workspace_size.argtypes = [SP, OP, ctypes.POINTER(ctypes.c_size_t)]
        L.pa_workspace_size.restype = ctypes.c_int
        for name in ("pa_decode", "pa_decode_split", "pa_decode_merge"):
            fn = getattr(L, name)
            fn.argtypes = [SP, OP, P, P, P, P, P, ctypes.c_float, P, P, ctypes.c_size_t, P]
            fn.restype = ctypes.c_int
        L.pa_decode_append.argtypes = [SP, OP, P, P, P, P, P, P, P, ctypes.c_float, P, P,
                                       ctypes.c_size_t, P]
        L.pa_decode_append.restype = ctypes.c_int
        L.pa_decode_noalloc.argtypes = [SP, OP, P, P, P, P, P, ctypes.c_float, P, P, P]
        L.pa_decode_noalloc.restype = ctypes.c_int
        L.pa_cache_append.argtypes = [SP, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.pa_cache_append.restype = ctypes.c_int
        L.pa_read_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
        L.pa_read_status.restype = ctypes.c_int
        L.pa_status_string.argtypes = [ctypes.c_int]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_plan_pieces.argtypes = [SP, OP, P, i32, i32, P, i32]
        L.pa_plan_pieces.restype = ctypes.c_int
        L.pa_plan_merge.argtypes = [SP, OP, P, i32, i32, P, P, i32]
        L.pa_plan_merge.restype = ctypes.c_int
        L.pa_bm_create.argtypes = [i32, i32, i32, i32]
        L.pa_bm_create.restype = P
        L.pa_bm_destroy.argtypes = [P]
        L.pa_bm_destroy.restype = None
        L.pa_bm_allocate.argtypes = [P, i32, i32]
        L.pa_bm_free_sequence.argtypes = [P, i32]
        L.pa_bm_share_prefix.argtypes = [P, i32, i32, i32]
        for name in ("pa_bm_copy_on_write", "pa_bm_reserve_slot"):
            getattr(L, name).argtypes = [P, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        L.pa_bm_block_table.argtypes = [P, P, i32, i32, P]
        L.pa_bm_query.argtypes = [P, i32, i32]
        for name in ("pa_bm_allocate", "pa_bm_free_sequence", "pa_bm_share_prefix",
                     "pa_bm_copy_on_write", "pa_bm_reserve_slot", "pa_bm_block_table",
                     "pa_bm_query"):
            getattr(L, name).restype = ctypes.c_int
        L.pa_copy_blocks.argtypes = [SP, P, P, P, i32, P, P]
        L.pa_copy_blocks.restype = ctypes.c_int
        L.pa_workspace_size_multi.argtypes = [SP, OP, i32, ctypes.POINTER(ctypes.c_size_t)]
        L.pa_workspace_size_multi.restype = ctypes.c_int
        L.pa_decode_multi.argtypes = [SP, OP, P, P, i32, i32, i32, P, P, P, P, ctypes.c_float, P,
                                      P, ctypes.c_size_t, P]
        L.pa_decode_multi.restype = ctypes.c_int
        L.pa_workspace_size_host.argtypes = [SP, OP, ctypes.POINTER(ctypes.c_size_t)]
        L.pa_workspace_size_host.restype = ctypes.c_int
        L.pa_decode_host.argtypes = [SP, OP, P, P, P, P, P, ctypes.c_float, P, P, P,
                                     ctypes.c_size_t, P]
        L.pa_decode_host.restype = ctypes.c_int
        L.pa_workspace_size_multi_host.argtypes = [SP, OP, i32, i32,
                                                   ctypes.POINTER(ctypes.c_size_t)]
        L.pa_workspace_size_multi_host.restype = ctypes.c_int
        L.pa_decode_multi_host.argtypes = [SP, OP, P, P, i32, i32, i32, P, P, P, P,
                                           ctypes.c_float, P, P, P, ctypes.c_size_t, P]
        L.pa_decode_multi_host.restype = ctypes.c_int
        L.pa_workspace_size_host_async.argtypes = [SP, OP, ctypes.POINTER(ctypes.c_size_t)]
        L.pa_workspace_size_host_async.restype = ctypes.c_int
        L.pa_decode_host_async.argtypes = [SP, OP, P, P, P, P, P, ctypes.c_float, P, P, i32, P,
                                           ctypes.c_size_t, P]
        L.pa_decode_host_async.restype = ctypes.c_int
        L.pa_workspace_size_multi_host_async.argtypes = [SP, OP, i32, i32,
                                                         ctypes.POINTER(ctypes.c_size_t)]
        L.pa_workspace_size_multi_host_async.restype = ctypes.c_int
        L.pa_decode_multi_host_async.argtypes = [SP, OP, P, P, i32, i32, i32, P, P, P, P,
                                                 ctypes.c_float, P, P, i32, P, ctypes.c_size_t, P]
        L.pa_decode_multi_host_async.restype = ctypes.c_int
        L.pa_launch_plan.argtypes = [SP, OP, i32, ctypes.POINTER(i32)]
        L.pa_launch_plan.restype = ctypes.c_int
        L.pa_version.argtypes = []
        L.pa_version.restype = ctypes.c_int
        _lib = L
        return L


def status_string(code: int) -> str:
    try:
        return lib().pa_status_string(int(code)).decode()
    except LibraryNotBuilt:
        return f"code {code}"


def _check(rc: int, where: str):
    if rc != PA_OK:
        raise PagedGQAError(rc, where)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"q/k/v must be float16 or bfloat16, got {t.dtype}")


def shape_of(q, k_cache, block_table) -> pa_shape:
    """pa_shape from q [B,H,d], k_cache [P,bs,Hkv,d], block_table [B,maxblk]."""
    B, H, d = q.shape
    P, bs, Hkv, d2 = k_cache.shape
    if d2 != d or block_table.shape[0] != B:
        raise ValueError("inconsistent q / k_cache / block_table shapes")
    return pa_shape(B, H, Hkv, d, bs, block_table.shape[1], P, _dtype_code(q))


def _check_tensors(q, k_cache, v_cache, block_table, cache_seqlens, out):
    import torch

    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("block_table", block_table), ("cache_seqlens", cache_seqlens),
                    ("out", out)):
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if k_cache is not None and (k_cache.dtype != q.dtype or v_cache.dtype != q.dtype
                                or v_cache.shape != k_cache.shape):
        raise ValueError("q, k_cache and v_cache must share dtype; k/v shapes must match")
    if block_table.dtype != torch.int32 or cache_seqlens.dtype != torch.int32:
        raise TypeError("block_table and cache_seqlens must be int32")
    if out is not None and (out.dtype != torch.float32 or tuple(out.shape) != tuple(q.shape)):
        raise TypeError("out must be float32 with q's shape")


def pa_launch_plan(shape: pa_shape, opts: Optional[pa_options] = None, max_q: int = 0) -> dict:
    """Which kernels a step launches on the current device (see
    include/pagedgqa.h): kernels per step, CTAs of the first kernel, CTAs per
    cluster (0 = none), ring slots per warp."""
    info = (ctypes.c_int32 * 4)()
    rc = lib().pa_launch_plan(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                              int(max_q), info)
    _check(rc, "pa_launch_plan")
    return {"kernels": int(info[0]), "ctas": int(info[1]), "cluster": int(info[2]),
            "ring": int(info[3])}


def pa_workspace_size(shape: pa_shape, opts: Optional[pa_options] = None) -> int:
    n = ctypes.c_size_t(0)
    rc = lib().pa_workspace_size(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                                 ctypes.byref(n))
    _check(rc, "pa_workspace_size")
    return int(n.value)


def alloc_workspace(shape: pa_shape, opts: Optional[pa_options] = None, device=None):
    """Zero-filled device workspace of pa_workspace_size bytes (torch uint8)."""
    import torch

    return torch.zeros(pa_workspace_size(shape, opts), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def shape_multi(q, k_cache, block_table) -> pa_shape:
    """pa_shape of a call with several query tokens per sequence: q is the
    packed [total_q, H, d]; B is the number of block-table rows."""
    _, H, d = q.shape
    P, bs, Hkv, d2 = k_cache.shape
    if d2 != d:
        raise ValueError("inconsistent q / k_cache shapes")
    return pa_shape(block_table.shape[0], H, Hkv, d, bs, block_table.shape[1], P, _dtype_code(q))


def pa_workspace_size_multi(shape: pa_shape, max_q: int,
                            opts: Optional[pa_options] = None) -> int:
    n = ctypes.c_size_t(0)
    rc = lib().pa_workspace_size_multi(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                                       int(max_q), ctypes.byref(n))
    _check(rc, "pa_workspace_size_multi")
    return int(n.value)


def alloc_workspace_multi(shape: pa_shape, max_q: int, opts: Optional[pa_options] = None,
                          device=None):
    """Zero-filled device workspace for pa_decode_multi (torch uint8)."""
    import torch

    return torch.zeros(pa_workspace_size_multi(shape, max_q, opts), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def pa_decode_multi(q, cu_seqlens_q, max_q, causal, k_cache, v_cache, block_table,
                    cache_seqlens, scale, out, workspace, opts: Optional[pa_options] = None,
                    stream=None) -> None:
    """out[total_q,H,d] (fp32) = attention of the packed query rows q
    [total_q,H,d]; sequence b owns rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
    (see include/pagedgqa.h)."""
    import torch

    _check_tensors(q, k_cache, v_cache, block_table, cache_seqlens, out)
    if not cu_seqlens_q.is_cuda or cu_seqlens_q.dtype != torch.int32:
        raise TypeError("cu_seqlens_q must be an int32 CUDA tensor")
    if tuple(cu_seqlens_q.shape) != (block_table.shape[0] + 1,):
        raise ValueError("cu_seqlens_q must be [B + 1]")
    shape = shape_multi(q, k_cache, block_table)
    rc = lib().pa_decode_multi(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                               _ptr(q), _ptr(cu_seqlens_q), int(q.shape[0]), int(max_q),
                               int(bool(causal)), _ptr(k_cache), _ptr(v_cache),
                               _ptr(block_table), _ptr(cache_seqlens), float(scale), _ptr(out),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream))
    _check(rc, "pa_decode_multi")


def _check_host(q, block_table, cache_seqlens, out, k_cache, v_cache, extra=()):
    import torch

    for name, t in (("q", q), ("block_table", block_table), ("cache_seqlens", cache_seqlens),
                    ("out", out)) + tuple(extra):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host (CPU) tensor")
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if k_cache.dtype != q.dtype or v_cache.dtype != q.dtype or v_cache.shape != k_cache.shape:
        raise ValueError("q, k_cache and v_cache must share dtype; k/v shapes must match")
    if block_table.dtype != torch.int32 or cache_seqlens.dtype != torch.int32:
        raise TypeError("block_table and cache_seqlens must be int32")
    if out.dtype != torch.float32 or tuple(out.shape) != tuple(q.shape):
        raise TypeError("out must be float32 with q's shape")


_tls = threading.local()


def _status_word():
    """This thread's page-locked host word that the host-buffer calls have
    the device publish their status into (no copy back needed), and a numpy
    view of it for reading."""
    import torch

    word = getattr(_tls, "status", None)
    if word is None:
        t = torch.zeros(1, dtype=torch.int32).pin_memory()
        word = (t, t.numpy().view("uint32"))
        _tls.status = word
    return word


def pa_workspace_size_host(shape: pa_shape, opts: Optional[pa_options] = None) -> int:
    n = ctypes.c_size_t(0)
    rc = lib().pa_workspace_size_host(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                                      ctypes.byref(n))
    _check(rc, "pa_workspace_size_host")
    return int(n.value)


def alloc_workspace_host(shape: pa_shape, opts: Optional[pa_options] = None, device=None):
    """Zero-filled device workspace for pa_decode_host (torch uint8)."""
    import torch

    return torch.zeros(pa_workspace_size_host(shape, opts), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def pa_decode_host(q, k_cache, v_cache, block_table, cache_seqlens, scale, out, workspace,
                   opts: Optional[pa_options] = None, stream=None) -> int:
    """pa_decode with q, block_table, cache_seqlens and out in host memory
    (CPU tensors; pinned ones copy fastest) and the pools on the device.
    Returns after out is filled; the result is this call's device status
    bits (0 = all well).  See include/pagedgqa.h."""
    _check_host(q, block_table, cache_seqlens, out, k_cache, v_cache)
    shape = shape_of(q, k_cache, block_table)
    st, view = _status_word()
    rc = lib().pa_decode_host(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                              _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                              _ptr(cache_seqlens), float(scale), _ptr(out), st.data_ptr(),
                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _stream(stream))
    _check(rc, "pa_decode_host")
    return int(view[0])


def pa_workspace_size_multi_host(shape: pa_shape, max_q: int, max_total_q: int,
                                 opts: Optional[pa_options] = None) -> int:
    n = ctypes.c_size_t(0)
    rc = lib().pa_workspace_size_multi_host(ctypes.byref(shape),
                                            ctypes.byref(opts) if opts else None, int(max_q),
                                            int(max_total_q), ctypes.byref(n))
    _check(rc, "pa_workspace_size_multi_host")
    return int(n.value)


def alloc_workspace_multi_host(shape: pa_shape, max_q: int, max_total_q: int,
                               opts: Optional[pa_options] = None, device=None):
    """Zero-filled device workspace for pa_decode_multi_host (torch uint8)."""
    import torch

    return torch.zeros(pa_workspace_size_multi_host(shape, max_q, max_total_q, opts),
                       dtype=torch.uint8, device=device if device is not None else "cuda")


def pa_decode_multi_host(q, cu_seqlens_q, max_q, causal, k_cache, v_cache, block_table,
                         cache_seqlens, scale, out, workspace, opts: Optional[pa_options] = None,
                         stream=None) -> int:
    """pa_decode_multi with q, cu_seqlens_q, block_table, cache_seqlens and out
    in host memory; returns this call's device status bits."""
    import torch

    _check_host(q, block_table, cache_seqlens, out, k_cache, v_cache,
                (("cu_seqlens_q", cu_seqlens_q),))
    if cu_seqlens_q.dtype != torch.int32 or tuple(cu_seqlens_q.shape) != (block_table.shape[0] + 1,):
        raise TypeError("cu_seqlens_q must be int32 [B + 1]")
    shape = shape_multi(q, k_cache, block_table)
    st, view = _status_word()
    rc = lib().pa_decode_multi_host(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                                    _ptr(q), _ptr(cu_seqlens_q), int(q.shape[0]), int(max_q),
                                    int(bool(causal)), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(block_table), _ptr(cache_seqlens), float(scale),
                                    _ptr(out), st.data_ptr(), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "pa_decode_multi_host")
    return int(view[0])


class _BoundCall:
    """One library entry point with its arguments marshalled once; calling
    it runs that entry point again on the same buffers (whose contents may
    have changed) and returns the call's device status bits.  Holds
    references to every tensor it points at."""

    def __init__(self, fn, name, args, keep, status):
        self._fn, self._name, self._args, self._keep = fn, name, args, keep
        self._status = status

    def __call__(self) -> int:
        rc = self._fn(*self._args)
        if rc != PA_OK:
            raise PagedGQAError(rc, self._name)
        return int(self._status[1][0])


def bind_decode_host(q, k_cache, v_cache, block_table, cache_seqlens, scale, out, workspace,
                     opts: Optional[pa_options] = None, stream=None) -> _BoundCall:
    """pa_decode_host on these buffers, checked and marshalled once: the
    returned callable runs one step per call (a serving loop rewrites q, the
    table and the lengths in place between steps) and returns its status.
    The stream (the current one when None) is taken at bind time."""
    _check_host(q, block_table, cache_seqlens, out, k_cache, v_cache)
    shape = shape_of(q, k_cache, block_table)
    st = _status_word()
    V = ctypes.c_void_p
    opt = pa_options.from_buffer_copy(opts) if opts else None
    args = (ctypes.byref(shape), ctypes.byref(opt) if opt else None, V(_ptr(q)), V(_ptr(k_cache)),
            V(_ptr(v_cache)), V(_ptr(block_table)), V(_ptr(cache_seqlens)),
            ctypes.c_float(scale), V(_ptr(out)), V(st[0].data_ptr()), V(_ptr(workspace)),
            ctypes.c_size_t(workspace.numel() * workspace.element_size()), V(_stream(stream)))
    keep = (shape, opt, q, k_cache, v_cache, block_table, cache_seqlens, out, workspace, st)
    return _BoundCall(lib().pa_decode_host, "pa_decode_host", args, keep, st)


def bind_decode_multi_host(q, cu_seqlens_q, max_q, causal, k_cache, v_cache, block_table,
                           cache_seqlens, scale, out, workspace,
                           opts: Optional[pa_options] = None, stream=None) -> _BoundCall:
    """pa_decode_multi_host on these buffers, checked and marshalled once
    (as bind_decode_host; total_q is q's row count, the stream is taken at
    bind time)."""
    import torch

    _check_host(q, block_table, cache_seqlens, out, k_cache, v_cache,
                (("cu_seqlens_q", cu_seqlens_q),))
    if cu_seqlens_q.dtype != torch.int32 or tuple(cu_seqlens_q.shape) != (block_table.shape[0] + 1,):
        raise TypeError("cu_seqlens_q must be int32 [B + 1]")
    shape = shape_multi(q, k_cache, block_table)
    st = _status_word()
    V = ctypes.c_void_p
    i32 = ctypes.c_int32
    opt = pa_options.from_buffer_copy(opts) if opts else None
    args = (ctypes.byref(shape), ctypes.byref(opt) if opt else None, V(_ptr(q)),
            V(_ptr(cu_seqlens_q)), i32(q.shape[0]), i32(max_q), i32(int(bool(causal))),
            V(_ptr(k_cache)), V(_ptr(v_cache)), V(_ptr(block_table)), V(_ptr(cache_seqlens)),
            ctypes.c_float(scale), V(_ptr(out)), V(st[0].data_ptr()), V(_ptr(workspace)),
            ctypes.c_size_t(workspace.numel() * workspace.element_size()), V(_stream(stream)))
    keep = (shape, opt, q, cu_seqlens_q, k_cache, v_cache, block_table, cache_seqlens, out,
            workspace, st)
    return _BoundCall(lib().pa_decode_multi_host, "pa_decode_multi_host", args, keep, st)


def pa_workspace_size_host_async(shape: pa_shape, opts: Optional[pa_options] = None) -> int:
    n = ctypes.c_size_t(0)
    rc = lib().pa_workspace_size_host_async(ctypes.byref(shape),
                                            ctypes.byref(opts) if opts else None, ctypes.byref(n))
    _check(rc, "pa_workspace_size_host_async")
    return int(n.value)


def alloc_workspace_host_async(shape: pa_shape, opts: Optional[pa_options] = None, device=None):
    """Zero-filled device workspace for pa_decode_host_async (two staging slots)."""
    import torch

    return torch.zeros(pa_workspace_size_host_async(shape, opts), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def pa_workspace_size_multi_host_async(shape: pa_shape, max_q: int, max_total_q: int,
                                       opts: Optional[pa_options] = None) -> int:
    n = ctypes.c_size_t(0)
    rc = lib().pa_workspace_size_multi_host_async(ctypes.byref(shape),
                                                  ctypes.byref(opts) if opts else None,
                                                  int(max_q), int(max_total_q), ctypes.byref(n))
    _check(rc, "pa_workspace_size_multi_host_async")
    return int(n.value)


def alloc_workspace_multi_host_async(shape: pa_shape, max_q: int, max_total_q: int,
                                     opts: Optional[pa_options] = None, device=None):
    """Zero-filled device workspace for pa_decode_multi_host_async."""
    import torch

    return torch.zeros(pa_workspace_size_multi_host_async(shape, max_q, max_total_q, opts),
                       dtype=torch.uint8, device=device if device is not None else "cuda")


class _BoundAsyncCall:
    """An asynchronous host-buffer entry point with its arguments marshalled
    once: calling it enqueues one step and returns at once.  status() reads
    the step's device status bits, valid once the stream has passed the call
    (e.g. after torch.cuda.synchronize()).  Holds references to every tensor
    it points at, its own page-locked status word included."""

    def __init__(self, fn, name, args, keep, status):
        self._fn, self._name, self._args, self._keep = fn, name, args, keep
        self._status = status

    def __call__(self) -> None:
        rc = self._fn(*self._args)
        if rc != PA_OK:
            raise PagedGQAError(rc, self._name)

    def status(self) -> int:
        return int(self._status[1][0])


def _own_status_word():
    import torch

    t = torch.zeros(1, dtype=torch.int32).pin_memory()
    return t, t.numpy().view("uint32")


def bind_decode_host_async(q, k_cache, v_cache, block_table, cache_seqlens, scale, out,
                           workspace, slot: int, opts: Optional[pa_options] = None,
                           stream=None) -> _BoundAsyncCall:
    """pa_decode_host_async on these buffers and this staging slot (0 or 1),
    checked and marshalled once.  A loop alternates two bound calls (slot 0
    and slot 1, each with its own host buffers) and synchronises only when
    it reads a result.  The stream is taken at bind time."""
    _check_host(q, block_table, cache_seqlens, out, k_cache, v_cache)
    if slot not in (0, 1):
        raise ValueError("slot must be 0 or 1")
    shape = shape_of(q, k_cache, block_table)
    st = _own_status_word()
    V = ctypes.c_void_p
    opt = pa_options.from_buffer_copy(opts) if opts else None
    args = (ctypes.byref(shape), ctypes.byref(opt) if opt else None, V(_ptr(q)), V(_ptr(k_cache)),
            V(_ptr(v_cache)), V(_ptr(block_table)), V(_ptr(cache_seqlens)),
            ctypes.c_float(scale), V(_ptr(out)), V(st[0].data_ptr()), ctypes.c_int32(slot),
            V(_ptr(workspace)), ctypes.c_size_t(workspace.numel() * workspace.element_size()),
            V(_stream(stream)))
    keep = (shape, opt, q, k_cache, v_cache, block_table, cache_seqlens, out, workspace, st)
    return _BoundAsyncCall(lib().pa_decode_host_async, "pa_decode_host_async", args, keep, st)


def bind_decode_multi_host_async(q, cu_seqlens_q, max_q, causal, k_cache, v_cache, block_table,
                                 cache_seqlens, scale, out, workspace, slot: int,
                                 opts: Optional[pa_options] = None,
                                 stream=None) -> _BoundAsyncCall:
    """pa_decode_multi_host_async on these buffers and this staging slot (as
    bind_decode_host_async; total_q is q's row count)."""
    import torch

    _check_host(q, block_table, cache_seqlens, out, k_cache, v_cache,
                (("cu_seqlens_q", cu_seqlens_q),))
    if cu_seqlens_q.dtype != torch.int32 or tuple(cu_seqlens_q.shape) != (block_table.shape[0] + 1,):
        raise TypeError("cu_seqlens_q must be int32 [B + 1]")
    if slot not in (0, 1):
        raise ValueError("slot must be 0 or 1")
    shape = shape_multi(q, k_cache, block_table)
    st = _own_status_word()
    V = ctypes.c_void_p
    i32 = ctypes.c_int32
    opt = pa_options.from_buffer_copy(opts) if opts else None
    args = (ctypes.byref(shape), ctypes.byref(opt) if opt else None, V(_ptr(q)),
            V(_ptr(cu_seqlens_q)), i32(q.shape[0]), i32(max_q), i32(int(bool(causal))),
            V(_ptr(k_cache)), V(_ptr(v_cache)), V(_ptr(block_table)), V(_ptr(cache_seqlens)),
            ctypes.c_float(scale), V(_ptr(out)), V(st[0].data_ptr()), i32(slot),
            V(_ptr(workspace)), ctypes.c_size_t(workspace.numel() * workspace.element_size()),
            V(_stream(stream)))
    keep = (shape, opt, q, cu_seqlens_q, k_cache, v_cache, block_table, cache_seqlens, out,
            workspace, st)
    return _BoundAsyncCall(lib().pa_decode_multi_host_async, "pa_decode_multi_host_async", args,
                           keep, st)


def _decode_call(name, q, k_cache, v_cache, block_table, cache_seqlens, scale, out,
                 workspace, opts, stream):
    _check_tensors(q, k_cache, v_cache, block_table, cache_seqlens, out)
    shape = shape_of(q, k_cache, block_table)
    fn = getattr(lib(), name)
    rc = fn(ctypes.byref(shape), ctypes.byref(opts) if opts else None, _ptr(q), _ptr(k_cache),
            _ptr(v_cache), _ptr(block_table), _ptr(cache_seqlens), float(scale), _ptr(out),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, name)


def pa_decode(q, k_cache, v_cache, block_table, cache_seqlens, scale, out, workspace,
              opts: Optional[pa_options] = None, stream=None) -> None:
    """out[B,H,d] (fp32) = paged GQA decode attention; see include/pagedgqa.h."""
    _decode_call("pa_decode", q, k_cache, v_cache, block_table, cache_seqlens, scale, out,
                 workspace, opts, stream)


class _BoundDeviceCall:
    """A device-buffer entry point with its arguments marshalled once:
    calling it enqueues the call again on the same buffers (whose contents
    may have changed in place).  Holds references to every tensor it points
    at.  The per-call Python checks cost tens of microseconds on the host,
    more than a small decode step takes on the GPU."""

    def __init__(self, fn, name, args, keep):
        self._fn, self._name, self._args, self._keep = fn, name, args, keep

    def __call__(self) -> None:
        rc = self._fn(*self._args)
        if rc != PA_OK:
            raise PagedGQAError(rc, self._name)


def bind_decode(q, k_cache, v_cache, block_table, cache_seqlens, scale, out, workspace,
                opts: Optional[pa_options] = None, stream=None,
                name: str = "pa_decode") -> _BoundDeviceCall:
    """pa_decode (or pa_decode_split / pa_decode_merge, by `name`) on these
    device buffers, checked and marshalled once; each call of the result
    enqueues one step.  The stream is taken at bind time."""
    if name not in ("pa_decode", "pa_decode_split", "pa_decode_merge"):
        raise ValueError(name)
    _check_tensors(q, k_cache, v_cache, block_table, cache_seqlens, out)
    shape = shape_of(q, k_cache, block_table)
    V = ctypes.c_void_p
    opt = pa_options.from_buffer_copy(opts) if opts else None
    args = (ctypes.byref(shape), ctypes.byref(opt) if opt else None, V(_ptr(q)), V(_ptr(k_cache)),
            V(_ptr(v_cache)), V(_ptr(block_table)), V(_ptr(cache_seqlens)),
            ctypes.c_float(scale), V(_ptr(out)), V(_ptr(workspace)),
            ctypes.c_size_t(workspace.numel() * workspace.element_size()), V(_stream(stream)))
    keep = (shape, opt, q, k_cache, v_cache, block_table, cache_seqlens, out, workspace)
    return _BoundDeviceCall(getattr(lib(), name), name, args, keep)


def bind_decode_multi(q, cu_seqlens_q, max_q, causal, k_cache, v_cache, block_table,
                      cache_seqlens, scale, out, workspace, opts: Optional[pa_options] = None,
                      stream=None) -> _BoundDeviceCall:
    """pa_decode_multi on these device buffers, checked and marshalled once
    (total_q is q's row count; the stream is taken at bind time)."""
    import torch

    _check_tensors(q, k_cache, v_cache, block_table, cache_seqlens, out)
    if not cu_seqlens_q.is_cuda or cu_seqlens_q.dtype != torch.int32:
        raise TypeError("cu_seqlens_q must be an int32 CUDA tensor")
    if tuple(cu_seqlens_q.shape) != (block_table.shape[0] + 1,):
        raise ValueError("cu_seqlens_q must be [B + 1]")
    shape = shape_multi(q, k_cache, block_table)
    V = ctypes.c_void_p
    i32 = ctypes.c_int32
    opt = pa_options.from_buffer_copy(opts) if opts else None
    args = (ctypes.byref(shape), ctypes.byref(opt) if opt else None, V(_ptr(q)),
            V(_ptr(cu_seqlens_q)), i32(q.shape[0]), i32(max_q), i32(int(bool(causal))),
            V(_ptr(k_cache)), V(_ptr(v_cache)), V(_ptr(block_table)), V(_ptr(cache_seqlens)),
            ctypes.c_float(scale), V(_ptr(out)), V(_ptr(workspace)),
            ctypes.c_size_t(workspace.numel() * workspace.element_size()), V(_stream(stream)))
    keep = (shape, opt, q, cu_seqlens_q, k_cache, v_cache, block_table, cache_seqlens, out,
            workspace)
    return _BoundDeviceCall(lib().pa_decode_multi, "pa_decode_multi", args, keep)


def bind_decode_append(q, k_new, v_new, k_cache, v_cache, block_table, cache_seqlens, scale,
                       out, workspace, opts: Optional[pa_options] = None,
                       stream=None) -> _BoundDeviceCall:
    """pa_decode_append on these device buffers, checked and marshalled once
    (the stream is taken at bind time)."""
    _check_tensors(q, k_cache, v_cache, block_table, cache_seqlens, out)
    P_, bs, Hkv, d = k_cache.shape
    for nm, t in (("k_new", k_new), ("v_new", v_new)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != k_cache.dtype:
            raise ValueError(f"{nm} must be a contiguous CUDA tensor of the cache dtype")
        if tuple(t.shape) != (q.shape[0], Hkv, d):
            raise ValueError(f"{nm} must be [B, Hkv, d]")
    shape = shape_of(q, k_cache, block_table)
    V = ctypes.c_void_p
    opt = pa_options.from_buffer_copy(opts) if opts else None
    args = (ctypes.byref(shape), ctypes.byref(opt) if opt else None, V(_ptr(q)), V(_ptr(k_new)),
            V(_ptr(v_new)), V(_ptr(k_cache)), V(_ptr(v_cache)), V(_ptr(block_table)),
            V(_ptr(cache_seqlens)), ctypes.c_float(scale), V(_ptr(out)), V(_ptr(workspace)),
            ctypes.c_size_t(workspace.numel() * workspace.element_size()), V(_stream(stream)))
    keep = (shape, opt, q, k_new, v_new, k_cache, v_cache, block_table, cache_seqlens, out,
            workspace)
    return _BoundDeviceCall(lib().pa_decode_append, "pa_decode_append", args, keep)


def pa_decode_split(q, k_cache, v_cache, block_table, cache_seqlens, scale, out, workspace,
                    opts: Optional[pa_options] = None, stream=None) -> None:
    _decode_call("pa_decode_split", q, k_cache, v_cache, block_table, cache_seqlens, scale, out,
                 workspace, opts, stream)


def pa_decode_merge(q, k_cache, v_cache, block_table, cache_seqlens, scale, out, workspace,
                    opts: Optional[pa_options] = None, stream=None) -> None:
    _decode_call("pa_decode_merge", q, k_cache, v_cache, block_table, cache_seqlens, scale, out,
                 workspace, opts, stream)


def pa_decode_append(q, k_new, v_new, k_cache, v_cache, block_table, cache_seqlens, scale, out,
                     workspace, opts: Optional[pa_options] = None, stream=None) -> None:
    """Write k_new/v_new [B,Hkv,d] at position cache_seqlens[b] and attend over
    cache_seqlens[b] + 1 tokens, in one pass (see include/pagedgqa.h)."""
    _check_tensors(q, k_cache, v_cache, block_table, cache_seqlens, out)
    P_, bs, Hkv, d = k_cache.shape
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != k_cache.dtype:
            raise ValueError(f"{name} must be a contiguous CUDA tensor of the cache dtype")
        if tuple(t.shape) != (q.shape[0], Hkv, d):
            raise ValueError(f"{name} must be [B, Hkv, d]")
    shape = shape_of(q, k_cache, block_table)
    rc = lib().pa_decode_append(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                                _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                _ptr(block_table), _ptr(cache_seqlens), float(scale), _ptr(out),
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream))
    _check(rc, "pa_decode_append")


def pa_decode_noalloc(q, k_cache, v_cache, block_table, cache_seqlens, scale, out, status=None,
                      opts: Optional[pa_options] = None, stream=None) -> None:
    """pa_decode for callers that cannot allocate device memory: the kernels'
    scratch lives in a fixed static device array inside the library (see
    include/pagedgqa.h).  `status` is an optional int32/uint32 CUDA tensor of
    one element that receives the device status bits."""
    import torch

    _check_tensors(q, k_cache, v_cache, block_table, cache_seqlens, out)
    if status is not None:
        # the kernels OR bits into this word from the device: it must be
        # device memory of q's GPU, 4-byte integers, at least one element
        if (not isinstance(status, torch.Tensor) or not status.is_cuda
                or status.device != q.device or status.numel() < 1
                or status.dtype not in (torch.int32, getattr(torch, "uint32", torch.int32))):
            raise PagedGQAError(PA_ERR_SHAPE, "pa_decode_noalloc: status must be an int32 or "
                                "uint32 CUDA tensor of at least one element on q's device")
    shape = shape_of(q, k_cache, block_table)
    rc = lib().pa_decode_noalloc(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                                 _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                 _ptr(cache_seqlens), float(scale), _ptr(out), _ptr(status),
                                 _stream(stream))
    _check(rc, "pa_decode_noalloc")


def pa_cache_append(k_new, v_new, k_cache, v_cache, block_table, cache_seqlens, workspace,
                    stream=None) -> None:
    """Write k_new/v_new [B,Hkv,d] at position cache_seqlens[b] (in place)."""
    import torch

    for name, t in (("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache),
                    ("v_cache", v_cache), ("block_table", block_table),
                    ("cache_seqlens", cache_seqlens)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if k_new.dtype != k_cache.dtype or v_new.dtype != k_cache.dtype:
        raise TypeError("k_new/v_new must have the cache dtype")
    if block_table.dtype != torch.int32 or cache_seqlens.dtype != torch.int32:
        raise TypeError("block_table and cache_seqlens must be int32")
    P, bs, Hkv, d = k_cache.shape
    B = block_table.shape[0]
    if tuple(k_new.shape) != (B, Hkv, d) or tuple(v_new.shape) != (B, Hkv, d):
        raise ValueError("k_new/v_new must be [B, Hkv, d]")
    shape = pa_shape(B, Hkv, Hkv, d, bs, block_table.shape[1], P, _dtype_code(k_cache))
    rc = lib().pa_cache_append(ctypes.byref(shape), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                               _ptr(v_cache), _ptr(block_table), _ptr(cache_seqlens),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream))
    _check(rc, "pa_cache_append")


def pa_read_status(workspace, stream=None) -> int:
    """Read and clear the sticky device status bits (synchronises the stream)."""
    v = ctypes.c_uint32(0)
    rc = lib().pa_read_status(_ptr(workspace), ctypes.byref(v), _stream(stream))
    _check(rc, "pa_read_status")
    return int(v.value)


def pa_plan_pieces(shape: pa_shape, opts: Optional[pa_options], lens_host, num_ctas: int,
                   cta: int):
    """Host replica of the work split: list of (b, j, blk0, blk1, slot)."""
    import numpy as np

    lens = np.ascontiguousarray(lens_host, dtype=np.int32)
    n = lib().pa_plan_pieces(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                             lens.ctypes.data, int(num_ctas), int(cta), None, 0)
    if n < 0:
        _check(n, "pa_plan_pieces")
    buf = np.zeros((max(n, 1), 5), dtype=np.int32)
    m = lib().pa_plan_pieces(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                             lens.ctypes.data, int(num_ctas), int(cta), buf.ctypes.data, n)
    assert m == n
    return [tuple(int(x) for x in row) for row in buf[:n]]


def pa_plan_merge(shape: pa_shape, opts: Optional[pa_options], lens_host, num_ctas: int,
                  seg: int, max_slots: int = 1 << 16):
    """Host replica of merge index `seg`: ((b, j), [slots]) or None."""
    import numpy as np

    lens = np.ascontiguousarray(lens_host, dtype=np.int32)
    bj = np.zeros(2, dtype=np.int32)
    slots = np.zeros(max_slots, dtype=np.int32)
    n = lib().pa_plan_merge(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                            lens.ctypes.data, int(num_ctas), int(seg), bj.ctypes.data,
                            slots.ctypes.data, max_slots)
    if n < 0:
        _check(n, "pa_plan_merge")
    if n == 0:
        return None
    return (int(bj[0]), int(bj[1])), [int(s) for s in slots[:n]]


class BlockManager:
    """Owner of a pa_block_manager handle (the C calls below take it as `bm`).

    Host allocator of the physical-block pool: free list, per-block reference
    count, per-sequence block lists; allocate / free_sequence / share_prefix /
    copy-on-write as the "paged-attention-runtime" design page's BlockManager
    section describes them."""

    def __init__(self, num_blocks: int, block_size: int, max_seqs: int,
                 max_blocks_per_seq: int):
        self.handle = pa_bm_create(num_blocks, block_size, max_seqs, max_blocks_per_seq)
        self.block_size = int(block_size)

    def close(self):
        if self.handle:
            pa_bm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def allocate(self, seq: int, n: int):
        pa_bm_allocate(self.handle, seq, n)

    def free_sequence(self, seq: int):
        pa_bm_free_sequence(self.handle, seq)

    def share_prefix(self, src: int, dst: int, n: int):
        pa_bm_share_prefix(self.handle, src, dst, n)

    def copy_on_write(self, seq: int, index: int):
        return pa_bm_copy_on_write(self.handle, seq, index)

    def reserve_slot(self, seq: int, pos: int):
        return pa_bm_reserve_slot(self.handle, seq, pos)

    def block_table(self, seq_ids, cols: int):
        return pa_bm_block_table(self.handle, seq_ids, cols)

    def free_blocks(self) -> int:
        return pa_bm_query(self.handle, PA_BM_FREE_BLOCKS, 0)

    def ref_count(self, block: int) -> int:
        return pa_bm_query(self.handle, PA_BM_REF_COUNT, block)

    def num_seq_blocks(self, seq: int) -> int:
        return pa_bm_query(self.handle, PA_BM_SEQ_BLOCKS, seq)


def pa_bm_create(num_blocks: int, block_size: int, max_seqs: int, max_blocks_per_seq: int):
    h = lib().pa_bm_create(int(num_blocks), int(block_size), int(max_seqs),
                           int(max_blocks_per_seq))
    if not h:
        raise PagedGQAError(PA_ERR_STATE, "pa_bm_create")
    return h


def pa_bm_destroy(bm) -> None:
    lib().pa_bm_destroy(bm)


def pa_bm_allocate(bm, seq: int, n: int) -> None:
    _check(lib().pa_bm_allocate(bm, int(seq), int(n)), "pa_bm_allocate")


def pa_bm_free_sequence(bm, seq: int) -> None:
    _check(lib().pa_bm_free_sequence(bm, int(seq)), "pa_bm_free_sequence")


def pa_bm_share_prefix(bm, src: int, dst: int, n: int) -> None:
    _check(lib().pa_bm_share_prefix(bm, int(src), int(dst), int(n)), "pa_bm_share_prefix")


def _bm_pair_call(name, bm, a: int, b: int):
    old, new = ctypes.c_int32(-1), ctypes.c_int32(-1)
    _check(getattr(lib(), name)(bm, int(a), int(b), ctypes.byref(old), ctypes.byref(new)), name)
    return int(old.value), int(new.value)


def pa_bm_copy_on_write(bm, seq: int, index: int):
    """(old_block, new_block); they differ when the caller must copy old -> new."""
    return _bm_pair_call("pa_bm_copy_on_write", bm, seq, index)


def pa_bm_reserve_slot(bm, seq: int, pos: int):
    """(old_block, new_block) for the block that will hold token `pos` of seq."""
    return _bm_pair_call("pa_bm_reserve_slot", bm, seq, pos)


def pa_bm_block_table(bm, seq_ids, cols: int):
    """int32 numpy array [len(seq_ids), cols], -1 past each sequence's blocks."""
    import numpy as np

    ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
    table = np.empty((ids.size, int(cols)), dtype=np.int32)
    _check(lib().pa_bm_block_table(bm, ids.ctypes.data, int(ids.size), int(cols),
                                   table.ctypes.data), "pa_bm_block_table")
    return table


def pa_bm_query(bm, what: int, arg: int = 0) -> int:
    r = lib().pa_bm_query(bm, int(what), int(arg))
    if r < 0:
        _check(r, "pa_bm_query")
    return int(r)


def pa_copy_blocks(k_cache, v_cache, pairs, status=None, stream=None) -> None:
    """Copy physical block pairs[i,0] onto pairs[i,1] in both pools (in place).

    pairs: int32 CUDA tensor [n, 2]; status: optional uint32-sized CUDA tensor
    that receives PA_STATUS_BAD_BLOCK for an out-of-range id."""
    import torch

    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("pairs", pairs)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if pairs.dtype != torch.int32 or pairs.dim() != 2 or pairs.shape[1] != 2:
        raise TypeError("pairs must be an int32 tensor [n, 2]")
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must match")
    P, bs, Hkv, d = k_cache.shape
    shape = pa_shape(0, Hkv, Hkv, d, bs, 1, P, _dtype_code(k_cache))
    rc = lib().pa_copy_blocks(ctypes.byref(shape), _ptr(k_cache), _ptr(v_cache), _ptr(pairs),
                              int(pairs.shape[0]), _ptr(status), _stream(stream))
    _check(rc, "pa_copy_blocks")


def pa_version() -> int:
    return int(lib().pa_version())
