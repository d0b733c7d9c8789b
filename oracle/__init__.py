"""Float64 CPU oracle for paged grouped-query decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The library never
imports this package, and this package never imports the library.

The arithmetic lives in ``pa_oracle.c`` (plain loops, IEEE double, ``exp``
from libm); this module compiles it with gcc on first use and marshals numpy
arrays.  Every function cites the page passage it follows in the C source.

Functions with no pin beyond the tests in ``tests/test_oracle_pins.py``:
none -- decode, decode_multi, partial/combine and append are all pinned there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None

F16 = 0
BF16 = 1

ERRORS = {
    -1: "unsupported shape",
    -2: "sequence length outside [0, max_blocks_per_seq*block_size]",
    -3: "unmapped or out-of-range block-table entry inside a sequence",
    -4: "out of memory",
    -5: "index out of range",
}


class OracleError(ValueError):
    pass


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into libpa_oracle.so (gcc, OpenMP)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.pa_oracle_decode.argtypes = [i] * 8 + [P, P, P, P, P, ctypes.c_double, i, P, P, i]
    lib.pa_oracle_decode.restype = i
    lib.pa_oracle_decode_multi.argtypes = ([i] * 8 + [P, i, P, i, P, P, P, P, ctypes.c_double,
                                            i, P, P, i])
    lib.pa_oracle_decode_multi.restype = i
    lib.pa_oracle_partial.argtypes = ([i] * 8 + [P, P, P, P, P, ctypes.c_double]
                                      + [i, i, i, i, P, P, P])
    lib.pa_oracle_partial.restype = i
    lib.pa_oracle_combine.argtypes = [i, i, P, P, P, P, P, P]
    lib.pa_oracle_combine.restype = None
    lib.pa_oracle_append.argtypes = [i] * 6 + [P] * 7
    lib.pa_oracle_append.restype = i
    lib.pa_oracle_widen.argtypes = [ctypes.c_uint16, i]
    lib.pa_oracle_widen.restype = ctypes.c_double
    lib.pa_oracle_max_threads.argtypes = []
    lib.pa_oracle_max_threads.restype = i
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are raw 16-bit storage (uint16 views)")
    return a


def _dtype_code(dtype) -> int:
    if dtype in (F16, "f16", "fp16", "float16"):
        return F16
    if dtype in (BF16, "bf16", "bfloat16"):
        return BF16
    raise ValueError(f"unknown dtype {dtype!r}")


def _check(rc: int):
    if rc != 0:
        raise OracleError(ERRORS.get(rc, f"oracle error {rc}"))


def max_threads() -> int:
    return int(_load().pa_oracle_max_threads())


def widen(bits: int, dtype) -> float:
    """Exact value of one stored 16-bit pattern."""
    return float(_load().pa_oracle_widen(int(bits), _dtype_code(dtype)))


def decode(q, k_cache, v_cache, block_table, cache_seqlens, scale, dtype,
           pairs=None, n_threads: int = 0) -> np.ndarray:
    """Float64 decode attention.

    q [B,H,d], k_cache/v_cache [P,bs,Hkv,d] as uint16 bit patterns;
    block_table [B,maxblk] int32; cache_seqlens [B] int32.
    Returns [B,H,d] float64, or [n,d] when ``pairs`` ([n,2] of (b,h)) is given.
    """
    lib = _load()
    q = _bits(q)
    k_cache = _bits(k_cache)
    v_cache = _bits(v_cache)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    B, H, d = q.shape
    P, bs, Hkv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("q/k/v shapes disagree")
    maxblk = bt.shape[1] if bt.ndim == 2 else 0
    if pairs is None:
        out = np.zeros((B, H, d), dtype=np.float64)
        n, pp = -1, None
    else:
        pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        out = np.zeros((pairs.shape[0], d), dtype=np.float64)
        n, pp = pairs.shape[0], _ptr(pairs)
    rc = lib.pa_oracle_decode(B, H, Hkv, d, bs, maxblk, P, _dtype_code(dtype),
                              _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(sl),
                              float(scale), n, pp, _ptr(out), int(n_threads))
    _check(rc)
    return out


def decode_multi(q, cu_q, causal, k_cache, v_cache, block_table, cache_seqlens, scale, dtype,
                 pairs=None, n_threads: int = 0) -> np.ndarray:
    """Float64 attention of packed query rows q [total_q, H, d]; sequence b
    owns rows cu_q[b] .. cu_q[b+1]-1 and its keys are its cache_seqlens[b]
    cached tokens (query i of n_q sees keys t < k_len - n_q + i + 1 when
    causal).  Returns [total_q, H, d] float64, or [n, d] for (row, h) pairs."""
    lib = _load()
    q = _bits(q)
    k_cache = _bits(k_cache)
    v_cache = _bits(v_cache)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    cu = np.ascontiguousarray(cu_q, dtype=np.int32)
    total_q, H, d = q.shape
    P, bs, Hkv, d2 = k_cache.shape
    B = sl.shape[0]
    if d2 != d or v_cache.shape != k_cache.shape or cu.shape != (B + 1,):
        raise ValueError("q/k/v/cu_q shapes disagree")
    maxblk = bt.shape[1] if bt.ndim == 2 else 0
    if pairs is None:
        out = np.zeros((total_q, H, d), dtype=np.float64)
        n, pp = -1, None
    else:
        pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        out = np.zeros((pairs.shape[0], d), dtype=np.float64)
        n, pp = pairs.shape[0], _ptr(pairs)
    rc = lib.pa_oracle_decode_multi(B, H, Hkv, d, bs, maxblk, P, _dtype_code(dtype), _ptr(q),
                                    total_q, _ptr(cu), int(bool(causal)), _ptr(k_cache),
                                    _ptr(v_cache), _ptr(bt), _ptr(sl), float(scale), n, pp,
                                    _ptr(out), int(n_threads))
    _check(rc)
    return out


def partial(q, k_cache, v_cache, block_table, cache_seqlens, scale, dtype, b, h, t0, t1):
    """Compound state (m, l, weighted_v[d]) of tokens [t0, t1) of (b, h)."""
    lib = _load()
    q = _bits(q)
    k_cache = _bits(k_cache)
    v_cache = _bits(v_cache)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    B, H, d = q.shape
    P, bs, Hkv, _ = k_cache.shape
    m = np.zeros(1)
    l = np.zeros(1)
    acc = np.zeros(d)
    rc = lib.pa_oracle_partial(B, H, Hkv, d, bs, bt.shape[1], P, _dtype_code(dtype),
                               _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(sl),
                               float(scale), int(b), int(h), int(t0), int(t1),
                               _ptr(m), _ptr(l), _ptr(acc))
    _check(rc)
    return float(m[0]), float(l[0]), acc


def combine(ms, ls, accs):
    """Fold compound states left to right with the combine op."""
    lib = _load()
    ms = np.ascontiguousarray(ms, dtype=np.float64)
    ls = np.ascontiguousarray(ls, dtype=np.float64)
    accs = np.ascontiguousarray(accs, dtype=np.float64)
    n, d = accs.shape
    m = np.zeros(1)
    l = np.zeros(1)
    acc = np.zeros(d)
    lib.pa_oracle_combine(n, d, _ptr(ms), _ptr(ls), _ptr(accs), _ptr(m), _ptr(l), _ptr(acc))
    return float(m[0]), float(l[0]), acc


def append(k_new, v_new, k_cache, v_cache, block_table, cache_seqlens):
    """Write new K/V rows into copies of the pools.

    Returns (k_cache', v_cache', slots[B,2] of (phys,row) with -1 for none,
    rc) where rc is 0 or the negative oracle code for a sequence with no slot.
    """
    lib = _load()
    k_new = _bits(k_new)
    v_new = _bits(v_new)
    kc = _bits(k_cache).copy()
    vc = _bits(v_cache).copy()
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    P, bs, Hkv, d = kc.shape
    B = sl.shape[0]
    slots = np.zeros((B, 2), dtype=np.int32)
    rc = lib.pa_oracle_append(B, Hkv, d, bs, bt.shape[1], P, _ptr(k_new), _ptr(v_new),
                              _ptr(kc), _ptr(vc), _ptr(bt), _ptr(sl), _ptr(slots))
    return kc, vc, slots, int(rc)
