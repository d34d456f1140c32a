"""CPU oracle for paged KV-cache attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The library's product path never touches it,
and it shares no code with the CUDA sources.

The arithmetic lives in ``pkv_oracle.c`` (plain C, double precision); this
module compiles it with gcc on first use (or via :func:`build`) and marshals
numpy arrays into it.  Every function cites the passage of the pages it
follows in the C source.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, a library attention routine, brute force, metamorphic
invariants and the pages' own numbers); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BLOCK_SIZE = 16


def build(force: bool = False) -> str:
    """Compile ``pkv_oracle.c`` into ``liboracle.so`` next to it (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [P, P, i64]
            lib.oracle_bf16_to_f64.restype = None
            lib.oracle_cache_write.argtypes = [P, P, i64, i32, i32, i32, P, P, P, i64]
            lib.oracle_cache_write.restype = ctypes.c_int
            lib.oracle_copy_blocks.argtypes = [P, P, i64, i32, i32, i32, P, P, i64]
            lib.oracle_copy_blocks.restype = ctypes.c_int
            lib.oracle_paged_attention.argtypes = [P, P, i64, i32, i32, i32, P, i32, P, P, i32, P, i32, f64,
                                                   P, i32]
            lib.oracle_paged_attention.restype = ctypes.c_int
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 exactly."""
    src = _c(bits, np.uint16)
    out = np.empty(src.shape, dtype=np.float64)
    _load().oracle_bf16_to_f64(_ptr(src), _ptr(out), src.size)
    return out


def _pool_dims(k_pool):
    nb, hkv, bs, d = k_pool.shape
    return nb, hkv, bs, d


def cache_write(k_pool, v_pool, k_new, v_new, slot_mapping):
    """In place: store row t of k_new/v_new ([T][Hkv][d]) at slot_mapping[t]."""
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    assert k_pool.dtype == np.uint16 and v_pool.dtype == np.uint16
    nb, hkv, bs, d = _pool_dims(k_pool)
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    sm = _c(slot_mapping, np.int32)
    rc = _load().oracle_cache_write(_ptr(k_pool), _ptr(v_pool), nb, hkv, d, bs, _ptr(kn), _ptr(vn), _ptr(sm),
                                    sm.size)
    if rc != 0:
        raise OracleError(f"oracle_cache_write -> {rc}")


def copy_blocks(k_pool, v_pool, src, dst):
    """In place: pool[dst[i]] <- pool[src[i]] for K and V, whole blocks."""
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    nb, hkv, bs, d = _pool_dims(k_pool)
    s, t = _c(src, np.int32), _c(dst, np.int32)
    rc = _load().oracle_copy_blocks(_ptr(k_pool), _ptr(v_pool), nb, hkv, d, bs, _ptr(s), _ptr(t), s.size)
    if rc != 0:
        raise OracleError(f"oracle_copy_blocks -> {rc}")


def swap_blocks(direction, k_pool, v_pool, blocks, slots, host):
    """In place, for every pair with blocks[i] >= 0: host[slots[i]] = (K, V) of
    pool block blocks[i] (direction 0), or the reverse (direction 1).  ``host``
    is uint16 [num_slots][2][Hkv][16][d]."""
    for b, h in zip(np.asarray(blocks).tolist(), np.asarray(slots).tolist()):
        if b < 0:
            continue
        if direction == 0:
            host[h, 0] = k_pool[b]
            host[h, 1] = v_pool[b]
        else:
            k_pool[b] = host[h, 0]
            v_pool[b] = host[h, 1]


def paged_attention(k_pool, v_pool, q, query_start_loc, context_lens, block_tables, scale, threads=1):
    """Causal attention of ``q`` ([Tq][Hq][d] bf16 bits) over the paged cache.

    Returns float64 ``[Tq][Hq][d]``.  Sequence s owns query rows
    query_start_loc[s]..query_start_loc[s+1]-1 at absolute positions
    context_lens[s]-query_len+i.
    """
    k_pool, v_pool = _c(k_pool, np.uint16), _c(v_pool, np.uint16)
    nb, hkv, bs, d = _pool_dims(k_pool)
    qq = _c(q, np.uint16)
    T, hq, dq = qq.shape
    assert dq == d
    qsl = _c(query_start_loc, np.int32)
    ctx = _c(context_lens, np.int32)
    bt = _c(block_tables, np.int32)
    if bt.ndim == 1:
        bt = bt.reshape(len(ctx), -1)
    out = np.zeros((T, hq, d), dtype=np.float64)
    rc = _load().oracle_paged_attention(_ptr(k_pool), _ptr(v_pool), nb, hkv, d, bs, _ptr(qq), hq, _ptr(qsl),
                                        _ptr(ctx), len(ctx), _ptr(bt), bt.shape[1] if bt.size else 0,
                                        float(scale), _ptr(out), int(threads))
    if rc != 0:
        raise OracleError(f"oracle_paged_attention -> {rc}")
    return out


def decode_attention(k_pool, v_pool, q, context_lens, block_tables, scale, threads=1):
    """One query row per sequence (``q`` is [B][Hq][d]); the decode case."""
    B = len(context_lens)
    qsl = np.arange(B + 1, dtype=np.int32)
    return paged_attention(k_pool, v_pool, q, qsl, context_lens, block_tables, scale, threads)


def run_step(w, threads=1, rows=None):
    """The whole step of a workload on copies of its pools: copy_blocks (if
    any), cache_write, then attention.  Returns (k_pool, v_pool, out).

    ``rows`` (optional) restricts attention to a subset of sequence indices:
    the output then only holds valid values for those sequences' rows.
    """
    k = w.k_pool.copy()
    v = w.v_pool.copy()
    if w.copy_src is not None:
        copy_blocks(k, v, w.copy_src, w.copy_dst)
    cache_write(k, v, w.k_new, w.v_new, w.slot_mapping)
    qsl = w.query_start_loc
    ctx = w.context_lens
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        ctx = np.zeros_like(ctx)
        ctx[rows] = w.context_lens[rows]
        # sequences outside `rows` keep their query rows but get zero-length
        # contexts only if they are decode rows; otherwise drop their rows.
        ql = np.diff(qsl)
        keep = np.zeros(len(ctx), dtype=bool)
        keep[rows] = True
        new_ql = np.where(keep, ql, 0)
        qsl2 = np.zeros_like(qsl)
        qsl2[1:] = np.cumsum(new_ql)
        # map the kept sequences' rows back to their positions in q
        idx = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in range(len(ctx)) if keep[s]] or
                             [np.zeros(0, dtype=np.int64)])
        sub = paged_attention(k, v, w.q[idx], qsl2, ctx, w.block_tables, w.scale, threads)
        out = np.full((w.q.shape[0], w.num_q_heads, w.head_dim), np.nan)
        out[idx] = sub
        return k, v, out
    out = paged_attention(k, v, w.q, qsl, ctx, w.block_tables, w.scale, threads)
    return k, v, out
