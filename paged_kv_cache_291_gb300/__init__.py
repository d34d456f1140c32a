"""paged_kv_cache_291_gb300 -- Python binding of libpagedkv (GB300, sm_103a).

A thin ctypes layer over the C-ABI declared in ``include/pkv.h``: it checks
tensor dtypes, shapes and devices, passes ``data_ptr()`` values and the
current CUDA stream, and raises :class:`PKVError` on a non-OK status.  Every
step of the computation runs in the library's CUDA kernels; there is no
fallback of any kind, and the binding refuses to work when ``libpagedkv.so``
has not been built (build it with ``python -m paged_kv_cache_291_gb300.build``
or ``__graft_entry__.build()``).

Tensors: K/V pools are 2-byte (bf16) CUDA tensors
``[num_blocks][num_kv_heads][16][head_dim]``; q/k_new/v_new bf16; index
arrays int32; outputs float32.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

__all__ = [
    "PKVError", "lib_path", "load", "version", "status_string", "cache_write", "copy_blocks",
    "decode_workspace_size", "decode_attention", "decode_step", "prefill_workspace_size",
    "chunked_prefill_attention",
    "get_error", "Cache", "Blocks", "prefix_keys", "swap_out", "swap_in", "test_arm_decode_stall",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpagedkv.so")
_lib = None

PKV_OK = 0
STATUS_NAMES = {
    0: "PKV_OK", 1: "PKV_ERR_NULL", 2: "PKV_ERR_SHAPE", 3: "PKV_ERR_HEADS", 4: "PKV_ERR_HEADDIM",
    5: "PKV_ERR_BLOCKSIZE", 6: "PKV_ERR_ALIAS", 7: "PKV_ERR_WORKSPACE", 8: "PKV_ERR_ALIGN", 9: "PKV_ERR_RANGE",
    10: "PKV_ERR_TIMEOUT", 11: "PKV_ERR_CUDA", 12: "PKV_ERR_UNSUPPORTED", 13: "PKV_ERR_SCRATCH_LIMIT",
    14: "PKV_ERR_NO_BLOCKS", 15: "PKV_ERR_HOST_MEMORY", 16: "PKV_ERR_DTYPE",
}
PKV_KV_BF16, PKV_KV_E4M3 = 0, 1


class PKVError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        msg = status_string(status) if _lib is not None else STATUS_NAMES.get(status, str(status))
        if self.status == 11 and _lib is not None:
            msg += f" ({_lib.pkv_last_cuda_error().decode()})"
        super().__init__(f"{what}: {msg}" if what else msg)


class Cache(ctypes.Structure):
    """Mirror of ``pkv_cache_t``."""
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("num_blocks", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


class BlocksState(ctypes.Structure):
    """Mirror of ``pkv_blocks_t``."""
    _fields_ = [("block_tables", ctypes.c_void_p), ("context_lens", ctypes.c_void_p),
                ("ref_counts", ctypes.c_void_p), ("free_ring", ctypes.c_void_p), ("ring_pos", ctypes.c_void_p),
                ("free_state", ctypes.c_void_p), ("scratch", ctypes.c_void_p), ("block_keys", ctypes.c_void_p),
                ("key_table", ctypes.c_void_p), ("cached", ctypes.c_void_p), ("num_blocks", ctypes.c_int32),
                ("max_seqs", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32), ("table_size", ctypes.c_int32)]


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libpagedkv.so (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"libpagedkv.so is not built ({_LIB_PATH}); run `python -m "
                           "paged_kv_cache_291_gb300.build` or __graft_entry__.build() first")
    lib = ctypes.CDLL(_LIB_PATH)
    P, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    CP = ctypes.POINTER(Cache)
    sigs = {
        "pkv_cache_write": ([CP, P, P, P, i32, P], ctypes.c_int),
        "pkv_copy_blocks": ([CP, P, P, i32, P, P, P], ctypes.c_int),
        "pkv_decode_workspace_size": ([i32, i32, i32, i32, i32, i32], sz),
        "pkv_decode_attention": ([CP, P, i32, P, i32, P, i32, i32, f32, P, P, sz, i32, P], ctypes.c_int),
        "pkv_decode_step": ([CP, P, P, P, P, i32, P, i32, P, i32, i32, f32, P, P, sz, i32, P], ctypes.c_int),
        "pkv_decode_shared_prefix_workspace_size": ([i32, i32, i32, i32, i32, i32], sz),
        "pkv_decode_attention_shared_prefix": ([CP, P, i32, P, i32, P, i32, i32, i32, f32, P, P, sz, P],
                                               ctypes.c_int),
        "pkv_common_prefix_blocks": ([P, i32, P, i32], i32),
        "pkv_copy": ([P, P, sz, P], ctypes.c_int),
        "pkv_prefill_workspace_size": ([i32, i32, i32, i32, i32, i32], sz),
        "pkv_chunked_prefill_attention": ([CP, P, i32, i32, P, P, P, i32, P, i32, i32, f32, P, P, sz, P],
                                          ctypes.c_int),
        "pkv_blocks_reset": ([ctypes.POINTER(BlocksState), P], ctypes.c_int),
        "pkv_blocks_append": ([ctypes.POINTER(BlocksState), P, i32, i32, P, P, P, P, P], ctypes.c_int),
        "pkv_blocks_fork": ([ctypes.POINTER(BlocksState), P, P, i32, P], ctypes.c_int),
        "pkv_blocks_release": ([ctypes.POINTER(BlocksState), P, i32, P], ctypes.c_int),
        "pkv_blocks_match": ([ctypes.POINTER(BlocksState), P, i32, P, i32, P, P], ctypes.c_int),
        "pkv_blocks_register": ([ctypes.POINTER(BlocksState), P, i32, P, i32, P], ctypes.c_int),
        "pkv_prefix_keys": ([P, P, P, P, i32, i32, P, P], ctypes.c_int),
        "pkv_swap_blocks": ([CP, i32, P, P, i32, P, ctypes.c_int64, P], ctypes.c_int),
        "pkv_get_error": ([P, ctypes.POINTER(i32)], ctypes.c_int),
        "pkv_test_arm_decode_stall": ([i32], ctypes.c_int),
        "pkv_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "pkv_last_cuda_error": ([], ctypes.c_char_p),
        "pkv_version": ([], ctypes.c_char_p),
    }
    for name, (argt, rest) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = argt
        fn.restype = rest
    _lib = lib
    return lib


def version() -> str:
    return load().pkv_version().decode()


def status_string(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


# ---------------------------------------------------------------- helpers

def _torch():
    import torch
    return torch


def _stream_handle(stream) -> ctypes.c_void_p:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t, name, elem_size=None, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if elem_size is not None and t.element_size() != elem_size:
        raise TypeError(f"{name} must have {elem_size}-byte elements")
    return ctypes.c_void_p(t.data_ptr())


def _out(t, name="out"):
    """An fp32 output tensor on the device or in page-locked host memory
    (``pin_memory()``), which the kernels then write directly."""
    torch = _torch()
    if isinstance(t, torch.Tensor) and not t.is_cuda:
        if not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or page-locked host memory")
        if not t.is_contiguous() or t.dtype != torch.float32:
            raise ValueError(f"{name} must be contiguous float32")
        return ctypes.c_void_p(t.data_ptr())
    return _dev(t, name, dtype=torch.float32)


def _cache(k_pool, v_pool, k_scale=None, v_scale=None, need_scales=False) -> Cache:
    """Descriptor of a pool pair: 2-byte elements are bf16, 1-byte elements
    (uint8 or float8_e4m3fn) e4m3 codes with one scale per pool."""
    if k_pool.shape != v_pool.shape or k_pool.dim() != 4:
        raise ValueError("k_pool and v_pool must both be [num_blocks][num_kv_heads][16][head_dim]")
    nb, hkv, bs, d = k_pool.shape
    es = k_pool.element_size()
    if es not in (1, 2):
        raise TypeError("pools must have 2-byte (bf16) or 1-byte (e4m3) elements")
    if es == 1 and need_scales and (k_scale is None or v_scale is None):
        raise ValueError("an e4m3 pool needs k_scale and v_scale")
    return Cache(_dev(k_pool, "k_pool", es).value, _dev(v_pool, "v_pool", es).value, nb, hkv, d, bs,
                 PKV_KV_E4M3 if es == 1 else PKV_KV_BF16,
                 1.0 if k_scale is None else float(k_scale), 1.0 if v_scale is None else float(v_scale))


def _check(status, what):
    if status != PKV_OK:
        raise PKVError(status, what)


def _host_i32(x):
    import numpy as np
    a = np.ascontiguousarray(x.cpu().numpy() if hasattr(x, "cpu") else x, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- calls

def cache_write(k_pool, v_pool, k_new, v_new, slot_mapping, stream=None, k_scale=None, v_scale=None) -> None:
    """Store rows k_new/v_new [T][Hkv][d] at ``slot_mapping`` [T] (negative = skip).
    e4m3 pools (1-byte elements) store code(x * (1/scale)) and need the scales."""
    torch = _torch()
    lib = load()
    c = _cache(k_pool, v_pool, k_scale, v_scale, need_scales=True)
    T = int(slot_mapping.shape[0])
    if k_new.shape != (T, c.num_kv_heads, c.head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [num_tokens][num_kv_heads][head_dim]")
    st = lib.pkv_cache_write(ctypes.byref(c), _dev(k_new, "k_new", 2), _dev(v_new, "v_new", 2),
                             _dev(slot_mapping, "slot_mapping", dtype=torch.int32), T, _stream_handle(stream))
    _check(st, "pkv_cache_write")


def copy_blocks(k_pool, v_pool, src, dst, check_host: bool = True, src_host=None, dst_host=None,
                stream=None) -> None:
    """Copy-on-write: pool[dst[i]] <- pool[src[i]] (K and V, whole blocks).

    The library rejects aliasing destinations before launching when it gets
    host copies of the id lists: pass them as ``src_host``/``dst_host``, or
    leave ``check_host`` on to have them copied from the device tensors
    (which synchronises).
    """
    torch = _torch()
    lib = load()
    c = _cache(k_pool, v_pool)
    n = int(src.shape[0])
    if dst.shape[0] != n:
        raise ValueError("src and dst must have the same length")
    sh = dh = None
    sp = dp = None
    if src_host is not None and dst_host is not None:
        sh, sp = _host_i32(src_host)
        dh, dp = _host_i32(dst_host)
        if sh.shape[0] != n or dh.shape[0] != n:
            raise ValueError("host id lists must match the device ones")
    elif check_host:
        sh, sp = _host_i32(src)
        dh, dp = _host_i32(dst)
    st = lib.pkv_copy_blocks(ctypes.byref(c), _dev(src, "src", dtype=torch.int32),
                             _dev(dst, "dst", dtype=torch.int32), n, sp, dp, _stream_handle(stream))
    _check(st, "pkv_copy_blocks")


def decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                          partition_blocks=0) -> int:
    n = load().pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                                         partition_blocks)
    if n == 0:
        raise PKVError(2, "pkv_decode_workspace_size")
    return int(n)


def new_workspace(nbytes: int, device=None):
    """A zero-filled, 256-byte aligned workspace (torch allocations are)."""
    torch = _torch()
    return torch.zeros(max(256, (nbytes + 255) // 256 * 256), dtype=torch.uint8, device=device or "cuda")


def decode_attention(k_pool, v_pool, q, block_tables, context_lens, max_context_len: int, scale: float,
                     out=None, workspace=None, partition_blocks: int = 0, stream=None, k_scale=None,
                     v_scale=None):
    """Paged decode attention; returns ``out`` float32 [B][Hq][d].  e4m3 pools
    (1-byte elements) need the scales they were written with."""
    torch = _torch()
    lib = load()
    c = _cache(k_pool, v_pool, k_scale, v_scale, need_scales=True)
    B, hq, d = q.shape
    if d != c.head_dim:
        raise ValueError("q head_dim does not match the pools")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables must be [B][max_blocks] and context_lens [B]")
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = load().pkv_decode_workspace_size(B, hq, c.num_kv_heads, d, int(max_context_len),
                                                int(partition_blocks))
        workspace = new_workspace(need, q.device)  # a size of 0 means bad arguments: the call reports them
    st = lib.pkv_decode_attention(ctypes.byref(c), _dev(q, "q", 2), hq,
                                  _dev(block_tables, "block_tables", dtype=torch.int32), int(block_tables.shape[1]),
                                  _dev(context_lens, "context_lens", dtype=torch.int32), B, int(max_context_len),
                                  float(scale), _out(out),
                                  _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                                  int(partition_blocks), _stream_handle(stream))
    _check(st, "pkv_decode_attention")
    return out


def decode_step(k_pool, v_pool, k_new, v_new, slot_mapping, q, block_tables, context_lens, max_context_len: int,
                scale: float, out=None, workspace=None, partition_blocks: int = 0, stream=None, k_scale=None,
                v_scale=None):
    """One decode step in one launch: store row s of k_new/v_new [B][Hkv][d]
    at slot_mapping[s] (the slot of position context_lens[s] - 1; negative =
    skip) and attend over the context; returns ``out`` float32 [B][Hq][d]."""
    torch = _torch()
    lib = load()
    c = _cache(k_pool, v_pool, k_scale, v_scale, need_scales=True)
    B, hq, d = q.shape
    if d != c.head_dim:
        raise ValueError("q head_dim does not match the pools")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables must be [B][max_blocks] and context_lens [B]")
    if k_new.shape != (B, c.num_kv_heads, d) or v_new.shape != k_new.shape or slot_mapping.shape[0] != B:
        raise ValueError("k_new/v_new must be [B][num_kv_heads][head_dim] and slot_mapping [B]")
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = lib.pkv_decode_workspace_size(B, hq, c.num_kv_heads, d, int(max_context_len), int(partition_blocks))
        workspace = new_workspace(need, q.device)
    st = lib.pkv_decode_step(ctypes.byref(c), _dev(k_new, "k_new", 2), _dev(v_new, "v_new", 2),
                             _dev(slot_mapping, "slot_mapping", dtype=torch.int32), _dev(q, "q", 2), hq,
                             _dev(block_tables, "block_tables", dtype=torch.int32), int(block_tables.shape[1]),
                             _dev(context_lens, "context_lens", dtype=torch.int32), B, int(max_context_len),
                             float(scale), _out(out), _dev(workspace, "workspace"),
                             workspace.numel() * workspace.element_size(), int(partition_blocks),
                             _stream_handle(stream))
    _check(st, "pkv_decode_step")
    return out


def copy(dst, src, stream=None) -> None:
    """Copy the bytes of tensor ``src`` into tensor ``dst`` (same byte size,
    contiguous) with a kernel; either may be on the device or in page-locked
    host memory (``pin_memory()``), which the GPU then reads or writes
    directly (pkv_copy)."""
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("copy needs contiguous tensors")
    nbytes = dst.numel() * dst.element_size()
    if nbytes != src.numel() * src.element_size():
        raise ValueError("copy needs tensors of the same byte size")
    st = load().pkv_copy(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()), nbytes,
                         _stream_handle(stream))
    _check(st, "pkv_copy")


def common_prefix_blocks(block_tables_host, context_lens_host) -> int:
    """The largest J such that every row of the host block table
    [B][max_blocks] starts with row 0's first J ids and every context holds
    16 J tokens (pkv_common_prefix_blocks; host arrays only)."""
    import numpy as np
    t = np.ascontiguousarray(block_tables_host, dtype=np.int32)
    n = np.ascontiguousarray(context_lens_host, dtype=np.int32)
    if t.ndim != 2 or n.ndim != 1 or n.shape[0] != t.shape[0]:
        raise ValueError("block_tables_host must be [B][max_blocks] and context_lens_host [B]")
    return int(load().pkv_common_prefix_blocks(t.ctypes.data, t.shape[1], n.ctypes.data, t.shape[0]))


def decode_shared_prefix_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                                        shared_blocks) -> int:
    n = load().pkv_decode_shared_prefix_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                       max_context_len, shared_blocks)
    if n == 0:
        raise PKVError(2, "pkv_decode_shared_prefix_workspace_size")
    return int(n)


def decode_attention_shared_prefix(k_pool, v_pool, q, block_tables, context_lens, max_context_len: int,
                                   shared_blocks: int, scale: float, out=None, workspace=None, stream=None,
                                   k_scale=None, v_scale=None):
    """Decode attention for a batch whose block tables all start with the
    same ``shared_blocks`` full blocks: those are read once per kv head for
    every sequence (tensor cores), the rest per sequence; returns ``out``
    float32 [B][Hq][d].  e4m3 pools (with their scales) attend the shared
    blocks per sequence."""
    torch = _torch()
    lib = load()
    c = _cache(k_pool, v_pool, k_scale, v_scale, need_scales=True)
    B, hq, d = q.shape
    if d != c.head_dim:
        raise ValueError("q head_dim does not match the pools")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables must be [B][max_blocks] and context_lens [B]")
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = lib.pkv_decode_shared_prefix_workspace_size(B, hq, c.num_kv_heads, d, int(max_context_len),
                                                           int(shared_blocks))
        workspace = new_workspace(need, q.device)
    st = lib.pkv_decode_attention_shared_prefix(
        ctypes.byref(c), _dev(q, "q", 2), hq, _dev(block_tables, "block_tables", dtype=torch.int32),
        int(block_tables.shape[1]), _dev(context_lens, "context_lens", dtype=torch.int32), B, int(max_context_len),
        int(shared_blocks), float(scale), _out(out), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "pkv_decode_attention_shared_prefix")
    return out


def prefill_workspace_size(num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, max_context_len) -> int:
    n = load().pkv_prefill_workspace_size(num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim,
                                          max_context_len)
    if n == 0:
        raise PKVError(2, "pkv_prefill_workspace_size")
    return int(n)


def chunked_prefill_attention(k_pool, v_pool, q, query_start_loc, context_lens, block_tables,
                              max_context_len: int, scale: float, out=None, workspace=None,
                              query_start_loc_host=None, stream=None):
    """Mixed batch of causal prefill chunks and decode rows; returns ``out``
    float32 [Tq][Hq][d]."""
    torch = _torch()
    lib = load()
    c = _cache(k_pool, v_pool)
    T, hq, d = q.shape
    S = int(context_lens.shape[0])
    if query_start_loc.shape[0] != S + 1:
        raise ValueError("query_start_loc must have num_seqs + 1 entries")
    if query_start_loc_host is None:
        query_start_loc_host = query_start_loc
    qh, qhp = _host_i32(query_start_loc_host)
    if out is None:
        out = torch.empty((T, hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = load().pkv_prefill_workspace_size(S, T, hq, c.num_kv_heads, d, int(max_context_len))
        workspace = new_workspace(need, q.device)
    st = lib.pkv_chunked_prefill_attention(
        ctypes.byref(c), _dev(q, "q", 2), hq, T, _dev(query_start_loc, "query_start_loc", dtype=torch.int32), qhp,
        _dev(context_lens, "context_lens", dtype=torch.int32), S,
        _dev(block_tables, "block_tables", dtype=torch.int32), int(block_tables.shape[1]), int(max_context_len),
        float(scale), _out(out), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "pkv_chunked_prefill_attention")
    return out


def _swap(direction, k_pool, v_pool, blocks, slots, host, stream):
    torch = _torch()
    lib = load()
    c = _cache(k_pool, v_pool)
    n = int(blocks.shape[0])
    if slots.shape[0] != n:
        raise ValueError("blocks and slots must have the same length")
    if not isinstance(host, torch.Tensor) or host.is_cuda or not host.is_contiguous():
        raise ValueError("host must be a contiguous CPU tensor in page-locked memory")
    slab = 2 * c.num_kv_heads * 16 * c.head_dim * k_pool.element_size()
    if host.numel() * host.element_size() % slab:
        raise ValueError("host must hold whole slabs of [2][num_kv_heads][16][head_dim] pool elements")
    num_slots = host.numel() * host.element_size() // slab
    st = lib.pkv_swap_blocks(ctypes.byref(c), int(direction), _dev(blocks, "blocks", dtype=torch.int32),
                             _dev(slots, "slots", dtype=torch.int32), n, ctypes.c_void_p(host.data_ptr()),
                             num_slots, _stream_handle(stream))
    _check(st, "pkv_swap_blocks")


def swap_out(k_pool, v_pool, blocks, slots, host, stream=None) -> None:
    """host slab slots[i] <- pool block blocks[i] (K then V); ``host`` is a
    pinned CPU tensor of whole [2][Hkv][16][d] slabs of the pools' elements."""
    _swap(0, k_pool, v_pool, blocks, slots, host, stream)


def swap_in(k_pool, v_pool, blocks, slots, host, stream=None) -> None:
    """pool block blocks[i] <- host slab slots[i]."""
    _swap(1, k_pool, v_pool, blocks, slots, host, stream)


def prefix_keys(token_ids, token_start_loc, max_blocks: int, extra=None, parent_keys=None, keys=None,
                stream=None):
    """Prefix-cache keys (uint8 [S][max_blocks][32]) of the full blocks of each
    token list: key_i = SHA-256(key_{i-1} || 16 token ids (<i4) || extra (<i8))."""
    torch = _torch()
    S = int(token_start_loc.shape[0]) - 1
    if keys is None:
        keys = torch.zeros((max(S, 1), max(max_blocks, 1), 32), dtype=torch.uint8, device=token_ids.device)
    ep = _dev(extra, "extra", dtype=torch.int64) if extra is not None else None
    pp = _dev(parent_keys, "parent_keys", dtype=torch.uint8) if parent_keys is not None else None
    st = load().pkv_prefix_keys(_dev(token_ids, "token_ids", dtype=torch.int32),
                                _dev(token_start_loc, "token_start_loc", dtype=torch.int32), ep, pp, S,
                                int(max_blocks), _dev(keys, "keys", dtype=torch.uint8), _stream_handle(stream))
    _check(st, "pkv_prefix_keys")
    return keys


class Blocks:
    """Block bookkeeping state on one GPU (``pkv_blocks_t``): block tables,
    context lengths, reference counts and the ring of free blocks, as int32
    CUDA tensors owned by this object.  ``block_tables`` and ``context_lens``
    are the arrays the attention calls read.  Every method is one launch on
    the current stream; device-side errors are read with :func:`get_error`."""

    def __init__(self, num_blocks: int, max_seqs: int, max_blocks_per_seq: int, device=None,
                 prefix_cache: bool = False):
        torch = _torch()
        device = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        i32 = dict(dtype=torch.int32, device=device)
        self.num_blocks, self.max_seqs, self.max_blocks_per_seq = num_blocks, max_seqs, max_blocks_per_seq
        n1 = max(num_blocks, 1)
        self.block_tables = torch.empty((max_seqs, max_blocks_per_seq), **i32)
        self.context_lens = torch.empty((max_seqs,), **i32)
        self.ref_counts = torch.empty((n1,), **i32)
        self.free_ring = torch.empty((2 * n1,), **i32)
        self.ring_pos = torch.empty((n1,), **i32)
        self.free_state = torch.empty((3,), **i32)
        self.scratch = torch.empty((3 * n1,), **i32)
        self.table_size = 0
        self.block_keys = self.key_table = self.cached = None
        if prefix_cache:
            self.table_size = 1 << max(1, (2 * n1 - 1).bit_length())
            self.block_keys = torch.zeros((n1, 32), dtype=torch.uint8, device=device)
            self.key_table = torch.empty((self.table_size,), **i32)
            self.cached = torch.empty((n1,), **i32)
        self.reset()

    def _state(self) -> BlocksState:
        ptr = lambda t: t.data_ptr() if t is not None else None
        return BlocksState(self.block_tables.data_ptr(), self.context_lens.data_ptr(), self.ref_counts.data_ptr(),
                           self.free_ring.data_ptr(), self.ring_pos.data_ptr(), self.free_state.data_ptr(),
                           self.scratch.data_ptr(), ptr(self.block_keys), ptr(self.key_table), ptr(self.cached),
                           self.num_blocks, self.max_seqs, self.max_blocks_per_seq, self.table_size)

    def free_queue(self) -> list:
        """The free block ids, least recently freed first (synchronises)."""
        ring, pos = self.free_ring.cpu().tolist(), self.ring_pos.cpu().tolist()
        head, entries, _ = self.free_state.cpu().tolist()
        cap = 2 * self.num_blocks
        out = []
        for e in range(entries):
            idx = (head + e) % cap
            b = ring[idx]
            if 0 <= b < self.num_blocks and pos[b] == idx:
                out.append(b)
        return out

    def match(self, keys, num_keys, matched=None, stream=None):
        """Prefix-cache hits for empty rows: returns matched [S] (int32 CUDA)."""
        torch = _torch()
        S = int(num_keys.shape[0])
        matched = matched if matched is not None else torch.empty((max(S, 1),), dtype=torch.int32,
                                                                  device=self.block_tables.device)
        st = load().pkv_blocks_match(ctypes.byref(self._state()), _dev(keys, "keys", dtype=torch.uint8),
                                     int(keys.shape[1]), _dev(num_keys, "num_keys", dtype=torch.int32), S,
                                     _dev(matched, "matched", dtype=torch.int32), _stream_handle(stream))
        _check(st, "pkv_blocks_match")
        return matched

    def register(self, keys, num_keys, stream=None) -> None:
        """Give rows' full blocks their prefix-cache keys."""
        torch = _torch()
        st = load().pkv_blocks_register(ctypes.byref(self._state()), _dev(keys, "keys", dtype=torch.uint8),
                                        int(keys.shape[1]), _dev(num_keys, "num_keys", dtype=torch.int32),
                                        int(num_keys.shape[0]), _stream_handle(stream))
        _check(st, "pkv_blocks_register")

    def reset(self, stream=None) -> None:
        """Every row empty, every block free (queued 0, 1, 2, ...)."""
        _check(load().pkv_blocks_reset(ctypes.byref(self._state()), _stream_handle(stream)), "pkv_blocks_reset")

    def append(self, query_start_loc, num_tokens: int, slot_mapping=None, cow_src=None, cow_dst=None,
               cow_count=None, stream=None):
        """Row s gains query_start_loc[s+1] - query_start_loc[s] tokens.

        Returns (slot_mapping [num_tokens], cow_src [S], cow_dst [S],
        cow_count [1]) as int32 CUDA tensors (allocated when not given)."""
        torch = _torch()
        S = int(query_start_loc.shape[0]) - 1
        dev = self.block_tables.device
        i32 = dict(dtype=torch.int32, device=dev)
        slot_mapping = slot_mapping if slot_mapping is not None else torch.empty((num_tokens,), **i32)
        cow_src = cow_src if cow_src is not None else torch.empty((max(S, 1),), **i32)
        cow_dst = cow_dst if cow_dst is not None else torch.empty((max(S, 1),), **i32)
        cow_count = cow_count if cow_count is not None else torch.empty((1,), **i32)
        if slot_mapping.shape[0] < num_tokens or cow_src.shape[0] < S or cow_dst.shape[0] < S:
            raise ValueError("output tensors are too small")
        sp = _dev(slot_mapping, "slot_mapping", dtype=torch.int32) if num_tokens > 0 else None
        st = load().pkv_blocks_append(ctypes.byref(self._state()),
                                      _dev(query_start_loc, "query_start_loc", dtype=torch.int32), S,
                                      int(num_tokens), sp, _dev(cow_src, "cow_src", dtype=torch.int32),
                                      _dev(cow_dst, "cow_dst", dtype=torch.int32),
                                      _dev(cow_count, "cow_count", dtype=torch.int32), _stream_handle(stream))
        _check(st, "pkv_blocks_append")
        return slot_mapping, cow_src, cow_dst, cow_count

    def fork(self, parents, children, stream=None) -> None:
        """Row children[i] takes row parents[i]'s blocks and length."""
        torch = _torch()
        n = int(parents.shape[0])
        if children.shape[0] != n:
            raise ValueError("parents and children must have the same length")
        st = load().pkv_blocks_fork(ctypes.byref(self._state()), _dev(parents, "parents", dtype=torch.int32),
                                    _dev(children, "children", dtype=torch.int32), n, _stream_handle(stream))
        _check(st, "pkv_blocks_fork")

    def release(self, rows, stream=None) -> None:
        """Rows drop their blocks (each row last block first) and end empty."""
        torch = _torch()
        st = load().pkv_blocks_release(ctypes.byref(self._state()), _dev(rows, "rows", dtype=torch.int32),
                                       int(rows.shape[0]), _stream_handle(stream))
        _check(st, "pkv_blocks_release")


def test_arm_decode_stall(launches: int) -> None:
    """Test hook: the next ``launches`` decode launches time out on purpose
    (their producer warp issues nothing; the bounded waits of the other warps
    expire after 2 s and record PKV_ERR_TIMEOUT).  0 disarms."""
    _check(load().pkv_test_arm_decode_stall(int(launches)), "pkv_test_arm_decode_stall")


def get_error(stream=None) -> Tuple[int, int]:
    """Synchronise the stream and return (status, detail) of the first
    device-side error since the last call, clearing it."""
    detail = ctypes.c_int32(0)
    st = load().pkv_get_error(_stream_handle(stream), ctypes.byref(detail))
    return int(st), int(detail.value)
