"""The allocation-free decode entry point.

pkv_decode_attention_static serves callers that may not call cudaMalloc
where they decode (host callbacks, plug-ins that do not own the process's
memory pool, runtimes that freeze device allocation): it runs the regular
decode on a scratch buffer built into the library.  These tests call it
through the C-ABI and check it against pkv_decode_attention with a
caller-provided workspace, twice in a row (the shared buffer keeps the
previous call's contents, so the second call checks that it is reset).

The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import pkv_workloads as W
from gpu_helpers import DeviceStep, assert_close

pytestmark = pytest.mark.gpu

PKV_ERR_SCRATCH_LIMIT = 13


@pytest.fixture(scope="module")
def lib():
    import paged_kv_cache_291_gb300 as pkv
    lib = pkv.load()
    P, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    lib.pkv_decode_attention_static.argtypes = [ctypes.POINTER(pkv.Cache), P, i32, P, i32, P, i32, i32, f32, P, P]
    lib.pkv_decode_attention_static.restype = ctypes.c_int
    lib.pkv_decode_static_scratch_bytes.argtypes = []
    lib.pkv_decode_static_scratch_bytes.restype = ctypes.c_size_t
    return lib


def _static_call(lib, pkv, ds, w, out, stream):
    cache = pkv._cache(ds.k, ds.v)
    return lib.pkv_decode_attention_static(
        ctypes.byref(cache), ctypes.c_void_p(ds.q.data_ptr()), w.num_q_heads, ctypes.c_void_p(ds.tables.data_ptr()),
        int(ds.tables.shape[1]), ctypes.c_void_p(ds.ctx.data_ptr()), w.num_seqs, w.max_context_len,
        ctypes.c_float(w.scale), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("cfg", [2, 4])
def test_static_scratch_matches_workspace_call(lib, cfg):
    import paged_kv_cache_291_gb300 as pkv
    w = W.build_config(cfg)
    ds = DeviceStep(w)
    ref = ds.run(pkv).clone()  # copy_blocks + cache_write + decode with a torch workspace
    stream = torch.cuda.current_stream()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        st = _static_call(lib, pkv, ds, w, out, stream)
        assert st == 0, pkv.status_string(st)
        torch.cuda.synchronize()
        assert pkv.get_error() == (0, 0)
        assert_close(out.cpu().numpy(), ref.cpu().numpy(), f"static scratch, config {cfg}")


def test_static_scratch_split_contexts(lib):
    """Long contexts (split across SMs, so the scratch holds partial results
    and arrival counters) on two calls in a row."""
    import paged_kv_cache_291_gb300 as pkv
    w = W.make_paged("split", 3, 16, 8, 128, [9000, 33, 4000, 1], [1] * 4)
    ds = DeviceStep(w)
    pkv.cache_write(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots)
    ref = pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale).clone()
    stream = torch.cuda.current_stream()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _static_call(lib, pkv, ds, w, out, stream) == 0
        torch.cuda.synchronize()
        assert pkv.get_error() == (0, 0)
        assert_close(out.cpu().numpy(), ref.cpu().numpy(), "static scratch, split contexts")


def test_static_scratch_rejects_batches_beyond_its_size(lib):
    """A batch whose workspace would exceed the built-in buffer is refused
    before anything is launched."""
    import paged_kv_cache_291_gb300 as pkv
    w = W.make_paged("tiny", 4, 8, 8, 128, [20], [1])
    ds = DeviceStep(w)
    out = torch.zeros((1, 8, 128), dtype=torch.float32, device="cuda")
    limit = lib.pkv_decode_static_scratch_bytes()
    assert limit == 4 << 20
    big_seqs = 200000  # one 4-byte arrival counter per (sequence, kv head) alone exceeds 4 MiB
    assert pkv.decode_workspace_size(big_seqs, 8, 8, 128, 20) > limit
    cache = pkv._cache(ds.k, ds.v)
    st = lib.pkv_decode_attention_static(
        ctypes.byref(cache), ctypes.c_void_p(ds.q.data_ptr()), 8, ctypes.c_void_p(ds.tables.data_ptr()), 2,
        ctypes.c_void_p(ds.ctx.data_ptr()), big_seqs, 20, ctypes.c_float(w.scale), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == PKV_ERR_SCRATCH_LIMIT
    assert "scratch" in pkv.status_string(st)
    torch.cuda.synchronize()
    assert torch.all(out == 0)
