"""GPU checks of pkv_copy (a kernel copy between device memory and page-locked
host memory that the GPU reaches directly): bit-exact in every direction,
refused for pageable host memory, and the end-to-end step pattern (inputs in
from pinned host memory, the decode step, the output back) captured in a CUDA
graph gives the direct calls' result."""
import numpy as np
import pytest
import torch

import pkv_workloads as W
from gpu_helpers import DeviceStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_291_gb300 as p
    p.load()
    return p


@pytest.mark.parametrize("nbytes", [16, 4096, 284928, 3 << 20])
def test_copy_directions_bit_exact(pkv, nbytes):
    rng = np.random.default_rng(nbytes)
    data = torch.from_numpy(rng.integers(0, 256, size=nbytes, dtype=np.uint8))
    host_in = data.pin_memory()
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dev2 = torch.empty_like(dev)
    host_out = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    pkv.copy(dev, host_in)
    pkv.copy(dev2, dev)
    pkv.copy(host_out, dev2)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), data) and torch.equal(host_out, data)


def test_copy_refuses_pageable_host_memory(pkv):
    dev = torch.empty(64, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(64, dtype=torch.uint8)
    with pytest.raises(pkv.PKVError) as e:
        pkv.copy(dev, pageable)
    assert pkv.STATUS_NAMES[e.value.status] == "PKV_ERR_HOST_MEMORY"


def test_step_with_host_io_in_a_graph(pkv):
    """The bench's end-to-end step: one staging copy in, the fused decode
    step, the output copy out, captured and replayed, equals the direct
    call on device inputs."""
    w = W.build_config(2)
    ds = DeviceStep(w)
    k0, v0 = ds.k.clone(), ds.v.clone()
    ref = pkv.decode_step(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots, ds.q, ds.tables, ds.ctx, w.max_context_len,
                          w.scale).clone()
    # The same step from host buffers: q staged through pinned memory.
    host_q = ds.q.cpu().pin_memory()
    dev_q = torch.empty_like(ds.q)
    out = torch.empty_like(ref)
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    ws = pkv.new_workspace(pkv.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                                     w.max_context_len))
    stream = torch.cuda.Stream()
    k, v = k0.clone(), v0.clone()
    torch.cuda.synchronize()

    def step():
        pkv.copy(dev_q, host_q, stream=stream)
        pkv.decode_step(k, v, ds.k_new, ds.v_new, ds.slots, dev_q, ds.tables, ds.ctx, w.max_context_len, w.scale,
                        out=out, workspace=ws, stream=stream)
        pkv.copy(host_out, out, stream=stream)
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    host_out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    assert torch.equal(host_out, ref.cpu())


def test_outputs_written_to_page_locked_host_memory(pkv):
    """An fp32 output in page-locked host memory is written by the kernels
    directly: the decode step, decode attention, the shared-prefix call and
    the mixed batch give the same rows as with device outputs."""
    w = W.build_config(2)
    ds = DeviceStep(w)
    ref = pkv.decode_step(ds.k.clone(), ds.v.clone(), ds.k_new, ds.v_new, ds.slots, ds.q, ds.tables, ds.ctx,
                          w.max_context_len, w.scale)
    host = torch.zeros(tuple(ref.shape), dtype=torch.float32).pin_memory()
    pkv.decode_step(ds.k.clone(), ds.v.clone(), ds.k_new, ds.v_new, ds.slots, ds.q, ds.tables, ds.ctx,
                    w.max_context_len, w.scale, out=host)
    torch.cuda.synchronize()
    assert torch.equal(host, ref.cpu())
    host.zero_()
    dev = pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale)
    pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale, out=host)
    torch.cuda.synchronize()
    assert torch.equal(host, dev.cpu())
    # shared prefix
    J = 10
    ws = W.make_paged("host-out-shared", 5005, 16, 8, 128, [16 * J + 3, 16 * J + 70, 16 * J + 200], [1] * 3,
                      share_prefix_blocks=J)
    d2 = DeviceStep(ws)
    pkv.cache_write(d2.k, d2.v, d2.k_new, d2.v_new, d2.slots)
    dev = pkv.decode_attention_shared_prefix(d2.k, d2.v, d2.q, d2.tables, d2.ctx, ws.max_context_len, J, ws.scale)
    host2 = torch.zeros(tuple(dev.shape), dtype=torch.float32).pin_memory()
    pkv.decode_attention_shared_prefix(d2.k, d2.v, d2.q, d2.tables, d2.ctx, ws.max_context_len, J, ws.scale,
                                       out=host2)
    torch.cuda.synchronize()
    assert torch.equal(host2, dev.cpu())
    # mixed batch (prefill tiles and decode rows)
    wm = W.build_config(5)
    d3 = DeviceStep(wm)
    pkv.cache_write(d3.k, d3.v, d3.k_new, d3.v_new, d3.slots)
    dev = pkv.chunked_prefill_attention(d3.k, d3.v, d3.q, d3.qsl, d3.ctx, d3.tables, wm.max_context_len, wm.scale,
                                        query_start_loc_host=wm.query_start_loc)
    host3 = torch.zeros(tuple(dev.shape), dtype=torch.float32).pin_memory()
    pkv.chunked_prefill_attention(d3.k, d3.v, d3.q, d3.qsl, d3.ctx, d3.tables, wm.max_context_len, wm.scale,
                                  out=host3, query_start_loc_host=wm.query_start_loc)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    assert torch.equal(host3, dev.cpu())
    with pytest.raises(ValueError):
        pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale,
                             out=torch.zeros(tuple(ref.shape), dtype=torch.float32))


def test_page_locked_output_for_e4m3_pools_and_the_static_entry_point(pkv):
    """The page-locked output also serves e4m3 pools (the tensor-core block
    math writes it) and pkv_decode_attention_static: the same rows as with a
    device output."""
    import ctypes
    w = W.build_config(2)
    ds = DeviceStep(w)
    pkv.cache_write(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots)
    nb, hkv, _, d = w.k_pool.shape
    k8 = torch.empty((nb, hkv, 16, d), dtype=torch.uint8, device="cuda")
    v8 = torch.empty_like(k8)
    slots = torch.arange(nb * 16, dtype=torch.int32, device="cuda")
    rk = ds.k.permute(0, 2, 1, 3).reshape(nb * 16, hkv, d).contiguous()
    rv = ds.v.permute(0, 2, 1, 3).reshape(nb * 16, hkv, d).contiguous()
    pkv.cache_write(k8, v8, rk, rv, slots, k_scale=1 / 64, v_scale=1 / 64)
    args = (ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale)
    dev = pkv.decode_attention(k8, v8, *args, k_scale=1 / 64, v_scale=1 / 64)
    host = torch.zeros(tuple(dev.shape), dtype=torch.float32).pin_memory()
    pkv.decode_attention(k8, v8, *args, out=host, k_scale=1 / 64, v_scale=1 / 64)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    assert torch.equal(host, dev.cpu())
    # the allocation-free entry point, bf16 pools
    lib = pkv.load()
    P, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    lib.pkv_decode_attention_static.argtypes = [ctypes.POINTER(pkv.Cache), P, i32, P, i32, P, i32, i32, f32, P, P]
    lib.pkv_decode_attention_static.restype = ctypes.c_int
    dev = pkv.decode_attention(ds.k, ds.v, *args)
    host.zero_()
    cache = pkv._cache(ds.k, ds.v, None, None)
    st = lib.pkv_decode_attention_static(ctypes.byref(cache), ctypes.c_void_p(ds.q.data_ptr()), w.num_q_heads,
                                         ctypes.c_void_p(ds.tables.data_ptr()), int(ds.tables.shape[1]),
                                         ctypes.c_void_p(ds.ctx.data_ptr()), w.num_seqs, w.max_context_len,
                                         ctypes.c_float(w.scale), ctypes.c_void_p(host.data_ptr()), None)
    assert st == 0, pkv.status_string(st)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    assert torch.equal(host, dev.cpu())
