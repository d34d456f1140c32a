"""GPU parity of the fused decode step (pkv_decode_step: the store of each
sequence's new row and decode attention in one launch) against the oracle's
cache write followed by attention, and against the library's own two-call
path, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
import pkv_workloads as W
from gpu_helpers import DeviceStep, assert_close, dev_tensor, host_bits

pytestmark = pytest.mark.gpu

PKV_ERR_RANGE = 9


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_291_gb300 as p
    p.load()
    return p


def fused(pkv, ds, partition_blocks=0, slots=None, workspace=None):
    w = ds.w
    return pkv.decode_step(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots if slots is None else slots, ds.q, ds.tables,
                           ds.ctx, w.max_context_len, w.scale, partition_blocks=partition_blocks,
                           workspace=workspace)


def check_fused(pkv, w, partition_blocks=0, threads=8):
    """Fused step on one copy of the pools, cache_write + decode_attention on
    another: pools bit-exact against the oracle, outputs within tolerance of
    the oracle and bit-identical between the two paths."""
    a, b = DeviceStep(w), DeviceStep(w)
    out_a = fused(pkv, a, partition_blocks)
    out_b = b.run(pkv, partition_blocks=partition_blocks)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    k_ref, v_ref, ref = oracle.run_step(w, threads=threads)
    assert np.array_equal(host_bits(a.k), k_ref) and np.array_equal(host_bits(a.v), v_ref), "pools differ"
    assert_close(out_a.cpu().numpy(), ref, w.name)
    assert torch.equal(out_a, out_b), "fused step and the two-call path differ"


@pytest.mark.parametrize("cfg", [1, 2])
def test_fused_step_configs(pkv, cfg):
    check_fused(pkv, W.build_config(cfg))


@pytest.mark.slow
def test_fused_step_long_contexts(pkv):
    """LLaMA-13B MHA shape in full: the new rows of the 32,768-token
    sequences fall in split pairs' last parts."""
    check_fused(pkv, W.build_config(3), threads=16)


@pytest.mark.parametrize("pb", [1, 2, 3, 7, 40])
def test_fused_step_forced_partitions(pkv, pb):
    """New rows at every offset of a block (n = 1, 15, 16, 17, 31, 32, 33 ...)
    and in parts of every size."""
    w = W.make_paged("fused parts", 78, 16, 8, 128, [1, 15, 16, 17, 31, 32, 33, 100, 640, 641], [1] * 10)
    check_fused(pkv, w, partition_blocks=pb)


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (16, 4, 128), (64, 8, 128), (8, 1, 64), (16, 8, 64),
                                      (32, 4, 64), (40, 40, 64)])
def test_fused_step_head_shapes(pkv, hq, hkv, d):
    ctx = [1, 2, 16, 17, 48, 250, 333]
    check_fused(pkv, W.make_paged("fused heads", hq * 101 + hkv + d, hq, hkv, d, ctx, [1] * len(ctx)))


def test_fused_step_many_sequences(pkv):
    ctx = W.randint_inclusive(6, 7, 300, 1, 700)
    check_fused(pkv, W.make_paged("fused ragged", 6, 16, 8, 128, ctx, [1] * 300))


def test_negative_slot_skips_the_store(pkv):
    """A negative slot leaves the pool's row as it is, and attention reads it
    there: rows written earlier with other values stay."""
    w = W.make_paged("fused skip", 31, 16, 8, 128, [5, 16, 40, 300], [1] * 4)
    skip = np.array([1, 3])
    other_k = W.normal_bf16(99, 1, w.k_new.size).reshape(w.k_new.shape)
    other_v = W.normal_bf16(99, 2, w.v_new.size).reshape(w.v_new.shape)
    ds = DeviceStep(w)
    pkv.cache_write(ds.k, ds.v, dev_tensor(other_k[skip]), dev_tensor(other_v[skip]), dev_tensor(w.slot_mapping[skip]))
    slots = w.slot_mapping.copy()
    slots[skip] = -1
    out = fused(pkv, ds, slots=dev_tensor(slots))
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    k, v = w.k_pool.copy(), w.v_pool.copy()
    oracle.cache_write(k, v, other_k[skip], other_v[skip], w.slot_mapping[skip])
    oracle.cache_write(k, v, w.k_new, w.v_new, slots)
    assert np.array_equal(host_bits(ds.k), k) and np.array_equal(host_bits(ds.v), v)
    ref = oracle.decode_attention(k, v, w.q, w.context_lens, w.block_tables, w.scale)
    assert_close(out.cpu().numpy(), ref, "skipped stores")


def test_slot_of_another_position_is_refused(pkv):
    """A slot that is not the last position's is reported (PKV_ERR_RANGE,
    detail: the sequence) and nothing is written there or at the right slot;
    the other sequences are unaffected."""
    w = W.make_paged("fused wrong slot", 32, 16, 8, 128, [40, 300, 77], [1] * 3)
    ds = DeviceStep(w)
    slots = w.slot_mapping.copy()
    wrong = int(w.block_tables[1, 3]) * 16 + 5   # a row of sequence 1's own context
    slots[1] = wrong
    out = fused(pkv, ds, slots=dev_tensor(slots))
    torch.cuda.synchronize()
    assert pkv.get_error() == (PKV_ERR_RANGE, 1)
    k, v = w.k_pool.copy(), w.v_pool.copy()
    keep = np.array([0, 2])
    oracle.cache_write(k, v, w.k_new[keep], w.v_new[keep], w.slot_mapping[keep])
    assert np.array_equal(host_bits(ds.k), k) and np.array_equal(host_bits(ds.v), v)
    ref = oracle.decode_attention(k, v, w.q, w.context_lens, w.block_tables, w.scale)
    assert_close(out.cpu().numpy()[keep], ref[keep], "sequences with right slots")


@pytest.mark.parametrize("cfg", [1, 2])
def test_fused_step_e4m3_pools(pkv, cfg):
    """e4m3 pools: the new rows are quantised as pkv_cache_write does (codes
    equal to the oracle's) and attention runs over those codes."""
    w = W.build_config(cfg)
    ks, vs = np.float32(0.0123), np.float32(0.0171)
    ik, iv = np.float32(1) / ks, np.float32(1) / vs
    k8, v8 = fp8.quantize_bf16_rows(w.k_pool, ik), fp8.quantize_bf16_rows(w.v_pool, iv)
    kd, vd = dev_tensor(k8), dev_tensor(v8)
    out = pkv.decode_step(kd, vd, dev_tensor(w.k_new), dev_tensor(w.v_new), dev_tensor(w.slot_mapping),
                          dev_tensor(w.q), dev_tensor(w.block_tables), dev_tensor(w.context_lens), w.max_context_len,
                          w.scale, k_scale=float(ks), v_scale=float(vs))
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    fp8.cache_write(k8, v8, w.k_new, w.v_new, w.slot_mapping, ik, iv)
    assert np.array_equal(kd.cpu().numpy(), k8) and np.array_equal(vd.cpu().numpy(), v8)
    ref = fp8.decode_attention(k8, v8, w.q, w.context_lens, w.block_tables, w.scale, float(ks), float(vs))
    assert_close(out.cpu().numpy(), ref, f"{w.name} (e4m3, fused)")


def test_fused_step_reuses_its_workspace_and_is_deterministic(pkv):
    w = W.make_paged("fused reuse", 33, 16, 8, 128, [5000, 17, 3000, 1], [1] * 4)
    ds = DeviceStep(w)
    need = pkv.decode_workspace_size(4, 16, 8, 128, w.max_context_len, 4)
    ws = pkv.new_workspace(need)
    a = fused(pkv, ds, partition_blocks=4, workspace=ws).clone()
    b = fused(pkv, ds, partition_blocks=4, workspace=ws).clone()
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    assert torch.equal(a, b)
    assert int(ws[:512].count_nonzero().item()) == 0
    _, _, ref = oracle.run_step(w)
    assert_close(a.cpu().numpy(), ref, "fused reuse")


def test_fused_step_checks_its_arguments(pkv):
    w = W.build_config(1)
    ds = DeviceStep(w)
    with pytest.raises(ValueError):
        pkv.decode_step(ds.k, ds.v, ds.k_new[:2], ds.v_new, ds.slots, ds.q, ds.tables, ds.ctx, w.max_context_len,
                        w.scale)
    lib = pkv.load()
    c = pkv._cache(ds.k, ds.v)
    import ctypes
    st = lib.pkv_decode_step(ctypes.byref(c), None, None, None, ds.q.data_ptr(), w.num_q_heads,
                             ds.tables.data_ptr(), w.max_blocks_per_seq, ds.ctx.data_ptr(), w.num_seqs,
                             w.max_context_len, w.scale, None, None, 0, 0, None)
    assert st == 1  # PKV_ERR_NULL
