"""GPU parity of cache_write and copy_blocks: bit-exact against the oracle on
whole pools (poison included, so a stray write anywhere shows up)."""
import numpy as np
import pytest
import torch

import oracle
import pkv_workloads as W
from gpu_helpers import dev_tensor, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_291_gb300 as p
    p.load()
    return p


def _pools(w):
    return dev_tensor(w.k_pool), dev_tensor(w.v_pool)


@pytest.mark.parametrize("cfg", [1, 2, 5])
def test_cache_write_bit_exact(pkv, cfg):
    w = W.build_config(cfg)
    k, v = _pools(w)
    pkv.cache_write(k, v, dev_tensor(w.k_new), dev_tensor(w.v_new), dev_tensor(w.slot_mapping))
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    k_ref, v_ref = w.k_pool.copy(), w.v_pool.copy()
    oracle.cache_write(k_ref, v_ref, w.k_new, w.v_new, w.slot_mapping)
    assert np.array_equal(host_bits(k), k_ref)
    assert np.array_equal(host_bits(v), v_ref)


@pytest.mark.parametrize("hkv,d", [(8, 128), (2, 64), (1, 128), (40, 128)])
def test_cache_write_skips_negative_and_ragged(pkv, hkv, d):
    nb = 37
    rng = np.random.default_rng(hkv * d)
    k0 = W.normal_bf16(1, 1, nb * hkv * 16 * d).reshape(nb, hkv, 16, d)
    v0 = W.normal_bf16(1, 2, nb * hkv * 16 * d).reshape(nb, hkv, 16, d)
    T = 301
    slots = rng.permutation(nb * 16)[:T].astype(np.int32)
    slots[rng.random(T) < 0.1] = -1
    kn = W.normal_bf16(2, 1, T * hkv * d).reshape(T, hkv, d)
    vn = W.normal_bf16(2, 2, T * hkv * d).reshape(T, hkv, d)
    k, v = dev_tensor(k0), dev_tensor(v0)
    pkv.cache_write(k, v, dev_tensor(kn), dev_tensor(vn), dev_tensor(slots))
    kr, vr = k0.copy(), v0.copy()
    oracle.cache_write(kr, vr, kn, vn, slots)
    assert np.array_equal(host_bits(k), kr) and np.array_equal(host_bits(v), vr)
    assert pkv.get_error() == (0, 0)


def test_cache_write_out_of_range_slot_reports_and_skips(pkv):
    nb, hkv, d = 4, 2, 64
    k0 = W.normal_bf16(3, 1, nb * hkv * 16 * d).reshape(nb, hkv, 16, d)
    k, v = dev_tensor(k0), dev_tensor(k0)
    kn = W.normal_bf16(3, 2, 2 * hkv * d).reshape(2, hkv, d)
    slots = np.array([5, nb * 16 + 3], np.int32)  # second slot is past the pool
    pkv.cache_write(k, v, dev_tensor(kn), dev_tensor(kn), dev_tensor(slots))
    st, detail = pkv.get_error()
    assert st == 9 and detail == 1
    kr = k0.copy()
    kr[0, :, 5, :] = kn[0]
    assert np.array_equal(host_bits(k), kr)
    assert pkv.get_error() == (0, 0)  # cleared


def test_copy_blocks_prefix_share_config(pkv):
    w = W.build_config(4)
    k, v = _pools(w)
    pkv.copy_blocks(k, v, dev_tensor(w.copy_src), dev_tensor(w.copy_dst))
    kr, vr = w.k_pool.copy(), w.v_pool.copy()
    oracle.copy_blocks(kr, vr, w.copy_src, w.copy_dst)
    assert np.array_equal(host_bits(k), kr) and np.array_equal(host_bits(v), vr)
    # every copy is byte-identical to the shared original
    src = w.copy_src[0]
    for dst in w.copy_dst:
        assert np.array_equal(kr[dst], w.k_pool[src])
    assert pkv.get_error() == (0, 0)


@pytest.mark.parametrize("hkv,d,n", [(8, 128, 1), (3, 64, 70), (40, 128, 5)])
def test_copy_blocks_shapes(pkv, hkv, d, n):
    nb = 2 * n + 3
    k0 = W.normal_bf16(4, 1, nb * hkv * 16 * d).reshape(nb, hkv, 16, d)
    v0 = W.normal_bf16(4, 2, nb * hkv * 16 * d).reshape(nb, hkv, 16, d)
    perm = W.permutation(4, 6, nb)
    src, dst = perm[:n].copy(), perm[n:2 * n].copy()
    k, v = dev_tensor(k0), dev_tensor(v0)
    pkv.copy_blocks(k, v, dev_tensor(src), dev_tensor(dst))
    kr, vr = k0.copy(), v0.copy()
    oracle.copy_blocks(kr, vr, src, dst)
    assert np.array_equal(host_bits(k), kr) and np.array_equal(host_bits(v), vr)


def test_copy_blocks_rejects_aliasing_on_host(pkv):
    w = W.build_config(1)
    k, v = _pools(w)
    before = host_bits(k).copy()
    for src, dst in (([1, 2], [3, 3]), ([1, 2], [2, 4])):
        with pytest.raises(pkv.PKVError) as e:
            pkv.copy_blocks(k, v, dev_tensor(np.array(src, np.int32)), dev_tensor(np.array(dst, np.int32)))
        assert e.value.status == 6
    with pytest.raises(pkv.PKVError) as e:
        pkv.copy_blocks(k, v, dev_tensor(np.array([0], np.int32)), dev_tensor(np.array([128], np.int32)))
    assert e.value.status == 9
    assert np.array_equal(host_bits(k), before)


def test_copy_blocks_device_range_check(pkv):
    """Without the host copies the kernel itself skips and reports bad ids."""
    w = W.build_config(1)
    k, v = _pools(w)
    before = host_bits(k).copy()
    pkv.copy_blocks(k, v, dev_tensor(np.array([0, 500], np.int32)), dev_tensor(np.array([1, 2], np.int32)),
                    check_host=False)
    st, detail = pkv.get_error()
    assert st == 9 and detail == 1
    want = before.copy()
    want[1] = before[0]
    assert np.array_equal(host_bits(k), want)
