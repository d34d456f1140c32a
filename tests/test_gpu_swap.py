"""GPU parity of pkv_swap_blocks (KV offloading to page-locked host memory)
against the oracle: bit-exact host slabs and pool blocks."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import dev_tensor, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_291_gb300 as p
    p.load()
    return p


def i32(x):
    return torch.tensor(np.asarray(x, dtype=np.int32), device="cuda")


@pytest.mark.parametrize("hkv,d", [(8, 128), (2, 64)])
def test_swap_out_and_in_match_the_oracle(pkv, hkv, d):
    rng = np.random.default_rng(hkv + d)
    NB, NS = 64, 40
    k = rng.integers(0, 2 ** 16, size=(NB, hkv, 16, d), dtype=np.uint16)
    v = rng.integers(0, 2 ** 16, size=(NB, hkv, 16, d), dtype=np.uint16)
    kd, vd = dev_tensor(k), dev_tensor(v)
    host = torch.zeros((NS, 2, hkv, 16, d), dtype=torch.int16).pin_memory()
    ref = np.zeros((NS, 2, hkv, 16, d), dtype=np.uint16)
    blocks = rng.choice(NB, size=30, replace=False)
    slots = rng.choice(NS, size=30, replace=False)
    blocks[[4, 17]] = -1                                        # skipped pairs
    pkv.swap_out(kd, vd, i32(blocks), i32(slots), host)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    oracle.swap_blocks(0, k, v, blocks, slots, ref)
    assert np.array_equal(host.numpy().view(np.uint16), ref)
    dst = rng.choice(NB, size=30, replace=False)
    pkv.swap_in(kd, vd, i32(dst), i32(slots), host)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    oracle.swap_blocks(1, k, v, np.where(blocks < 0, -1, dst), slots, ref)
    # pairs skipped on the way out were swapped in from zero slabs on the device
    for i in np.flatnonzero(blocks < 0):
        k[dst[i]], v[dst[i]] = ref[slots[i], 0], ref[slots[i], 1]
    assert np.array_equal(host_bits(kd), k) and np.array_equal(host_bits(vd), v)


def test_out_of_range_slot_is_a_range_error_and_the_rest_moves(pkv):
    k = np.arange(4 * 2 * 16 * 64, dtype=np.uint16).reshape(4, 2, 16, 64)
    kd, vd = dev_tensor(k), dev_tensor(k.copy())
    host = torch.zeros((2, 2, 2, 16, 64), dtype=torch.int16).pin_memory()
    pkv.swap_out(kd, vd, i32([0, 1]), i32([1, 2]), host)        # slot 2 does not exist
    torch.cuda.synchronize()
    assert pkv.get_error() == (9, 1)
    assert np.array_equal(host.numpy().view(np.uint16)[1, 0], k[0])


def test_memory_that_is_not_mapped_pinned_host_memory_is_refused(pkv):
    k = np.zeros((4, 2, 16, 64), dtype=np.uint16)
    kd, vd = dev_tensor(k), dev_tensor(k)
    pageable = torch.zeros((2, 2, 2, 16, 64), dtype=torch.int16)
    with pytest.raises(pkv.PKVError) as e:
        pkv.swap_out(kd, vd, i32([0]), i32([0]), pageable)
    assert e.value.status == 15
    lib = pkv.load()
    c = pkv._cache(kd, vd)
    on_device = torch.zeros(2 * 2 * 16 * 64 * 2, dtype=torch.int16, device="cuda")
    st = lib.pkv_swap_blocks(ctypes.byref(c), 0, ctypes.c_void_p(i32([0]).data_ptr()),
                             ctypes.c_void_p(i32([0]).data_ptr()), 1, ctypes.c_void_p(on_device.data_ptr()), 1,
                             None)
    assert st == 15
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
