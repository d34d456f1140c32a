"""Pins for the oracle's block swap (no GPU): swapping a block out and into
another block is copy_blocks; out and back in is the identity; a negative
block id skips the pair ([ENG] "traffic characteristics": KV moved to CPU
memory while a request is idle and brought back for the next turn)."""
import numpy as np

import oracle


def pools(seed, nb=12, hkv=2, d=64):
    rng = np.random.default_rng(seed)
    k = rng.integers(0, 2 ** 16, size=(nb, hkv, 16, d), dtype=np.uint16)
    v = rng.integers(0, 2 ** 16, size=(nb, hkv, 16, d), dtype=np.uint16)
    return k, v


def test_out_then_in_elsewhere_is_copy_blocks():
    k, v = pools(1)
    k2, v2 = k.copy(), v.copy()
    host = np.zeros((5, 2) + k.shape[1:], dtype=np.uint16)
    oracle.swap_blocks(0, k, v, [3, 7, -1, 0], [4, 1, 2, 0], host)
    oracle.swap_blocks(1, k, v, [9, 10, 11], [4, 1, 0], host)
    oracle.copy_blocks(k2, v2, np.array([3, 7, 0], np.int32), np.array([9, 10, 11], np.int32))
    assert np.array_equal(k, k2) and np.array_equal(v, v2)
    assert not host[2].any()                                    # skipped pair wrote nothing


def test_round_trip_restores_a_released_block():
    k, v = pools(2)
    saved_k, saved_v = k[5].copy(), v[5].copy()
    host = np.zeros((1, 2) + k.shape[1:], dtype=np.uint16)
    oracle.swap_blocks(0, k, v, [5], [0], host)
    k[5], v[5] = 0, 0                                           # the block is reused meanwhile
    oracle.swap_blocks(1, k, v, [5], [0], host)
    assert np.array_equal(k[5], saved_k) and np.array_equal(v[5], saved_v)
