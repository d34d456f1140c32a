"""CPU checks of the shared-prefix decode's host side: pkv_common_prefix_blocks
(host arrays only) against a brute-force definition, and the argument checks
that pkv_decode_attention_shared_prefix makes before touching a device."""
import ctypes

import numpy as np
import pytest

import pkv_workloads as W


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_291_gb300 as p
    from paged_kv_cache_291_gb300 import build
    build.build()
    p.load()
    return p


def brute_force(tables, lens):
    """Largest J with every row's first J ids equal to row 0's and every
    context holding 16 J tokens, by trying each J."""
    S, MB = tables.shape
    best = 0
    for J in range(MB + 1):
        if all(int(lens[s]) >= 16 * J for s in range(S)) and all(
                np.array_equal(tables[s, :J], tables[0, :J]) for s in range(S)):
            best = J
    return best


def test_common_prefix_of_workloads(pkv):
    w = W.build_config(4)
    assert pkv.common_prefix_blocks(w.block_tables, w.context_lens) == 187
    w2 = W.build_config(2)
    assert pkv.common_prefix_blocks(w2.block_tables, w2.context_lens) == 0


@pytest.mark.parametrize("seed", range(12))
def test_common_prefix_random_tables(pkv, seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 9))
    MB = int(rng.integers(1, 12))
    J0 = int(rng.integers(0, MB + 1))
    base = rng.integers(0, 1000, size=MB).astype(np.int32)
    tables = np.tile(base, (S, 1))
    # break the shared part at a random place in some rows, keep the rest random
    for s in range(1, S):
        cut = int(rng.integers(J0, MB + 1))
        if cut < MB:
            tables[s, cut:] = rng.integers(1000, 2000, size=MB - cut)
    lens = rng.integers(0, 16 * MB + 1, size=S).astype(np.int32)
    assert pkv.common_prefix_blocks(tables, lens) == brute_force(tables, lens)


def test_common_prefix_edge_cases(pkv):
    t = np.array([[5, 6, 7], [5, 6, 8]], dtype=np.int32)
    assert pkv.common_prefix_blocks(t, np.array([48, 48], np.int32)) == 2
    assert pkv.common_prefix_blocks(t, np.array([48, 31], np.int32)) == 1   # second context holds 1 full block
    assert pkv.common_prefix_blocks(t, np.array([0, 48], np.int32)) == 0
    assert pkv.common_prefix_blocks(t[:1], np.array([47], np.int32)) == 2    # one sequence: its own full blocks
    lib = pkv.load()
    assert lib.pkv_common_prefix_blocks(None, 3, None, 2) == 0


def test_shared_blocks_argument_checks_without_gpu(pkv):
    """shared_blocks < 0, past the table width, or more tokens than
    max_context_len: PKV_ERR_SHAPE (2) before any device work."""
    lib = pkv.load()
    fake = ctypes.c_void_p(1 << 20)
    c = pkv.Cache(1 << 20, 1 << 20, 64, 8, 128, 16, pkv.PKV_KV_BF16, 1.0, 1.0)

    def call(J, max_blocks=10, max_ctx=160):
        return lib.pkv_decode_attention_shared_prefix(ctypes.byref(c), fake, 16, fake, max_blocks, fake, 4, max_ctx,
                                                      J, 0.1, fake, fake, 1 << 20, None)
    assert call(-1) == 2
    assert call(11) == 2
    assert call(10, max_ctx=159) == 2
