"""Host-side checks of the seeded workload builder (no GPU, no attention math)."""
import numpy as np
import pytest

import pkv_workloads as W


def test_generator_is_deterministic_and_counter_based():
    a = W.normal_bf16(5, 1, 10001)
    b = W.normal_bf16(5, 1, 10001)
    assert np.array_equal(a, b)
    # element i does not depend on how many elements were asked for
    assert np.array_equal(W.normal_bf16(5, 1, 100), a[:100])
    assert not np.array_equal(W.normal_bf16(6, 1, 100), a[:100])
    assert not np.array_equal(W.normal_bf16(5, 2, 100), a[:100])


def test_generator_is_standard_normal():
    import torch
    x = torch.from_numpy(W.normal_bf16(9, 3, 1 << 20).view(np.int16)).view(torch.bfloat16).double().numpy()
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    assert abs(np.mean(np.abs(x) < 1.0) - 0.6827) < 3e-3


def test_multithreaded_generation_matches_serial():
    n = (1 << 22) * 2 + 123
    assert np.array_equal(W.normal_bf16(1, 1, n, threads=1), W.normal_bf16(1, 1, n, threads=4))


def test_permutation_and_randint():
    p = W.permutation(3, 6, 1000)
    assert sorted(p.tolist()) == list(range(1000))
    r = W.randint_inclusive(3, 7, 5000, 300, 4096)
    assert r.min() >= 300 and r.max() <= 4096 and len(set(r.tolist())) > 1000


def _check_layout(w):
    """Every cached slot holds data, every other slot is NaN; tables valid."""
    nb = w.num_blocks
    used = np.zeros((nb, 16), bool)
    for s in range(w.num_seqs):
        n = int(w.context_lens[s])
        ql = int(w.query_lens[s])
        pos = np.arange(n - ql)
        used[w.block_tables[s][pos // 16], pos % 16] = True
    if w.copy_src is not None:  # the original shared partial block is the only extra data
        pass
    k = w.k_pool.transpose(0, 2, 1, 3)
    is_nan = (k == W.BF16_NAN).all(axis=(2, 3))
    return used, is_nan


@pytest.mark.parametrize("cfg", [1, 2, 5])
def test_config_layouts(cfg):
    w = W.build_config(cfg)
    used, is_nan = _check_layout(w)
    assert not (used & is_nan).any()
    assert (is_nan | used).all()
    assert w.block_tables.max() < w.num_blocks
    # each sequence's blocks are distinct and no two sequences share a block
    ids = np.concatenate([w.block_tables[s][:W.blocks_for(w.context_lens[s])] for s in range(w.num_seqs)])
    assert len(np.unique(ids)) == len(ids)
    # new rows land in their own sequence's next slots
    T = w.slot_mapping.shape[0]
    assert T == w.query_start_loc[-1] == w.q.shape[0]
    for s in range(w.num_seqs):
        n, ql = int(w.context_lens[s]), int(w.query_lens[s])
        pos = np.arange(n - ql, n)
        want = w.block_tables[s][pos // 16] * 16 + pos % 16
        r0 = w.query_start_loc[s]
        assert np.array_equal(w.slot_mapping[r0:r0 + ql], want)


def test_config_shapes():
    w1 = W.build_config(1)
    assert (w1.num_q_heads, w1.num_kv_heads, w1.head_dim, w1.num_blocks) == (32, 8, 64, 128)
    assert w1.context_lens.tolist() == [1, 17, 100, 512]
    w2 = W.build_config(2)
    assert (w2.num_q_heads, w2.num_kv_heads, w2.head_dim, w2.num_blocks) == (16, 8, 128, 1378)
    assert w2.num_seqs == 34 and (w2.context_lens == 640).all() and w2.is_decode
    w5 = W.build_config(5)
    assert w5.num_seqs == 35 and w5.num_tokens == 3 * 512 + 32
    assert w5.query_lens.tolist()[:3] == [512] * 3 and w5.context_lens.tolist()[:4] == [1536] * 3 + [300]
    assert w5.num_tokens <= 2048
    dec = w5.context_lens[3:]
    assert dec.min() >= 300 and dec.max() <= 4096


def test_mha_config_shape_small():
    w = W.llama13b_mha_decode(long_len=600, n_short=6, n_long=2)
    assert (w.num_q_heads, w.num_kv_heads) == (40, 40)
    assert w.context_lens.tolist()[-2:] == [600, 600]
    assert all(128 <= n <= 2048 for n in w.context_lens[:6])


def test_prefix_share_config():
    w = W.build_config(4)
    assert w.num_seqs == 32 and (w.context_lens == 3032).all()
    assert (w.block_tables[:, :187] == w.block_tables[0, :187]).all()
    assert len(np.unique(w.block_tables[:, 187:])) == 32 * 3
    assert (w.copy_dst == w.block_tables[:, 187]).all()
    assert (w.copy_src == w.meta["orig_partial"]).all()
    assert w.slot_mapping.shape[0] == 32 * 32
    # the original partial block holds 8 valid rows, then poison
    kp = w.k_pool[w.meta["orig_partial"]]
    assert not (kp[:, :8] == W.BF16_NAN).all()
    assert (kp[:, 8:] == W.BF16_NAN).all()
    # the copy destinations start fully poisoned
    assert (w.k_pool[w.copy_dst] == W.BF16_NAN).all()
