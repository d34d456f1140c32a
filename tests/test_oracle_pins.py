"""Pins for the CPU oracle: each test checks the oracle against something
other than itself -- a library attention routine, a closed form, numpy
indexing, exact invariants the pages state, or brute force.

Page citations:
  [KV2]  "LLM KV cache part 2: KV management in serving engines" (ttlab.hopto.org)
  [ENG]  "How LLM inference engines work: from one token to agent caches"
         (xiaohu-jiedu.pages.dev)
"""
import math

import numpy as np
import pytest
import torch

import oracle
import pkv_workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def bf16_bits(x):
    """float array -> bf16 bits via torch (round to nearest even)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def widen(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def sdpa_reference(k_pool, v_pool, q, qsl, ctx, tables, scale):
    """Independent reference: numpy fancy-index gather + torch SDPA in float64
    with an explicit causal mask and contiguous GQA groups."""
    nb, hkv, bs, d = k_pool.shape
    T, hq, _ = q.shape
    G = hq // hkv
    K = widen(k_pool)
    V = widen(v_pool)
    Q = widen(q)
    out = np.zeros((T, hq, d))
    for s in range(len(ctx)):
        n = int(ctx[s])
        r0, r1 = int(qsl[s]), int(qsl[s + 1])
        if r1 == r0 or n == 0:
            continue
        j = np.arange(n)
        phys = tables[s][j // bs]
        Kc = K[phys, :, j % bs, :]  # [n][hkv][d]
        Vc = V[phys, :, j % bs, :]
        Kh = torch.from_numpy(np.repeat(Kc.transpose(1, 0, 2), G, axis=0))  # [hq][n][d]
        Vh = torch.from_numpy(np.repeat(Vc.transpose(1, 0, 2), G, axis=0))
        Qh = torch.from_numpy(Q[r0:r1].transpose(1, 0, 2).copy())  # [hq][qlen][d]
        qlen = r1 - r0
        pos = n - qlen + np.arange(qlen)
        mask = torch.from_numpy(j[None, :] <= pos[:, None])
        o = torch.nn.functional.scaled_dot_product_attention(Qh, Kh, Vh, attn_mask=mask, scale=scale)
        out[r0:r1] = o.numpy().transpose(1, 0, 2)
    return out


def random_case(seed, ctx, qlens, hq, hkv, d, slack=1.5):
    w = W.make_paged("pin", seed, hq, hkv, d, ctx, qlens, slack=slack)
    k, v = w.k_pool.copy(), w.v_pool.copy()
    oracle.cache_write(k, v, w.k_new, w.v_new, w.slot_mapping)
    return w, k, v


# --------------------------------------------------------------------------
# bf16 widening
# --------------------------------------------------------------------------

def test_bf16_widening_matches_known_values():
    bits = np.array([0x3F80, 0xC000, 0x3F00, 0x4049, 0x0001, 0x7F80, 0xFF80, 0x0000, 0x8000], dtype=np.uint16)
    got = oracle.bf16_to_f64(bits)
    want = [1.0, -2.0, 0.5, 3.140625, 2.0 ** -133, math.inf, -math.inf, 0.0, -0.0]
    assert list(got) == want
    assert math.copysign(1.0, got[-1]) == -1.0
    assert np.isnan(oracle.bf16_to_f64(np.array([0x7FC0], dtype=np.uint16))[0])
    rnd = W.normal_bf16(7, 1, 4096)
    assert np.array_equal(oracle.bf16_to_f64(rnd), widen(rnd))


# --------------------------------------------------------------------------
# cache_write / copy_blocks against numpy indexing (bit exact)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("hkv,d", [(8, 64), (2, 128), (3, 16)])
def test_cache_write_matches_numpy_indexing(hkv, d):
    nb = 9
    rng = np.random.default_rng(1)
    k = rng.integers(0, 65535, size=(nb, hkv, 16, d), dtype=np.uint16)
    v = rng.integers(0, 65535, size=(nb, hkv, 16, d), dtype=np.uint16)
    T = 40
    slots = rng.permutation(nb * 16)[:T].astype(np.int32)
    slots[[3, 17, 25]] = -1  # skipped tokens
    kn = rng.integers(0, 65535, size=(T, hkv, d), dtype=np.uint16)
    vn = rng.integers(0, 65535, size=(T, hkv, d), dtype=np.uint16)
    k_ref, v_ref = k.copy(), v.copy()
    keep = slots >= 0
    k_ref[slots[keep] // 16, :, slots[keep] % 16, :] = kn[keep]
    v_ref[slots[keep] // 16, :, slots[keep] % 16, :] = vn[keep]
    oracle.cache_write(k, v, kn, vn, slots)
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def test_cache_write_rejects_out_of_range_slot():
    k = np.zeros((2, 1, 16, 8), dtype=np.uint16)
    v = k.copy()
    with pytest.raises(oracle.OracleError):
        oracle.cache_write(k, v, np.ones((1, 1, 8), np.uint16), np.ones((1, 1, 8), np.uint16),
                           np.array([32], np.int32))


def test_copy_blocks_matches_numpy_slicing():
    rng = np.random.default_rng(2)
    k = rng.integers(0, 65535, size=(20, 4, 16, 32), dtype=np.uint16)
    v = rng.integers(0, 65535, size=(20, 4, 16, 32), dtype=np.uint16)
    src = np.array([3, 3, 3, 7, 0], np.int32)      # one shared block copied three times
    dst = np.array([10, 11, 12, 19, 5], np.int32)
    k_ref, v_ref = k.copy(), v.copy()
    k_ref[dst] = k[src]
    v_ref[dst] = v[src]
    oracle.copy_blocks(k, v, src, dst)
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


# --------------------------------------------------------------------------
# Attention against a library routine
# --------------------------------------------------------------------------

@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 4), (8, 2, 64), (6, 3, 16), (32, 8, 64)])
def test_decode_matches_torch_sdpa(hq, hkv, d):
    ctx = [1, 15, 16, 17, 40, 33]
    w, k, v = random_case(11 + hq, ctx, [1] * len(ctx), hq, hkv, d)
    got = oracle.decode_attention(k, v, w.q, w.context_lens, w.block_tables, w.scale)
    ref = sdpa_reference(k, v, w.q, w.query_start_loc, w.context_lens, w.block_tables, w.scale)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("hq,hkv,d", [(4, 2, 16), (2, 1, 64)])
def test_mixed_prefill_matches_torch_sdpa(hq, hkv, d):
    # two chunks over a cached prefix, decode rows around them
    ctx = [40, 23, 1, 17, 36]
    ql = [8, 1, 1, 17, 1]
    w, k, v = random_case(5, ctx, ql, hq, hkv, d)
    got = oracle.paged_attention(k, v, w.q, w.query_start_loc, w.context_lens, w.block_tables, w.scale,
                                 threads=3)
    ref = sdpa_reference(k, v, w.q, w.query_start_loc, w.context_lens, w.block_tables, w.scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_large_logits_are_stable():
    """Scores near +-1000 overflow exp() unless the maximum is subtracted."""
    w, k, v = random_case(3, [20, 9], [1, 1], 2, 1, 8)
    got = oracle.decode_attention(k, v, w.q, w.context_lens, w.block_tables, scale=300.0)
    ref = sdpa_reference(k, v, w.q, w.query_start_loc, w.context_lens, w.block_tables, 300.0)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-9)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

def test_single_token_context_returns_v_exactly():
    w, k, v = random_case(21, [1, 1, 1], [1, 1, 1], 8, 2, 64)
    got = oracle.decode_attention(k, v, w.q, w.context_lens, w.block_tables, w.scale)
    for s in range(3):
        phys = w.block_tables[s][0]
        for h in range(8):
            assert np.array_equal(got[s, h], oracle.bf16_to_f64(v[phys, h // 4, 0]))


def test_zero_query_gives_mean_of_v():
    w, k, v = random_case(22, [37], [1], 2, 1, 16)
    q = np.zeros_like(w.q)
    got = oracle.decode_attention(k, v, q, w.context_lens, w.block_tables, w.scale)
    j = np.arange(37)
    Vc = oracle.bf16_to_f64(v[w.block_tables[0][j // 16], 0, j % 16])
    np.testing.assert_allclose(got[0, 0], Vc.mean(axis=0), rtol=0, atol=1e-14)
    np.testing.assert_allclose(got[0, 1], Vc.mean(axis=0), rtol=0, atol=1e-14)


def test_two_key_worked_example():
    """q = e0, k0 = e0, k1 = 0, scale = ln 3: scores (ln 3, 0), weights (3/4, 1/4)."""
    d = 4
    k = np.full((2, 1, 16, d), W.BF16_NAN, np.uint16)
    v = np.full((2, 1, 16, d), W.BF16_NAN, np.uint16)
    k[1, 0, 0] = bf16_bits([1, 0, 0, 0])
    k[1, 0, 1] = bf16_bits([0, 0, 0, 0])
    v[1, 0, 0] = bf16_bits([4, 8, -4, 1])
    v[1, 0, 1] = bf16_bits([0, 4, 4, -3])
    q = bf16_bits([[[1, 0, 0, 0]]]).reshape(1, 1, d)
    got = oracle.decode_attention(k, v, q, np.array([2], np.int32), np.array([[1]], np.int32), math.log(3.0))
    want = 0.75 * np.array([4, 8, -4, 1.0]) + 0.25 * np.array([0, 4, 4, -3.0])
    np.testing.assert_allclose(got[0, 0], want, rtol=0, atol=1e-15)


def test_dominant_key_selects_its_value():
    w, k, v = random_case(23, [30], [1], 1, 1, 16)
    j = 13
    phys, off = w.block_tables[0][j // 16], j % 16
    q = k[phys, 0, off].reshape(1, 1, 16).copy()
    got = oracle.decode_attention(k, v, q, w.context_lens, w.block_tables, scale=200.0)
    np.testing.assert_allclose(got[0, 0], oracle.bf16_to_f64(v[phys, 0, off]), rtol=0, atol=1e-9)


# --------------------------------------------------------------------------
# Invariants the pages state ([KV2] section 2)
# --------------------------------------------------------------------------

def test_paged_equals_contiguous():
    """Reading through a scattered block table gives the same result as one
    contiguous array ([KV2] section 2, "Blocks and block tables")."""
    ctx = [50, 3, 64, 17]
    w, k, v = random_case(31, ctx, [1] * 4, 4, 2, 32)
    got = oracle.decode_attention(k, v, w.q, w.context_lens, w.block_tables, w.scale)
    # lay every sequence out in consecutive physical blocks, in logical order
    nblk = [W.blocks_for(n) for n in ctx]
    k2 = np.full((sum(nblk),) + k.shape[1:], W.BF16_NAN, np.uint16)
    v2 = k2.copy()
    tables2 = np.full_like(w.block_tables, -1)
    base = 0
    for s, nb in enumerate(nblk):
        for i in range(nb):
            k2[base + i] = k[w.block_tables[s][i]]
            v2[base + i] = v[w.block_tables[s][i]]
            tables2[s, i] = base + i
        base += nb
    got2 = oracle.decode_attention(k2, v2, w.q, w.context_lens, tables2, w.scale)
    assert np.array_equal(got, got2)


def test_physical_placement_is_irrelevant():
    """Blocks may sit anywhere in free memory ([KV2] section 2): relabelling
    the physical ids (pool and tables together) leaves the output bit-identical."""
    w, k, v = random_case(32, [70, 16, 5], [1] * 3, 8, 4, 16)
    got = oracle.decode_attention(k, v, w.q, w.context_lens, w.block_tables, w.scale)
    perm = np.random.default_rng(0).permutation(k.shape[0])  # new id of old block b is perm[b]
    k2, v2 = np.empty_like(k), np.empty_like(v)
    k2[perm], v2[perm] = k, v
    t2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    got2 = oracle.decode_attention(k2, v2, w.q, w.context_lens, t2, w.scale)
    assert np.array_equal(got, got2)


def test_shared_prefix_equals_unshared_copies():
    """Requests may point at the same physical blocks ([KV2] section 2,
    "Sharing blocks"): shared tables give bit-identical results to private copies."""
    hq, hkv, d = 4, 2, 16
    ctx = [45, 45, 45]
    w = W.make_paged("share", 41, hq, hkv, d, ctx, [1, 1, 1], share_prefix_blocks=2, slack=2.0)
    k, v = w.k_pool.copy(), w.v_pool.copy()
    oracle.cache_write(k, v, w.k_new, w.v_new, w.slot_mapping)
    assert (w.block_tables[:, :2] == w.block_tables[0, :2]).all()
    got = oracle.decode_attention(k, v, w.q, w.context_lens, w.block_tables, w.scale)
    # give each sequence private copies of the shared blocks
    free = [b for b in range(k.shape[0]) if b not in set(w.block_tables.ravel())]
    t2 = w.block_tables.copy()
    for s in range(1, 3):
        for i in range(2):
            nbid = free.pop()
            oracle.copy_blocks(k, v, [w.block_tables[s, i]], [nbid])
            t2[s, i] = nbid
    got2 = oracle.decode_attention(k, v, w.q, w.context_lens, t2, w.scale)
    assert np.array_equal(got, got2)


def test_poisoned_slots_never_reach_the_output():
    ctx = [1, 15, 17, 31, 33]
    w, k, v = random_case(42, ctx, [1] * 5, 4, 4, 8)
    out = oracle.decode_attention(k, v, w.q, w.context_lens, w.block_tables, w.scale)
    assert np.all(np.isfinite(out))
    # the poison really is there: the slot right after each context is NaN
    for s, n in enumerate(ctx):
        if n % 16:
            assert np.isnan(oracle.bf16_to_f64(k[w.block_tables[s][n // 16], 0, n % 16])).all()


def test_chunked_prefill_equals_one_shot():
    """Splitting a prompt into consecutive slices ([ENG] "Chunked Prefill")
    and attending each slice over the cached prefix gives the rows of one-shot
    causal attention over the whole prompt."""
    hq, hkv, d = 4, 2, 16
    n = 70
    w, k, v = random_case(51, [n], [n], hq, hkv, d)
    one = oracle.paged_attention(k, v, w.q, w.query_start_loc, w.context_lens, w.block_tables, w.scale)
    for first, last in W.chunk_slices(n, 24):
        ql = last - first + 1
        sub = oracle.paged_attention(k, v, w.q[first:last + 1], np.array([0, ql], np.int32),
                                     np.array([last + 1], np.int32), w.block_tables, w.scale)
        assert np.array_equal(sub, one[first:last + 1])


def test_decode_row_in_mixed_batch_equals_pure_decode():
    ctx = [30, 48, 9]
    ql = [1, 16, 1]
    w, k, v = random_case(52, ctx, ql, 4, 2, 16)
    mixed = oracle.paged_attention(k, v, w.q, w.query_start_loc, w.context_lens, w.block_tables, w.scale)
    for s in (0, 2):
        r = w.query_start_loc[s]
        dec = oracle.decode_attention(k, v, w.q[r:r + 1], w.context_lens[s:s + 1], w.block_tables[s:s + 1],
                                      w.scale)
        assert np.array_equal(dec[0], mixed[r])


def test_empty_context_gives_zero_row():
    w, k, v = random_case(53, [5, 7], [1, 1], 2, 2, 8)
    ctx = w.context_lens.copy()
    ctx[1] = 0
    out = oracle.decode_attention(k, v, w.q, ctx, w.block_tables, w.scale)
    assert np.all(out[1] == 0) and np.all(np.isfinite(out[0]))


def test_threads_do_not_change_the_result():
    ctx = list(range(1, 40, 3))
    w, k, v = random_case(54, ctx, [1] * len(ctx), 4, 1, 16)
    a = oracle.decode_attention(k, v, w.q, w.context_lens, w.block_tables, w.scale, threads=1)
    b = oracle.decode_attention(k, v, w.q, w.context_lens, w.block_tables, w.scale, threads=5)
    assert np.array_equal(a, b)


def test_brute_force_tiny():
    """Triple loop in pure Python (no library) on a tiny case."""
    w, k, v = random_case(55, [3, 19], [1, 2], 2, 1, 4)
    got = oracle.paged_attention(k, v, w.q, w.query_start_loc, w.context_lens, w.block_tables, w.scale)
    K, V, Q = widen(k), widen(v), widen(w.q)
    for s in range(2):
        n = int(w.context_lens[s])
        r0, r1 = int(w.query_start_loc[s]), int(w.query_start_loc[s + 1])
        for r in range(r0, r1):
            pos = n - (r1 - r0) + (r - r0)
            for h in range(2):
                sc = []
                for j in range(pos + 1):
                    b = w.block_tables[s][j // 16]
                    sc.append(sum(Q[r, h, c] * K[b, 0, j % 16, c] for c in range(4)) * w.scale)
                e = [math.exp(x - max(sc)) for x in sc]
                for c in range(4):
                    num = sum(e[j] * V[w.block_tables[s][j // 16], 0, j % 16, c] for j in range(pos + 1))
                    assert abs(got[r, h, c] - num / sum(e)) < 1e-13


# --------------------------------------------------------------------------
# The pages' own numbers (tests/golden)
# --------------------------------------------------------------------------

def _golden(name):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    return rows


def test_golden_chunk_slices():
    rows = _golden("chunk_slices_8k_budget_2k.txt")
    prompt, budget = map(int, rows[0])
    want = [tuple(map(int, r)) for r in rows[1:]]
    assert W.chunk_slices(prompt, budget) == want


def test_golden_kv_capacity():
    g = {r[0]: int(r[1]) for r in _golden("kv_capacity_qwen3_1p7b.txt")}
    assert g["kv_capacity_tokens"] // g["block_size"] == g["pool_blocks"]
    assert W.blocks_for(g["request_tokens"]) == g["blocks_per_request"]
    fit = g["pool_blocks"] // W.blocks_for(g["request_tokens"])
    assert fit == g["requests_that_fit"]
    assert fit * W.blocks_for(g["request_tokens"]) == g["blocks_for_34"]
    w = W.make_paged("cap", 1, 2, 1, 8, [g["request_tokens"]] * fit, [1] * fit,
                     num_blocks=g["pool_blocks"])
    assert w.num_blocks == 1378 and w.block_tables.shape == (34, 40)
    with pytest.raises(ValueError):
        W.make_paged("cap", 1, 2, 1, 8, [640] * 35, [1] * 35, num_blocks=1378)


def test_golden_prefix_share_shape():
    g = {r[0]: int(r[1]) for r in _golden("prefix_3000_blocks.txt")}
    assert g["prefix_tokens"] // 16 == g["full_shared_blocks"]
    assert g["prefix_tokens"] % 16 == g["tokens_in_partial_block"]
    assert W.blocks_for(g["context_tokens"]) == g["blocks_per_sequence"]


def test_last_block_waste_is_under_one_block():
    """The only waste left is the unused tail of each request's last block,
    under 16 tokens ([KV2] section 2)."""
    for n in range(1, 200):
        waste = W.blocks_for(n) * 16 - n
        assert 0 <= waste < 16
