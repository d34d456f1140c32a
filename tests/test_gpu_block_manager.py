"""GPU parity of the device block bookkeeping (pkv_blocks_*) against the
sequential oracle: bit-exact tables, lengths, counts, free ring, slot
mappings, copy-on-write pairs and error codes after every call; and a whole
step (append -> copy_blocks -> cache_write -> attention) through the state."""
import numpy as np
import pytest
import torch

import oracle
from oracle import block_manager as bm
from oracle import prefix_keys as pk
import pkv_workloads as W
from gpu_helpers import assert_close, dev_tensor, host_bits

pytestmark = pytest.mark.gpu

B = bm.BLOCK_SIZE


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_291_gb300 as p
    p.load()
    return p


def i32(x):
    return torch.tensor(np.asarray(x, dtype=np.int32), device="cuda")


def u8(x):
    return torch.tensor(np.ascontiguousarray(x, dtype=np.uint8), device="cuda")


def assert_same_state(blocks, st, what):
    assert np.array_equal(blocks.block_tables.cpu().numpy(), st.tables), f"{what}: tables"
    assert np.array_equal(blocks.context_lens.cpu().numpy(), st.context_lens), f"{what}: lengths"
    n = st.num_blocks
    assert np.array_equal(blocks.ref_counts.cpu().numpy()[:n], st.ref_counts), f"{what}: counts"
    assert blocks.free_queue() == st.free_queue(), f"{what}: free queue"
    assert blocks.free_state.cpu().tolist()[2] == st.free_count, f"{what}: free count"
    assert not blocks.scratch.cpu().numpy()[:2 * n].any(), f"{what}: scratch not left zero"
    if blocks.cached is not None:
        cached = blocks.cached.cpu().numpy()[:n]
        keys = blocks.block_keys.cpu().numpy()
        assert set(np.flatnonzero(cached).tolist()) == set(st.block_key), f"{what}: cached blocks"
        for b, k in st.block_key.items():
            assert bytes(keys[b]) == k, f"{what}: key of block {b}"
        table = blocks.key_table.cpu().numpy()
        assert sorted(table[table >= 0].tolist()) == sorted(st.block_key), f"{what}: table contents"


def run_append(pkv, blocks, st, qsl, what):
    T = int(qsl[-1])
    slots, cs, cd, cc = blocks.append(i32(qsl), T)
    err = pkv.get_error()
    status, o_slots, o_cs, o_cd = bm.append(st, qsl)
    assert err[0] == status, f"{what}: device {err} vs oracle {status}"
    S = len(qsl) - 1
    if status == bm.OK:
        assert np.array_equal(slots.cpu().numpy(), o_slots), f"{what}: slot mapping"
        k = int(cc.item())
        assert k == len(o_cs)
        assert np.array_equal(cs.cpu().numpy()[:k], o_cs) and np.array_equal(cd.cpu().numpy()[:k], o_cd)
        assert np.all(cs.cpu().numpy()[k:S] == -1) and np.all(cd.cpu().numpy()[k:S] == -1)
    else:
        assert np.all(slots.cpu().numpy() == -1) and np.all(cs.cpu().numpy()[:S] == -1)
        assert int(cc.item()) == 0
    assert_same_state(blocks, st, what)
    return status


@pytest.mark.parametrize("seed,rows,num_blocks", [(0, 48, 256), (1, 48, 96), (2, 1500, 4000), (3, 64, 2000)])
def test_random_lifecycles_match_oracle(pkv, seed, rows, num_blocks):
    rng = np.random.default_rng(seed)
    MB = 24
    blocks = pkv.Blocks(num_blocks, rows, MB)
    st = bm.BlockState(num_blocks, rows, MB)
    assert_same_state(blocks, st, "reset")
    seen = set()
    for step in range(40):
        op = rng.integers(0, 10)
        live = [r for r in range(rows) if st.context_lens[r] > 0]
        empty = [r for r in range(rows) if st.context_lens[r] == 0]
        what = f"seed {seed} step {step}"
        if op < 6:
            S = int(rng.integers(1, rows + 1))
            q = rng.integers(0, 3, size=S) * rng.integers(0, 2, size=S)
            q[rng.integers(0, S)] = rng.integers(1, 3 * B)           # one chunk
            if rng.integers(0, 8) == 0:
                q[rng.integers(0, S)] = MB * B                      # past the table: range error
            qsl = np.concatenate([[0], np.cumsum(q)]).astype(np.int64)
            seen.add(run_append(pkv, blocks, st, qsl, what))
        elif op < 8 and live and empty:
            k = min(len(empty), int(rng.integers(1, 5)))
            children = rng.choice(empty, size=k, replace=False)
            parents = rng.choice(live, size=k)
            if rng.integers(0, 6) == 0 and len(live) > 0:
                children[0] = live[0]                                # not empty (or a parent): an error
            blocks.fork(i32(parents), i32(children))
            err = pkv.get_error()
            status = bm.fork(st, parents, children)
            assert err[0] == status, f"{what}: fork device {err} vs oracle {status}"
            seen.add(status)
            assert_same_state(blocks, st, what)
        elif live:
            k = min(len(live), int(rng.integers(1, 4)))
            rel = list(rng.choice(live, size=k, replace=False))
            if rng.integers(0, 6) == 0:
                rel.append(rel[0])                                   # repeated row: alias error
            blocks.release(i32(rel))
            err = pkv.get_error()
            status = bm.release(st, rel)
            assert err[0] == status, f"{what}: release device {err} vs oracle {status}"
            seen.add(status)
            assert_same_state(blocks, st, what)
    assert bm.OK in seen


def test_every_holder_appends_and_the_last_keeps_the_block(pkv):
    blocks = pkv.Blocks(16, 8, 4)
    st = bm.BlockState(16, 8, 4)
    run_append(pkv, blocks, st, [0, 5], "prompt")
    blocks.fork(i32([0] * 5), i32([1, 2, 3, 4, 5]))
    assert pkv.get_error() == (0, 0)
    bm.fork(st, [0] * 5, [1, 2, 3, 4, 5])
    assert_same_state(blocks, st, "fork")
    run_append(pkv, blocks, st, [0, 1, 2, 3, 4, 5, 6], "all six append")
    assert st.tables[5, 0] == 0 and st.ref_counts[0] == 1


def test_out_of_blocks_changes_nothing(pkv):
    blocks = pkv.Blocks(3, 4, 4)
    st = bm.BlockState(3, 4, 4)
    run_append(pkv, blocks, st, [0, 20, 36], "fill")             # row 0: 2 blocks, row 1: 1 full block
    status = run_append(pkv, blocks, st, [0, 0, 1], "needs a 4th block")
    assert status == bm.ERR_NO_BLOCKS


def test_step_through_the_state_matches_the_oracle(pkv):
    """Prompts are appended, two samples fork from each, and a decode step
    appends one token to every row (copy-on-write of the shared partly filled
    block): copy_blocks with the emitted pairs, cache_write at the emitted
    slots and decode attention over blocks.block_tables give the oracle's
    attention over the oracle's state."""
    rng = np.random.default_rng(11)
    hq, hkv, d, NB, R, MB = 16, 8, 128, 160, 12, 16
    blocks = pkv.Blocks(NB, R, MB)
    st = bm.BlockState(NB, R, MB)
    k_pool = np.full((NB, hkv, B, d), 0x7FC0, dtype=np.uint16)      # NaN everywhere unused
    v_pool = k_pool.copy()
    kd, vd = dev_tensor(k_pool), dev_tensor(v_pool)

    def step(qsl, seed):
        T = int(qsl[-1])
        k_new = W.normal_bf16(seed, 1, T * hkv * d).reshape(T, hkv, d)
        v_new = W.normal_bf16(seed, 2, T * hkv * d).reshape(T, hkv, d)
        slots, cs, cd, cc = blocks.append(i32(qsl), T)
        S = len(qsl) - 1
        pkv.copy_blocks(kd, vd, cs[:S], cd[:S], check_host=False)
        pkv.cache_write(kd, vd, dev_tensor(k_new), dev_tensor(v_new), slots)
        status, o_slots, o_cs, o_cd = bm.append(st, qsl)
        assert status == bm.OK
        oracle.copy_blocks(k_pool, v_pool, o_cs, o_cd)
        oracle.cache_write(k_pool, v_pool, k_new, v_new, o_slots)
        assert pkv.get_error() == (0, 0)

    prompts = [37, 16, 5, 50]
    step(np.concatenate([[0], np.cumsum(prompts)]), 1)
    parents = [0, 0, 1, 1, 2, 2, 3, 3]
    children = [4, 5, 6, 7, 8, 9, 10, 11]
    blocks.fork(i32(parents), i32(children))
    assert bm.fork(st, parents, children) == bm.OK
    for t in range(3):
        step(np.arange(R + 1), 10 + t)                              # one token per row
    assert_same_state(blocks, st, "after the steps")
    assert np.array_equal(host_bits(kd), k_pool) and np.array_equal(host_bits(vd), v_pool)

    q = W.normal_bf16(99, 3, R * hq * d).reshape(R, hq, d)
    out = pkv.decode_attention(kd, vd, dev_tensor(q), blocks.block_tables, blocks.context_lens,
                               int(st.context_lens.max()), 1.0 / np.sqrt(d))
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    ref = oracle.decode_attention(k_pool, v_pool, q, st.context_lens, st.tables, 1.0 / np.sqrt(d), threads=8)
    assert_close(out.cpu().numpy(), ref, "blocks step")


def _keys(tokens, n, stride):
    out = np.zeros((stride, 32), dtype=np.uint8)
    for i, k in enumerate(pk.sequence_keys(np.asarray(tokens, dtype=np.int64))[:n]):
        out[i] = np.frombuffer(k, dtype=np.uint8)
    return out


@pytest.mark.parametrize("seed,rows,num_blocks", [(0, 8, 40), (1, 8, 24), (2, 24, 120)])
def test_prefix_cache_lifecycles_match_oracle(pkv, seed, rows, num_blocks):
    """Requests with prompts from a few shared prefixes come and go (match,
    append of the rest, register, decode steps, release), with the pool small
    enough that cached blocks get evicted: after every call the device state
    (tables, counts, free queue in LRU order, cached keys) equals the
    oracle's."""
    rng = np.random.default_rng(200 + seed)
    MB = 12
    blocks = pkv.Blocks(num_blocks, rows, MB, prefix_cache=True)
    st = bm.BlockState(num_blocks, rows, MB)
    assert_same_state(blocks, st, "reset")
    hist = {r: [] for r in range(rows)}
    prefixes = [rng.integers(0, 1000, size=int(rng.integers(16, 70))) for _ in range(3)]
    hits = evictions_seen = 0
    for step in range(60):
        what = f"seed {seed} step {step}"
        op = rng.integers(0, 10)
        empty = [r for r in range(rows) if st.context_lens[r] == 0]
        live = [r for r in range(rows) if st.context_lens[r] > 0]
        if op < 4 and empty:
            r = int(rng.choice(empty))
            prompt = np.concatenate([prefixes[rng.integers(0, 3)], rng.integers(0, 1000, size=rng.integers(0, 20))])
            nf = len(prompt) // B
            keys = np.zeros((rows, MB, 32), dtype=np.uint8)
            keys[r] = _keys(prompt, nf, MB)
            nk = np.zeros(rows, dtype=np.int32)
            nk[r] = nf
            m = blocks.match(u8(keys), i32(nk))
            status, om = bm.match(st, keys, nk)
            assert pkv.get_error() == (0, 0) and status == bm.OK
            assert np.array_equal(m.cpu().numpy()[:rows], om), f"{what}: matched"
            hits += int(om[r])
            assert_same_state(blocks, st, what + " match")
            q = np.zeros(rows, dtype=np.int64)
            q[r] = len(prompt) - om[r] * B
            status = run_append(pkv, blocks, st, np.concatenate([[0], np.cumsum(q)]), what + " prompt")
            if status != bm.OK:
                blocks.release(i32([r]))
                assert pkv.get_error() == (0, 0) and bm.release(st, [r]) == bm.OK
                hist[r] = []
                continue
            hist[r] = list(prompt)
        elif op < 8 and live:
            q = np.zeros(rows, dtype=np.int64)
            q[live] = 1
            status = run_append(pkv, blocks, st, np.concatenate([[0], np.cumsum(q)]), what + " decode")
            if status == bm.OK:
                for r in live:
                    hist[r].append(int(rng.integers(0, 1000)))
        elif live:
            r = int(rng.choice(live))
            blocks.release(i32([r]))
            assert pkv.get_error() == (0, 0) and bm.release(st, [r]) == bm.OK
            hist[r] = []
            assert_same_state(blocks, st, what + " release")
        cached_before = len(st.block_key)
        keys = np.zeros((rows, MB, 32), dtype=np.uint8)
        nk = np.zeros(rows, dtype=np.int32)
        for r in range(rows):
            nk[r] = int(st.context_lens[r]) // B
            keys[r] = _keys(hist[r], int(nk[r]), MB)
        blocks.register(u8(keys), i32(nk))
        assert pkv.get_error() == (0, 0) and bm.register(st, keys, nk) == bm.OK
        assert_same_state(blocks, st, what + " register")
        evictions_seen += max(0, cached_before - len(st.block_key))
    assert hits > 0


def test_stale_entries_are_compacted_away(pkv):
    """A prompt's blocks are released (content kept) and matched back again
    and again: every match leaves stale ring entries, so the ring of
    2 * num_blocks entries must be compacted on release; the free queue stays
    the oracle's throughout."""
    NB, MB = 6, 4
    blocks = pkv.Blocks(NB, 2, MB, prefix_cache=True)
    st = bm.BlockState(NB, 2, MB)
    prompt = np.arange(48)                                     # 3 full blocks
    run_append(pkv, blocks, st, [0, 48], "prompt")
    keys = np.zeros((2, MB, 32), dtype=np.uint8)
    keys[0] = _keys(prompt, 3, MB)
    blocks.register(u8(keys), i32([3, 0]))
    assert bm.register(st, keys, [3, 0]) == bm.OK
    most = 0
    for cycle in range(12):
        blocks.release(i32([0]))
        assert pkv.get_error() == (0, 0) and bm.release(st, [0]) == bm.OK
        assert_same_state(blocks, st, f"cycle {cycle} release")
        most = max(most, blocks.free_state.cpu().tolist()[1])
        m = blocks.match(u8(keys), i32([3, 0]))
        status, om = bm.match(st, keys, [3, 0])
        assert pkv.get_error() == (0, 0) and status == bm.OK and om.tolist() == [3, 0]
        assert m.cpu().tolist()[:2] == [3, 0]
        assert_same_state(blocks, st, f"cycle {cycle} match")
    assert most == 2 * NB, "the ring never filled, so compaction was not exercised"


def test_equal_prompts_registered_together_keep_the_first_rows_blocks(pkv):
    """Rows 0 and 2 computed the same 40-token prompt separately and row 1 is
    a fork of row 0: one register call gives each key to row 0's block (row
    1's entries are the same blocks, row 2's equal keys lose and are removed
    from the table again)."""
    NB, MB, R = 16, 4, 3
    blocks = pkv.Blocks(NB, R, MB, prefix_cache=True)
    st = bm.BlockState(NB, R, MB)
    prompt = np.arange(500, 540)
    run_append(pkv, blocks, st, [0, 40], "row 0")
    blocks.fork(i32([0]), i32([1]))
    assert pkv.get_error() == (0, 0) and bm.fork(st, [0], [1]) == bm.OK
    run_append(pkv, blocks, st, [0, 0, 0, 40], "row 2")
    keys = np.stack([_keys(prompt, 2, MB)] * R)
    for trial in range(3):                                      # the race between equal keys varies
        blocks.register(u8(keys), i32([2, 2, 2]))
        assert pkv.get_error() == (0, 0)
        if trial == 0:
            assert bm.register(st, keys, [2, 2, 2]) == bm.OK
        assert_same_state(blocks, st, f"register, trial {trial}")
    assert sorted(st.block_key) == sorted(st.tables[0, :2].tolist())
    m = blocks.match(u8(np.stack([np.zeros((MB, 32), np.uint8)] * R)), i32([0, 0, 0]))
    assert pkv.get_error() == (0, 0)
