"""GPU parity of the device block bookkeeping (pkv_blocks_*) against the
sequential oracle: bit-exact tables, lengths, counts, free ring, slot
mappings, copy-on-write pairs and error codes after every call; and a whole
step (append -> copy_blocks -> cache_write -> attention) through the state."""
import numpy as np
import pytest
import torch

import oracle
from oracle import block_manager as bm
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


def assert_same_state(blocks, st, what):
    assert np.array_equal(blocks.block_tables.cpu().numpy(), st.tables), f"{what}: tables"
    assert np.array_equal(blocks.context_lens.cpu().numpy(), st.context_lens), f"{what}: lengths"
    n = st.num_blocks
    assert np.array_equal(blocks.ref_counts.cpu().numpy()[:n], st.ref_counts), f"{what}: counts"
    assert np.array_equal(blocks.free_ids.cpu().numpy()[:n], st.free_ids), f"{what}: free ring"
    assert blocks.free_state.cpu().tolist() == [st.free_head, st.free_count], f"{what}: ring head/count"
    assert not blocks.scratch.cpu().numpy().any(), f"{what}: scratch not left zero"


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
