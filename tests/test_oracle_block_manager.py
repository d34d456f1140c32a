"""Pins for the block bookkeeping oracle (no GPU).

What fixes the oracle, independently of its own code:
- token replay: a pool of token ids written through the slot mapping (after
  the copy-on-write copies) must give every row back exactly its own token
  history when read through its table: the paged cache holds the same
  content as one contiguous array per request ("Blocks and block tables" and
  "Sharing blocks", section 2 of the serving-engine KV blog);
- invariants: a block's count is the number of table entries pointing at it,
  the free queue holds exactly the blocks nobody holds, each once, and a row
  holds exactly ceil(len / 16) blocks (allocation on fill, no reservation);
- hand-worked examples with the values written out below.
"""
import numpy as np
import pytest

from oracle import block_manager as bm
from oracle import prefix_keys as pk

B = bm.BLOCK_SIZE


def check_invariants(st):
    refs = np.zeros(st.num_blocks, dtype=np.int64)
    for r in range(st.tables.shape[0]):
        nb = bm.blocks_for(st.context_lens[r])
        assert np.all(st.tables[r, nb:] == -1), f"row {r} holds blocks past its length"
        for li in range(nb):
            refs[st.tables[r, li]] += 1
    assert np.array_equal(refs, st.ref_counts), "counts differ from table references"
    q = st.free_queue()
    assert len(q) == len(set(q)), "a block is queued twice"
    assert set(q) == set(np.flatnonzero(refs == 0).tolist()), "free queue != unheld blocks"


class Replay:
    """Token ids written into a pool through the oracle's slot mappings."""

    def __init__(self, st):
        self.pool = np.full(st.num_blocks * B, -1, dtype=np.int64)
        self.hist = {r: [] for r in range(st.tables.shape[0])}
        self.next_tok = 1000

    def apply_append(self, st, qsl, slots, cow_src, cow_dst):
        for s, d in zip(cow_src, cow_dst):
            self.pool[d * B:(d + 1) * B] = self.pool[s * B:(s + 1) * B]
        for r in range(len(qsl) - 1):
            for i in range(qsl[r], qsl[r + 1]):
                self.pool[slots[i]] = self.next_tok
                self.hist[r].append(self.next_tok)
                self.next_tok += 1

    def check(self, st):
        for r, h in self.hist.items():
            n = int(st.context_lens[r])
            assert n == len(h)
            got = [int(self.pool[st.tables[r, p // B] * B + p % B]) for p in range(n)]
            assert got == h, f"row {r} reads back other tokens"


def test_fresh_state_allocates_on_fill_in_queue_order():
    st = bm.BlockState(4, 4, 4)
    status, slots, cs, cd = bm.append(st, [0, 5, 21, 41])       # rows get 5, 16, 20 tokens
    assert status == bm.OK
    assert slots.tolist() == [0, 1, 2, 3, 4] + list(range(16, 32)) + list(range(32, 48)) + [48, 49, 50, 51]
    assert st.tables[:3, :2].tolist() == [[0, -1], [1, -1], [2, 3]]
    assert cs.size == 0 and st.free_count == 0 and st.ref_counts.tolist() == [1, 1, 1, 1]
    status, slots, _, _ = bm.append(st, [0, 1])                  # row 0's 6th token: same block
    assert status == bm.OK and slots.tolist() == [5]
    before = st.clone()
    status, *_ = bm.append(st, [0, 0, 1])                        # row 1 is full: needs a 5th block
    assert status == bm.ERR_NO_BLOCKS
    assert np.array_equal(st.tables, before.tables) and st.free_count == 0
    assert np.array_equal(st.context_lens, before.context_lens)


def test_fork_then_all_holders_append_copies_all_but_the_last():
    st = bm.BlockState(8, 4, 2)
    assert bm.append(st, [0, 5])[0] == bm.OK                     # row 0: block 0, 5 tokens
    assert bm.fork(st, [0, 0], [2, 3]) == bm.OK
    assert st.ref_counts[0] == 3 and st.context_lens.tolist() == [5, 0, 5, 5]
    status, slots, cs, cd = bm.append(st, [0, 1, 1, 2, 3])       # rows 0, 2, 3 append; row 1 nothing
    assert status == bm.OK
    # row 0 (count 3) copies into block 1, row 2 (count now 2) into block 2,
    # row 3 (count now 1) writes in place.
    assert cs.tolist() == [0, 0] and cd.tolist() == [1, 2]
    assert slots.tolist() == [1 * B + 5, 2 * B + 5, 0 * B + 5]
    assert st.ref_counts[:3].tolist() == [1, 1, 1]
    assert st.tables[[0, 2, 3], 0].tolist() == [1, 2, 0]


def test_fork_then_one_holder_appends_copies():
    st = bm.BlockState(8, 2, 2)
    bm.append(st, [0, 3])
    bm.fork(st, [0], [1])
    status, slots, cs, cd = bm.append(st, [0, 0, 1])             # only row 1 appends
    assert status == bm.OK and cs.tolist() == [0] and cd.tolist() == [1] and slots.tolist() == [B + 3]
    assert st.ref_counts[:2].tolist() == [1, 1]


def test_full_shared_block_is_not_copied():
    st = bm.BlockState(8, 2, 3)
    bm.append(st, [0, 16])                                      # exactly one full block
    bm.fork(st, [0], [1])
    status, slots, cs, _ = bm.append(st, [0, 1, 2])
    assert status == bm.OK and cs.size == 0
    assert slots.tolist() == [B * 1, B * 2]                      # new blocks 1 and 2
    assert st.ref_counts[:3].tolist() == [2, 1, 1]


def test_release_queues_blocks_last_first_when_the_count_reaches_zero():
    st = bm.BlockState(6, 3, 3)
    bm.append(st, [0, 40])                                      # row 0: blocks 0, 1, 2
    bm.fork(st, [0], [1])
    assert bm.release(st, [0]) == bm.OK                         # still held by row 1
    assert st.free_queue() == [3, 4, 5]
    assert bm.release(st, [1]) == bm.OK
    assert st.free_queue() == [3, 4, 5, 2, 1, 0]
    status, slots, _, _ = bm.append(st, [0, 1])
    assert slots.tolist() == [3 * B]


def test_errors_leave_the_state_unchanged():
    st = bm.BlockState(4, 3, 2)
    bm.append(st, [0, 17])
    snap = st.clone()
    assert bm.append(st, [0, 16])[0] == bm.ERR_RANGE             # 17 + 16 > 2 blocks
    assert bm.fork(st, [0], [0]) == bm.ERR_ALIAS
    assert bm.fork(st, [1, 1], [2, 2]) == bm.ERR_ALIAS
    bm.append(st, [0, 0, 3])
    snap = st.clone()
    assert bm.fork(st, [0], [1]) == bm.ERR_RANGE                 # child is not empty
    assert bm.release(st, [1, 1]) == bm.ERR_ALIAS
    assert bm.release(st, [5]) == bm.ERR_RANGE
    for a in ("tables", "context_lens", "ref_counts"):
        assert np.array_equal(getattr(st, a), getattr(snap, a))
    assert st.free_queue() == snap.free_queue()


@pytest.mark.parametrize("seed", range(6))
def test_random_lifecycles_replay_and_invariants(seed):
    rng = np.random.default_rng(seed)
    R, NB, MB = 12, 96, 10
    st = bm.BlockState(NB, R, MB)
    rp = Replay(st)
    copies = 0
    for _ in range(60):
        op = rng.integers(0, 10)
        live = [r for r in range(R) if st.context_lens[r] > 0]
        empty = [r for r in range(R) if st.context_lens[r] == 0]
        if op < 6:
            q = rng.integers(0, 3, size=R) * rng.integers(0, 2, size=R)
            q[rng.integers(0, R)] = rng.integers(1, 40)          # one longer chunk
            qsl = np.concatenate([[0], np.cumsum(q)]).astype(np.int64)
            snap = st.clone()
            status, slots, cs, cd = bm.append(st, qsl)
            if status == bm.OK:
                rp.apply_append(st, qsl, slots, cs, cd)
                copies += len(cs)
                assert len(set(slots.tolist())) == len(slots), "two new tokens share a slot"
            else:
                assert status in (bm.ERR_NO_BLOCKS, bm.ERR_RANGE)
                assert np.array_equal(st.tables, snap.tables)
        elif op < 8 and live and empty:
            k = min(len(empty), int(rng.integers(1, 4)))
            children = list(rng.choice(empty, size=k, replace=False))
            parents = list(rng.choice(live, size=k))
            assert bm.fork(st, parents, children) == bm.OK
            for p, c in zip(parents, children):
                rp.hist[int(c)] = list(rp.hist[int(p)])
        elif live:
            k = min(len(live), int(rng.integers(1, 3)))
            rows = list(rng.choice(live, size=k, replace=False))
            assert bm.release(st, rows) == bm.OK
            for r in rows:
                rp.hist[int(r)] = []
        check_invariants(st)
        rp.check(st)
    assert copies > 0, "the random walk never exercised copy-on-write"


def keys_of(tokens, n):
    ks = pk.sequence_keys(tokens)[:n]
    return [np.frombuffer(k, dtype=np.uint8) for k in ks]


def test_a_reused_prompt_takes_its_cached_blocks_and_allocation_follows_lru():
    st = bm.BlockState(8, 3, 4)
    prompt = np.arange(100, 140)                                 # 40 tokens: 2 full blocks + 8
    assert bm.append(st, [0, 40])[0] == bm.OK                    # blocks 0, 1, 2
    assert bm.register(st, [keys_of(prompt, 2)], [2]) == bm.OK
    assert bm.release(st, [0]) == bm.OK
    assert st.free_queue() == [3, 4, 5, 6, 7, 2, 1, 0]           # content kept, last block first
    status, m = bm.match(st, [keys_of(prompt, 2), []], [2, 0])
    assert status == bm.OK and m.tolist() == [2, 0]
    assert st.tables[0, :2].tolist() == [0, 1] and st.context_lens[0] == 32
    assert st.free_queue() == [3, 4, 5, 6, 7, 2]
    status, slots, _, _ = bm.append(st, [0, 8])                 # the 8 tokens left: block 3
    assert slots.tolist() == list(range(3 * B, 3 * B + 8))


def test_match_stops_at_the_first_key_not_cached():
    """A key stands for its whole prefix (section 4 of the serving-engine KV
    blog), so a row's cached blocks are a leading run: with the second key
    unknown, the third block is not taken even though its key is cached."""
    st = bm.BlockState(6, 2, 4)
    prompt = np.arange(48)
    bm.append(st, [0, 48])                                       # blocks 0, 1, 2
    ks = keys_of(prompt, 3)
    bm.register(st, [ks], [3])
    bm.release(st, [0])                                          # queue: 3, 4, 5, 2, 1, 0
    other = keys_of(np.arange(1000, 1016), 1)[0]
    status, m = bm.match(st, [[ks[0], other, ks[2]]], [3])
    assert status == bm.OK and m.tolist() == [1]
    assert st.tables[0].tolist() == [0, -1, -1, -1] and st.context_lens[0] == 16
    assert st.free_queue() == [3, 4, 5, 2, 1]


def test_reusing_a_freed_block_drops_its_key():
    st = bm.BlockState(3, 3, 4)
    prompt = np.arange(32)
    bm.append(st, [0, 32])                                       # blocks 0, 1
    bm.register(st, [keys_of(prompt, 2)], [2])
    bm.release(st, [0])                                          # queue: 2, 1, 0
    bm.append(st, [0, 0, 20])                                    # row 1 takes 2 and 1 (1 loses its key)
    assert st.tables[1, :2].tolist() == [2, 1]
    status, m = bm.match(st, [[], [], keys_of(prompt, 2)], [0, 0, 2])
    assert status == bm.OK and m.tolist() == [0, 0, 1]           # block 0 still cached; block 1's key is gone
    assert st.tables[2, 0] == 0 and st.context_lens[1] == 20 and st.free_queue() == []


@pytest.mark.parametrize("seed", range(4))
def test_random_requests_with_shared_prefixes_replay(seed):
    """Requests with prompts from a few shared prefixes come and go: cached
    blocks are reused, evicted under pressure, and every row still reads its
    own tokens; every cached key's block holds the tokens it was given."""
    rng = np.random.default_rng(100 + seed)
    R, NB, MB = 8, 40, 12
    st = bm.BlockState(NB, R, MB)
    rp = Replay(st)
    hist = {r: [] for r in range(R)}                               # token ids per row
    prefixes = [rng.integers(0, 1000, size=int(rng.integers(16, 70))) for _ in range(3)]
    key_tokens = {}
    hits = 0
    for _ in range(80):
        op = rng.integers(0, 10)
        empty = [r for r in range(R) if st.context_lens[r] == 0]
        live = [r for r in range(R) if st.context_lens[r] > 0]
        if op < 4 and empty:                                       # a new request
            r = int(rng.choice(empty))
            prompt = np.concatenate([prefixes[rng.integers(0, 3)], rng.integers(0, 1000, size=rng.integers(0, 20))])
            nf = len(prompt) // B
            ks = [[] for _ in range(R)]
            nk = [0] * R
            ks[r], nk[r] = keys_of(prompt, nf), nf
            status, m = bm.match(st, ks, nk)
            assert status == bm.OK
            hits += int(m[r])
            hist[r] = list(prompt[:m[r] * B])
            rp.hist[r] = list(prompt[:m[r] * B])
            q = np.zeros(R, dtype=np.int64)
            q[r] = len(prompt) - m[r] * B
            qsl = np.concatenate([[0], np.cumsum(q)])
            status, slots, cs, cd = bm.append(st, qsl)
            if status != bm.OK:                                    # pool exhausted: drop the request
                assert status == bm.ERR_NO_BLOCKS
                assert bm.release(st, [r]) == bm.OK
                hist[r], rp.hist[r] = [], []
                continue
            for s_, d_ in zip(cs, cd):
                rp.pool[d_ * B:(d_ + 1) * B] = rp.pool[s_ * B:(s_ + 1) * B]
            tail = prompt[m[r] * B:]
            for i, sl in enumerate(slots):
                rp.pool[sl] = tail[i]
            hist[r] = list(prompt)
            rp.hist[r] = list(prompt)
        elif op < 8 and live:                                      # a decode step for every live row
            q = np.zeros(R, dtype=np.int64)
            q[live] = 1
            qsl = np.concatenate([[0], np.cumsum(q)])
            snap = st.clone()
            status, slots, cs, cd = bm.append(st, qsl)
            if status != bm.OK:
                assert status == bm.ERR_NO_BLOCKS and st.free_queue() == snap.free_queue()
                continue
            for s_, d_ in zip(cs, cd):
                rp.pool[d_ * B:(d_ + 1) * B] = rp.pool[s_ * B:(s_ + 1) * B]
            for i, r in enumerate(live):
                t = int(rng.integers(0, 1000))
                rp.pool[slots[i]] = t
                hist[r].append(t)
                rp.hist[r].append(t)
        elif live:                                                 # a request ends
            r = int(rng.choice(live))
            assert bm.release(st, [r]) == bm.OK
            hist[r], rp.hist[r] = [], []
        # every row registers its full blocks
        ks, nk = [], []
        for r in range(R):
            nf = int(st.context_lens[r]) // B
            ks.append(keys_of(np.array(hist[r], dtype=np.int64), nf))
            nk.append(nf)
            for i in range(nf):
                key_tokens.setdefault(bytes(ks[r][i]), list(hist[r][i * B:(i + 1) * B]))
        assert bm.register(st, ks, nk) == bm.OK
        check_invariants(st)
        rp.check(st)
        for k, b in st.cache.items():
            assert st.block_key[b] == k
            assert rp.pool[b * B:(b + 1) * B].tolist() == key_tokens[k], "a cached key's block was overwritten"
    assert hits > 0, "no prefix was ever reused"


def test_equal_keys_in_one_register_call_go_to_the_first_row():
    st = bm.BlockState(16, 3, 4)
    prompt = np.arange(500, 540)
    bm.append(st, [0, 40])                                       # row 0: blocks 0, 1, 2
    bm.fork(st, [0], [1])
    bm.append(st, [0, 0, 0, 40])                                 # row 2: blocks 3, 4, 5
    ks = [keys_of(prompt, 2)] * 3
    assert bm.register(st, ks, [2, 2, 2]) == bm.OK
    assert sorted(st.block_key) == [0, 1]
    assert all(st.cache[bytes(k)] == b for k, b in zip(keys_of(prompt, 2), [0, 1]))
