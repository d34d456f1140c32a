"""Block bookkeeping oracle for a paged KV cache -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  It shares no code with the CUDA library.

A plain sequential model of the bookkeeping around the cache:

- "PagedAttention: splitting KV into blocks", section 2 of the serving-engine
  KV blog, subsection "Blocks and block tables": the KV of a request is cut
  into fixed blocks of 16 tokens that may sit anywhere in free memory; each
  request keeps a table from logical to physical blocks, and a new block is
  allocated at the moment the tokens fill the last one (nothing is reserved
  ahead).
- Same section, subsection "Sharing blocks": several requests may point at
  the same block (parallel sampling, beam search share a prompt); blocks
  carry a reference count, and a shared block is copied only when one of its
  holders has to append to it (copy-on-write).
- Section 4 ("Prefix cache") of the same blog: blocks of a finished request
  go back to the free queue tail block first.

Readings where the pages leave a step open:

- Sequences of one call are processed in index order.  A holder of a
  shared, partly filled last block copies it when the block's count is above
  1 at that moment, so when every holder appends in the same call, the last
  one (highest index) writes in place and all others copy.
- Free blocks form a FIFO queue: allocation takes from the head, release
  appends at the tail.  A fresh state queues blocks 0, 1, 2, ... in order.
  Within one call, allocation goes in sequence order; within a sequence, the
  copy-on-write block comes first, then new blocks in logical order.
- Release processes rows in the given order, each row's blocks from its last
  logical block to its first; a block is queued when its count reaches 0.
- Fork gives a child row all of its parent's blocks (the partly filled last
  block included), each block's count going up by one.
- Prefix cache (section 4): a freed block keeps its content and its key
  ("empty but content kept") and stays in the free queue in LRU order; a
  new row whose leading block keys are cached takes those blocks (a block
  with no holder leaves the free queue); allocation takes the least recently
  freed block first and drops its key.  Match is per row, in row order, and
  stops at the first key not cached.  Register gives a row's full blocks their
  keys in (row, block) order; a block that already has a key keeps it, and a
  key that is already cached keeps its first block.
- A call that cannot be completed (too few free blocks, a length beyond the
  table, an inconsistent table or count, a repeated row) changes nothing and
  returns its error code.

Parity status: pinned by ``tests/test_oracle_block_manager.py``: brute-force
token replay (every sequence reads back exactly its own tokens through its
table), reference-count and free-queue invariants, hand-worked examples.
"""
from __future__ import annotations

import copy

import numpy as np

BLOCK_SIZE = 16

OK = 0
ERR_SHAPE = 2
ERR_ALIAS = 6
ERR_RANGE = 9
ERR_NO_BLOCKS = 14


def blocks_for(n_tokens: int) -> int:
    """Blocks needed to hold n_tokens (ceil(n / 16))."""
    return -(-int(n_tokens) // BLOCK_SIZE)


class BlockState:
    """Tables, lengths, reference counts and the free queue."""

    def __init__(self, num_blocks: int, max_seqs: int, max_blocks_per_seq: int):
        self.num_blocks = int(num_blocks)
        self.tables = np.full((max_seqs, max_blocks_per_seq), -1, dtype=np.int32)
        self.context_lens = np.zeros(max_seqs, dtype=np.int32)
        self.ref_counts = np.zeros(num_blocks, dtype=np.int32)
        self.queue = list(range(num_blocks))   # free blocks, least recently freed first
        self.cache = {}                        # key (bytes) -> block
        self.block_key = {}                    # block -> its key, for cached blocks

    @property
    def free_count(self) -> int:
        return len(self.queue)

    def clone(self) -> "BlockState":
        return copy.deepcopy(self)

    def free_queue(self) -> list:
        """The free block ids, least recently freed first."""
        return list(self.queue)

    def _pop(self) -> int:
        b = self.queue.pop(0)
        if b in self.block_key:                # reused: its cached content is gone
            del self.cache[self.block_key.pop(b)]
        return b

    def _push(self, b: int) -> None:
        self.queue.append(b)


def _row_blocks_valid(st: BlockState, r: int) -> bool:
    nb = blocks_for(st.context_lens[r])
    if nb > st.tables.shape[1]:
        return False
    for li in range(nb):
        b = int(st.tables[r, li])
        if b < 0 or b >= st.num_blocks or st.ref_counts[b] <= 0:
            return False
    return True


def append(st: BlockState, query_start_loc):
    """Add query_start_loc[s+1] - query_start_loc[s] tokens to row s, for
    rows 0 .. len(query_start_loc) - 2.

    Returns (status, slot_mapping, cow_src, cow_dst): the slot of every new
    token (block * 16 + row, in token order) and the copy-on-write pairs in
    the order they were made.  On an error the state is unchanged."""
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    S = len(qsl) - 1
    if S < 0 or S > st.tables.shape[0]:
        return ERR_SHAPE, None, None, None
    q = qsl[1:] - qsl[:-1]
    if np.any(q < 0) or (S > 0 and qsl[0] != 0):
        return ERR_RANGE, None, None, None
    cap = st.tables.shape[1] * BLOCK_SIZE
    appenders = {}
    for s in range(S):
        if q[s] == 0:
            continue
        # Only what the append touches is checked: the length and, when the
        # last block is partly filled, that block.
        n0 = int(st.context_lens[s])
        if n0 < 0 or n0 + int(q[s]) > cap:
            return ERR_RANGE, None, None, None
        if n0 % BLOCK_SIZE:
            b = int(st.tables[s, n0 // BLOCK_SIZE])
            if b < 0 or b >= st.num_blocks or st.ref_counts[b] <= 0:
                return ERR_RANGE, None, None, None
            appenders[b] = appenders.get(b, 0) + 1
    for b, k in appenders.items():
        if k > st.ref_counts[b]:   # more holders append than hold the block
            return ERR_RANGE, None, None, None

    w = st.clone()
    slots = np.zeros(int(qsl[-1]) if S > 0 else 0, dtype=np.int32)
    cow_src, cow_dst = [], []
    for s in range(S):
        if q[s] == 0:
            continue
        n0 = int(w.context_lens[s])
        n1 = n0 + int(q[s])
        if n0 % BLOCK_SIZE:
            li = n0 // BLOCK_SIZE
            b = int(w.tables[s, li])
            if w.ref_counts[b] > 1:
                if w.free_count == 0:
                    return ERR_NO_BLOCKS, None, None, None
                nb = w._pop()
                w.ref_counts[b] -= 1
                w.ref_counts[nb] = 1
                w.tables[s, li] = nb
                cow_src.append(b)
                cow_dst.append(nb)
        for li in range(blocks_for(n0), blocks_for(n1)):
            if w.free_count == 0:
                return ERR_NO_BLOCKS, None, None, None
            nb = w._pop()
            w.ref_counts[nb] = 1
            w.tables[s, li] = nb
        for i in range(int(q[s])):
            pos = n0 + i
            slots[qsl[s] + i] = w.tables[s, pos // BLOCK_SIZE] * BLOCK_SIZE + pos % BLOCK_SIZE
        w.context_lens[s] = n1
    st.__dict__.update(w.__dict__)
    return OK, slots, np.array(cow_src, dtype=np.int32), np.array(cow_dst, dtype=np.int32)


def fork(st: BlockState, parents, children) -> int:
    """Row children[i] becomes a copy of row parents[i] sharing its blocks.
    Children must be empty, distinct, and not parents of the same call."""
    parents = [int(p) for p in parents]
    children = [int(c) for c in children]
    if len(parents) != len(children):
        return ERR_SHAPE
    R = st.tables.shape[0]
    if any(not (0 <= r < R) for r in parents + children):
        return ERR_RANGE
    if len(set(children)) != len(children) or set(children) & set(parents):
        return ERR_ALIAS
    for p, c in zip(parents, children):
        if st.context_lens[c] != 0 or not _row_blocks_valid(st, p):
            return ERR_RANGE
    for p, c in zip(parents, children):
        nb = blocks_for(st.context_lens[p])
        for li in range(nb):
            b = int(st.tables[p, li])
            st.tables[c, li] = b
            st.ref_counts[b] += 1
        st.context_lens[c] = st.context_lens[p]
    return OK


def release(st: BlockState, rows) -> int:
    """Drop rows (in the given order): each row's blocks, last first, lose a
    reference, and a block whose count reaches 0 joins the free queue's tail."""
    rows = [int(r) for r in rows]
    R = st.tables.shape[0]
    if any(not (0 <= r < R) for r in rows):
        return ERR_RANGE
    if len(set(rows)) != len(rows):
        return ERR_ALIAS
    held = {}
    for r in rows:
        if not _row_blocks_valid(st, r):
            return ERR_RANGE
        for li in range(blocks_for(st.context_lens[r])):
            b = int(st.tables[r, li])
            held[b] = held.get(b, 0) + 1
    for b, k in held.items():
        if k > st.ref_counts[b]:
            return ERR_RANGE
    for r in rows:
        nb = blocks_for(st.context_lens[r])
        for li in reversed(range(nb)):
            b = int(st.tables[r, li])
            st.ref_counts[b] -= 1
            if st.ref_counts[b] == 0:
                st._push(b)
            st.tables[r, li] = -1
        st.context_lens[r] = 0
    return OK


def match(st: BlockState, keys, num_keys):
    """Rows s = 0 .. S-1 with num_keys[s] > 0 (each empty) take the cached
    blocks of their leading keys keys[s][0 .. m_s) (m_s <= num_keys[s],
    stopping at the first key that is not cached); a block with no holder
    leaves the free queue.  Rows with num_keys[s] == 0 are untouched.
    Returns (status, m)."""
    num_keys = [int(n) for n in num_keys]
    S = len(num_keys)
    if S > st.tables.shape[0]:
        return ERR_SHAPE, None
    for s in range(S):
        if num_keys[s] < 0 or num_keys[s] > st.tables.shape[1] or (num_keys[s] > 0 and st.context_lens[s] != 0):
            return ERR_RANGE, None
    m = np.zeros(S, dtype=np.int32)
    for s in range(S):
        if num_keys[s] == 0:
            continue
        for i in range(num_keys[s]):
            b = st.cache.get(bytes(np.asarray(keys[s][i], dtype=np.uint8)))
            if b is None:
                break
            if st.ref_counts[b] == 0:
                st.queue.remove(b)
            st.ref_counts[b] += 1
            st.tables[s, i] = b
            m[s] = i + 1
        st.context_lens[s] = m[s] * BLOCK_SIZE
    return OK, m


def register(st: BlockState, keys, num_keys) -> int:
    """Give the full blocks of rows s = 0 .. S-1 their keys keys[s][0 ..
    num_keys[s]), in (row, block) order: a block that already has a key keeps
    it, and a key already cached keeps its block."""
    num_keys = [int(n) for n in num_keys]
    S = len(num_keys)
    if S > st.tables.shape[0]:
        return ERR_SHAPE
    for s in range(S):
        if num_keys[s] < 0 or num_keys[s] > int(st.context_lens[s]) // BLOCK_SIZE:
            return ERR_RANGE
    for s in range(S):
        for i in range(num_keys[s]):
            b = int(st.tables[s, i])
            k = bytes(np.asarray(keys[s][i], dtype=np.uint8))
            if b in st.block_key or k in st.cache:
                continue
            st.cache[k] = b
            st.block_key[b] = k
    return OK
