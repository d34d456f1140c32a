"""Prefix-cache block keys oracle -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  It shares no code with the CUDA library.

Section 4 ("Prefix cache") of the serving-engine KV blog: every full block
gets a key that hashes the previous block's key, this block's token ids and
extra information (adapter, multimodal input hashes, a per-user cache salt).
Because the previous key is part of it, one key stands for the whole prefix
up to its block: the same 16 tokens after a different prefix get a different
key.  Only full blocks are keyed.  The default hash is SHA-256.

Readings taken where the pages give the parts of a key but not its bytes:
- the hashed message is parent key (32 bytes) || the block's 16 token ids as
  little-endian int32 (64 bytes) || the sequence's extra value as a
  little-endian int64 (8 bytes), 104 bytes;
- the first block's parent key is 32 zero bytes, unless a parent key is
  given (continuing a chain from an earlier call);
- the key is the 32-byte SHA-256 digest (hashlib provides SHA-256 here).

Parity status: pinned by ``tests/test_oracle_prefix_keys.py`` (the message
rebuilt byte by byte with struct, chaining and sharing properties).
"""
from __future__ import annotations

import hashlib

import numpy as np

BLOCK_SIZE = 16
ROOT = bytes(32)


def block_key(parent: bytes, tokens, extra: int) -> bytes:
    """Key of one full block: SHA-256(parent || tokens (16 x <i4) || extra (<i8))."""
    t = np.asarray(tokens, dtype="<i4")
    assert t.shape == (BLOCK_SIZE,) and len(parent) == 32
    msg = bytes(parent) + t.tobytes() + np.asarray([extra], dtype="<i8").tobytes()
    return hashlib.sha256(msg).digest()


def sequence_keys(tokens, extra: int = 0, parent: bytes = ROOT) -> list:
    """Keys of every full block of one token list, chained from `parent`."""
    tokens = np.asarray(tokens, dtype=np.int64)
    keys = []
    for i in range(len(tokens) // BLOCK_SIZE):
        parent = block_key(parent, tokens[i * BLOCK_SIZE:(i + 1) * BLOCK_SIZE], extra)
        keys.append(parent)
    return keys


def batch_keys(token_ids, query_start_loc, max_blocks: int, extra=None, parents=None) -> np.ndarray:
    """keys[s][i] (uint8 [S][max_blocks][32]) for the full blocks of sequence s,
    whose tokens are token_ids[query_start_loc[s]:query_start_loc[s+1]];
    entries past a sequence's full blocks are zero."""
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    S = len(qsl) - 1
    out = np.zeros((S, max_blocks, 32), dtype=np.uint8)
    for s in range(S):
        e = int(extra[s]) if extra is not None else 0
        p = bytes(np.asarray(parents[s], dtype=np.uint8)) if parents is not None else ROOT
        ks = sequence_keys(np.asarray(token_ids)[qsl[s]:qsl[s + 1]], e, p)
        assert len(ks) <= max_blocks
        for i, k in enumerate(ks):
            out[s, i] = np.frombuffer(k, dtype=np.uint8)
    return out
