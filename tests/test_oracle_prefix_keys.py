"""Pins for the prefix-cache key oracle (no GPU).

The message is rebuilt here byte by byte with struct (an encoding written
independently of the oracle's numpy one), and the properties the pages state
are checked: a key stands for the whole prefix up to its block, equal
prefixes give equal keys (the sharing the cache exists for), the extra value
separates users, and only full blocks are keyed ("Prefix cache", section 4
of the serving-engine KV blog)."""
import hashlib
import struct

import numpy as np

from oracle import prefix_keys as pk


def test_message_encoding_rebuilt_with_struct():
    rng = np.random.default_rng(1)
    toks = rng.integers(-2 ** 31, 2 ** 31, size=48).tolist()
    parent = bytes(32)
    for i in range(3):
        msg = parent + struct.pack("<16i", *toks[16 * i:16 * i + 16]) + struct.pack("<q", -77)
        assert len(msg) == 104
        parent = hashlib.sha256(msg).digest()
        assert pk.sequence_keys(toks, extra=-77)[i] == parent


def test_sha256_itself_on_the_standard_vector():
    assert hashlib.sha256(b"abc").hexdigest() == \
        "ba7816bf8f01cfea414140de5dae2223b00361a396177a9cb410ff61f20015ad"


def test_a_key_stands_for_its_whole_prefix():
    rng = np.random.default_rng(2)
    a = rng.integers(0, 50000, size=80)
    b = a.copy()
    b[3] += 1                                    # differs in block 0 only
    ka, kb = pk.sequence_keys(a), pk.sequence_keys(b)
    assert len(ka) == 5
    assert all(x != y for x, y in zip(ka, kb))   # every later key changes too
    c = a.copy()
    c[70] += 1                                   # differs in block 4 only
    kc = pk.sequence_keys(c)
    assert kc[:4] == ka[:4] and kc[4] != ka[4]


def test_equal_prefixes_share_keys_and_same_tokens_elsewhere_do_not():
    rng = np.random.default_rng(3)
    prefix = rng.integers(0, 50000, size=48)
    x = np.concatenate([prefix, rng.integers(0, 50000, size=37)])
    y = np.concatenate([prefix, rng.integers(0, 50000, size=20)])
    assert pk.sequence_keys(x)[:3] == pk.sequence_keys(y)[:3]
    blk = prefix[16:32]
    alone = pk.sequence_keys(blk)[0]                 # same 16 tokens, empty prefix
    assert alone != pk.sequence_keys(prefix)[1]


def test_extra_value_separates_users_and_partial_blocks_are_not_keyed():
    toks = np.arange(40)
    assert pk.sequence_keys(toks, extra=1)[0] != pk.sequence_keys(toks, extra=2)[0]
    assert len(pk.sequence_keys(toks)) == 2          # 40 tokens: 2 full blocks


def test_continuing_a_chain_equals_hashing_at_once():
    rng = np.random.default_rng(4)
    toks = rng.integers(0, 50000, size=96)
    whole = pk.sequence_keys(toks, extra=9)
    first = pk.sequence_keys(toks[:32], extra=9)
    rest = pk.sequence_keys(toks[32:], extra=9, parent=first[-1])
    assert first + rest == whole
