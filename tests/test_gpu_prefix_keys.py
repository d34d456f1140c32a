"""GPU parity of pkv_prefix_keys (SHA-256 block-key chains) against the
oracle (hashlib over the same 104-byte messages): bit-exact keys."""
import numpy as np
import pytest
import torch

from oracle import prefix_keys as pk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_291_gb300 as p
    p.load()
    return p


def _t(a, dtype):
    return torch.tensor(np.asarray(a), dtype=dtype, device="cuda")


@pytest.mark.parametrize("seed,lens", [(0, [0, 15, 16, 17, 33, 100]), (1, [3000] * 4 + [31] * 40),
                                        (2, list(range(0, 700, 7)))])
def test_keys_match_the_oracle(pkv, seed, lens):
    rng = np.random.default_rng(seed)
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    toks = rng.integers(-2 ** 31, 2 ** 31, size=int(qsl[-1]), dtype=np.int64).astype(np.int32)
    extra = rng.integers(-2 ** 63, 2 ** 63, size=len(lens), dtype=np.int64)
    MB = max(1, max(lens) // 16)
    keys = pkv.prefix_keys(_t(toks, torch.int32), _t(qsl, torch.int32), MB, extra=_t(extra, torch.int64))
    assert pkv.get_error() == (0, 0)
    ref = pk.batch_keys(toks, qsl, MB, extra=extra)
    assert np.array_equal(keys.cpu().numpy(), ref)


def test_parent_keys_continue_a_chain(pkv):
    rng = np.random.default_rng(5)
    toks = rng.integers(0, 150000, size=(3, 96)).astype(np.int32)
    whole = [pk.sequence_keys(t, extra=4) for t in toks]
    parents = np.stack([np.frombuffer(w[1], dtype=np.uint8) for w in whole])
    rest = toks[:, 32:].reshape(-1)
    qsl = np.arange(0, 3 * 64 + 1, 64, dtype=np.int32)
    keys = pkv.prefix_keys(_t(rest, torch.int32), _t(qsl, torch.int32), 4, extra=_t([4, 4, 4], torch.int64),
                           parent_keys=_t(parents, torch.uint8))
    assert pkv.get_error() == (0, 0)
    got = keys.cpu().numpy()
    for s in range(3):
        for i in range(4):
            assert bytes(got[s, i]) == whole[s][2 + i]


def test_too_many_blocks_is_a_range_error(pkv):
    qsl = _t([0, 16, 64], torch.int32)
    keys = pkv.prefix_keys(_t(np.arange(64), torch.int32), qsl, 2)
    assert pkv.get_error() == (9, 1)                  # sequence 1 has 3 full blocks
    assert bytes(keys.cpu().numpy()[0, 0]) == pk.sequence_keys(np.arange(16))[0]
