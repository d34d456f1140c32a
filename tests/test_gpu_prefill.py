"""GPU parity of chunked-prefill attention (tcgen05 tiles for the prompt
chunks, the decode kernel for the single-token rows of the mixed batch)
against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import pkv_workloads as W
from gpu_helpers import DeviceStep, assert_close, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_291_gb300 as p
    p.load()
    return p


def run_and_check(pkv, w, threads=16):
    ds = DeviceStep(w)
    out = ds.run(pkv)
    torch.cuda.synchronize()
    st = pkv.get_error()
    assert st == (0, 0), f"device error {st}"
    k_ref, v_ref, ref = oracle.run_step(w, threads=threads)
    got = out.cpu().numpy()
    assert np.array_equal(host_bits(ds.k), k_ref) and np.array_equal(host_bits(ds.v), v_ref)
    return assert_close(got, ref, w.name), out


def test_chunked_mixed_config_full(pkv):
    """3 prompts x 512-token chunk at offset 1,024 + 32 decode rows."""
    w = W.build_config(5)
    run_and_check(pkv, w)


@pytest.mark.parametrize("qlen,prefix", [(2, 0), (127, 0), (128, 0), (129, 0), (300, 0), (16, 1), (64, 15),
                                         (200, 17), (128, 128), (333, 1024), (1, 700)])
def test_prefill_edges(pkv, qlen, prefix):
    """Tile and block edges: chunks shorter/longer than a 128-row tile,
    prefixes ending inside a block, keys past the last position."""
    w = W.make_paged("edge", 1000 + qlen + prefix, 16, 8, 128, [prefix + qlen], [qlen])
    run_and_check(pkv, w)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (32, 4), (16, 2)])
def test_prefill_head_groups(pkv, hq, hkv):
    w = W.make_paged("gqa", hq * 10 + hkv, hq, hkv, 128, [300, 1, 450, 77], [150, 1, 200, 1])
    run_and_check(pkv, w)


def test_mixed_order_and_many_sequences(pkv):
    """Decode rows before, between and after several prefill chunks."""
    ctx = [40, 900, 5, 260, 1300, 33, 129, 2]
    ql = [1, 256, 1, 260, 100, 1, 129, 2]
    w = W.make_paged("order", 4242, 16, 8, 128, ctx, ql)
    run_and_check(pkv, w)


def test_chunked_equals_one_shot_on_gpu(pkv):
    """A prompt processed in consecutive slices (each over the cached
    prefix) gives the rows of one-shot causal prefill."""
    n = 700
    w = W.make_paged("whole", 77, 16, 8, 128, [n], [n])
    ds = DeviceStep(w)
    one = ds.run(pkv).clone()
    parts = []
    for first, last in W.chunk_slices(n, 256):
        ql = last - first + 1
        qsl = torch.tensor([0, ql], dtype=torch.int32, device="cuda")
        ctx = torch.tensor([last + 1], dtype=torch.int32, device="cuda")
        parts.append(pkv.chunked_prefill_attention(ds.k, ds.v, ds.q[first:last + 1].contiguous(), qsl, ctx,
                                                   ds.tables, n, w.scale,
                                                   query_start_loc_host=np.array([0, ql], np.int32)))
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    chunked = torch.cat(parts)
    # each row sees the same keys in the same tiles order only up to the
    # tile alignment, so compare within the tolerance, and both to the oracle
    _, _, ref = oracle.run_step(w, threads=16)
    assert_close(one.cpu().numpy(), ref, "one-shot")
    assert_close(chunked.cpu().numpy(), ref, "chunked")


def test_prefill_head_dim_64_is_rejected_cleanly(pkv):
    w = W.make_paged("d64", 5, 8, 2, 64, [40], [20])
    ds = DeviceStep(w)
    with pytest.raises(pkv.PKVError) as e:
        ds.run(pkv)
    assert e.value.status == 12
