"""GPU parity of shared-prefix decode (pkv_decode_attention_shared_prefix:
the blocks every sequence's table starts with are attended once per kv head
for all sequences on tensor cores, the rest per sequence, then merged)
against the CPU oracle, which attends each sequence over its whole context."""
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


def prepare(pkv, w):
    """The step's copy-on-write and cache write, as the decode step runs them."""
    ds = DeviceStep(w)
    if ds.src is not None:
        pkv.copy_blocks(ds.k, ds.v, ds.src, ds.dst)
    pkv.cache_write(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots)
    return ds


def shared(pkv, ds, J, workspace=None):
    w = ds.w
    return pkv.decode_attention_shared_prefix(ds.k, ds.v, ds.q, ds.tables, ds.ctx, w.max_context_len, J, w.scale,
                                              workspace=workspace)


def check(pkv, w, J=None, threads=8):
    ds = prepare(pkv, w)
    if J is None:
        J = pkv.common_prefix_blocks(w.block_tables, w.context_lens)
    out = shared(pkv, ds, J)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    k_ref, v_ref, ref = oracle.run_step(w, threads=threads)
    assert_close(out.cpu().numpy(), ref, f"{w.name} J={J}")
    assert np.array_equal(host_bits(ds.k), k_ref) and np.array_equal(host_bits(ds.v), v_ref)
    return ds, out, ref


def test_prefix_share_config(pkv):
    """Qwen3-1.7B, 32 sequences over a 3,000-token shared prefix (187 full
    shared blocks, then each sequence's copy of the partial block and its
    suffix): every output row against the oracle."""
    w = W.build_config(4)
    J = pkv.common_prefix_blocks(w.block_tables, w.context_lens)
    assert J == w.meta["shared_blocks"] == 187
    ds, out, ref = check(pkv, w, J)
    plain = pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale)
    torch.cuda.synchronize()
    assert_close(plain.cpu().numpy(), ref, "plain decode")


@pytest.mark.parametrize("hq,hkv,d", [(16, 8, 128), (8, 8, 128), (32, 8, 128), (64, 8, 128), (16, 8, 64),
                                      (8, 1, 64), (40, 40, 64), (32, 4, 128)])
def test_head_shapes(pkv, hq, hkv, d):
    """Every GQA group size and both head sizes; contexts from the prefix
    alone plus one token to the prefix plus 700."""
    J = 9
    ctx = [16 * J + x for x in (1, 2, 15, 16, 17, 100, 333, 700)]
    w = W.make_paged("shared-heads", hq * 100 + hkv + d, hq, hkv, d, ctx, [1] * len(ctx), share_prefix_blocks=J)
    check(pkv, w, J)


@pytest.mark.parametrize("B,G", [(1, 2), (31, 2), (32, 2), (33, 2), (70, 1), (130, 1), (17, 4), (9, 8)])
def test_query_tiles(pkv, B, G):
    """Batches whose B x G query rows fill 64-row tiles exactly, leave a
    ragged last tile, or need one row only."""
    J = 13
    ctx = W.randint_inclusive(B * 7 + G, 3, B, 16 * J + 1, 16 * J + 300)
    w = W.make_paged("shared-tiles", 1000 + B * 10 + G, 8 * G, 8, 128, ctx, [1] * B, share_prefix_blocks=J)
    check(pkv, w, J)


@pytest.mark.parametrize("J", [1, 3, 4, 5, 64, 311])
def test_prefix_lengths(pkv, J):
    """One chunk of the shared blocks per kv head (small prefixes) up to
    many chunks of uneven size."""
    ctx = [16 * J + 1, 16 * J + 40, 16 * J + 97, 16 * J + 16, 16 * J + 250]
    w = W.make_paged("shared-len", 2000 + J, 16, 8, 128, ctx, [1] * len(ctx), share_prefix_blocks=J)
    check(pkv, w, J)


def test_fewer_shared_blocks_than_the_tables_share(pkv):
    """Any J up to the common prefix is valid: the blocks past J are attended
    per sequence."""
    J = 40
    ctx = [16 * J + x for x in (5, 77, 300)]
    w = W.make_paged("shared-partial", 3001, 16, 8, 128, ctx, [1] * 3, share_prefix_blocks=J)
    for j in (0, 1, 17, J):
        check(pkv, w, j)


def test_context_ending_at_the_prefix(pkv):
    """A sequence whose context is exactly the shared blocks (its own part is
    empty) merges the shared states alone."""
    J = 6
    ctx = [16 * J, 16 * J + 3, 16 * J + 50]
    w = W.make_paged("shared-edge", 3002, 16, 8, 128, ctx, [1] * 3, share_prefix_blocks=J)
    check(pkv, w, J)


def test_zero_shared_blocks_is_plain_decode(pkv):
    ctx = [17, 300, 1000]
    w = W.make_paged("shared-zero", 3003, 16, 8, 128, ctx, [1] * 3, share_prefix_blocks=1)
    ds = prepare(pkv, w)
    a = shared(pkv, ds, 0).clone()
    b = pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_repeatable_and_workspace_left_zeroed(pkv):
    """Two calls on one workspace give bit-identical results (every merge
    runs in a fixed order) and leave the arrival counters at zero."""
    J = 30
    ctx = [16 * J + x for x in (1, 4000, 17, 2500)]
    w = W.make_paged("shared-repeat", 3004, 16, 8, 128, ctx, [1] * 4, share_prefix_blocks=J)
    ds = prepare(pkv, w)
    need = pkv.decode_shared_prefix_workspace_size(4, 16, 8, 128, w.max_context_len, J)
    ws = pkv.new_workspace(need)
    a = shared(pkv, ds, J, workspace=ws).clone()
    b = shared(pkv, ds, J, workspace=ws).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert int(ws[:512].count_nonzero().item()) == 0
    _, _, ref = oracle.run_step(w)
    assert_close(a.cpu().numpy(), ref, "repeat")


def test_broken_promise_is_reported(pkv):
    """A sequence whose table differs inside the claimed shared part, or
    whose context is shorter than it, raises PKV_ERR_RANGE with its index;
    nothing faults and the next call is clean."""
    J = 8
    ctx = [16 * J + 5, 16 * J + 9, 16 * J + 30]
    w = W.make_paged("shared-bad", 3005, 16, 8, 128, ctx, [1] * 3, share_prefix_blocks=J)
    ds = prepare(pkv, w)
    tables = ds.tables.clone()
    tables[2, 3] = tables[2, J]  # another valid block id
    pkv.decode_attention_shared_prefix(ds.k, ds.v, ds.q, tables, ds.ctx, w.max_context_len, J, w.scale)
    torch.cuda.synchronize()
    assert pkv.get_error() == (9, 2)
    ctx_short = ds.ctx.clone()
    ctx_short[1] = 16 * J - 1
    pkv.decode_attention_shared_prefix(ds.k, ds.v, ds.q, ds.tables, ctx_short, w.max_context_len, J, w.scale)
    torch.cuda.synchronize()
    assert pkv.get_error() == (9, 1)
    out = shared(pkv, ds, J)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    _, _, ref = oracle.run_step(w)
    assert_close(out.cpu().numpy(), ref, "after errors")


def test_e4m3_pools_attend_the_prefix_per_sequence(pkv):
    """e4m3 pools take the per-sequence path: the result is bit-identical
    to pkv_decode_attention on the same pools."""
    J = 10
    ctx = [16 * J + x for x in (1, 33, 200)]
    w = W.make_paged("shared-e4m3", 3006, 16, 8, 128, ctx, [1] * 3, share_prefix_blocks=J)
    ds = prepare(pkv, w)
    nb, hkv, _, d = w.k_pool.shape
    k8 = torch.empty((nb, hkv, 16, d), dtype=torch.uint8, device="cuda")
    v8 = torch.empty_like(k8)
    slots = torch.arange(nb * 16, dtype=torch.int32, device="cuda")
    rk = ds.k.permute(0, 2, 1, 3).reshape(nb * 16, hkv, d).contiguous()
    rv = ds.v.permute(0, 2, 1, 3).reshape(nb * 16, hkv, d).contiguous()
    pkv.cache_write(k8, v8, rk, rv, slots, k_scale=1 / 64, v_scale=1 / 64)
    a = pkv.decode_attention_shared_prefix(k8, v8, ds.q, ds.tables, ds.ctx, w.max_context_len, J, w.scale,
                                           k_scale=1 / 64, v_scale=1 / 64)
    b = pkv.decode_attention(k8, v8, ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale, k_scale=1 / 64,
                             v_scale=1 / 64)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    assert torch.equal(a, b)
