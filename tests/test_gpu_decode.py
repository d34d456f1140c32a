"""GPU parity of paged decode attention (with split-KV and the in-launch
log-sum-exp merge) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import pkv_workloads as W
from gpu_helpers import DeviceStep, assert_close, dev_tensor, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_291_gb300 as p
    p.load()
    return p


def run_and_check(pkv, w, partition_blocks=0, rows=None, threads=8):
    ds = DeviceStep(w)
    out = ds.run(pkv, partition_blocks=partition_blocks)
    torch.cuda.synchronize()
    st = pkv.get_error()
    assert st == (0, 0), f"device error {st}"
    k_ref, v_ref, ref = oracle.run_step(w, threads=threads, rows=rows)
    got = out.cpu().numpy()
    if rows is not None:
        sel = np.concatenate([np.arange(w.query_start_loc[s], w.query_start_loc[s + 1]) for s in rows])
        got, ref = got[sel], ref[sel]
    return assert_close(got, ref, w.name), ds, k_ref, v_ref


@pytest.mark.parametrize("cfg", [1, 2])
def test_decode_configs_full(pkv, cfg):
    w = W.build_config(cfg)
    _, ds, k_ref, v_ref = run_and_check(pkv, w)
    assert np.array_equal(host_bits(ds.k), k_ref) and np.array_equal(host_bits(ds.v), v_ref)


def test_prefix_share_config_full(pkv):
    """copy_blocks (32 CoW copies) + cache_write of the suffixes + decode at 3,032."""
    w = W.build_config(4)
    _, ds, k_ref, v_ref = run_and_check(pkv, w)
    assert np.array_equal(host_bits(ds.k), k_ref) and np.array_equal(host_bits(ds.v), v_ref)


@pytest.mark.slow
def test_mha_long_context_config_full(pkv):
    """LLaMA-13B MHA shape at full size (4 x 32,768 + 64 short, 4.1 GB of
    K/V): every output row of all 68 sequences against the oracle, the four
    long ones included (split-KV + merge), and both pools bit-exact after the
    step's cache write."""
    w = W.build_config(3)
    _, ds, k_ref, v_ref = run_and_check(pkv, w, threads=16)
    assert np.array_equal(host_bits(ds.k), k_ref) and np.array_equal(host_bits(ds.v), v_ref)


@pytest.mark.parametrize("pb", [1, 2, 3, 7, 40])
def test_forced_partitions_match(pkv, pb):
    """Partition sizes from one block up to the whole context all agree with
    the unsplit definition (the log-sum-exp merge is exact in real arithmetic)."""
    w = W.make_paged("parts", 77, 16, 8, 128, [1, 15, 16, 17, 31, 32, 33, 100, 640, 641], [1] * 10)
    run_and_check(pkv, w, partition_blocks=pb)


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (16, 4, 128), (64, 8, 128), (8, 1, 64), (16, 8, 64),
                                      (32, 4, 64), (40, 40, 64)])
def test_head_shapes(pkv, hq, hkv, d):
    ctx = [1, 2, 16, 17, 48, 250, 333]
    w = W.make_paged("heads", hq * 100 + hkv + d, hq, hkv, d, ctx, [1] * len(ctx))
    run_and_check(pkv, w)


@pytest.mark.parametrize("B,n", [(34, 640), (20, 640), (50, 320), (7, 2000), (300, 48), (152, 17)])
def test_equal_contexts(pkv, B, n):
    """Batches whose pairs all span the same blocks: the automatic plan then
    takes ranges of whole pairs when that costs at most 15% more units per
    range (no pair split), else the usual cut."""
    w = W.make_paged("equal", 4000 + B + n, 16, 8, 128, [n] * B, [1] * B)
    run_and_check(pkv, w)


def test_many_sequences_ragged(pkv):
    """More than one 32-sequence window in the work decoder, random lengths."""
    ctx = W.randint_inclusive(5, 7, 300, 1, 700)
    w = W.make_paged("ragged", 5, 16, 8, 128, ctx, [1] * 300)
    run_and_check(pkv, w)


def test_workspace_reuse_is_deterministic(pkv):
    """The workspace is left zeroed: a second call reuses it and gives the
    bit-identical result (partials are merged in a fixed order)."""
    w = W.make_paged("reuse", 9, 16, 8, 128, [5000, 17, 3000, 1], [1] * 4)
    ds = DeviceStep(w)
    pkv.cache_write(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots)
    need = pkv.decode_workspace_size(4, 16, 8, 128, w.max_context_len, 4)
    ws = pkv.new_workspace(need)
    a = pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale, workspace=ws,
                             partition_blocks=4).clone()
    b = pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale, workspace=ws,
                             partition_blocks=4).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    # the header (work counters) and the per-(sequence, kv head) arrival counters are zero again
    assert int(ws[:512].count_nonzero().item()) == 0
    _, _, ref = oracle.run_step(w)
    assert_close(a.cpu().numpy(), ref, "reuse")


def test_empty_context_gives_zero_row(pkv):
    w = W.make_paged("empty", 10, 8, 2, 128, [7, 20], [1, 1])
    ds = DeviceStep(w)
    pkv.cache_write(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots)
    ctx = ds.ctx.clone()
    ctx[0] = 0
    out = pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ctx, w.max_context_len, w.scale)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    assert torch.all(out[0] == 0)
    _, _, ref = oracle.run_step(w)
    assert_close(out[1].cpu().numpy(), ref[1], "row 1")


def test_bad_block_id_reports_range_error_without_fault(pkv):
    """An id outside the pool is never dereferenced: the kernel reads block 0
    instead and records PKV_ERR_RANGE with the sequence index."""
    w = W.make_paged("badid", 11, 8, 2, 128, [40, 40], [1, 1])
    ds = DeviceStep(w)
    tables = ds.tables.clone()
    tables[1, 1] = w.num_blocks + 1000
    pkv.decode_attention(ds.k, ds.v, ds.q, tables, ds.ctx, w.max_context_len, w.scale)
    st, detail = pkv.get_error()
    assert st == 9 and detail == 1
    assert pkv.get_error() == (0, 0)


def test_context_longer_than_table_is_clamped_and_reported(pkv):
    w = W.make_paged("clamp", 12, 8, 2, 128, [40, 40], [1, 1])
    ds = DeviceStep(w)
    ctx = ds.ctx.clone()
    ctx[0] = 40 + 16 * 10  # beyond max_blocks_per_seq * 16
    pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ctx, 40 + 160, w.scale)
    st, detail = pkv.get_error()
    assert st == 9 and detail == 0


def test_host_argument_errors(pkv):
    w = W.build_config(1)
    ds = DeviceStep(w)
    with pytest.raises(pkv.PKVError) as e:  # 32 q heads over 8 kv heads is fine; 12 is not a multiple
        pkv.decode_attention(ds.k, ds.v, ds.q[:, :12].contiguous(), ds.tables, ds.ctx, 512, 0.125)
    assert e.value.status == 3
    ws = pkv.new_workspace(256)
    with pytest.raises(pkv.PKVError) as e:
        pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ds.ctx, 4096 * 16, 0.125, workspace=ws)
    assert e.value.status == 7


def test_decode_rows_through_mixed_batch_api(pkv):
    """A batch whose every query_len is 1 through the chunked-prefill call
    takes the decode kernel with the rows located by query_start_loc."""
    w = W.make_paged("mixed-decode", 13, 16, 8, 128, [5, 900, 33], [1, 1, 1])
    ds = DeviceStep(w)
    pkv.cache_write(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots)
    out = pkv.chunked_prefill_attention(ds.k, ds.v, ds.q, ds.qsl, ds.ctx, ds.tables, w.max_context_len, w.scale,
                                        query_start_loc_host=w.query_start_loc)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    _, _, ref = oracle.run_step(w)
    assert_close(out.cpu().numpy(), ref, "mixed decode rows")


def _lengths_from_previous_kernel(pkv, fresh: list, stale_value: int):
    """A fake two-block pool whose block 0 holds stale int32 values and block 1
    the fresh ones; returns (k_fake, v_fake, view of block 0, launch) where
    launch() rewrites block 0 from block 1 with pkv_copy_blocks.  The decode
    call made right after may start before that copy ends (both launch
    overlapped), so it can see the stale values before its wait."""
    n = len(fresh)
    fk = torch.zeros((2, 1, 16, 128), dtype=torch.bfloat16, device="cuda")
    fv = torch.zeros_like(fk)
    flat = fk.view(torch.int32).view(-1)  # 1,024 int32 per block
    assert n <= 1024
    flat[1024:1024 + n] = torch.tensor(fresh, dtype=torch.int32, device="cuda")
    src = torch.tensor([1], dtype=torch.int32, device="cuda")
    dst = torch.tensor([0], dtype=torch.int32, device="cuda")
    one, zero = np.array([1], dtype=np.int32), np.array([0], dtype=np.int32)

    def launch():
        flat[0:n] = stale_value
        pkv.copy_blocks(fk, fv, src, dst, src_host=one, dst_host=zero)

    return flat[0:n], launch


def test_lengths_written_by_the_previous_kernel(pkv):
    """context_lens produced by the kernel launched just before decode: the
    decode plan may be worked out from stale lengths before the wait, and must
    be redone from the fresh ones after it."""
    w = W.make_paged("prev-kernel lengths", 21, 16, 8, 128, [640] * 20 + [37, 1000, 3, 129], [1] * 24)
    ds = DeviceStep(w)
    pkv.cache_write(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots)
    _, _, ref = oracle.run_step(w)
    ctx_view, launch = _lengths_from_previous_kernel(pkv, w.context_lens.tolist(), 1)
    for _ in range(6):
        launch()
        out = pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ctx_view, w.max_context_len, w.scale)
        torch.cuda.synchronize()
        assert pkv.get_error() == (0, 0)
        assert_close(out.cpu().numpy(), ref, "lengths from the previous kernel")


def test_row_offsets_written_by_the_previous_kernel(pkv):
    """The same through the mixed-batch call: query_start_loc (which decides
    which rows are decode rows) comes from the kernel launched just before."""
    w = W.make_paged("prev-kernel qsl", 22, 16, 8, 128, [300, 2000, 90, 640], [1, 1, 1, 1])
    ds = DeviceStep(w)
    pkv.cache_write(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots)
    _, _, ref = oracle.run_step(w)
    qsl_view, launch = _lengths_from_previous_kernel(pkv, w.query_start_loc.tolist(), 0)
    for _ in range(6):
        launch()
        out = pkv.chunked_prefill_attention(ds.k, ds.v, ds.q, qsl_view, ds.ctx, ds.tables, w.max_context_len,
                                            w.scale, query_start_loc_host=w.query_start_loc)
        torch.cuda.synchronize()
        assert pkv.get_error() == (0, 0)
        assert_close(out.cpu().numpy(), ref, "row offsets from the previous kernel")
