"""Over-write guards: every output buffer of the library is passed as a view
inside a larger buffer whose borders hold a sentinel bit pattern, and every
workspace is followed by sentinel bytes; after the calls the sentinels must
be intact (and the outputs still right)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import block_manager as bm
from oracle import prefix_keys as pk
import pkv_workloads as W
from gpu_helpers import DeviceStep, assert_close, dev_tensor

pytestmark = pytest.mark.gpu

GUARD = 64                 # rows of guard on each side
SENT_F32 = 0x7FA5A5A5      # a NaN payload no kernel writes
SENT_U8 = 0xA5


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_291_gb300 as p
    p.load()
    return p


def guarded_f32(shape):
    full = torch.full((shape[0] + 2 * GUARD,) + tuple(shape[1:]), 0, dtype=torch.int32, device="cuda")
    full.fill_(SENT_F32)
    return full, full.view(torch.float32)[GUARD:GUARD + shape[0]]


def guard_intact_i32(full, n):
    a = full.cpu().numpy()
    return bool(np.all(a[:GUARD] == SENT_F32) and np.all(a[GUARD + n:] == SENT_F32))


def guarded_workspace(pkv, nbytes):
    ws = torch.zeros(nbytes + 4096, dtype=torch.uint8, device="cuda")
    ws[nbytes:] = SENT_U8
    return ws


@pytest.mark.parametrize("cfg", [1, 2])
def test_decode_writes_only_its_output_rows_and_workspace(pkv, cfg):
    w = W.build_config(cfg)
    ds = DeviceStep(w)
    pkv.cache_write(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots)
    need = pkv.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_context_len)
    ws = guarded_workspace(pkv, need)
    full, out = guarded_f32((w.num_seqs, w.num_q_heads, w.head_dim))
    pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale, out=out,
                         workspace=ws[:need])
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    assert guard_intact_i32(full, w.num_seqs), "decode wrote outside its output rows"
    wsn = ws.cpu().numpy()
    assert np.all(wsn[need:] == SENT_U8), "decode wrote past its workspace"
    counters_end = 256 + -(-w.num_seqs * w.num_kv_heads * 4 // 256) * 256
    assert not wsn[:counters_end].any(), "decode left its header or arrival counters non-zero"
    _, _, ref = oracle.run_step(w, threads=16)
    assert_close(out.cpu().numpy(), ref, f"config {cfg}")


def test_chunked_prefill_writes_only_its_output_rows_and_workspace(pkv):
    w = W.make_paged("guards", 9, 16, 8, 128, [300, 40, 700, 5], [150, 1, 300, 1])
    ds = DeviceStep(w)
    pkv.cache_write(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots)
    need = pkv.prefill_workspace_size(w.num_seqs, w.num_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                      w.max_context_len)
    ws = guarded_workspace(pkv, need)
    full, out = guarded_f32((w.num_tokens, w.num_q_heads, w.head_dim))
    pkv.chunked_prefill_attention(ds.k, ds.v, ds.q, ds.qsl, ds.ctx, ds.tables, w.max_context_len, w.scale,
                                  out=out, workspace=ws[:need], query_start_loc_host=w.query_start_loc)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    assert guard_intact_i32(full, w.num_tokens), "prefill wrote outside its output rows"
    wsn = ws.cpu().numpy()
    assert np.all(wsn[need:] == SENT_U8), "prefill wrote past its workspace"
    counters_end = 256 + -(-w.num_seqs * w.num_kv_heads * 4 // 256) * 256
    assert not wsn[:counters_end].any(), "prefill left its header or arrival counters non-zero"
    _, _, ref = oracle.run_step(w, threads=16)
    assert_close(out.cpu().numpy(), ref, "guarded prefill")


def test_block_and_key_outputs_stay_in_bounds(pkv):
    S, T = 5, 45
    qsl = np.array([0, 20, 20, 21, 40, 45], np.int32)
    blocks = pkv.Blocks(40, S, 6, prefix_cache=True)
    full = torch.full((T + 2 * GUARD,), SENT_F32, dtype=torch.int32, device="cuda")
    pairs = torch.full((S + 2 * GUARD,), SENT_F32, dtype=torch.int32, device="cuda")
    pairs2 = torch.full((S + 2 * GUARD,), SENT_F32, dtype=torch.int32, device="cuda")
    slots, _, _, _ = blocks.append(dev_tensor(qsl), T, slot_mapping=full[GUARD:GUARD + T],
                                   cow_src=pairs[GUARD:GUARD + S], cow_dst=pairs2[GUARD:GUARD + S])
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    assert guard_intact_i32(full, T) and guard_intact_i32(pairs, S) and guard_intact_i32(pairs2, S)
    st = bm.BlockState(40, S, 6)
    _, o_slots, _, _ = bm.append(st, qsl)
    assert np.array_equal(slots.cpu().numpy(), o_slots)

    toks = np.arange(3000, 3077, dtype=np.int32)                # 4 full blocks and 13 tokens
    MB = 6
    kbuf = torch.full((1, MB, 32), SENT_U8, dtype=torch.uint8, device="cuda")
    pkv.prefix_keys(dev_tensor(toks), dev_tensor(np.array([0, 77], np.int32)), MB, keys=kbuf)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    got = kbuf.cpu().numpy()[0]
    assert got[:4].tobytes() == b"".join(pk.sequence_keys(toks))
    assert np.all(got[4:] == SENT_U8), "keys written past the sequence's full blocks"
