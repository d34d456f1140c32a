"""The bounded waits inside the decode kernel, made to expire without a
fault: the test hook leaves the producer warp idle, so the consumer and
merger warps wait for work descriptors that never arrive.  Their waits give
up after the bounded time, the launch records PKV_ERR_TIMEOUT, nothing is in
flight when the kernel ends, and the context stays usable: the next ordinary
call on the same workspace is right."""
import pytest
import torch

import oracle
import pkv_workloads as W
from gpu_helpers import DeviceStep, assert_close

pytestmark = pytest.mark.gpu

PKV_ERR_TIMEOUT = 10
CONSUMER_SITE, MERGER_SITE = 2, 3  # details the decode kernel records for its waits


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_291_gb300 as p
    p.load()
    return p


def test_expired_wait_reports_timeout_and_next_call_is_right(pkv):
    w = W.make_paged("stall", 23, 16, 8, 128, [40, 300, 1500], [1, 1, 1])
    ds = DeviceStep(w)
    pkv.cache_write(ds.k, ds.v, ds.k_new, ds.v_new, ds.slots)
    need = pkv.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_context_len)
    ws = pkv.new_workspace(need)
    sentinel = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), 7.0, dtype=torch.float32, device="cuda")
    out = sentinel.clone()
    assert pkv.get_error() == (0, 0)
    pkv.test_arm_decode_stall(1)
    pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale, out=out, workspace=ws)
    torch.cuda.synchronize()
    status, detail = pkv.get_error()
    assert status == PKV_ERR_TIMEOUT and detail in (CONSUMER_SITE, MERGER_SITE), (status, detail)
    assert torch.equal(out, sentinel), "a launch that timed out wrote output rows"
    assert int(ws.count_nonzero().item()) == 0, "the stalled launch touched the workspace"
    # The hook was armed for one launch only: the next call runs normally.
    pkv.decode_attention(ds.k, ds.v, ds.q, ds.tables, ds.ctx, w.max_context_len, w.scale, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    _, _, ref = oracle.run_step(w)
    assert_close(out.cpu().numpy(), ref, "decode after a timeout")


def test_stall_hook_rejects_negative_counts(pkv):
    with pytest.raises(pkv.PKVError):
        pkv.test_arm_decode_stall(-1)
    pkv.test_arm_decode_stall(0)
