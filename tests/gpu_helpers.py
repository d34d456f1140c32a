"""Helpers shared by the GPU parity tests (host <-> device marshalling and
the tolerance check).  Tolerance: max-abs 2e-3 and max-rel 1e-2 against the
oracle, relative error measured against max(|oracle|, 0.2) so that elements
near zero are held to the absolute bound (0.2 = 2e-3 / 1e-2)."""
import numpy as np
import torch

ATOL = 2e-3
RTOL = 1e-2
REL_FLOOR = 0.2


def dev_tensor(a, device="cuda"):
    x = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        x = x.view(torch.int16).view(torch.bfloat16)
    return x.to(device)


def host_bits(t):
    """bf16 CUDA tensor -> uint16 numpy bit patterns."""
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mabs = float(err.max()) if err.size else 0.0
    mrel = float((err / np.maximum(np.abs(ref), REL_FLOOR)).max()) if err.size else 0.0
    assert mabs <= ATOL and mrel <= RTOL, f"{what}: max-abs {mabs:.3e} (<= {ATOL}), max-rel {mrel:.3e} (<= {RTOL})"
    return mabs, mrel


class DeviceStep:
    """A workload's tensors on the GPU."""

    def __init__(self, w, device="cuda"):
        self.w = w
        self.k = dev_tensor(w.k_pool, device)
        self.v = dev_tensor(w.v_pool, device)
        self.q = dev_tensor(w.q, device)
        self.k_new = dev_tensor(w.k_new, device)
        self.v_new = dev_tensor(w.v_new, device)
        self.slots = dev_tensor(w.slot_mapping, device)
        self.tables = dev_tensor(w.block_tables, device)
        self.ctx = dev_tensor(w.context_lens, device)
        self.qsl = dev_tensor(w.query_start_loc, device)
        self.src = dev_tensor(w.copy_src, device) if w.copy_src is not None else None
        self.dst = dev_tensor(w.copy_dst, device) if w.copy_dst is not None else None

    def run(self, pkv, partition_blocks=0, workspace=None):
        w = self.w
        if self.src is not None:
            pkv.copy_blocks(self.k, self.v, self.src, self.dst)
        pkv.cache_write(self.k, self.v, self.k_new, self.v_new, self.slots)
        if w.is_decode:
            return pkv.decode_attention(self.k, self.v, self.q, self.tables, self.ctx, w.max_context_len, w.scale,
                                        partition_blocks=partition_blocks, workspace=workspace)
        return pkv.chunked_prefill_attention(self.k, self.v, self.q, self.qsl, self.ctx, self.tables,
                                             w.max_context_len, w.scale, workspace=workspace,
                                             query_start_loc_host=w.query_start_loc)
