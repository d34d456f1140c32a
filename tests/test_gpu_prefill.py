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


def test_prefill_grid_of_several_waves(pkv):
    """Enough row tiles that the grid needs more than one CTA per SM: no
    row tile is split into one-head CTAs and the CTAs run in several waves
    (the batches above are small enough that their longest tiles are
    split)."""
    ctx = [400 + 37 * i for i in range(14)]
    ql = [400 - 13 * i for i in range(14)]
    w = W.make_paged("waves", 515, 16, 8, 128, ctx, ql)
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


def test_prefill_head_dim_64_mixed_batch(pkv):
    """The Llama-3.2-1B attention shape (32 q / 8 kv heads, head_dim 64) in a
    mixed batch: chunks on the tensor cores (one 64-dim panel per tile),
    decode rows beside them."""
    w = W.make_paged("llama1b mixed", 64, 32, 8, 64, [300, 40, 700, 1, 513, 17], [150, 1, 300, 1, 129, 1])
    run_and_check(pkv, w)


@pytest.mark.parametrize("hq,hkv,qlen,prefix", [(8, 8, 128, 0), (16, 4, 129, 15), (8, 1, 200, 17),
                                                (16, 8, 2, 1024)])
def test_prefill_head_dim_64_edges(pkv, hq, hkv, qlen, prefix):
    w = W.make_paged("d64 edge", 640 + hq + hkv + qlen, hq, hkv, 64, [prefix + qlen, 33], [qlen, 1])
    run_and_check(pkv, w)


def _bf16(x):
    return W._f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _pool_index(w, s, pos):
    blk = int(w.block_tables[s][pos // W.BLOCK_SIZE])
    return blk, pos % W.BLOCK_SIZE


def test_prefill_dominant_keys_and_tiny_weights(pkv):
    """P V runs with P in fp16.  Scores are built so that two keys carry
    most of the weight (the second at 2^0.51 times the first, so its P is
    not a power of two, with V = +3 and -3) while the ~2,100 others sit 14-15
    binary orders below: under the fp16 normal range once P is formed, yet
    about 4% of the row sum, with V near 1.  Flushing those weights to zero
    moves the output by ~4e-2; P rounded to bf16 by ~2.7e-3 (both beyond
    the tolerance); fp16 P by ~3.5e-4."""
    prefix, ql, d = 2048, 128, 128
    w = W.make_paged("tiny-p", 31, 16, 8, d, [prefix + ql], [ql])
    rng = np.random.default_rng(7)
    # q = (8, 0, ...), k = (beta, 0, ...): log2-domain score 8*beta*scale*log2(e)
    w.q[:] = 0
    w.q[:, :, 0] = _bf16(8.0)
    beta = rng.uniform(5.4, 6.3, size=prefix + ql)
    vals = 1.0 + 0.1 * rng.standard_normal((prefix + ql, w.num_kv_heads, d))
    for pos, b, v in ((0, 20.0, 3.0), (700, 20.5, -3.0)):
        beta[pos], vals[pos] = b, v
    for pos in range(prefix):
        blk, row = _pool_index(w, 0, pos)
        w.k_pool[blk, :, row, :] = 0
        w.k_pool[blk, :, row, 0] = _bf16(beta[pos])
        w.v_pool[blk, :, row, :] = _bf16(vals[pos])
    w.k_new[:] = 0
    w.k_new[:, :, 0] = _bf16(beta[prefix:])[:, None]
    w.v_new[:] = _bf16(vals[prefix:])
    run_and_check(pkv, w)


def test_prefill_v_beyond_fp16_range_is_exact(pkv):
    """A V entry of a visible key that fp16 cannot hold (|v| > 65504): the
    CTA recomputes its rows exactly, with no error."""
    w = W.make_paged("v-range", 32, 16, 8, 128, [300], [200])
    blk, row = _pool_index(w, 0, 5)
    w.v_pool[blk, 3, row, 7] = _bf16(70000.0)
    run_and_check(pkv, w)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("log2_scale", [17, -20])
def test_prefill_v_magnitudes(pkv, d, log2_scale):
    """Every V value multiplied by 2^17 (|v| up to ~5e5, beyond fp16) or by
    2^-20 (|v| ~1e-6, fp16 subnormals): scaling V by a power of two scales the
    exact result by the same power, so the output divided by it is held to
    the usual tolerance against the oracle's, with no error reported."""
    w = W.make_paged("v-scale", 90 + d + log2_scale, 16, 8, d, [700, 40, 300], [300, 1, 129])
    f = np.float32(2.0 ** log2_scale)

    def scaled(bits):  # exact for every finite bf16 value here; the NaN poison stays NaN
        return W._f32_to_bf16_bits((bits.astype(np.uint32) << 16).view(np.float32) * f)

    w.v_pool[:] = scaled(w.v_pool)
    w.v_new[:] = scaled(w.v_new)
    ds = DeviceStep(w)
    out = ds.run(pkv)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    _, _, ref = oracle.run_step(w, threads=16)
    assert_close(out.cpu().numpy() / float(f), ref / float(f), f"V x 2^{log2_scale}")
