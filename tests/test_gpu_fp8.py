"""GPU parity of the e4m3 (fp8) pools against the fp8 oracle: the write is
compared code for code, decode attention within the attention tolerance,
and the byte-moving calls byte for byte."""
import numpy as np
import pytest
import torch

from oracle import fp8
import pkv_workloads as W
from gpu_helpers import assert_close, dev_tensor

pytestmark = pytest.mark.gpu

K_SCALE = np.float32(0.0123)
V_SCALE = np.float32(0.0171)


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_291_gb300 as p
    p.load()
    return p


def inv(scale):
    return np.float32(1.0) / np.float32(scale)


def codes_of(pool_bits, scale):
    """Codes of a whole bf16 pool (the context already in the cache),
    quantised by the oracle; unused slots hold bf16 NaN and get NaN codes,
    which neither side reads."""
    return fp8.quantize_bf16_rows(pool_bits, inv(scale))


def run_fp8_step(pkv, w, ks=K_SCALE, vs=V_SCALE, partition_blocks=0, seqs=None):
    """Device: upload the cached context's codes, write this step's rows with
    the e4m3 cache write, decode.  Oracle: the same from the same codes."""
    if seqs is None:
        k8 = codes_of(w.k_pool, ks)
        v8 = codes_of(w.v_pool, vs)
    else:  # only the blocks the compared sequences read; the others hold zero codes
        used = np.unique(w.block_tables[np.asarray(seqs)])
        used = used[used >= 0]
        k8 = np.zeros(w.k_pool.shape, np.uint8)
        v8 = np.zeros(w.v_pool.shape, np.uint8)
        k8[used] = codes_of(w.k_pool[used], ks)
        v8[used] = codes_of(w.v_pool[used], vs)
    kd, vd = dev_tensor(k8), dev_tensor(v8)
    pkv.cache_write(kd, vd, dev_tensor(w.k_new), dev_tensor(w.v_new), dev_tensor(w.slot_mapping),
                    k_scale=float(ks), v_scale=float(vs))
    out = pkv.decode_attention(kd, vd, dev_tensor(w.q), dev_tensor(w.block_tables), dev_tensor(w.context_lens),
                               w.max_context_len, w.scale, partition_blocks=partition_blocks,
                               k_scale=float(ks), v_scale=float(vs))
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    fp8.cache_write(k8, v8, w.k_new, w.v_new, w.slot_mapping, inv(ks), inv(vs))
    assert np.array_equal(kd.cpu().numpy(), k8), "e4m3 K pool differs from the oracle's write"
    assert np.array_equal(vd.cpu().numpy(), v8), "e4m3 V pool differs from the oracle's write"
    sel = np.arange(w.num_seqs) if seqs is None else np.asarray(seqs)
    ref = fp8.decode_attention(k8, v8, w.q[sel], w.context_lens[sel], w.block_tables[sel], w.scale,
                               float(ks), float(vs))
    return assert_close(out.cpu().numpy()[sel], ref, f"{w.name} (e4m3)")


def test_write_rounds_ties_saturates_and_keeps_subnormals(pkv):
    """Scale 1: every code value, every midpoint between neighbours (exact
    ties, which go to the even code), values past 448, zeros of both signs
    and values below half the smallest subnormal."""
    vals = fp8.decode_codes()[:127]
    mids = (vals[:-1] + vals[1:]) / 2
    extra = np.array([0.0, -0.0, 448.0, 450.0, 464.0, 480.0, 2.0 ** 13, 2.0 ** 127, 2.0 ** -10, 2.0 ** -11,
                      2.0 ** -9 * 1.5, 2.0 ** -9 * 0.75, 2.0 ** -100])
    x = np.concatenate([vals, mids, extra])
    x = np.concatenate([x, -x])
    f32 = x.astype(np.float32)
    bits = (f32.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), f32)   # all exact in bf16
    hkv, d = 2, 64
    T = -(-bits.size // (hkv * d))
    rows = np.zeros(T * hkv * d, np.uint16)
    rows[:bits.size] = bits
    rows = rows.reshape(T, hkv, d)
    nb = -(-T // 16) + 1
    slots = np.random.default_rng(0).permutation(nb * 16)[:T].astype(np.int32)
    k8 = np.zeros((nb, hkv, 16, d), np.uint8)
    kd, vd = dev_tensor(k8), dev_tensor(k8)
    pkv.cache_write(kd, vd, dev_tensor(rows), dev_tensor(rows), dev_tensor(slots), k_scale=1.0, v_scale=1.0)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    ref = k8.copy()
    fp8.cache_write(ref, ref.copy(), rows, rows, slots, np.float32(1), np.float32(1))
    assert np.array_equal(kd.cpu().numpy(), ref)
    assert np.array_equal(vd.cpu().numpy(), ref)


def test_write_of_random_rows_with_a_scale(pkv):
    rng = np.random.default_rng(3)
    T, hkv, d = 300, 4, 128
    k = W.normal_bf16(11, 1, T * hkv * d).reshape(T, hkv, d)
    v = W.normal_bf16(11, 2, T * hkv * d).reshape(T, hkv, d)
    nb = 40
    slots = rng.permutation(nb * 16)[:T].astype(np.int32)
    slots[::17] = -1                                           # skipped rows
    k8 = rng.integers(0, 256, size=(nb, hkv, 16, d)).astype(np.uint8)
    v8 = rng.integers(0, 256, size=(nb, hkv, 16, d)).astype(np.uint8)
    kd, vd = dev_tensor(k8), dev_tensor(v8)
    pkv.cache_write(kd, vd, dev_tensor(k), dev_tensor(v), dev_tensor(slots), k_scale=float(K_SCALE),
                    v_scale=float(V_SCALE))
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    fp8.cache_write(k8, v8, k, v, slots, inv(K_SCALE), inv(V_SCALE))
    assert np.array_equal(kd.cpu().numpy(), k8) and np.array_equal(vd.cpu().numpy(), v8)


def test_nan_input_gives_a_nan_code(pkv):
    nan = np.full((1, 1, 64), 0x7FC0, np.uint16)
    kd = torch.zeros((1, 1, 16, 64), dtype=torch.uint8, device="cuda")
    vd = torch.zeros_like(kd)
    pkv.cache_write(kd, vd, dev_tensor(nan), dev_tensor(nan), dev_tensor(np.array([5], np.int32)),
                    k_scale=1.0, v_scale=1.0)
    torch.cuda.synchronize()
    row = kd.cpu().numpy()[0, 0, 5]
    assert np.all((row & 0x7F) == 0x7F)


@pytest.mark.parametrize("cfg", [1, 2])
def test_fp8_decode_configs(pkv, cfg):
    run_fp8_step(pkv, W.build_config(cfg))


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (16, 8, 128), (32, 8, 128), (32, 4, 128),
                                      (8, 8, 64), (16, 8, 64), (32, 8, 64), (64, 8, 64)])
def test_fp8_head_shapes(pkv, hq, hkv, d):
    w = W.make_paged(f"fp8 shapes {hq}/{hkv}/{d}", 17 + hq + d, hq, hkv, d, [1, 17, 100, 300, 33, 16], [1] * 6)
    run_fp8_step(pkv, w)


@pytest.mark.parametrize("pb", [1, 3, 7])
def test_fp8_split_kv_merge(pkv, pb):
    w = W.make_paged("fp8 split", 23, 16, 8, 128, [700, 5, 260, 1024], [1] * 4)
    run_fp8_step(pkv, w, partition_blocks=pb)


def test_fp8_small_and_large_scales(pkv):
    """Scales far from 1 (q is pre-multiplied by k_scale inside the kernel,
    the V scale is applied with 1/l at the end), with many subnormal codes
    under the large scales."""
    w = W.make_paged("fp8 scales", 29, 16, 8, 128, [333, 64, 1], [1] * 3)
    run_fp8_step(pkv, w, ks=np.float32(3.1e-4), vs=np.float32(2.7e-5))
    run_fp8_step(pkv, w, ks=np.float32(5.3), vs=np.float32(9.1))


@pytest.mark.slow
def test_fp8_long_context_sampled(pkv):
    """LLaMA-13B MHA shape at full size; sampled sequences, a 32,768-token
    one among them (split-KV and merge)."""
    w = W.build_config(3)
    rows = [0, 5, 33, 64]
    run_fp8_step(pkv, w, seqs=rows)


def test_fp8_equals_the_bf16_path_on_exact_values(pkv):
    """With power-of-two scales every dequantised element is exactly a bf16
    value; decode over the e4m3 pools must then agree with decode over bf16
    pools holding those values, up to how each path carries P into its P.V
    MMAs (a hi + lo pair: 2^-18 relative in bf16, 2^-22 in f16), that is
    within 2^-17 of the largest |v|, and the final division's rounding."""
    w = W.make_paged("fp8 vs bf16", 31, 32, 8, 128, [500, 77, 1, 260], [1] * 4)
    rng = np.random.default_rng(5)
    k8 = rng.integers(0, 256, size=w.k_pool.shape).astype(np.uint8)
    v8 = rng.integers(0, 256, size=w.v_pool.shape).astype(np.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x3A
    v8[(v8 & 0x7F) == 0x7F] = 0x45
    ks, vs = 2.0 ** -4, 2.0 ** -6

    def bf16_of(c, s):
        return ((fp8.value(c) * s).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    args = (dev_tensor(w.q), dev_tensor(w.block_tables), dev_tensor(w.context_lens), w.max_context_len, w.scale)
    a = pkv.decode_attention(dev_tensor(k8), dev_tensor(v8), *args, k_scale=ks, v_scale=vs)
    b = pkv.decode_attention(dev_tensor(bf16_of(k8, ks)), dev_tensor(bf16_of(v8, vs)), *args)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    a, b = a.cpu().numpy(), b.cpu().numpy()
    vmax = float(np.abs(fp8.value(v8)).max() * vs)
    assert np.allclose(a, b, rtol=2e-6, atol=2.0 ** -17 * vmax), float(np.abs(a - b).max())


def test_fp8_copy_blocks_and_swap_move_bytes(pkv):
    rng = np.random.default_rng(7)
    nb, hkv, d = 20, 8, 128
    k8 = rng.integers(0, 256, size=(nb, hkv, 16, d)).astype(np.uint8)
    v8 = rng.integers(0, 256, size=(nb, hkv, 16, d)).astype(np.uint8)
    kd, vd = dev_tensor(k8), dev_tensor(v8)
    src, dst = np.array([3, 3, 11, -1], np.int32), np.array([7, 8, 0, 19], np.int32)
    pkv.copy_blocks(kd, vd, dev_tensor(src), dev_tensor(dst))
    for s_, d_ in zip(src, dst):
        if s_ >= 0:
            k8[d_], v8[d_] = k8[s_], v8[s_]
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy(), k8) and np.array_equal(vd.cpu().numpy(), v8)
    host = torch.zeros((4, 2, hkv, 16, d), dtype=torch.uint8).pin_memory()
    blocks, slots = dev_tensor(np.array([5, 0, 13], np.int32)), dev_tensor(np.array([2, 0, 3], np.int32))
    pkv.swap_out(kd, vd, blocks, slots, host)
    torch.cuda.synchronize()
    h = host.numpy()
    for b_, s_ in [(5, 2), (0, 0), (13, 3)]:
        assert np.array_equal(h[s_, 0], k8[b_]) and np.array_equal(h[s_, 1], v8[b_])
    assert not h[1].any()
    kd.zero_()
    vd.zero_()
    pkv.swap_in(kd, vd, blocks, slots, host)
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    got_k = kd.cpu().numpy()
    assert np.array_equal(got_k[[5, 0, 13]], k8[[5, 0, 13]]) and not got_k[1].any()


def test_fp8_pools_rejected_where_not_supported(pkv):
    w = W.make_paged("fp8 reject", 37, 16, 8, 128, [40, 30], [20, 1])
    kd = torch.zeros(w.k_pool.shape, dtype=torch.uint8, device="cuda")
    vd = torch.zeros_like(kd)
    with pytest.raises(pkv.PKVError) as e:
        pkv.chunked_prefill_attention(kd, vd, dev_tensor(w.q), dev_tensor(w.query_start_loc),
                                      dev_tensor(w.context_lens), dev_tensor(w.block_tables), w.max_context_len,
                                      w.scale, query_start_loc_host=w.query_start_loc)
    assert e.value.status == 16
    for bad in (0.0, -1.0, float("inf"), float("nan"), 1e-45):
        with pytest.raises(pkv.PKVError) as e:
            pkv.cache_write(kd, vd, dev_tensor(w.k_new), dev_tensor(w.v_new), dev_tensor(w.slot_mapping),
                            k_scale=bad, v_scale=1.0)
        assert e.value.status == 16
    with pytest.raises(ValueError):
        pkv.decode_attention(kd, vd, dev_tensor(w.q[:2]), dev_tensor(w.block_tables), dev_tensor(w.context_lens),
                             w.max_context_len, w.scale)


def test_fp8_empty_context_and_output_bounds(pkv):
    """An empty context gives a zero row; decode writes only its own output
    rows (sentinel rows around them stay intact)."""
    w = W.make_paged("fp8 empty", 41, 16, 8, 128, [5, 40, 1], [1] * 3)
    ctx = w.context_lens.copy()
    ctx[1] = 0
    k8, v8 = codes_of(w.k_pool, K_SCALE), codes_of(w.v_pool, V_SCALE)
    fp8.cache_write(k8, v8, w.k_new, w.v_new, w.slot_mapping, inv(K_SCALE), inv(V_SCALE))  # this step's rows
    G = 8
    full = torch.full((3 + 2 * G, 16, 128), float("nan"), dtype=torch.float32, device="cuda")
    out = full[G:G + 3]
    pkv.decode_attention(dev_tensor(k8), dev_tensor(v8), dev_tensor(w.q), dev_tensor(w.block_tables), dev_tensor(ctx),
                         w.max_context_len, w.scale, out=out, k_scale=float(K_SCALE), v_scale=float(V_SCALE))
    torch.cuda.synchronize()
    assert pkv.get_error() == (0, 0)
    f = full.cpu().numpy()
    assert np.all(np.isnan(f[:G])) and np.all(np.isnan(f[G + 3:])), "decode wrote outside its rows"
    got = f[G:G + 3]
    assert not got[1].any(), "empty context must give a zero row"
    ref = fp8.decode_attention(k8, v8, w.q, ctx, w.block_tables, w.scale, float(K_SCALE), float(V_SCALE))
    assert_close(got, ref, "fp8 empty context")


def test_fp8_allocation_free_entry_point(pkv):
    """pkv_decode_attention_static takes the same e4m3 descriptor."""
    import ctypes
    lib = pkv.load()
    P, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    lib.pkv_decode_attention_static.argtypes = [ctypes.POINTER(pkv.Cache), P, i32, P, i32, P, i32, i32, f32, P, P]
    lib.pkv_decode_attention_static.restype = ctypes.c_int
    w = W.make_paged("fp8 static", 43, 32, 8, 128, [700, 33, 260, 1], [1] * 4)
    k8, v8 = codes_of(w.k_pool, K_SCALE), codes_of(w.v_pool, V_SCALE)
    fp8.cache_write(k8, v8, w.k_new, w.v_new, w.slot_mapping, inv(K_SCALE), inv(V_SCALE))  # this step's rows
    kd, vd = dev_tensor(k8), dev_tensor(v8)
    q, t, c = dev_tensor(w.q), dev_tensor(w.block_tables), dev_tensor(w.context_lens)
    cache = pkv._cache(kd, vd, float(K_SCALE), float(V_SCALE))
    out = torch.full((4, 32, 128), float("nan"), dtype=torch.float32, device="cuda")
    for _ in range(2):
        st = lib.pkv_decode_attention_static(ctypes.byref(cache), ctypes.c_void_p(q.data_ptr()), 32,
                                             ctypes.c_void_p(t.data_ptr()), int(t.shape[1]),
                                             ctypes.c_void_p(c.data_ptr()), 4, w.max_context_len,
                                             ctypes.c_float(w.scale), ctypes.c_void_p(out.data_ptr()), None)
        assert st == 0, pkv.status_string(st)
        torch.cuda.synchronize()
        assert pkv.get_error() == (0, 0)
        ref = fp8.decode_attention(k8, v8, w.q, w.context_lens, w.block_tables, w.scale, float(K_SCALE),
                                   float(V_SCALE))
        assert_close(out.cpu().numpy(), ref, "fp8 static entry point")
