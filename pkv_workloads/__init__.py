"""Seeded synthetic inputs for paged KV-cache attention.

This module plays the part of the serving engine's scheduler (which picks the
KV blocks a step uses) and of the model (which produces q, K and V); it does
no attention arithmetic.  The CUDA library, the CPU oracle, the tests and the
benchmark all take their inputs from here, so both sides see the same bytes.

Random numbers: a counter-based generator.  Element ``i`` of stream ``s`` under
seed ``seed`` is ``splitmix64(base(seed, s) + i)`` (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014); normals come
from the Box-Muller transform (Box and Muller, 1958) applied to the two 24-bit
halves of each 64-bit draw, and are rounded to bfloat16 with
round-to-nearest-even.  Everything is integer arithmetic except the
Box-Muller step, so the draws are identical on x86 and Arm up to the last bit
of libm's log/cos/sin.

Pool layout (the one the library uses): K and V pools are each
``[num_blocks][num_kv_heads][16][head_dim]`` bfloat16 (stored here as uint16
bit patterns).  A token at logical position ``p`` of a sequence lives in
physical block ``block_table[p // 16]`` at offset ``p % 16``; the unused tail
of each sequence's last block and every block nobody owns hold bfloat16 NaN
(0x7FC0), so any read of a slot outside the context shows up as a NaN.

The five workload shapes follow the pages on paged KV caches
("PagedAttention: splitting KV into blocks", section 2 of the serving-engine
KV blog: 16-token blocks, per-request block tables, a 22,048-token pool and
34 requests of 512+128 tokens; section 4 for the 3,000-token shared prefix
with 32-token suffixes; section 3 for 3 x 3,500-token prompts inserted beside
a 300-token decode under a 2,048-token budget).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

BLOCK_SIZE = 16
BF16_NAN = np.uint16(0x7FC0)
_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

# Stream ids: one per kind of array a workload draws.
STREAM_K_POOL, STREAM_V_POOL, STREAM_Q, STREAM_K_NEW, STREAM_V_NEW = 1, 2, 3, 4, 5
STREAM_PERM, STREAM_LENS, STREAM_MISC = 6, 7, 8


def splitmix64(x: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser applied elementwise to ``x + golden`` (uint64, wraps)."""
    with np.errstate(over="ignore"):
        z = x.astype(np.uint64, copy=False) + _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
        return z ^ (z >> np.uint64(31))


def _base(seed: int, stream: int) -> np.uint64:
    s = np.array([(int(seed) * 0x10001 + int(stream) * 0x632BE59BD9B4E019) & 0xFFFFFFFFFFFFFFFF],
                 dtype=np.uint64)
    return splitmix64(s)[0]


def uniform_u64(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """``count`` raw 64-bit draws of stream ``stream``, starting at counter ``offset``."""
    base = _base(seed, stream)
    with np.errstate(over="ignore"):
        idx = np.arange(offset, offset + count, dtype=np.uint64) + base
    return splitmix64(idx)


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit pattern, round to nearest even (inputs are finite)."""
    b = x.astype(np.float32, copy=False).view(np.uint32)
    rnd = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + rnd) >> np.uint32(16)).astype(np.uint16)


def _normal_chunk(seed: int, stream: int, offset: int, count: int) -> np.ndarray:
    """Normals ``offset .. offset+count`` (count even, offset even) as bf16 bits."""
    z = uniform_u64(seed, stream, count // 2, offset // 2)
    u1 = ((z >> np.uint64(40)).astype(np.float64) + 1.0) * (1.0 / 16777216.0)  # (0, 1]
    u2 = ((z >> np.uint64(16)) & np.uint64(0xFFFFFF)).astype(np.float64) * (1.0 / 16777216.0)
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    out = np.empty(count, dtype=np.float32)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return _f32_to_bf16_bits(out)


def normal_bf16(seed: int, stream: int, count: int, threads: Optional[int] = None) -> np.ndarray:
    """``count`` iid N(0,1) samples rounded to bf16, as uint16 bit patterns."""
    n2 = count + (count & 1)
    out = np.empty(n2, dtype=np.uint16)
    chunk = 1 << 22
    starts = list(range(0, n2, chunk))

    def work(s):
        e = min(n2, s + chunk)
        out[s:e] = _normal_chunk(seed, stream, s, e - s)

    nthr = threads or min(16, os.cpu_count() or 1)
    if len(starts) == 1 or nthr == 1:
        for s in starts:
            work(s)
    else:
        with ThreadPoolExecutor(nthr) as ex:
            list(ex.map(work, starts))
    return out[:count]


def randint_inclusive(seed: int, stream: int, count: int, lo: int, hi: int) -> np.ndarray:
    """``count`` integers uniform in [lo, hi] (modulo reduction of 64-bit draws)."""
    z = uniform_u64(seed, stream, count)
    return (lo + (z % np.uint64(hi - lo + 1)).astype(np.int64)).astype(np.int64)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """A seeded permutation of 0..n-1: sort the indices by 64-bit random keys."""
    keys = uniform_u64(seed, stream, n)
    return np.argsort(keys, kind="stable").astype(np.int32)


def blocks_for(n_tokens: int) -> int:
    """Blocks a sequence of ``n_tokens`` occupies: ceil(n / 16)."""
    return -(-int(n_tokens) // BLOCK_SIZE)


def chunk_slices(prompt_len: int, budget: int) -> List[tuple]:
    """Split a prompt into consecutive inclusive slices of at most ``budget``
    tokens: an 8K prompt under a 2K budget becomes 0-2047, 2048-4095,
    4096-6143, 6144-8191 (the chunked-prefill example of the inference-engine
    talk write-up, section "Chunked Prefill")."""
    return [(s, min(prompt_len, s + budget) - 1) for s in range(0, prompt_len, budget)]


@dataclass
class Workload:
    """One synthetic step.  Arrays are numpy; bf16 tensors are uint16 bit patterns.

    ``k_pool``/``v_pool`` hold the cache *before* the step (the new rows'
    slots still poisoned).  A step is: copy_blocks (if ``copy_src`` is given),
    then cache_write of ``k_new``/``v_new`` into ``slot_mapping``, then
    attention of ``q`` over ``context_lens`` tokens gathered via
    ``block_tables`` (decode when every query_len is 1, otherwise the mixed
    chunked-prefill batch described by ``query_start_loc``).
    """
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_blocks: int
    k_pool: np.ndarray
    v_pool: np.ndarray
    block_tables: np.ndarray          # int32 [S][max_blocks_per_seq], -1 padded
    context_lens: np.ndarray          # int32 [S], includes this step's rows
    query_start_loc: np.ndarray       # int32 [S+1]
    q: np.ndarray                     # uint16 [Tq][Hq][d]
    k_new: np.ndarray                 # uint16 [T][Hkv][d]
    v_new: np.ndarray
    slot_mapping: np.ndarray          # int32 [T]
    copy_src: Optional[np.ndarray] = None
    copy_dst: Optional[np.ndarray] = None
    seed: int = 0
    meta: Dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def query_lens(self) -> np.ndarray:
        return np.diff(self.query_start_loc).astype(np.int32)

    @property
    def is_decode(self) -> bool:
        return bool(np.all(self.query_lens == 1))


def default_seed(config: int) -> int:
    return 0x291 * 1000 + int(config)


def _pool_arrays(seed, num_blocks, hkv, d, threads=None):
    n = num_blocks * hkv * BLOCK_SIZE * d
    k = normal_bf16(seed, STREAM_K_POOL, n, threads).reshape(num_blocks, hkv, BLOCK_SIZE, d)
    v = normal_bf16(seed, STREAM_V_POOL, n, threads).reshape(num_blocks, hkv, BLOCK_SIZE, d)
    return k, v


def _poison_unused(k_pool, v_pool, valid_slots: np.ndarray):
    """Set every slot not listed in ``valid_slots`` (flat slot ids) to bf16 NaN."""
    nb = k_pool.shape[0]
    used = np.zeros(nb * BLOCK_SIZE, dtype=bool)
    used[valid_slots] = True
    used = used.reshape(nb, BLOCK_SIZE)
    kv = k_pool.transpose(0, 2, 1, 3)  # view [nb][16][hkv][d]
    vv = v_pool.transpose(0, 2, 1, 3)
    kv[~used] = BF16_NAN
    vv[~used] = BF16_NAN


def _slots_of(table_row: np.ndarray, positions: np.ndarray) -> np.ndarray:
    return table_row[positions // BLOCK_SIZE].astype(np.int64) * BLOCK_SIZE + positions % BLOCK_SIZE


def make_paged(name, seed, hq, hkv, d, context_lens, query_lens, num_blocks=None,
               slack=1.25, table_pad=0, threads=None, share_prefix_blocks=0, meta=None):
    """General builder: sequences with ``context_lens[s]`` tokens of which the
    last ``query_lens[s]`` are this step's new rows (written by cache_write,
    so their slots start poisoned).  Block ids come from a seeded permutation
    of the pool; ``share_prefix_blocks`` > 0 makes every sequence's first
    that many table entries point at the same physical blocks."""
    context_lens = np.asarray(context_lens, dtype=np.int64)
    query_lens = np.asarray(query_lens, dtype=np.int64)
    S = len(context_lens)
    nblk = np.array([blocks_for(n) for n in context_lens], dtype=np.int64)
    shared = int(share_prefix_blocks)
    need = shared + int(np.sum(nblk - shared)) if S else 0
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(slack * need)))
    if need > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {need}")
    perm = permutation(seed, STREAM_PERM, num_blocks)
    max_blocks = int(nblk.max()) + table_pad if S else 1
    tables = np.full((S, max(1, max_blocks)), -1, dtype=np.int32)
    cursor = shared
    for s in range(S):
        tables[s, :shared] = perm[:shared]
        k = int(nblk[s]) - shared
        tables[s, shared:shared + k] = perm[cursor:cursor + k]
        cursor += k
    k_pool, v_pool = _pool_arrays(seed, num_blocks, hkv, d, threads)
    cached, new_slots, rows = [], [], []
    for s in range(S):
        n, ql = int(context_lens[s]), int(query_lens[s])
        pos_old = np.arange(0, n - ql)
        pos_new = np.arange(n - ql, n)
        cached.append(_slots_of(tables[s], pos_old))
        new_slots.append(_slots_of(tables[s], pos_new))
    cached_slots = np.concatenate(cached) if cached else np.zeros(0, np.int64)
    _poison_unused(k_pool, v_pool, cached_slots)
    slot_mapping = (np.concatenate(new_slots) if new_slots else np.zeros(0, np.int64)).astype(np.int32)
    T = int(np.sum(query_lens))
    qsl = np.zeros(S + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(query_lens)
    q = normal_bf16(seed, STREAM_Q, T * hq * d, threads).reshape(T, hq, d)
    k_new = normal_bf16(seed, STREAM_K_NEW, T * hkv * d, threads).reshape(T, hkv, d)
    v_new = normal_bf16(seed, STREAM_V_NEW, T * hkv * d, threads).reshape(T, hkv, d)
    return Workload(name=name, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_blocks=num_blocks,
                    k_pool=k_pool, v_pool=v_pool, block_tables=tables,
                    context_lens=context_lens.astype(np.int32), query_start_loc=qsl, q=q,
                    k_new=k_new, v_new=v_new, slot_mapping=slot_mapping, seed=seed,
                    meta=dict(meta or {}))


# --------------------------------------------------------------------------
# The five workload shapes
# --------------------------------------------------------------------------

def llama1b_decode(seed=None, threads=None):
    """Llama-3.2-1B attention shape: 4 decode sequences, 32 q / 8 kv heads,
    head_dim 64, contexts {1, 17, 100, 512}, a 128-block pool."""
    seed = default_seed(1) if seed is None else seed
    ctx = [1, 17, 100, 512]
    return make_paged("llama3.2-1b decode, 4 seqs, ctx {1,17,100,512}", seed, 32, 8, 64, ctx,
                      [1] * 4, num_blocks=128, threads=threads)


def qwen17b_decode(seed=None, threads=None):
    """Qwen3-1.7B attention shape: 16 q / 8 kv heads, head_dim 128; a
    22,048-token pool (1,378 blocks) holding 34 sequences of 512 + 128 = 640
    tokens, each decoding its 640th token (cache_write of 34 rows)."""
    seed = default_seed(2) if seed is None else seed
    return make_paged("qwen3-1.7b decode, 34 seqs x 640 ctx", seed, 16, 8, 128, [640] * 34,
                      [1] * 34, num_blocks=22048 // BLOCK_SIZE, threads=threads)


def llama13b_mha_decode(seed=None, threads=None, long_len=32768, n_short=64, n_long=4):
    """LLaMA-13B MHA shape: 40 q = 40 kv heads, head_dim 128; 64 sequences
    with context uniform in [128, 2048] plus 4 at 32,768 tokens."""
    seed = default_seed(3) if seed is None else seed
    short = randint_inclusive(seed, STREAM_LENS, n_short, 128, 2048)
    ctx = list(short) + [long_len] * n_long
    return make_paged("llama-13b mha decode, 64 x U[128,2048] + 4 x 32768", seed, 40, 40, 128, ctx,
                      [1] * len(ctx), threads=threads)


def qwen17b_prefix_share(seed=None, threads=None, n_seqs=32, prefix=3000, suffix=32):
    """32 sequences sharing a 3,000-token prefix: 187 full blocks mapped to
    the same physical ids, then the partially filled block 188 (0-based 187)
    which every sequence copies on write before appending its own 32-token
    suffix.  The step is copy_blocks (32 copies of the shared partial block)
    + cache_write of 32 x 32 suffix rows + decode at context 3,032."""
    seed = default_seed(4) if seed is None else seed
    hq, hkv, d = 16, 8, 128
    full = prefix // BLOCK_SIZE                # 187 shared full blocks
    n = prefix + suffix                        # 3,032
    nblk = blocks_for(n)                       # 190 table entries per sequence
    private = nblk - full                      # 3: CoW copy + 2 fresh
    need = full + 1 + n_seqs * private
    num_blocks = int(math.ceil(1.25 * need))
    perm = permutation(seed, STREAM_PERM, num_blocks)
    shared_ids = perm[:full]
    orig_partial = int(perm[full])
    priv = perm[full + 1: full + 1 + n_seqs * private].reshape(n_seqs, private)
    tables = np.empty((n_seqs, nblk), dtype=np.int32)
    tables[:, :full] = shared_ids
    tables[:, full:] = priv
    k_pool, v_pool = _pool_arrays(seed, num_blocks, hkv, d, threads)
    # Before the step: shared full blocks + the first prefix%16 rows of the
    # original partial block hold data; everything else is poison.
    valid = [(shared_ids[:, None].astype(np.int64) * BLOCK_SIZE + np.arange(BLOCK_SIZE)).ravel(),
             orig_partial * BLOCK_SIZE + np.arange(prefix % BLOCK_SIZE)]
    _poison_unused(k_pool, v_pool, np.concatenate(valid))
    # Suffix rows land in each sequence's private blocks.
    pos = np.arange(prefix, n)
    slot_mapping = np.concatenate([_slots_of(tables[s], pos) for s in range(n_seqs)]).astype(np.int32)
    T = n_seqs * suffix
    q = normal_bf16(seed, STREAM_Q, n_seqs * hq * d, threads).reshape(n_seqs, hq, d)
    k_new = normal_bf16(seed, STREAM_K_NEW, T * hkv * d, threads).reshape(T, hkv, d)
    v_new = normal_bf16(seed, STREAM_V_NEW, T * hkv * d, threads).reshape(T, hkv, d)
    qsl = np.arange(n_seqs + 1, dtype=np.int32)
    return Workload(name="qwen3-1.7b prefix share, 32 seqs, 3000 shared + 32 suffix", num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=d, num_blocks=num_blocks, k_pool=k_pool, v_pool=v_pool,
                    block_tables=tables, context_lens=np.full(n_seqs, n, dtype=np.int32),
                    query_start_loc=qsl, q=q, k_new=k_new, v_new=v_new, slot_mapping=slot_mapping,
                    copy_src=np.full(n_seqs, orig_partial, dtype=np.int32),
                    copy_dst=priv[:, 0].astype(np.int32).copy(), seed=seed,
                    meta=dict(shared_blocks=full, orig_partial=orig_partial, suffix=suffix))


def qwen17b_chunked_mixed(seed=None, threads=None, n_prompts=3, chunk=512, offset=1024, n_decode=32):
    """Mixed chunked-prefill batch under a 2,048-token budget: 3 prompts of
    3,500 tokens each contribute the 512-token causal chunk at offset 1,024
    (context 1,536), beside 1 decode sequence at context 300 and 31 with
    context uniform in [300, 4096]."""
    seed = default_seed(5) if seed is None else seed
    dec = [300] + list(randint_inclusive(seed, STREAM_LENS, n_decode - 1, 300, 4096))
    ctx = [offset + chunk] * n_prompts + dec
    ql = [chunk] * n_prompts + [1] * n_decode
    return make_paged("qwen3-1.7b chunked-prefill mixed batch, 3 x 512 chunk + 32 decode", seed, 16, 8,
                      128, ctx, ql, threads=threads,
                      meta=dict(n_prompts=n_prompts, chunk=chunk, offset=offset, prompt_len=3500,
                                budget=2048))


CONFIGS = {1: llama1b_decode, 2: qwen17b_decode, 3: llama13b_mha_decode, 4: qwen17b_prefix_share,
           5: qwen17b_chunked_mixed}


def build_config(k: int, seed=None, threads=None) -> Workload:
    return CONFIGS[int(k)](seed=seed, threads=threads)

