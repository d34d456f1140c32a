"""Planted mistakes in the oracle must fail its pins (no GPU).

Each case plants one plausible mistake in a scratch copy of the oracle
package: a dropped term, a wrong index, sign or stride, a transposed operand,
an off-by-one, a wrong rounding rule.  The pin tests of that part of the
oracle then run against the copy in a child process, and at least one pin has
to fail.  The committed oracle is never modified: the copies live in pytest's
temporary folder, and the child finds them first on its module path.  An
unmodified copy passes every pin (the control case), so a pin run that fails
for another reason cannot pass for a caught mistake.

Every mutation names text that must occur exactly once in its file, so an
edit of the oracle that moves it makes the case fail loudly instead of
testing nothing.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")

PINS = {
    "pkv_oracle.c": ["test_oracle_pins.py"],
    "fp8.py": ["test_oracle_fp8.py"],
    "prefix_keys.py": ["test_oracle_prefix_keys.py"],
    "block_manager.py": ["test_oracle_block_manager.py"],
    "__init__.py": ["test_oracle_swap.py"],
}

# (name, file, text, replacement)
MUTANTS = [
    # paged attention (C): the definition softmax(scale q K^T) V read through the block table
    ("scale_dropped", "pkv_oracle.c", "x[j] = J->scale * dot;", "x[j] = dot;"),
    ("max_not_subtracted", "pkv_oracle.c", "x[j] = exp(x[j] - m);", "x[j] = exp(x[j]);"),
    ("min_taken_for_max", "pkv_oracle.c", "if (x[j] > m) m = x[j];", "if (x[j] < m) m = x[j];"),
    ("not_normalised", "pkv_oracle.c", "orow[c] = acc[c] / L;", "orow[c] = acc[c];"),
    ("sum_skips_first_key", "pkv_oracle.c", "L += x[j];", "if (j > 0) L += x[j];"),
    ("no_causal_mask", "pkv_oracle.c", "const int64_t pos = n - qlen + i;", "const int64_t pos = n - 1;"),
    ("position_off_by_one", "pkv_oracle.c", "const int64_t pos = n - qlen + i;",
     "const int64_t pos = n - qlen + i - 1;"),
    ("gqa_groups_interleaved", "pkv_oracle.c", "for (int32_t h = g * group; h < (g + 1) * group; ++h) {",
     "for (int32_t h = g; h < J->hq; h += J->hkv) {"),
    ("q_row_of_the_kv_head", "pkv_oracle.c", "J->q + ((row0 + i) * J->hq + h) * J->d;",
     "J->q + ((row0 + i) * J->hq + g) * J->d;"),
    ("v_in_the_scores", "pkv_oracle.c", "dot += qd[c] * Kc[j * J->d + c];", "dot += qd[c] * Vc[j * J->d + c];"),
    ("pool_rows_and_heads_swapped", "pkv_oracle.c", "((int64_t)h * J->bs + off) * J->d;",
     "((int64_t)off * J->hkv + h) * J->d;"),
    ("table_row_of_sequence_0", "pkv_oracle.c", "J->tables[(int64_t)s * J->max_blocks + logical];",
     "J->tables[logical];"),
    ("bf16_widened_with_half_an_ulp", "pkv_oracle.c", "uint32_t u = ((uint32_t)b) << 16;",
     "uint32_t u = (((uint32_t)b) << 16) | 0x8000u;"),
    ("write_row_from_the_block_index", "pkv_oracle.c", "int64_t off = slot % block_size;",
     "int64_t off = (slot / block_size) % block_size;"),
    ("write_rows_read_head_major", "pkv_oracle.c", "int64_t src = (t * num_kv_heads + h) * row;",
     "int64_t src = (h * num_tokens + t) * row;"),
    ("write_v_from_k", "pkv_oracle.c", "memcpy(v_pool + dst, v_new + src,", "memcpy(v_pool + dst, k_new + src,"),
    ("copy_moves_k_only", "pkv_oracle.c",
     "memmove(v_pool + (int64_t)dst[i] * block_elems, v_pool + (int64_t)src[i] * block_elems,",
     "memmove(v_pool + (int64_t)dst[i] * block_elems, v_pool + (int64_t)dst[i] * block_elems,"),
    ("exp2_for_exp", "pkv_oracle.c", "x[j] = exp(x[j] - m);", "x[j] = exp2(x[j] - m);"),
    ("last_dim_dropped", "pkv_oracle.c", "for (int32_t c = 0; c < J->d; ++c) dot += qd[c] * Kc[j * J->d + c];",
     "for (int32_t c = 0; c < J->d - 1; ++c) dot += qd[c] * Kc[j * J->d + c];"),
    ("write_skips_the_first_token", "pkv_oracle.c", "for (int64_t t = 0; t < num_tokens; ++t) {",
     "for (int64_t t = 1; t < num_tokens; ++t) {"),
    ("copy_direction_reversed", "pkv_oracle.c",
     "memmove(k_pool + (int64_t)dst[i] * block_elems, k_pool + (int64_t)src[i] * block_elems,",
     "memmove(k_pool + (int64_t)src[i] * block_elems, k_pool + (int64_t)dst[i] * block_elems,"),
    # e4m3 format, rounding and the dequantised decode
    ("e4m3_exponent_bias_8", "fp8.py", "2.0 ** (e - 7)", "2.0 ** (e - 8)"),
    ("e4m3_subnormal_scale", "fp8.py", "(m / 8.0) * 2.0 ** -6", "(m / 8.0) * 2.0 ** -7"),
    ("e4m3_ties_to_odd", "fp8.py", "(_FINITE[i] % 2 == 0)", "(_FINITE[i] % 2 == 1)"),
    ("e4m3_sign_dropped", "fp8.py", "code = code | np.where(np.signbit(x), 0x80, 0)", "code = code | 0"),
    ("e4m3_nan_code", "fp8.py", "code = np.where(np.isnan(x), 0x7F |", "code = np.where(np.isnan(x), 0x7E |"),
    ("e4m3_product_in_fp64", "fp8.py", "prod = (f * np.float32(inv_scale)).astype(np.float32)",
     "prod = f.astype(np.float64) * inv_scale"),
    ("e4m3_v_dequantised_with_k_scale", "fp8.py", "V = value(v_pool[blocks, :, pos % 16, :]) * v_scale",
     "V = value(v_pool[blocks, :, pos % 16, :]) * k_scale"),
    ("e4m3_gqa_interleaved", "fp8.py", "x = scale * (K[:, h // G, :] @ q[s, h])",
     "x = scale * (K[:, h % hkv, :] @ q[s, h])"),
    ("e4m3_negative_nan_decoded_as_a_number", "fp8.py", "if e == 0xF and m == 0x7:", "if c == 0x7F:"),
    ("e4m3_k_scale_not_applied", "fp8.py", "K = value(k_pool[blocks, :, pos % 16, :]) * k_scale",
     "K = value(k_pool[blocks, :, pos % 16, :])"),
    # prefix-cache keys
    ("key_not_chained", "prefix_keys.py",
     "parent = block_key(parent, tokens[i * BLOCK_SIZE:(i + 1) * BLOCK_SIZE], extra)",
     "parent = block_key(ROOT, tokens[i * BLOCK_SIZE:(i + 1) * BLOCK_SIZE], extra)"),
    ("key_extra_as_int32", "prefix_keys.py", 'np.asarray([extra], dtype="<i8")', 'np.asarray([extra], dtype="<i4")'),
    ("key_tokens_big_endian", "prefix_keys.py", 't = np.asarray(tokens, dtype="<i4")',
     't = np.asarray(tokens, dtype=">i4")'),
    ("key_parent_after_tokens", "prefix_keys.py", "msg = bytes(parent) + t.tobytes() +",
     "msg = t.tobytes() + bytes(parent) +"),
    # block bookkeeping
    ("cow_of_unshared_blocks", "block_manager.py", "if w.ref_counts[b] > 1:", "if w.ref_counts[b] >= 1:"),
    ("cow_keeps_the_old_count", "block_manager.py", "                w.ref_counts[b] -= 1\n",
     "                w.ref_counts[b] -= 0\n"),
    ("free_queue_lifo", "block_manager.py", "b = self.queue.pop(0)", "b = self.queue.pop()"),
    ("release_first_block_first", "block_manager.py", "for li in reversed(range(nb)):", "for li in range(nb):"),
    ("fork_takes_no_reference", "block_manager.py", "            st.tables[c, li] = b\n            st.ref_counts[b] += 1",
     "            st.tables[c, li] = b\n            st.ref_counts[b] += 0"),
    ("match_leaves_the_block_queued", "block_manager.py", "st.queue.remove(b)", "pass"),
    ("register_overwrites_a_cached_key", "block_manager.py", "if b in st.block_key or k in st.cache:",
     "if b in st.block_key:"),
    ("slot_row_off_by_one", "block_manager.py", "* BLOCK_SIZE + pos % BLOCK_SIZE", "* BLOCK_SIZE + (pos + 1) % BLOCK_SIZE"),
    ("allocation_one_block_ahead", "block_manager.py", "for li in range(blocks_for(n0), blocks_for(n1)):",
     "for li in range(blocks_for(n0), blocks_for(n1 + 1)):"),
    ("release_queues_at_the_head", "block_manager.py", "self.queue.append(b)", "self.queue.insert(0, b)"),
    ("match_skips_a_missing_key", "block_manager.py", "            if b is None:\n                break",
     "            if b is None:\n                continue"),
    ("blocks_for_rounds_down", "block_manager.py", "return -(-int(n_tokens) // BLOCK_SIZE)",
     "return int(n_tokens) // BLOCK_SIZE"),
    # block swap
    ("swap_out_v_from_k", "__init__.py", "host[h, 1] = v_pool[b]", "host[h, 1] = k_pool[b]"),
    ("swap_in_k_from_v", "__init__.py", "k_pool[b] = host[h, 0]", "k_pool[b] = host[h, 1]"),
]


def _copy_oracle(dst_parent):
    dst = os.path.join(dst_parent, "oracle")
    shutil.copytree(os.path.join(ROOT, "oracle"), dst,
                    ignore=shutil.ignore_patterns("__pycache__", "liboracle.so*"))
    return dst


def _run_pins(workdir, pin_files):
    """Run pin files against the oracle copy under workdir; return (rc, tail of output)."""
    env = dict(os.environ)
    # The copy first, then the repository (for the workload generators); the
    # repository is on the path already, so the test configuration does not
    # put it in front of the copy.
    env["PYTHONPATH"] = os.pathsep.join([workdir, ROOT] + ([env["PYTHONPATH"]] if env.get("PYTHONPATH") else []))
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu",
           "--rootdir", ROOT, "-c", os.path.join(ROOT, "pytest.ini")] + [os.path.join(TESTS, f) for f in pin_files]
    r = subprocess.run(cmd, cwd=workdir, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, (r.stdout + r.stderr)[-3000:]


def _case(tmp_root, name, fname, text, repl):
    workdir = os.path.join(tmp_root, name)
    os.makedirs(workdir)
    pkg = _copy_oracle(workdir)
    if fname is not None:
        path = os.path.join(pkg, fname)
        with open(path) as f:
            src = f.read()
        if src.count(text) != 1:
            return "anchor", f"{fname}: the mutated text occurs {src.count(text)} times"
        with open(path, "w") as f:
            f.write(src.replace(text, repl))
        pins = PINS[fname]
    else:
        pins = sorted({p for v in PINS.values() for p in v})
    return _run_pins(workdir, pins)


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    tmp_root = str(tmp_path_factory.mktemp("oracle_mutants"))
    cases = [("control", None, None, None)] + MUTANTS
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        futs = {c[0]: ex.submit(_case, tmp_root, *c) for c in cases}
        return {k: f.result() for k, f in futs.items()}


def test_mutant_names_are_distinct():
    assert len({m[0] for m in MUTANTS}) == len(MUTANTS)


def test_unmodified_copy_passes_every_pin(results):
    rc, out = results["control"]
    assert rc == 0, out


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(results, name):
    rc, out = results[name]
    assert rc != "anchor", out
    # pytest exits with 1 when a test failed; any other code is a broken run
    assert rc == 1, f"{name}: pins exited {rc}\n{out}"
