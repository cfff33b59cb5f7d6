"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one.  Each mutant is a one-line edit of oracle.c (wrong step
index, wrong mantissa scale, ties away from zero, off-by-one exponent, wrong
clamp, wrong threshold tie, wrong header size, reversed tree levels, swapped
difference, wrong subnormal scaling in the fp16 conversion, error-feedback sign,
owner without error feedback, flush tie in the codec statistics, wrong chunk or an
owner that keeps its input in the compressed allgather, a root that keeps its input
in the compressed broadcast, a dropped base or average in the difference epilogue,
swapped or unsigned BFP4 nibbles, -0.0 taken for a zero, a chunk's sparse
message cut into 256-element pieces, sparse values restored at the wrong
index, a receiver that adds only nonzero message values, standalone decoders
that overwrite instead of adding or keep acc where they should clear it, a
shifted sparse index, a broadcast that ignores its root, a swapped standalone
difference, either chunk index of the plain allgather, chunks of floor(T/N)
elements, a tree that counts half its bytes); the mutated copy
is compiled into a temporary directory and the pin suite is run against it in
a child process.  The real oracle is never modified."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "rs_send_index": ("int c = mod((long)r - s, N);", "int c = mod((long)r - s + 1, N);", 1),
    "ag_recv_index": ("int c = mod((long)r - s, N);", "int c = mod((long)r - s + 1, N);", 2),
    "mantissa_scale": ("int q = bits - 2;", "int q = bits - 1;", 1),
    "ties_away": ("float r = nearbyintf(scaled);", "float r = roundf(scaled);", 1),
    "exponent_off_by_one": ("    frexpf(amax, &E);\n    return E - 1;", "    frexpf(amax, &E);\n    return E;", 1),
    "subnormal_exponent": ("        return -126;\n    int E;", "        return -127;\n    int E;", 1),
    "clamp_limit": ("return (1 << (bits - 1)) - 1;", "return (1 << (bits - 1));", 1),
    "threshold_tie": ("return (double)nnz < (1.0 - threshold)", "return (double)nnz <= (1.0 - threshold)", 1),
    "sparse_header_bytes": ("m->bytes += 8 + 8 * nnz;", "m->bytes += 4 + 8 * nnz;", 1),
    "tree_level_order": ("    for (int k = 0; k < L; k++) {\n        int step = 1 << k;",
                         "    for (int k = L - 1; k >= 0; k--) {\n        int step = 1 << k;", 1),
    "diff_sign": ("((const float *)in[r])[i] - diff_prev[r][i]", "diff_prev[r][i] - ((const float *)in[r])[i]", 1),
    "average_by_reciprocal": ("w = w / (float)N;", "w = w * (1.0f / (float)N);", 1),
    "f16_subnormal_scale": ("float q = nearbyintf(ldexpf(a, 24));", "float q = nearbyintf(ldexpf(a, 23));", 1),
    "ef_residual_sign": ("e[i] = u[i] - d;", "e[i] = d - u[i];", 1),
    "stats_flush_tie": ("if (fabsf(blk[i]) <= ldexpf(1.0f, e - 7))", "if (fabsf(blk[i]) < ldexpf(1.0f, e - 7))", 1),
    "ef_owner_skipped": ("            if (resid)\n                msg_encode_ef(&held[r]",
                         "            if (0)\n                msg_encode_ef(&held[r]", 1),
    "agc_recv_index": ("int c = mod((long)r - s, N);", "int c = mod((long)r - s + 1, N);", 4),
    "bcc_root_keeps_input": ("    for (int r = 0; r < N; r++)\n        for (size_t i = 0; i < T; i++)\n            store_from_f32(buf[r], i, t, msg_value(&m, &cd, i));",
                             "    for (int r = 0; r < N; r++)\n        for (size_t i = 0; i < T * (r != root); i++)\n            store_from_f32(buf[r], i, t, msg_value(&m, &cd, i));", 1),
    "base_dropped": ("                if (diff_base)\n                    w = diff_base[i] + w;",
                     "                if (0)\n                    w = diff_base[i] + w;", 1),
    "average_dropped": ("                if (average)\n                    w = w / (float)N;",
                        "                if (0)\n                    w = w / (float)N;", 1),
    "nibble_order": ("                if (i % 2 == 0)\n                    mants[i / 2] |= nib;",
                     "                if (i % 2 == 1)\n                    mants[i / 2] |= nib;", 1),
    "nibble_unsigned": ("return nib >= 8 ? nib - 16 : nib;", "return nib;", 1),
    "minus_zero_is_zero": ("    memcpy(&u, &v, 4);\n    return u != 0u;",
                           "    memcpy(&u, &v, 4);\n    return (u << 1) != 0u;", 1),
    "sparse_chunk_cut_in_slices": ("const size_t step = cd->slice ? cd->slice : (len ? len : 1);",
                                   "const size_t step = cd->slice ? cd->slice : 256;", 1),
    "sparse_restored_at_wrong_index": ("m->f[lo + (size_t)pi[k]] = pv[k];", "m->f[lo + k] = pv[k];", 1),
    "receiver_skips_zero_values": ("local[r][lo + i] = local[r][lo + i] + v; /* S4 */",
                                   "if (is_nonzero(v)) local[r][lo + i] = local[r][lo + i] + v; /* S4 */", 1),
    "bfp_decode_accumulate_overwrites": ("out[i] = accumulate ? out[i] + v : v;", "out[i] = v;", 1),
    "sparse_dense_accumulate_overwrites": ("acc[i] = accumulate ? acc[i] + v : v;", "acc[i] = v;", 1),
    "sparse_listed_accumulate_overwrites": ("acc[i] = accumulate ? acc[i] + v : v;", "acc[i] = v;", 2),
    "sparse_decode_keeps_acc": ("    if (!accumulate)\n        for (size_t i = 0; i < n; i++)\n            acc[i] = 0.0f;",
                                "    if (0)\n        for (size_t i = 0; i < n; i++)\n            acc[i] = 0.0f;", 1),
    "sparse_encode_index_shift": ("idx[k] = (int32_t)i;", "idx[k] = (int32_t)(i + 1);", 1),
    "broadcast_ignores_root": ("int src = (q + root) % N, dst = (qd + root) % N;", "int src = q, dst = qd;", 1),
    "diff_encode_swapped": ("diff[i] = cur[i] - prev[i];", "diff[i] = prev[i] - cur[i];", 1),
    "plain_ag_send_index": ("int c = mod((long)r - s + 1, N);", "int c = mod((long)r - s, N);", 1),
    "plain_ag_recv_index": ("int c = mod((long)r - s, N);", "int c = mod((long)r - s + 1, N);", 3),
    "chunk_len_floor": ("size_t n = (T + (size_t)N - 1) / (size_t)N; /* R3 */", "size_t n = T / (size_t)N; /* R3 */", 1),
    "tree_bytes_halved": ("            sent[src] += 4 * T;", "            sent[src] += 2 * T;", 1),
    "agc_owner_keeps_input": ("/* the owner's own chunk becomes the decoded codes as well */\n    for (int r = 0; r < N; r++) {",
                              "/* the owner's own chunk becomes the decoded codes as well */\n    for (int r = 0; r < 0; r++) {", 1),
}


def _mutate(src, old, new, occurrence):
    pos = -1
    for _ in range(occurrence):
        pos = src.index(old, pos + 1)
    return src[:pos] + new + src[pos + len(old):]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new, occ = MUTANTS[name]
    src = open(SRC).read()
    mutated = _mutate(src, old, new, occ)
    assert mutated != src
    c = tmp_path / "oracle_mutant.c"
    c.write_text(mutated)
    so = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", str(so), str(c), "-lm"], check=True)
    env = dict(os.environ, RRA_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
