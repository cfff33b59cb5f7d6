"""CPU-side checks of the boundary: the library builds for sm_103a, loads,
exports every entry point include/rra.h declares, rejects bad arguments on the
host before touching the device, and the oracle and the CUDA path share no
code (neither imports, includes or links the other)."""
import ctypes as C
import os
import re
import subprocess

import pytest

import ring_allreduce_compressed_gb300 as rra

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rra.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rra_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    rra.build()
    return rra.lib()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ["rra_ring_allreduce", "rra_reduce_scatter", "rra_allgather", "rra_broadcast",
                 "rra_tree_allreduce", "rra_bfp_encode", "rra_bfp_decode", "rra_sparse_encode",
                 "rra_sparse_decode", "rra_diff_encode", "rra_get_bytes", "rra_comm_create",
                 "rra_comm_destroy", "rra_comm_status", "rra_set_timeout"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    raw = C.CDLL(rra.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def declared_arity():
    """Parameter count of every function include/rra.h declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(rra_[a-z_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_declares_every_signature(lib):
    """The binding gives ctypes each entry point's full signature (a missing
    argtypes would pass 64-bit pointers and sizes as C int)."""
    arity = declared_arity()
    assert set(arity) == set(declared_functions())
    for name, n in arity.items():
        f = getattr(lib, name)
        assert f.argtypes is not None and len(f.argtypes) == n, name
        assert f.restype is (C.c_char_p if name == "rra_status_string" else C.c_int), name


def test_status_strings(lib):
    assert rra.status_string(rra.RRA_OK) == "RRA_OK"
    assert rra.status_string(rra.RRA_ERR_TIMEOUT) == "RRA_ERR_TIMEOUT"


def test_host_side_argument_checks(lib):
    """Invalid arguments are rejected before any CUDA call."""
    L = lib
    assert L.rra_bfp_encode(None, 10, 0, 8, None, None, None) == rra.RRA_ERR_INVALID
    assert L.rra_bfp_encode(C.c_void_p(16), 10, 0, 5, C.c_void_p(16), C.c_void_p(16),
                            None) == rra.RRA_ERR_INVALID
    assert L.rra_bfp_decode(None, None, 0, 8, None, 0, None) == rra.RRA_ERR_INVALID
    assert L.rra_sparse_encode(C.c_void_p(16), 10, 0, C.c_float(1.5), C.c_void_p(16),
                               C.c_void_p(16), C.c_void_p(16), None) == rra.RRA_ERR_INVALID
    assert L.rra_diff_encode(None, None, None, 4, None) == rra.RRA_ERR_INVALID
    h = C.c_void_p()
    assert L.rra_comm_create(0, 10, 0, C.byref(h)) == rra.RRA_ERR_INVALID
    assert L.rra_comm_create(65, 10, 0, C.byref(h)) == rra.RRA_ERR_INVALID
    assert L.rra_comm_create(4, 0, 0, C.byref(h)) == rra.RRA_ERR_INVALID
    assert L.rra_ring_allreduce(None, None, None, 10, 0, 0, None, None) == rra.RRA_ERR_INVALID
    assert L.rra_get_bytes(None, None, None) == rra.RRA_ERR_INVALID
    assert L.rra_comm_destroy(None) == rra.RRA_OK
    assert L.rra_comm_last_shape(None, None, None, None, None) == rra.RRA_ERR_INVALID
    assert L.rra_autotune(None, None, None, 10, 0, 0, None, None) == rra.RRA_ERR_INVALID
    assert L.rra_allreduce_auto(None, None, 10, 0, None, None) == rra.RRA_ERR_INVALID
    assert L.rra_set_crossover(None, 0) == rra.RRA_ERR_INVALID
    assert L.rra_get_crossover(None, None) == rra.RRA_ERR_INVALID
    assert L.rra_autotune_crossover(None, None, 10, 0, None, None) == rra.RRA_ERR_INVALID
    assert L.rra_codec_measure(None, None, 10, 0, None, None) == rra.RRA_ERR_INVALID
    assert L.rra_codec_advise(None, None, 10, 0, C.c_float(0.5), C.c_float(0.01), None, None,
                              None) == rra.RRA_ERR_INVALID
    assert L.rra_allgather_codec(None, None, 10, 0, None, None) == rra.RRA_ERR_INVALID
    bfp, keep = rra.Codec("bfp", bits=8)._marshal()
    assert L.rra_allgather_codec(None, None, 10, 0, C.byref(bfp), None) == rra.RRA_ERR_INVALID
    avg, keep2 = rra.Codec("bfp", bits=8, average=True)._marshal()
    assert L.rra_allgather_codec(None, None, 10, 0, C.byref(avg), None) == rra.RRA_ERR_INVALID
    assert L.rra_broadcast_codec(None, None, 10, 0, 0, None, None) == rra.RRA_ERR_INVALID
    assert L.rra_broadcast_codec(None, None, 10, 0, 0, C.byref(bfp), None) == rra.RRA_ERR_INVALID
    assert L.rra_broadcast_codec(None, None, 10, 0, 0, C.byref(avg), None) == rra.RRA_ERR_INVALID
    sp, keep3 = rra.Codec("sparse", sparsity_threshold=0.5)._marshal()
    assert L.rra_broadcast_codec(None, None, 10, 0, 0, C.byref(sp), None) == rra.RRA_ERR_UNSUPPORTED
    assert L.rra_codec_measure_op(None, 1, 0, None, 10, 0, None, None) == rra.RRA_ERR_INVALID
    assert L.rra_codec_advise_op(None, 2, 0, None, 10, 0, C.c_float(0.5), C.c_float(0.01), 1,
                                 None, None, None) == rra.RRA_ERR_INVALID


def test_header_constants_match_the_binding():
    text = open(HEADER).read()
    consts = dict(re.findall(r"#define (RRA_[A-Z_]+) \(?([0-9a-fx]+)", text))
    assert int(consts["RRA_ALGO_RING"]) == rra.RRA_ALGO_RING
    assert int(consts["RRA_ALGO_TREE"]) == rra.RRA_ALGO_TREE
    for name in ("RRA_OP_ALLREDUCE", "RRA_OP_ALLGATHER", "RRA_OP_BROADCAST"):
        assert int(consts[name]) == getattr(rra, name)
    m = re.search(r"#define RRA_DEFAULT_CROSSOVER \((\d+)ull << (\d+)\)", text)
    assert int(m.group(1)) << int(m.group(2)) == rra.RRA_DEFAULT_CROSSOVER
    m = re.search(r"#define RRA_DEFAULT_CROSSOVER_WIDE \(\(1ull << (\d+)\) \+ 1\)", text)
    assert (1 << int(m.group(1))) + 1 == rra.RRA_DEFAULT_CROSSOVER_WIDE
    assert int(consts["RRA_RING_SLICE"]) == rra.RING_SLICE
    assert int(consts["RRA_BFP_BLOCK"]) == rra.BFP_BLOCK
    assert int(consts["RRA_SPARSE_PER_CHUNK"]) == rra.SPARSE_PER_CHUNK
    assert int(consts["RRA_SPARSE_PER_SLICE"]) == rra.SPARSE_PER_SLICE


def test_codec_struct_layout_matches_the_binding(tmp_path):
    """Every field of rra_codec sits at the offset the ctypes binding uses."""
    fields = [f for f, _ in rra._Codec._fields_]
    prog = tmp_path / "layout.c"
    prog.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "rra.h"\nint main(void){\n' +
                    f'printf("%zu\\n", sizeof(rra_codec));\n' +
                    "".join(f'printf("%zu\\n", offsetof(rra_codec, {f}));\n' for f in fields) +
                    "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), "-o", str(exe), str(prog)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert got[0] == C.sizeof(rra._Codec)
    assert got[1:] == [getattr(rra._Codec, f).offset for f in fields]


def _sources(folder, exts):
    out = []
    for dp, _, fs in os.walk(os.path.join(ROOT, folder)):
        if "_build" in dp or "__pycache__" in dp:
            continue
        out += [os.path.join(dp, f) for f in fs if f.endswith(exts)]
    return out


def test_oracle_and_cuda_path_share_no_code():
    for f in _sources("oracle", (".c", ".h", ".py")):
        text = open(f).read()
        assert "ring_allreduce_compressed_gb300" not in text.replace(
            "GPU library (``ring_allreduce_compressed_gb300``)", ""), f
        assert "rra.h" not in text and "rra_device" not in text, f
    for f in _sources("ring_allreduce_compressed_gb300", (".cu", ".cuh", ".h", ".py")):
        text = open(f).read()
        assert "import oracle" not in text and "oracle.h" not in text and \
            "liboracle" not in text, f
    wl = open(os.path.join(ROOT, "workloads", "__init__.py")).read()
    assert "import oracle" not in wl and "ring_allreduce_compressed_gb300" not in wl


def test_product_path_never_calls_the_oracle():
    """Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
    reference legs may touch oracle/."""
    bench = open(os.path.join(ROOT, "bench.py")).read()
    uses = [m.start() for m in re.finditer(r"import oracle", bench)]
    for pos in uses:
        fn = bench.rfind("\ndef ", 0, pos)
        name = bench[fn + 5:bench.index("(", fn)]
        assert name in ("oracle_sample_ring", "run_reference"), name


def test_header_is_plain_c(tmp_path):
    """include/rra.h is a C ABI: it compiles as strict C99 and as C++, and a C
    translation unit can name every entry point it declares."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    src = tmp_path / "use_rra.c"
    refs = "\n".join(f"    (void)&{n};" for n in declared_functions())
    src.write_text('#include "rra.h"\nvoid use_all(void)\n{\n' + refs + "\n}\n")
    for lang in (["-x", "c", "-std=c99", "-pedantic-errors"], ["-x", "c++", "-std=c++17"]):
        r = subprocess.run([gcc, *lang, "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                            "-I", cuda_inc, "-c", str(src), "-o", str(tmp_path / "u.o")],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
