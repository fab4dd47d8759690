"""The C-ABI library on the host: it loads, exports every symbol the header declares, and
its host-side argument validation rejects bad calls before launching anything (these
calls never reach the GPU, so they run without one)."""
import ctypes
import os
import re

import pytest

import speculative_decoding_03_gb300 as ds
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED = 0, 1, 2
FAKE = 0x10000000          # an aligned address that is never dereferenced by these calls


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "dspark.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    L = ds.lib()
    declared = _declared_symbols()
    assert len(declared) >= 8
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(n for n, _, _ in ds.SIGNATURES) == declared


def test_status_strings():
    L = ds.lib()
    for code, name in ds.STATUS.items():
        assert L.dspark_status_string(code).decode() == name
    assert L.dspark_status_string(99).decode() == "DSPARK_ERR_UNKNOWN"


def test_workspace_bytes():
    L = ds.lib()
    for w in workloads.WORKLOADS:
        n = L.dspark_workspace_bytes(w.B, w.gamma, w.V, w.r, w.H)
        assert n >= w.B * w.V * 4 and n % 256 == 0
    assert L.dspark_workspace_bytes(0, 4, 1000, 16, 64) == 0
    assert L.dspark_workspace_bytes(4, 4, 1001, 16, 64) == 0      # V % 8 != 0
    assert L.dspark_workspace_bytes(4, 4, 1000, 24, 64) == 0      # r % 16 != 0
    assert L.dspark_workspace_bytes(4, 33, 1000, 16, 64) == 0     # gamma > 32
    # the largest accepted batches: B * gamma beyond a 65535-CTA grid dimension is accepted
    # (the verification folds its rows into the grid), B * (gamma + 1) >= 2^21 is not
    assert L.dspark_workspace_bytes(4096, 16, 64, 16, 0) > 0
    assert L.dspark_workspace_bytes(65535, 31, 8, 16, 0) > 0
    assert L.dspark_workspace_bytes(65535, 32, 8, 16, 0) == 0


def _draft(L, U=FAKE, W1=FAKE, W2=FAKE, anchor=FAKE, B=4, gamma=4, V=1000, r=16, out=FAKE,
           ws=FAKE, ws_bytes=1 << 30):
    return L.dspark_draft(U, W1, W2, anchor, B, gamma, V, r, 0, out, out, out, out, ws, ws_bytes, None)


def test_draft_validation():
    L = ds.lib()
    assert _draft(L, U=None) == INVALID
    assert _draft(L, U=FAKE + 4) == INVALID              # logits not 16-byte aligned
    assert _draft(L, ws=FAKE + 16) == INVALID            # workspace not 256-byte aligned
    assert _draft(L, ws_bytes=100) == INVALID            # workspace too small
    assert _draft(L, B=0) == INVALID
    assert _draft(L, V=1004) == UNSUPPORTED
    assert _draft(L, r=300) == UNSUPPORTED
    assert _draft(L, gamma=40) == UNSUPPORTED
    assert _draft(L, B=70000) == UNSUPPORTED


def test_schedule_validation():
    L = ds.lib()
    call = lambda R=4, gamma=4, sps_len=21, a=FAKE, ws=FAKE: L.dspark_schedule(
        a, R, gamma, FAKE, sps_len, FAKE, FAKE, FAKE, ws, 1 << 20, None)
    assert call(sps_len=20) == INVALID                   # table shorter than R (gamma+1) + 1
    assert call(a=None) == INVALID
    assert call(R=1024, gamma=17) == UNSUPPORTED         # more than 16384 items
    assert call(ws=None) == INVALID


def test_verify_confidence_and_bias_validation():
    L = ds.lib()
    assert L.dspark_verify(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 4, 4, 1000,
                           16, 0, FAKE, FAKE, FAKE, FAKE, 1 << 30, None) == INVALID
    assert L.dspark_confidence(FAKE + 8, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(1.0), 4, 4, 64, 16,
                               1000, FAKE, FAKE, FAKE, 1 << 20, None) == INVALID
    assert L.dspark_confidence(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(1.0), 4, 4, 66, 16,
                               1000, FAKE, FAKE, FAKE, 1 << 20, None) == UNSUPPORTED
    assert L.dspark_markov_bias(FAKE, FAKE, FAKE, 0, 4, 1000, 16, FAKE, FAKE, 1 << 20, None) == INVALID
    assert L.dspark_markov_bias(FAKE, FAKE, FAKE, 1, 4, 1000, 16, FAKE, None, 1 << 20, None) == INVALID


def test_copy_target_rows_validation():
    L = ds.lib()
    # null source, misaligned destination, workspace without a status word, bad shapes
    assert L.dspark_copy_target_rows(None, FAKE, FAKE, 4, 4, 1000, FAKE, 256, None) == INVALID
    assert L.dspark_copy_target_rows(FAKE, FAKE + 4, FAKE, 4, 4, 1000, FAKE, 256, None) == INVALID
    assert L.dspark_copy_target_rows(FAKE, FAKE, FAKE, 4, 4, 1000, FAKE, 128, None) == INVALID
    assert L.dspark_copy_target_rows(FAKE, FAKE, FAKE, 0, 4, 1000, FAKE, 256, None) == INVALID
    assert L.dspark_copy_target_rows(FAKE, FAKE, FAKE, 4, 33, 1000, FAKE, 256, None) == UNSUPPORTED
    assert L.dspark_copy_target_rows(FAKE, FAKE, FAKE, 4, 4, 1004, FAKE, 256, None) == UNSUPPORTED


def _compile(compiler, std, source, extra=()):
    import shutil
    import subprocess
    import tempfile
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not found")
    with tempfile.TemporaryDirectory() as d:
        ext = ".c" if compiler == "gcc" else ".cpp"
        src = os.path.join(d, "use" + ext)
        with open(src, "w") as f:
            f.write(source)
        cmd = [compiler, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-c", src,
               "-o", os.path.join(d, "use.o"), "-I", os.path.join(ROOT, "include"), *extra]
        res = subprocess.run(cmd, capture_output=True, text=True)
        assert res.returncode == 0, res.stderr


def _use_every_entry_point(prefix=""):
    names = _declared_symbols()
    body = "\n".join(f"  (void *)&{n}," for n in names)
    return (prefix + '#include "dspark.h"\n'
            "void *dspark_entry_points[] = {\n" + body + "\n};\n")


def test_header_is_plain_c():
    """include/dspark.h compiles as C11 on its own (no CUDA headers needed) and declares
    every entry point the library exports."""
    _compile("gcc", "c11", _use_every_entry_point())


def test_header_is_valid_cpp_with_and_without_the_cuda_runtime():
    """From C++ (extern "C" guard), alone and after cuda_runtime.h, whose cudaStream_t the
    header's own typedef must match."""
    _compile("g++", "c++17", _use_every_entry_point())
    cuda_inc = "/usr/local/cuda/include"
    if os.path.exists(os.path.join(cuda_inc, "cuda_runtime.h")):
        _compile("g++", "c++17", _use_every_entry_point("#include <cuda_runtime.h>\n"),
                 ("-I", cuda_inc, "-Wno-unused-parameter"))


def test_readme_c_example_compiles():
    """The C example of one step in the user documentation compiles as C11 against the
    header."""
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```c\n(.*?)```", text, flags=re.S)
    assert blocks, "no C example in the user documentation"
    for block in blocks:
        _compile("gcc", "c11", block)
