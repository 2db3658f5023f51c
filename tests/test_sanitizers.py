"""AddressSanitizer, UndefinedBehaviorSanitizer and ThreadSanitizer builds (CPU, no GPU).

The oracle's C source and the library's host-side code (every translation unit
of libkbattn, with its device code compiled as usual) are rebuilt with
``-fsanitize=address`` and ``-fsanitize=undefined`` and linked into the two drivers under
``tests/sanitize/``. The oracle driver runs every oracle function on small
problems held in exactly sized heap blocks; the host driver runs the argument
validation of every entry point, the workspace sizing, the tensor-core path's
work lists over a grid of shapes, and the small host-only calls. Any invalid
access, overflow or undefined operation aborts the driver. Nothing here
launches a kernel (every attention call is rejected by validation first), so
a GPU is neither needed nor touched. A third build under ``-fsanitize=thread``
runs the host-only calls from eight threads at once (``thread_driver.cpp``): the
work lists' shared per-shape cache, validation, the status strings and the
per-thread last error. This is the substitute for the sanitizer runs of the GPU
code, which are not available here.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

import pytest

from roofline_benchmarking_gb300 import build as kb_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.join(ROOT, "tests", "sanitize")
SAN = ["-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer", "-g"]
ENV = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0:halt_on_error=1",
           UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")


def run(cmd, **kw):
    r = subprocess.run(cmd, capture_output=True, text=True, **kw)
    assert r.returncode == 0, f"{' '.join(cmd[:3])} ... failed ({r.returncode}):\n{r.stdout[-3000:]}\n{r.stderr[-6000:]}"
    return r


def cuda_lib_dir() -> str:
    nvcc = kb_build.nvcc()
    home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        if os.path.exists(os.path.join(home, sub, "libcudart_static.a")):
            return os.path.join(home, sub)
    pytest.skip("libcudart_static.a not found")


@pytest.fixture(scope="module")
def gcc():
    if shutil.which("gcc") is None or shutil.which("g++") is None:
        pytest.skip("gcc/g++ not available")


def test_oracle_under_address_and_undefined_sanitizers(gcc, tmp_path):
    exe = str(tmp_path / "oracle_asan")
    run(["gcc", *SAN, "-O1", "-std=c11", "-ffp-contract=off", os.path.join(HERE, "oracle_driver.c"),
         os.path.join(ROOT, "oracle", "attn_oracle.c"), "-lm", "-o", exe])
    r = run([exe], env=ENV, timeout=300)
    assert "all checks passed" in r.stdout


def test_library_host_code_under_address_and_undefined_sanitizers(gcc, tmp_path):
    cudalib = cuda_lib_dir()
    nvcc = kb_build.nvcc()
    xsan = [x for f in SAN for x in ("-Xcompiler", f)]

    def compile_one(src):
        obj = str(tmp_path / (os.path.splitext(src)[0] + ".o"))
        run([nvcc, *kb_build.ARCH, *kb_build.NVCC_FLAGS, *xsan, "-I", kb_build.INCLUDE, "-c",
             os.path.join(kb_build.CSRC, src), "-o", obj])
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(kb_build.SOURCES)) as ex:
        objs = list(ex.map(compile_one, kb_build.SOURCES))
    exe = str(tmp_path / "host_asan")
    run(["g++", *SAN, "-O1", "-std=c++17", "-I", kb_build.INCLUDE, os.path.join(HERE, "host_driver.cpp"), *objs,
         "-L", cudalib, "-lcudart_static", "-ldl", "-lpthread", "-lrt", "-o", exe])
    r = run([exe], env=ENV, timeout=600)
    assert "all checks passed" in r.stdout


def test_library_host_code_under_thread_sanitizer(gcc, tmp_path):
    cudalib = cuda_lib_dir()
    nvcc = kb_build.nvcc()
    tsan = ["-fsanitize=thread", "-fno-omit-frame-pointer", "-g"]
    xsan = [x for f in tsan for x in ("-Xcompiler", f)]

    def compile_one(src):
        obj = str(tmp_path / (os.path.splitext(src)[0] + ".o"))
        run([nvcc, *kb_build.ARCH, *kb_build.NVCC_FLAGS, *xsan, "-I", kb_build.INCLUDE, "-c",
             os.path.join(kb_build.CSRC, src), "-o", obj])
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(kb_build.SOURCES)) as ex:
        objs = list(ex.map(compile_one, kb_build.SOURCES))
    exe = str(tmp_path / "host_tsan")
    run(["g++", *tsan, "-O1", "-std=c++17", "-I", kb_build.INCLUDE, os.path.join(HERE, "thread_driver.cpp"), *objs,
         "-L", cudalib, "-lcudart_static", "-ldl", "-lpthread", "-lrt", "-o", exe])
    env = dict(os.environ, TSAN_OPTIONS="halt_on_error=1:second_deadlock_stack=1")
    r = run([exe], env=env, timeout=600)
    assert "all checks passed" in r.stdout
