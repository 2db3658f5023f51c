"""The C-ABI boundary without a GPU: the library builds, loads, exports every
entry point include/kbattn.h declares, and rejects invalid requests before any
CUDA call (so these run on a CPU-only host)."""
import ctypes
import os
import re
import subprocess

import pytest

from roofline_benchmarking_gb300 import build as kb_build
from roofline_benchmarking_gb300 import kbattn
from roofline_benchmarking_gb300.kbattn import DType, Status, Variant

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kbattn.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kb_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    kb_build.build()
    return kbattn.load()


def test_header_declares_the_documented_calls():
    names = header_functions()
    for want in ("kb_attn_fwd", "kb_attn_fwd_ws", "kb_attn_workspace_bytes", "kb_attn_bench", "kb_triad",
                 "kb_triad_bench", "kb_device_info", "kb_status_string", "kb_last_cuda_error"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", kbattn.LIBRARY], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\S+)$", out, flags=re.M))
    missing = [n for n in header_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    # and the binding covers exactly the declared set
    assert sorted(kbattn.SIGNATURES) == header_functions()
    # only the ABI is exported (hidden visibility for everything else)
    extra = sorted(n for n in exported if n.startswith("kb") and n not in header_functions())
    assert not extra, extra


def test_build_targets_sm103a_only():
    """Every translation unit and the link get exactly one target: sm_103a
    machine code, no PTX and no other architecture."""
    assert kb_build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert not any("arch" in f or "code=" in f for f in kb_build.NVCC_FLAGS)


@pytest.mark.gpu
def test_runtime_reports_sm103_code(lib):
    """The CUDA runtime's view of the loaded kernels: binaryVersion 103."""
    assert kbattn.binary_version() == 103


def test_binary_version_rejects_a_null_pointer(lib):
    assert lib.kb_binary_version(None) == Status.INVALID_ARG


FAKE = 1 << 20  # an aligned, never-dereferenced address


def attn(q=FAKE, k=FAKE, v=FAKE, o=FAKE, B=1, H=1, S=64, d=64, causal=0, scale=0.125, dtype=DType.F32,
         variant=Variant.FLASH):
    return kbattn.kb_attn_fwd_ptr(q, k, v, o, B, H, S, d, causal, scale, dtype, variant, None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), Status.INVALID_ARG),
    (dict(o=0), Status.INVALID_ARG),
    (dict(v=FAKE + 4), Status.INVALID_ARG),          # not 16-byte aligned
    (dict(B=0), Status.INVALID_ARG),
    (dict(H=-1), Status.INVALID_ARG),
    (dict(S=0), Status.INVALID_ARG),
    (dict(d=0), Status.INVALID_ARG),
    (dict(causal=2), Status.INVALID_ARG),
    (dict(scale=0.0), Status.INVALID_ARG),
    (dict(scale=-1.0), Status.INVALID_ARG),
    (dict(scale=float("nan")), Status.INVALID_ARG),
    (dict(scale=float("inf")), Status.INVALID_ARG),
    (dict(dtype=7), Status.INVALID_ARG),
    (dict(variant=9), Status.INVALID_ARG),
    (dict(B=1 << 20, H=1 << 20, S=1 << 20, d=64), Status.INVALID_ARG),   # B*H overflows int32
    (dict(B=1 << 15, H=1 << 15, S=1 << 30, d=128), Status.INVALID_ARG),  # bytes overflow int64
    (dict(B=2, H=1, S=(1 << 31) - 1, d=32, variant=Variant.NAIVE), Status.UNSUPPORTED),  # score grid
    (dict(d=48), Status.UNSUPPORTED),
    (dict(d=256), Status.UNSUPPORTED),                                  # fp32 at d = 256: tensor cores only
    (dict(d=512, dtype=DType.BF16, variant=Variant.TC), Status.UNSUPPORTED),
    (dict(B=1 << 15, H=1 << 15, S=1 << 11, d=32, dtype=DType.BF16, variant=Variant.TC),
     Status.UNSUPPORTED),  # 2^30 heads x 8 pairs: work items overflow int32
    (dict(dtype=DType.F32, variant=Variant.TC), Status.UNSUPPORTED),
    (dict(dtype=DType.BF16, variant=Variant.FLASH), Status.UNSUPPORTED),
    (dict(dtype=DType.F16, variant=Variant.NAIVE), Status.UNSUPPORTED),
])
def test_invalid_requests_are_rejected_before_any_launch(lib, kw, want):
    assert attn(**kw) == want


def test_valid_request_without_a_device_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for variant, dtype in ((Variant.FLASH, DType.F32), (Variant.FUSED, DType.F32), (Variant.TC, DType.BF16),
                           (Variant.AUTO, DType.F16)):
        assert attn(variant=variant, dtype=dtype) == Status.NO_DEVICE
    st = kbattn.load().kb_triad(FAKE, FAKE, FAKE, 1.0, 1024, 256, None)
    assert st == Status.NO_DEVICE
    info = kbattn.DeviceInfo()
    assert kbattn.load().kb_device_info(0, ctypes.byref(info)) == Status.NO_DEVICE


def test_naive_workspace_contract(lib):
    assert kbattn.kb_attn_workspace_bytes(1, 8, 1024, 64, DType.F32, Variant.NAIVE) == 8 * 1024 * 1024 * 4
    assert kbattn.kb_attn_workspace_bytes(2, 3, 5, 32, DType.F32, Variant.NAIVE) == 6 * 25 * 4
    assert kbattn.kb_attn_workspace_bytes(1, 8, 1024, 64, DType.F32, Variant.FUSED) == 0
    # KB_AUTO picks the flash kernel for fp32 inputs, and so its workspace
    assert (kbattn.kb_attn_workspace_bytes(1, 8, 1024, 64, DType.F32, Variant.AUTO) ==
            kbattn.kb_attn_workspace_bytes(1, 8, 1024, 64, DType.F32, Variant.FLASH))
    # fp32 flash: the partial states (m, l and 64 x d O values of 64 rows) of the
    # two halves of its split causal query tiles, the heavier T - ceil(T / 2) of
    # the T = ceil(S / 64) tiles of each head
    for B, H, S, d in ((1, 8, 1024, 64), (2, 3, 300, 128), (1, 1, 64, 32)):
        T = -(-S // 64)
        want = B * H * (T - (T + 1) // 2) * 2 * 64 * (d + 2) * 4
        assert kbattn.kb_attn_workspace_bytes(B, H, S, d, DType.F32, Variant.FLASH) == want
    assert kbattn.kb_attn_workspace_bytes(1, 8, 1024, 64, DType.BF16, Variant.TC) == 0
    assert kbattn.kb_attn_workspace_bytes(0, 8, 1024, 64, DType.F32, Variant.NAIVE) == 0
    # a score matrix too large to address is refused, never a wrapped-around size
    assert kbattn.kb_attn_workspace_bytes(2, 1, (1 << 31) - 1, 32, DType.F32, Variant.NAIVE) == 0
    # too small a workspace is refused before the device is touched
    st = kbattn.load().kb_attn_fwd_ws(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, 0.125, DType.F32, Variant.NAIVE,
                                      None, FAKE, 64 * 64 * 4 - 1)
    assert st == Status.NO_MEMORY
    st = kbattn.load().kb_attn_fwd_ws(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, 0.125, DType.F32, Variant.NAIVE,
                                      None, None, 0)
    assert st == Status.NO_MEMORY


def test_triad_and_bench_argument_checks(lib):
    L = kbattn.load()
    assert L.kb_triad(FAKE, FAKE, FAKE, 1.0, 0, 256, None) == Status.OK      # n = 0 is a no-op
    assert L.kb_triad(0, FAKE, FAKE, 1.0, 16, 256, None) == Status.INVALID_ARG
    assert L.kb_triad(FAKE + 8, FAKE, FAKE, 1.0, 16, 256, None) == Status.INVALID_ARG
    assert L.kb_triad(FAKE, FAKE, FAKE, 1.0, 16, 384, None) == Status.INVALID_ARG
    ms = (ctypes.c_float * 1)()
    assert L.kb_triad_bench(FAKE, FAKE, FAKE, 1.0, 16, 256, None, 0, 0, ms) == Status.INVALID_ARG
    assert L.kb_attn_bench(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, 0.125, 0, 3, None, None, 0, -1, 2,
                           ms) == Status.INVALID_ARG


def test_graph_bench_argument_checks(lib):
    L = lib
    ms = (ctypes.c_float * 4)()
    base = (FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 32, 0, 0.125, DType.F32, Variant.FLASH, None, None, 0)
    for launches, warmup, iters in ((0, 1, 1), (100001, 1, 1), (10, -1, 1), (10, 1, 0)):
        assert L.kb_attn_bench_graph(*base, launches, warmup, iters, ms) == Status.INVALID_ARG
    assert L.kb_attn_bench_graph(*base, 10, 1, 1, None) == Status.INVALID_ARG
    bad = base[:6] + (0,) + base[7:]  # S = 0
    assert L.kb_attn_bench_graph(*bad, 10, 1, 1, ms) == Status.INVALID_ARG


def test_fixed_point_support_matrix(lib):
    L = lib
    args = (FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0)
    assert L.kb_attn_fwd(*args, 0.125, DType.Q15, Variant.TC, None) == Status.UNSUPPORTED
    assert L.kb_attn_fwd(*args, 0.125, DType.Q15, Variant.FLASH, None) == Status.UNSUPPORTED
    assert L.kb_attn_fwd(*args, 0.125, DType.F32, Variant.FIXEDPOINT, None) == Status.UNSUPPORTED
    assert L.kb_attn_fwd(*args, 0.125, DType.BF16, Variant.FIXEDPOINT, None) == Status.UNSUPPORTED
    assert L.kb_attn_fwd(*args, 1e5, DType.Q15, Variant.FIXEDPOINT, None) == Status.INVALID_ARG  # C > 2^30
    big = (FAKE, FAKE, FAKE, FAKE, 1, 1, 65537, 64, 0, 0.125)
    assert L.kb_attn_fwd(*big, DType.Q15, Variant.AUTO, None) == Status.INVALID_ARG
    assert L.kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 48, 0, 0.125, DType.Q15, Variant.AUTO,
                         None) == Status.UNSUPPORTED
    ms = (ctypes.c_float * 1)()
    assert L.kb_attn_fwd_lse(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, 0.125, DType.Q15, Variant.AUTO,
                             None) == Status.UNSUPPORTED
    import torch
    if not torch.cuda.is_available():  # never launch on the fake pointers where a GPU exists
        assert L.kb_attn_fwd(*args, 0.125, DType.Q15, Variant.AUTO, None) == Status.NO_DEVICE


def test_fixed_point_table_is_exact(lib):
    import mpmath
    mpmath.mp.dps = 50
    want = [int(mpmath.nint(32768 * mpmath.power(2, mpmath.mpf(-f) / 64))) for f in range(64)]
    assert kbattn.kb_q15_exp_table() == want


def test_lse_argument_checks(lib):
    L = kbattn.load()
    args = (FAKE, FAKE, FAKE, FAKE)
    assert L.kb_attn_fwd_lse(*args, None, 1, 1, 64, 64, 0, 0.125, DType.BF16, Variant.TC, None) == Status.INVALID_ARG
    assert L.kb_attn_fwd_lse(*args, FAKE + 2, 1, 1, 64, 64, 0, 0.125, DType.BF16, Variant.TC, None) == Status.INVALID_ARG
    for v in (Variant.NAIVE, Variant.FUSED):
        assert L.kb_attn_fwd_lse(*args, FAKE, 1, 1, 64, 64, 0, 0.125, DType.F32, v, None) == Status.UNSUPPORTED
    assert L.kb_attn_fwd_lse(*args, FAKE, 1, 1, 0, 64, 0, 0.125, DType.F32, Variant.FLASH, None) == Status.INVALID_ARG


def test_hbm_argument_checks(lib):
    L = kbattn.load()
    assert L.kb_hbm_copy(FAKE, FAKE, 0, 256, None) == Status.OK          # n = 0 is a no-op
    assert L.kb_hbm_copy(FAKE, 0, 16, 256, None) == Status.INVALID_ARG
    assert L.kb_hbm_copy(FAKE, FAKE + 4, 16, 256, None) == Status.INVALID_ARG
    assert L.kb_hbm_write(FAKE, 1.0, 16, 96, None) == Status.INVALID_ARG
    assert L.kb_hbm_read(FAKE, 16, 256, None, None) == Status.INVALID_ARG
    assert L.kb_hbm_read(FAKE, 16, 256, FAKE + 2, None) == Status.INVALID_ARG
    ms = (ctypes.c_float * 1)()
    assert L.kb_hbm_bench(7, FAKE, FAKE, FAKE, 1.0, 16, 256, FAKE, None, 0, 1, ms) == Status.INVALID_ARG
    assert L.kb_hbm_bench(0, FAKE, FAKE, FAKE, 1.0, 16, 256, FAKE, None, 0, 0, ms) == Status.INVALID_ARG


def test_status_strings(lib):
    for s in Status:
        assert kbattn.status_string(s) == "KB_" + ("OK" if s == Status.OK else "ERR_" + s.name)
    assert kbattn.status_string(99) == "KB_UNKNOWN_STATUS"
    assert kbattn.version() == 101


def test_binding_refuses_to_run_without_the_library(tmp_path):
    # the product path fails loudly instead of falling back
    code = ("import roofline_benchmarking_gb300.kbattn as k\n"
            f"k.LIBRARY = {str(tmp_path / 'missing.so')!r}\n"
            "try:\n    k.load(k.LIBRARY)\nexcept RuntimeError as e:\n    print('raised', e)\n")
    r = subprocess.run(["python", "-c", code], capture_output=True, text=True, cwd=ROOT)
    assert "raised" in r.stdout and "not built" in r.stdout


def test_host_call_validates_before_copying(lib):
    """kb_attn_fwd_host rejects null host pointers and every kb_attn_fwd argument
    error before it issues any copy (so no device is needed here)."""
    f = ctypes.c_void_p(FAKE)
    args = [f] * 8 + [1, 1, 64, 64, 0, ctypes.c_float(0.125), DType.F32, Variant.FLASH, None]
    for i in range(8):
        a = list(args)
        a[i] = None
        assert lib.kb_attn_fwd_host(*a) == Status.INVALID_ARG, i
    a = list(args)
    a[11] = 48  # d
    assert lib.kb_attn_fwd_host(*a) == Status.UNSUPPORTED
    a = list(args)
    a[13] = ctypes.c_float(0.0)  # scale
    assert lib.kb_attn_fwd_host(*a) == Status.INVALID_ARG
