"""kb_attn_fwd_naive_noalloc: the naive fp32 forward for callers that cannot
allocate device memory (their memory is all reserved by their own pool, or they
must not pay cudaMalloc's cost and implicit synchronisation). Its score
workspace is a fixed array inside the library instead of a cudaMalloc.

Checked here, through the C ABI: two calls in a row (different shapes, so the
second runs over what the first left in the array) each match the allocating
entry point kb_attn_fwd(variant=KB_NAIVE) within the fp32 tolerance; requests
larger than the array are refused before any device work; and a call leaves
the device's free memory unchanged. This file is named to be collected last.
"""
import ctypes

import pytest
import torch

from roofline_benchmarking_gb300 import inputs
from roofline_benchmarking_gb300 import kbattn
from roofline_benchmarking_gb300.kbattn import DType, Status, Variant

F32_TOL = 1e-4


@pytest.fixture(scope="module")
def lib():
    from roofline_benchmarking_gb300 import build
    build.build()
    return kbattn.load()


def noalloc(lib, q, k, v, o, causal, scale):
    B, H, S, d = q.shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.kb_attn_fwd_naive_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, S, d,
                                         int(causal), ctypes.c_float(scale), stream)


@pytest.mark.gpu
def test_two_calls_in_a_row_match_the_allocating_entry_point(lib):
    # the first workload fills the whole array (8 heads x 1024^2 x 4 bytes = 32 MiB)
    first = inputs.F32_S1024
    second = inputs.Workload("ragged_causal", 1, 3, 300, 32, True, "f32", 31, "uniform")
    assert first.N * first.S * first.S * 4 == kbattn.NAIVE_NOALLOC_MAX_BYTES
    for w in (first, second):
        q, k, v = (t.cuda() for t in inputs.make_qkv(w))
        want = kbattn.kb_attn_fwd(q, k, v, causal=w.causal, scale=w.scale, variant=Variant.NAIVE)
        got = torch.full_like(q, float("nan"))
        assert noalloc(lib, q, k, v, got, w.causal, w.scale) == Status.OK
        torch.cuda.synchronize()
        assert kbattn.kb_check_device_error() == Status.OK
        err = float((got - want).abs().max())
        assert err <= F32_TOL, (w.name, err)


@pytest.mark.gpu
def test_a_call_allocates_no_device_memory(lib):
    w = inputs.F32_S1024_CAUSAL
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    o = torch.empty_like(q)
    assert noalloc(lib, q, k, v, o, True, w.scale) == Status.OK  # set-up call on this device
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert noalloc(lib, q, k, v, o, True, w.scale) == Status.OK
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before


FAKE = 1 << 20  # aligned, never dereferenced: the size check comes before any device work


def test_requests_beyond_the_array_are_refused(lib):
    fake = ctypes.c_void_p(FAKE)
    # 8 heads x 1025^2 x 4 bytes is just over 32 MiB
    st = lib.kb_attn_fwd_naive_noalloc(fake, fake, fake, fake, 1, 8, 1025, 64, 0, ctypes.c_float(0.125), None)
    assert st == Status.NO_MEMORY
    st = lib.kb_attn_fwd_naive_noalloc(fake, fake, fake, fake, 1, 1, 4096, 64, 1, ctypes.c_float(0.125), None)
    assert st == Status.NO_MEMORY
    # argument errors are reported as for kb_attn_fwd
    st = lib.kb_attn_fwd_naive_noalloc(None, fake, fake, fake, 1, 1, 64, 64, 0, ctypes.c_float(0.125), None)
    assert st == Status.INVALID_ARG
    st = lib.kb_attn_fwd_naive_noalloc(fake, fake, fake, fake, 1, 1, 64, 48, 0, ctypes.c_float(0.125), None)
    assert st == Status.UNSUPPORTED
