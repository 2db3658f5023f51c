"""kb_attn_fwd_naive_noalloc: the naive fp32 forward for callers that cannot
allocate device memory (their memory is all reserved by their own pool, or they
must not pay cudaMalloc's cost and implicit synchronisation). Its score
workspace is a fixed array inside the library instead of a cudaMalloc.

Checked here, through the C ABI: two calls in a row (different shapes, so the
second runs over what the first left in the array) each write exactly their
output (poisoned guards before and after it), match the oracle within the fp32
tolerance, and match the allocating entry point kb_attn_fwd(variant=KB_NAIVE);
requests larger than the array are refused before any device work; and, in a
fresh process, free device memory is recorded around the first call on the
device (where the module holding the array is loaded and the array committed)
and around later calls (which commit nothing). This file is named to be
collected last.
"""
import ctypes
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from roofline_benchmarking_gb300 import inputs
from roofline_benchmarking_gb300 import kbattn
from roofline_benchmarking_gb300.kbattn import Status, Variant
from tests.gpu_util import Guarded, errors

F32_TOL = 1e-4
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
def test_two_calls_in_a_row_match_the_oracle_and_the_allocating_entry_point(lib, oracle):
    # the first workload fills the whole array (8 heads x 1024^2 x 4 bytes = 32 MiB)
    first = inputs.F32_S1024
    second = inputs.Workload("ragged_causal", 1, 3, 300, 32, True, "f32", 31, "uniform")
    assert first.N * first.S * first.S * 4 == kbattn.NAIVE_NOALLOC_MAX_BYTES
    for w in (first, second):
        qh, kh, vh = inputs.make_qkv(w)
        q, k, v = qh.cuda(), kh.cuda(), vh.cuda()
        g = Guarded(q.shape, q.dtype)
        assert noalloc(lib, q, k, v, g.out, w.causal, w.scale) == Status.OK
        got = g.check()
        assert kbattn.kb_check_device_error() == Status.OK
        mx, _, _ = errors(got.cpu().numpy(), oracle.attn(qh, kh, vh, w.causal, w.scale))
        assert mx <= F32_TOL, (w.name, "vs oracle", mx)
        want = kbattn.kb_attn_fwd(q, k, v, causal=w.causal, scale=w.scale, variant=Variant.NAIVE)
        err = float((got - want).abs().max())
        assert err <= F32_TOL, (w.name, "vs kb_attn_fwd", err)


# Run in a fresh process, so that no earlier test has loaded the library's
# modules on the device: free memory before the library is loaded, after it is
# loaded, after the first call and after three more calls.
FIRST_CALL_PROBE = r"""
import ctypes, json, sys, torch
sys.path.insert(0, sys.argv[1])
from roofline_benchmarking_gb300 import inputs, kbattn
w = inputs.F32_S1024_CAUSAL
q, k, v = (t.cuda() for t in inputs.make_qkv(w))
o = torch.empty_like(q)
torch.cuda.synchronize()
free = lambda: torch.cuda.mem_get_info()[0]
f_ctx = free()
lib = kbattn.load()
f_loaded = free()
stream = torch.cuda.current_stream().cuda_stream
call = lambda: lib.kb_attn_fwd_naive_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                             w.B, w.H, w.S, w.d, 1, ctypes.c_float(w.scale), stream)
st = [call()]
torch.cuda.synchronize()
f_first = free()
st += [call() for _ in range(3)]
torch.cuda.synchronize()
f_later = free()
print(json.dumps({"status": st, "free": [f_ctx, f_loaded, f_first, f_later]}))
"""


@pytest.mark.gpu
def test_where_the_array_is_committed_and_later_calls_allocate_nothing(lib):
    from roofline_benchmarking_gb300 import build
    build.build()
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY")
    r = subprocess.run([sys.executable, "-c", FIRST_CALL_PROBE, ROOT], capture_output=True, text=True, env=env,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    rec = json.loads(r.stdout.strip().splitlines()[-1])
    assert rec["status"] == [Status.OK] * 4
    f_ctx, f_loaded, f_first, f_later = rec["free"]
    print(f"free device memory (bytes): context {f_ctx}, library loaded {f_loaded}, after the first call "
          f"{f_first}, after three more {f_later}")
    # lazy loading: the 32 MiB lands in the first call (with the kernels' modules), not at the library's load
    assert f_ctx - f_loaded < kbattn.NAIVE_NOALLOC_MAX_BYTES
    assert f_loaded - f_first >= kbattn.NAIVE_NOALLOC_MAX_BYTES
    # later calls commit nothing
    assert f_later == f_first


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
    assert np.isfinite(o.cpu().numpy()).all()


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
