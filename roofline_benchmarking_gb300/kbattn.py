"""ctypes binding of libkbattn (include/kbattn.h): the same entry points, with
argument marshalling only. Every step of the computation runs in the CUDA
library; there is no fallback. If the library has not been built, loading it
raises.

Tensors are passed as torch tensors (device memory and streams come from
PyTorch); the ``*_ptr`` forms take raw integers for callers that manage memory
themselves.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(HERE, "libkbattn.so")


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED = 2
    CUDA = 3
    NO_MEMORY = 4
    TIMEOUT = 5
    NO_DEVICE = 6


class DType(enum.IntEnum):
    F32 = 0
    BF16 = 1
    F16 = 2
    Q15 = 3


class Variant(enum.IntEnum):
    AUTO = 0
    NAIVE = 1
    FUSED = 2
    FLASH = 3
    TC = 4
    FIXEDPOINT = 5


class DeviceInfo(ctypes.Structure):
    _fields_ = [
        ("device", ctypes.c_int),
        ("cc_major", ctypes.c_int),
        ("cc_minor", ctypes.c_int),
        ("sm_count", ctypes.c_int),
        ("sm_clock_khz", ctypes.c_int),
        ("mem_clock_khz", ctypes.c_int),
        ("mem_bus_width_bits", ctypes.c_int),
        ("l2_bytes", ctypes.c_int),
        ("smem_per_block_optin", ctypes.c_int),
        ("smem_per_sm", ctypes.c_int),
        ("total_mem_bytes", ctypes.c_size_t),
        ("name", ctypes.c_char * 256),
    ]

    def as_dict(self) -> dict:
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["name"] = self.name.decode(errors="replace")
        return d


class KbError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}"
                         + (f" (cudaError {last_cuda_error()})" if status == Status.CUDA else ""))


# Entry points and their C signatures (names identical to include/kbattn.h).
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_FP = ctypes.POINTER(ctypes.c_float)
SIGNATURES = {
    "kb_attn_fwd": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "kb_attn_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "kb_attn_fwd_lse": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "kb_attn_fwd_ws": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _P, _SZ]),
    "kb_attn_fwd_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "kb_attn_bench": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _P, _SZ, _I, _I, _FP]),
    "kb_attn_bench_graph": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _P, _SZ, _I, _I, _I, _FP]),
    "kb_triad": (_I, [_P, _P, _P, _F, _SZ, _I, _P]),
    "kb_triad_bench": (_I, [_P, _P, _P, _F, _SZ, _I, _P, _I, _I, _FP]),
    "kb_device_info": (_I, [_I, ctypes.POINTER(DeviceInfo)]),
    "kb_check_device_error": (_I, [_P]),
    "kb_selftest_timeout": (_I, [ctypes.c_ulonglong, _P]),
    "kb_status_string": (ctypes.c_char_p, [_I]),
    "kb_last_cuda_error": (_I, []),
    "kb_version": (_I, []),
    "kb_binary_version": (_I, [ctypes.POINTER(ctypes.c_int)]),
    "kb_q15_exp_table": (_I, [ctypes.POINTER(ctypes.c_uint16)]),
    "kb_attn_work_lists": (_I, [ctypes.c_longlong, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int),
                                ctypes.POINTER(ctypes.c_uint32), _I, ctypes.POINTER(ctypes.c_int)]),
    "kb_attn_fwd_naive_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "kb_hbm_copy": (_I, [_P, _P, _SZ, _I, _P]),
    "kb_hbm_write": (_I, [_P, _F, _SZ, _I, _P]),
    "kb_hbm_read": (_I, [_P, _SZ, _I, _P, _P]),
    "kb_hbm_bench": (_I, [_I, _P, _P, _P, _F, _SZ, _I, _P, _P, _I, _I, _FP]),
}


class HbmOp(enum.IntEnum):
    TRIAD = 0
    COPY = 1
    READ = 2
    WRITE = 3


# Bytes each HBM kernel moves per float element.
HBM_BYTES_PER_ELEMENT = {HbmOp.TRIAD: 12, HbmOp.COPY: 8, HbmOp.READ: 4, HbmOp.WRITE: 4}

# Bytes of the library-owned score array of kb_attn_fwd_naive_noalloc.
NAIVE_NOALLOC_MAX_BYTES = 32 * 1024 * 1024

_lib = None
_lock = threading.Lock()


def load(path: str = LIBRARY) -> ctypes.CDLL:
    """Load libkbattn (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libkbattn is not built ({path} missing); run "
                    "`python -m roofline_benchmarking_gb300.build`")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def status_string(status: int) -> str:
    return load().kb_status_string(int(status)).decode()


def last_cuda_error() -> int:
    return load().kb_last_cuda_error()


def version() -> int:
    return load().kb_version()


def binary_version() -> int:
    """10 * major + minor of the architecture the kernels were compiled for
    (cudaFuncAttributes::binaryVersion on the current device)."""
    out = ctypes.c_int(0)
    _check(load().kb_binary_version(ctypes.byref(out)), "kb_binary_version")
    return out.value


def _check(status: int, what: str) -> None:
    if status != Status.OK:
        raise KbError(status, what)


def _stream_ptr(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


_DTYPES = None


def _dtype_code(t) -> int:
    global _DTYPES
    if _DTYPES is None:
        import torch
        _DTYPES = {torch.float32: DType.F32, torch.bfloat16: DType.BF16, torch.float16: DType.F16,
                   torch.int16: DType.Q15}
    try:
        return int(_DTYPES[t.dtype])
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}") from None


def _attn_args(q, k, v, o):
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if t.dim() != 4 or t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must be [B, H, S, d] like q, with q's dtype")
    B, H, S, d = q.shape
    return B, H, S, d, _dtype_code(q)


# ---------------------------------------------------------------- attention
def kb_attn_fwd_ptr(q: int, k: int, v: int, o: int, B: int, H: int, S: int, d: int, causal: bool,
                    scale: float, dtype: int, variant: int = Variant.AUTO, stream: int | None = 0) -> int:
    """Raw form: device pointers as integers; returns the kb_status (no raise)."""
    return load().kb_attn_fwd(q, k, v, o, B, H, S, d, int(causal), float(scale), int(dtype),
                              int(variant), stream)


def kb_attn_fwd(q, k, v, o=None, causal: bool = False, scale: float | None = None,
                variant: int = Variant.AUTO, stream=None):
    """O = softmax(Q K^T * scale [+ causal mask]) V on the current CUDA device.

    q, k, v: contiguous CUDA tensors [B, H, S, d] (fp32, bf16 or f16). ``o`` is
    written if given, else allocated. ``scale`` defaults to 1/sqrt(d).
    """
    import torch
    if o is None:
        o = torch.empty_like(q)
    B, H, S, d, dt = _attn_args(q, k, v, o)
    if scale is None:
        scale = d ** -0.5
    st = load().kb_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, S, d,
                            int(bool(causal)), float(scale), dt, int(variant), _stream_ptr(stream))
    _check(st, "kb_attn_fwd")
    return o


def kb_attn_fwd_host(qh, kh, vh, oh, q, k, v, o, causal: bool = False, scale: float | None = None,
                     variant: int = Variant.AUTO, stream=None):
    """kb_attn_fwd from host tensors to a host tensor: ``qh``, ``kh``, ``vh`` are
    copied into the device staging tensors ``q``, ``k``, ``v`` on ``stream``,
    the forward pass runs into ``o`` and ``o`` is copied back into ``oh``
    (asynchronously: ``oh`` is valid once the stream gets there). Host tensors
    should be pinned (``Tensor.pin_memory()``) for the copies to be asynchronous."""
    B, H, S, d, dt = _attn_args(q, k, v, o)
    for name, t in (("qh", qh), ("kh", kh), ("vh", vh), ("oh", oh)):
        if t.is_cuda or not t.is_contiguous() or t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must be a contiguous host tensor shaped and typed like q")
    if scale is None:
        scale = d ** -0.5
    st = load().kb_attn_fwd_host(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(), q.data_ptr(),
                                 k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, S, d, int(bool(causal)),
                                 float(scale), dt, int(variant), _stream_ptr(stream))
    _check(st, "kb_attn_fwd_host")
    return oh


def kb_attn_fwd_lse(q, k, v, o=None, lse=None, causal: bool = False, scale: float | None = None,
                    variant: int = Variant.AUTO, stream=None):
    """kb_attn_fwd that also returns the natural-log log-sum-exp of every score
    row, an fp32 [B, H, S] tensor (written into ``lse`` if given)."""
    import torch
    if o is None:
        o = torch.empty_like(q)
    B, H, S, d, dt = _attn_args(q, k, v, o)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if not lse.is_cuda or lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * S:
        raise ValueError("lse must be a contiguous fp32 CUDA tensor of B*H*S elements")
    if scale is None:
        scale = d ** -0.5
    st = load().kb_attn_fwd_lse(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, S,
                                d, int(bool(causal)), float(scale), dt, int(variant), _stream_ptr(stream))
    _check(st, "kb_attn_fwd_lse")
    return o, lse


def kb_attn_workspace_bytes(B: int, H: int, S: int, d: int, dtype: int, variant: int) -> int:
    return int(load().kb_attn_workspace_bytes(B, H, S, d, int(dtype), int(variant)))


def kb_attn_fwd_ws(q, k, v, o, workspace, causal: bool = False, scale: float | None = None,
                   variant: int = Variant.AUTO, stream=None):
    """kb_attn_fwd with a caller-owned workspace tensor (any dtype, on the device)."""
    B, H, S, d, dt = _attn_args(q, k, v, o)
    if scale is None:
        scale = d ** -0.5
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().kb_attn_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, S, d,
                               int(bool(causal)), float(scale), dt, int(variant), _stream_ptr(stream),
                               ws_ptr, ws_bytes)
    _check(st, "kb_attn_fwd_ws")
    return o


def kb_attn_bench(q, k, v, o, causal: bool, scale: float | None = None, variant: int = Variant.AUTO,
                  warmup: int = 3, iters: int = 10, workspace=None, stream=None) -> list[float]:
    """Per-call device times in ms of ``iters`` timed calls after ``warmup`` untimed ones."""
    B, H, S, d, dt = _attn_args(q, k, v, o)
    if scale is None:
        scale = d ** -0.5
    ms = (ctypes.c_float * iters)()
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().kb_attn_bench(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, S, d,
                              int(bool(causal)), float(scale), dt, int(variant), _stream_ptr(stream),
                              ws_ptr, ws_bytes, warmup, iters, ms)
    _check(st, "kb_attn_bench")
    return list(ms)


def kb_q15_exp_table() -> list[int]:
    """The 64-entry table of the fixed-point path, round(2^15 * 2^(-f/64))."""
    out = (ctypes.c_uint16 * 64)()
    _check(load().kb_q15_exp_table(out), "kb_q15_exp_table")
    return list(out)


def kb_attn_work_lists(N: int, S: int, d: int, causal: bool, grid: int):
    """The tensor-core path's per-CTA work lists: a list of ``grid`` lists of
    (head, unit) pairs in run order, or None when the kernel orders the units
    itself (see include/kbattn.h)."""
    cap = 4096
    start = (ctypes.c_int * (grid + 1))()
    items = (ctypes.c_uint32 * cap)()
    count = ctypes.c_int(0)
    _check(load().kb_attn_work_lists(N, S, d, int(bool(causal)), grid, start, items, cap, ctypes.byref(count)),
           "kb_attn_work_lists")
    if count.value == 0:
        return None
    return [[(items[k] >> 16, items[k] & 0xFFFF) for k in range(start[c], start[c + 1])] for c in range(grid)]


def kb_attn_bench_graph(q, k, v, o, causal: bool, scale: float | None = None, variant: int = Variant.AUTO,
                        launches: int = 200, warmup: int = 3, iters: int = 10, workspace=None,
                        stream=None) -> list[float]:
    """Device times in ms of ``iters`` replays of one CUDA graph holding
    ``launches`` captured calls (per call: divide by ``launches``)."""
    B, H, S, d, dt = _attn_args(q, k, v, o)
    if scale is None:
        scale = d ** -0.5
    ms = (ctypes.c_float * iters)()
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().kb_attn_bench_graph(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, S, d,
                                    int(bool(causal)), float(scale), dt, int(variant), _stream_ptr(stream),
                                    ws_ptr, ws_bytes, launches, warmup, iters, ms)
    _check(st, "kb_attn_bench_graph")
    return list(ms)


def kb_attn_fwd_naive_noalloc(q, k, v, o, causal: bool = False, scale: float | None = None, stream=None):
    """The naive fp32 forward with its score workspace in the library's fixed
    array: for callers that cannot allocate device memory (their memory is all
    reserved by their own pool, or they must not pay cudaMalloc's cost and
    implicit synchronisation). ``o`` must be given; nothing is allocated.
    Calls that overlap on the GPU share the array and race on it."""
    B, H, S, d, dt = _attn_args(q, k, v, o)
    if scale is None:
        scale = d ** -0.5
    st = load().kb_attn_fwd_naive_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, S, d,
                                          int(bool(causal)), float(scale), _stream_ptr(stream))
    _check(st, "kb_attn_fwd_naive_noalloc")
    return o


# ---------------------------------------------------------------- triad
def kb_triad(a, b, c, s: float, block: int = 256, stream=None):
    """a = b + s*c (fp32, one rounding) over every element of the CUDA tensors."""
    n = a.numel()
    if b.numel() != n or c.numel() != n:
        raise ValueError("a, b, c must have the same number of elements")
    st = load().kb_triad(a.data_ptr(), b.data_ptr(), c.data_ptr(), float(s), n, block, _stream_ptr(stream))
    _check(st, "kb_triad")
    return a


def kb_triad_bench(a, b, c, s: float, block: int = 256, warmup: int = 3, iters: int = 10,
                   stream=None) -> list[float]:
    n = a.numel()
    ms = (ctypes.c_float * iters)()
    st = load().kb_triad_bench(a.data_ptr(), b.data_ptr(), c.data_ptr(), float(s), n, block,
                               _stream_ptr(stream), warmup, iters, ms)
    _check(st, "kb_triad_bench")
    return list(ms)


def kb_hbm_copy(a, b, block: int = 256, stream=None):
    """a = b over every element (fp32 CUDA tensors of equal size)."""
    if b.numel() != a.numel():
        raise ValueError("a and b must have the same number of elements")
    _check(load().kb_hbm_copy(a.data_ptr(), b.data_ptr(), a.numel(), block, _stream_ptr(stream)), "kb_hbm_copy")
    return a


def kb_hbm_write(a, s: float, block: int = 256, stream=None):
    """a = s over every element."""
    _check(load().kb_hbm_write(a.data_ptr(), float(s), a.numel(), block, _stream_ptr(stream)), "kb_hbm_write")
    return a


def kb_hbm_read(b, out, block: int = 256, stream=None):
    """out[0] = sum of b (fp32 partial sums); ``out`` is a 1-element fp32 CUDA tensor."""
    _check(load().kb_hbm_read(b.data_ptr(), b.numel(), block, out.data_ptr(), _stream_ptr(stream)), "kb_hbm_read")
    return out


def kb_hbm_bench(op: int, a, b, c, s: float, out, block: int = 256, warmup: int = 3, iters: int = 10,
                 stream=None) -> list[float]:
    """Per-call device times (ms) of one HBM kernel over a.numel() floats."""
    ms = (ctypes.c_float * iters)()
    st = load().kb_hbm_bench(int(op), a.data_ptr(), b.data_ptr(), c.data_ptr(), float(s), a.numel(), block,
                             out.data_ptr(), _stream_ptr(stream), warmup, iters, ms)
    _check(st, "kb_hbm_bench")
    return list(ms)


# ---------------------------------------------------------------- device
def kb_device_info(device: int = 0) -> dict:
    info = DeviceInfo()
    _check(load().kb_device_info(device, ctypes.byref(info)), "kb_device_info")
    return info.as_dict()


def kb_check_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load().kb_check_device_error(_stream_ptr(stream)))


def kb_selftest_timeout(limit_ns: int = 1_000_000, stream=None) -> None:
    _check(load().kb_selftest_timeout(int(limit_ns), _stream_ptr(stream)), "kb_selftest_timeout")
