"""TEST INFRASTRUCTURE ONLY: ctypes front end of the plain C oracle.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The attention library never imports it, and this
package never imports the library: the two share nothing but the seeded input
generators, which hold none of the method's arithmetic.

The oracle (``attn_oracle.c``) restates, single-threaded and in double
precision, the attention forward O = softmax(Q K^T * scale [+ causal mask]) V
of the kbench page ("kbench -- Transformer Attention Micro-benchmark Harness",
section "Implementation details / The three GPU kernels") and the STREAM Triad
a = b + s*c of the TileOPs "Hardware Microbenchmarks" README (section
"HBM Bandwidth"), and the page's Q15 fixed-point model of the microcontroller
path (section "CPU reference + cache profiling").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "attn_oracle.c")
LIBRARY = os.path.join(HERE, "libkboracle.so")

# Flags: plain -O2, no FMA contraction (x86_64 and aarch64 then agree bit for bit).
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(source: str = SOURCE, out: str = LIBRARY, force: bool = False) -> str:
    """Compile the oracle with gcc into a shared library; return its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(source):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, source, "-lm"], check=True)
    os.replace(tmp, out)
    return out


_I64 = ctypes.c_int64
_DP = ctypes.POINTER(ctypes.c_double)
_FP = ctypes.POINTER(ctypes.c_float)
_I64P = ctypes.POINTER(ctypes.c_int64)
_I16P = ctypes.POINTER(ctypes.c_int16)
_U16P = ctypes.POINTER(ctypes.c_uint16)


class Oracle:
    """Handle on one compiled copy of the oracle (the tests also load mutants)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.kb_oracle_attn.argtypes = [_DP, _DP, _DP, _DP, _I64, _I64, _I64, _I64,
                                       ctypes.c_int, ctypes.c_double]
        lib.kb_oracle_attn.restype = ctypes.c_int
        lib.kb_oracle_attn_rows.argtypes = [_DP, _DP, _DP, _DP, _I64, _I64, _I64,
                                            ctypes.c_int, ctypes.c_double, _I64P, _I64P, _I64]
        lib.kb_oracle_attn_rows.restype = ctypes.c_int
        lib.kb_oracle_triad.argtypes = [_FP, _FP, _FP, ctypes.c_float, _I64]
        lib.kb_oracle_triad.restype = ctypes.c_int
        lib.kb_oracle_lse.argtypes = [_DP, _DP, _DP, _I64, _I64, _I64, ctypes.c_int, ctypes.c_double]
        lib.kb_oracle_lse.restype = ctypes.c_int
        lib.kb_oracle_copy.argtypes = [_FP, _FP, _I64]
        lib.kb_oracle_copy.restype = ctypes.c_int
        lib.kb_oracle_fill.argtypes = [_FP, ctypes.c_float, _I64]
        lib.kb_oracle_fill.restype = ctypes.c_int
        lib.kb_oracle_sum.argtypes = [_FP, _I64, _DP]
        lib.kb_oracle_sum.restype = ctypes.c_int
        lib.kb_oracle_attn_q15.argtypes = [_I16P, _I16P, _I16P, _I16P, _I64, _I64, _I64, ctypes.c_int,
                                           ctypes.c_double]
        lib.kb_oracle_attn_q15.restype = ctypes.c_int
        lib.kb_oracle_q15_exp_table.argtypes = [_U16P]
        lib.kb_oracle_q15_exp_table.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    @staticmethod
    def _f64(x) -> np.ndarray:
        # Exact widening: fp32 and bf16 values are all representable in fp64.
        if hasattr(x, "detach"):  # a torch tensor on the CPU
            x = x.detach().to("cpu").double().numpy()
        return np.ascontiguousarray(np.asarray(x, dtype=np.float64))

    def attn(self, q, k, v, causal: bool, scale: float) -> np.ndarray:
        """O for q, k, v of shape [B, H, S, d]; returns float64 [B, H, S, d]."""
        q, k, v = self._f64(q), self._f64(k), self._f64(v)
        if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
            raise ValueError(f"q, k, v must share one [B,H,S,d] shape, got {q.shape} {k.shape} {v.shape}")
        B, H, S, d = q.shape
        o = np.empty_like(q)
        rc = self.lib.kb_oracle_attn(q.ctypes.data_as(_DP), k.ctypes.data_as(_DP),
                                     v.ctypes.data_as(_DP), o.ctypes.data_as(_DP),
                                     B, H, S, d, int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"kb_oracle_attn returned {rc}")
        return o

    def attn_rows(self, q, k, v, causal: bool, scale: float, heads, rows) -> np.ndarray:
        """Rows (heads[t], rows[t]) of O, each exactly as the full evaluation gives it.

        q, k, v are [B, H, S, d] (or [N, S, d]); heads index the flattened
        b*H + h axis. Returns float64 [count, d].
        """
        q, k, v = self._f64(q), self._f64(k), self._f64(v)
        S, d = q.shape[-2], q.shape[-1]
        N = int(np.prod(q.shape[:-2]))
        heads = np.ascontiguousarray(np.asarray(heads, dtype=np.int64))
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        if heads.shape != rows.shape or heads.ndim != 1:
            raise ValueError("heads and rows must be 1-D and of equal length")
        o = np.empty((heads.size, d), dtype=np.float64)
        rc = self.lib.kb_oracle_attn_rows(q.ctypes.data_as(_DP), k.ctypes.data_as(_DP),
                                          v.ctypes.data_as(_DP), o.ctypes.data_as(_DP),
                                          N, S, d, int(bool(causal)), float(scale),
                                          heads.ctypes.data_as(_I64P), rows.ctypes.data_as(_I64P),
                                          heads.size)
        if rc != 0:
            raise ValueError(f"kb_oracle_attn_rows returned {rc}")
        return o

    def attn_threads(self, q, k, v, causal: bool, scale: float, threads: int | None = None) -> np.ndarray:
        """The same result as ``attn``, with the heads dealt out to host threads.

        Heads are independent problems (each one's rows read only its own Q, K
        and V), so every thread runs the unchanged single-threaded oracle on a
        contiguous range of heads; the ctypes calls release the GIL. Returns
        float64 [B, H, S, d], element for element what ``attn`` returns.
        """
        import concurrent.futures as cf

        q, k, v = self._f64(q), self._f64(k), self._f64(v)
        if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
            raise ValueError(f"q, k, v must share one [B,H,S,d] shape, got {q.shape} {k.shape} {v.shape}")
        B, H, S, d = q.shape
        N = B * H
        qf, kf, vf = (x.reshape(N, S, d) for x in (q, k, v))
        o = np.empty((N, S, d), dtype=np.float64)
        if threads is None:
            threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        threads = max(1, min(int(threads), N))
        bounds = [N * t // threads for t in range(threads + 1)]

        def run(t):
            n0, n1 = bounds[t], bounds[t + 1]
            if n1 == n0:
                return 0
            return self.lib.kb_oracle_attn(qf[n0:n1].ctypes.data_as(_DP), kf[n0:n1].ctypes.data_as(_DP),
                                           vf[n0:n1].ctypes.data_as(_DP), o[n0:n1].ctypes.data_as(_DP),
                                           1, n1 - n0, S, d, int(bool(causal)), float(scale))

        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            rcs = list(ex.map(run, range(threads)))
        if any(rcs):
            raise ValueError(f"kb_oracle_attn returned {rcs}")
        return o.reshape(B, H, S, d)

    def triad(self, b, c, s: float) -> np.ndarray:
        """a = b + s*c in fp32, rounded once."""
        b = np.ascontiguousarray(np.asarray(b, dtype=np.float32))
        c = np.ascontiguousarray(np.asarray(c, dtype=np.float32))
        if b.shape != c.shape:
            raise ValueError("b and c must have the same shape")
        a = np.empty_like(b)
        rc = self.lib.kb_oracle_triad(a.ctypes.data_as(_FP), b.ctypes.data_as(_FP),
                                      c.ctypes.data_as(_FP), ctypes.c_float(s), b.size)
        if rc != 0:
            raise ValueError(f"kb_oracle_triad returned {rc}")
        return a


    def lse(self, q, k, causal: bool, scale: float) -> np.ndarray:
        """log(sum_j exp(score_ij)) over the visible keys; q, k [B, H, S, d] -> [B, H, S]."""
        q, k = self._f64(q), self._f64(k)
        if q.ndim != 4 or q.shape != k.shape:
            raise ValueError("q and k must share one [B,H,S,d] shape")
        B, H, S, d = q.shape
        out = np.empty((B, H, S), dtype=np.float64)
        rc = self.lib.kb_oracle_lse(q.ctypes.data_as(_DP), k.ctypes.data_as(_DP), out.ctypes.data_as(_DP),
                                    B * H, S, d, int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"kb_oracle_lse returned {rc}")
        return out

    def attn_q15(self, q, k, v, causal: bool, scale: float) -> np.ndarray:
        """The Q15 fixed-point model: int16 q, k, v [..., S, d] -> int16 O of the same shape."""
        q, k, v = (np.ascontiguousarray(np.asarray(x.numpy() if hasattr(x, "numpy") else x, dtype=np.int16))
                   for x in (q, k, v))
        if q.ndim < 2 or q.shape != k.shape or q.shape != v.shape:
            raise ValueError("q, k, v must share one [..., S, d] shape")
        S, d = q.shape[-2], q.shape[-1]
        N = int(np.prod(q.shape[:-2])) if q.ndim > 2 else 1
        o = np.empty_like(q)
        rc = self.lib.kb_oracle_attn_q15(q.ctypes.data_as(_I16P), k.ctypes.data_as(_I16P),
                                         v.ctypes.data_as(_I16P), o.ctypes.data_as(_I16P),
                                         N, S, d, int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"kb_oracle_attn_q15 returned {rc}")
        return o

    def q15_exp_table(self) -> np.ndarray:
        out = np.empty(64, dtype=np.uint16)
        if self.lib.kb_oracle_q15_exp_table(out.ctypes.data_as(_U16P)) != 0:
            raise ValueError("kb_oracle_q15_exp_table failed")
        return out

    def copy(self, b) -> np.ndarray:
        b = np.ascontiguousarray(np.asarray(b, dtype=np.float32))
        a = np.empty_like(b)
        if self.lib.kb_oracle_copy(a.ctypes.data_as(_FP), b.ctypes.data_as(_FP), b.size) != 0:
            raise ValueError("kb_oracle_copy failed")
        return a

    def fill(self, n: int, s: float) -> np.ndarray:
        a = np.empty(n, dtype=np.float32)
        if self.lib.kb_oracle_fill(a.ctypes.data_as(_FP), ctypes.c_float(s), n) != 0:
            raise ValueError("kb_oracle_fill failed")
        return a

    def sum(self, b) -> float:
        b = np.ascontiguousarray(np.asarray(b, dtype=np.float32))
        out = ctypes.c_double()
        if self.lib.kb_oracle_sum(b.ctypes.data_as(_FP), b.size, ctypes.byref(out)) != 0:
            raise ValueError("kb_oracle_sum failed")
        return out.value


_default: Oracle | None = None
_lock = threading.Lock()


def get() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def attn(q, k, v, causal: bool, scale: float) -> np.ndarray:
    return get().attn(q, k, v, causal, scale)


def attn_rows(q, k, v, causal: bool, scale: float, heads, rows) -> np.ndarray:
    return get().attn_rows(q, k, v, causal, scale, heads, rows)


def triad(b, c, s: float) -> np.ndarray:
    return get().triad(b, c, s)
