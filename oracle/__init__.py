"""fp64 CPU oracle for exact scaled dot-product attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. It shares no code with the CUDA library: the
arithmetic lives in ``attn_oracle.c`` (plain C, fp64), and this module only
compiles it with gcc and marshals numpy arrays into it.

What it computes is stated in the header of ``attn_oracle.c``: the plain
definition O = softmax(scale * Q K^T + mask) V row by row, with the two-pass
(max, normaliser, divide) softmax of "Tensor Parallelism with CUDA - Standard
Attention", section "Step 2: Softmax", and the logsumexp of each row.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "libattn_oracle.so")
_default = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle source into a shared library (skipped when up to date)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """ctypes handle on one compiled copy of the oracle."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_attn.restype = ctypes.c_int
        lib.oracle_attn.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_double, ctypes.c_int, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
        ]
        lib.oracle_attn_ex.restype = ctypes.c_int
        lib.oracle_attn_ex.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
        ]
        self._lib = lib

    def half_to_double(self, bits: int) -> float:
        """Decode one binary16 bit pattern with the oracle's own decoder."""
        return self._lib.oracle_half_to_double(bits)

    def bf16_to_double(self, bits: int) -> float:
        """Decode one bfloat16 bit pattern with the oracle's own decoder."""
        return self._lib.oracle_bf16_to_double(bits)

    def attn(self, q, k, v, *, sm_scale: float, causal: bool = False, key_lengths=None,
             rows=None, threads: int | None = None, dtype: str = "f16"):
        """Oracle forward.

        dtype "f16": q, k, v are numpy float16 arrays; "bf16": numpy uint16 (or int16) arrays
        of bfloat16 bit patterns; "f32": numpy float32 arrays.
        q: [B, H, N, d] (N query rows per head); k, v: [B, Hkv, Nk, d]
        with H a multiple of Hkv (query head h reads key/value head h // (H // Hkv)).
        Self-attention is k, v of q's shape. With causal and Nk != N, query i sees
        keys j <= i + Nk - N.
        key_lengths: int array [B] or None. rows: ascending flat row ids
        ((b*H + h)*N + i) or None for every row.
        Returns (o, lse) as float64: o is [B,H,N,d] (or [len(rows), d]), lse is
        [B,H,N] (or [len(rows)]).
        """
        if dtype == "f16":
            code = 0
            q, k, v = (np.ascontiguousarray(x, dtype=np.float16) for x in (q, k, v))
        elif dtype == "bf16":
            code = 1
            for x in (q, k, v):
                if np.asarray(x).dtype not in (np.uint16, np.int16):
                    raise TypeError("bf16 inputs are uint16/int16 arrays of bit patterns")
            q, k, v = (np.ascontiguousarray(x).view(np.uint16) for x in (q, k, v))
        elif dtype == "f32":
            code = 2
            q, k, v = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v))
        else:
            raise ValueError("dtype must be 'f16', 'bf16' or 'f32'")
        if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape:
            raise ValueError("q must be [B,H,N,d] and k, v one [B,Hkv,Nk,d] shape")
        B, H, N, d = q.shape
        Hkv, Nk = k.shape[1], k.shape[2]
        if k.shape[0] != B or k.shape[3] != d or Hkv < 1 or H % Hkv != 0:
            raise ValueError("k, v must be [B,Hkv,Nk,d] with H a multiple of Hkv")
        kl = None
        if key_lengths is not None:
            kl = np.ascontiguousarray(key_lengths, dtype=np.int32)
            if kl.shape != (B,):
                raise ValueError("key_lengths must have shape [B]")
        if rows is None:
            n_rows = B * H * N
            o = np.empty((B, H, N, d), np.float64)
            lse = np.empty((B, H, N), np.float64)
            rows_arr = None
        else:
            rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
            n_rows = rows_arr.size
            o = np.empty((n_rows, d), np.float64)
            lse = np.empty((n_rows,), np.float64)
        rc = self._lib.oracle_attn_ex(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, Hkv, N, Nk, d, code, float(sm_scale),
            int(bool(causal)), None if kl is None else kl.ctypes.data,
            None if rows_arr is None else rows_arr.ctypes.data, n_rows,
            o.ctypes.data, lse.ctypes.data, int(threads or default_threads()))
        if rc != 0:
            raise RuntimeError(f"oracle_attn_ex failed with code {rc}")
        return o, lse


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def half_to_double(bits: int) -> float:
    return default().half_to_double(bits)


def attn(q, k, v, **kw):
    """Oracle forward with the default build; see ``Oracle.attn``."""
    return default().attn(q, k, v, **kw)
