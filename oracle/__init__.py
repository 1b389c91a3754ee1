"""CPU oracle for the MSA index-branch block score -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``block_score_gb300``) never imports it and shares no code with it.

Two independent formulations live here:

* ``msa_oracle.c`` (wrapped by :func:`oracle_full` / :func:`oracle_rows`):
  the per-block formula of the feature request "MsaIndexScore"
  (gitcode.com/cann/ops-transformer/issues/4117, section "calculation"),
  in plain C with fp64 accumulation and one final rounding to fp32.
* :mod:`oracle.bruteforce`: the mask-then-block-max definition of the
  "DSA / GQA forward" notes (section 3, "from token score to block
  selection"): a dense masked token-score matrix reshaped into blocks and
  reduced with ``amax``.  It exists to pin the C oracle.

Parity pins: see ``tests/test_oracle_pins.py``.  No function here is
"parity unpinned" except the two conventions the pages leave open (the
local-mask scope for rows with no visible key and the exact fill constant),
which the tests pin as chosen readings.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_LIB = os.path.join(_HERE, "libmsa_oracle.so")
_lock = threading.Lock()
_lib = None

_DT = {torch.float16: 0, torch.bfloat16: 1, torch.int8: 2,
       torch.float8_e4m3fn: 3, torch.float8_e5m2: 4}
_LAYOUT = {"BBND": 0, "BNBD": 1, "TND": 2}


class _Args(ctypes.Structure):
    _fields_ = [
        ("query", ctypes.c_void_p), ("q_dtype", ctypes.c_int32), ("T", ctypes.c_int64),
        ("H_q", ctypes.c_int32), ("D", ctypes.c_int32),
        ("key", ctypes.c_void_p), ("k_dtype", ctypes.c_int32), ("layout", ctypes.c_int32),
        ("NP", ctypes.c_int64), ("P", ctypes.c_int32), ("H_kv", ctypes.c_int32),
        ("page_stride", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("B", ctypes.c_int32), ("MB", ctypes.c_int32),
        ("cu_q", ctypes.c_void_p), ("kv_len", ctypes.c_void_p), ("cu_k", ctypes.c_void_p),
        ("start_loc", ctypes.c_void_p), ("scale", ctypes.c_void_p),
        ("sparse_mode", ctypes.c_int32), ("init_blocks", ctypes.c_int32),
        ("local_blocks", ctypes.c_int32), ("fill_value", ctypes.c_float),
        ("q_scale", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
        ("fp4_format", ctypes.c_int32),
    ]

_FP4_FORMAT = {"mx": 0, "nv": 1}


def build(force: bool = False) -> str:
    """Compile ``msa_oracle.c`` into ``libmsa_oracle.so`` (gcc, OpenMP)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.msa_oracle_rows.argtypes = [ctypes.POINTER(_Args), ctypes.c_void_p,
                                        ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        lib.msa_oracle_rows.restype = ctypes.c_int
        lib.msa_oracle_full.argtypes = [ctypes.POINTER(_Args), ctypes.c_void_p, ctypes.c_int]
        lib.msa_oracle_full.restype = ctypes.c_int
        lib.msa_oracle_threads.argtypes = [ctypes.c_int]
        lib.msa_oracle_threads.restype = ctypes.c_int
        lib.msa_oracle_decode.argtypes = [ctypes.c_int32, ctypes.c_uint32]
        lib.msa_oracle_decode.restype = ctypes.c_double
        _lib = lib
    return _lib


def _cpu(x: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    if x is None:
        return None
    return x.detach().cpu()


def _make_args(case, fill_value: float, keep: list) -> _Args:
    q = _cpu(case.query).contiguous()
    k = _cpu(case.key)
    layout = case.layout.upper()
    if layout == "TND":
        k = k.contiguous()
        page_stride = int(k.shape[1] * k.shape[2])
    else:
        # inner three dims must be compact; dim0 may carry a gap
        inner = k.shape[1] * k.shape[2] * k.shape[3]
        want = (k.shape[2] * k.shape[3], k.shape[3], 1)
        if tuple(k.stride()[1:]) != want or k.stride(0) < inner:
            k = k.contiguous()
        page_stride = int(k.stride(0))
    keep += [q, k]
    a = _Args()
    fp4 = getattr(case, "fp4", None)
    a.query = q.data_ptr()
    a.q_dtype = 5 if fp4 else _DT[q.dtype]
    a.T = int(q.shape[0])
    a.H_q = int(q.shape[1])
    a.D = int(q.shape[2]) * (2 if fp4 else 1)      # FP4: two elements per byte
    a.key = k.data_ptr()
    a.k_dtype = 5 if fp4 else _DT[k.dtype]
    a.layout = _LAYOUT[layout]
    a.NP = int(k.shape[0])
    if layout == "BBND":
        a.P, a.H_kv = int(k.shape[1]), int(k.shape[2])
    elif layout == "BNBD":
        a.H_kv, a.P = int(k.shape[1]), int(k.shape[2])
    else:
        a.P, a.H_kv = int(case.P), int(k.shape[1])
    a.page_stride = page_stride

    def ptr(t, dtype):
        if t is None:
            return None
        t = _cpu(t).to(dtype).contiguous()
        keep.append(t)
        return t.data_ptr()

    a.block_table = ptr(case.block_table, torch.int32)
    a.B = int(case.cu_seqlens_q.shape[0]) - 1
    a.MB = int(case.MB)
    a.cu_q = ptr(case.cu_seqlens_q, torch.int32)
    a.kv_len = ptr(case.kv_len, torch.int32)
    a.cu_k = ptr(case.cu_seqlens_k, torch.int32)
    a.start_loc = ptr(case.start_loc, torch.int32)
    a.scale = ptr(case.scale, torch.float32)
    a.sparse_mode = int(case.sparse_mode)
    a.init_blocks = int(case.init_blocks)
    a.local_blocks = int(case.local_blocks)
    a.fill_value = float(fill_value)
    if fp4:
        a.q_scale = ptr(case.q_scale, torch.uint8)
        a.k_scale = ptr(case.k_scale, torch.uint8)
        a.fp4_format = _FP4_FORMAT[fp4]
    return a


def oracle_full(case, nthreads: int = 0, fill_value: float = float("-inf")) -> torch.Tensor:
    """Whole output ``[H_q, T, RoundUp(MB,16)]`` as a float32 CPU tensor."""
    lib = _load()
    keep: list = []
    a = _make_args(case, fill_value, keep)
    MBp = (int(case.MB) + 15) // 16 * 16
    out = torch.empty((a.H_q, a.T, MBp), dtype=torch.float32)
    if a.T > 0:
        nbad = lib.msa_oracle_full(ctypes.byref(a), out.data_ptr(), int(nthreads))
        if nbad:
            raise ValueError(f"oracle: {nbad} rows read an out-of-range table entry")
    return out


def oracle_rows(case, rows: Sequence[int], nthreads: int = 0,
                fill_value: float = float("-inf")) -> torch.Tensor:
    """Selected output rows; ``rows[i] = h * T + t``.  Returns ``[len(rows), MBp]``."""
    lib = _load()
    keep: list = []
    a = _make_args(case, fill_value, keep)
    MBp = (int(case.MB) + 15) // 16 * 16
    r = torch.as_tensor(np.asarray(rows, dtype=np.int64))
    out = torch.empty((len(r), MBp), dtype=torch.float32)
    if len(r):
        nbad = lib.msa_oracle_rows(ctypes.byref(a), r.data_ptr(), len(r), out.data_ptr(),
                                   int(nthreads))
        if nbad:
            raise ValueError(f"oracle: {nbad} rows read an out-of-range table entry")
    return out


def decode(dtype, bits: int) -> float:
    """The oracle's decoding of one element bit pattern of ``dtype`` (a torch
    dtype, or "e2m1" for an FP4 code / "e8m0" for an MX scale byte)."""
    code = {"e2m1": 5, "e8m0": 6}.get(dtype) if isinstance(dtype, str) else _DT[dtype]
    return float(_load().msa_oracle_decode(code, bits))


def oracle_threads(nthreads: int = 0) -> int:
    """Threads the oracle's parallel region actually runs with."""
    return int(_load().msa_oracle_threads(int(nthreads)))
