"""MSA index-branch block score on GB300 -- thin Python binding of the C ABI.

Every step of the computation runs in the CUDA library
``libmsa_index_score.so`` (declared in ``include/msa_index_score.h``); this
module only turns torch tensors into pointers, sizes and the current stream.
There is no CPU fallback: if the library is missing, importing the binding
raises.

The call mirrors the torch API of the reference op (guide "CANN
ops-transformer ... msa_index_score", sec. 3 "function prototype"):

    score = msa_index_score(query, key, start_loc, *, block_table=None, scale=None,
                            actual_seq_qlen, actual_seq_klen, layout_key="BBND",
                            sparse_mode=3, init_blocks=0, local_blocks=1)

``atten_mask`` is not taken: the reference uses it only for host-side
validation and the device never reads it (same guide, sec. 4).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

__all__ = [
    "msa_index_score", "msa_index_score_plan", "msa_index_score_run",
    "msa_index_score_workspace_size", "msa_index_score_out_shape", "msa_get_device_error",
    "MsaError", "library_path", "load_library", "DEVERR", "msa_index_score_noalloc",
    "noalloc_device_error",
    "msa_block_topk",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libmsa_index_score.so")

MSA_OK = 0
_STATUS_EXC = {1: ValueError, 2: NotImplementedError}
DEVERR = {0x01: "cu_seqlens_q", 0x02: "kv_len", 0x04: "cu_seqlens_k",
          0x08: "block_table", 0x10: "timeout"}
_DT = {torch.float16: 0, torch.bfloat16: 1, torch.int8: 2,
       torch.float8_e4m3fn: 3, torch.float8_e5m2: 4}
_LAYOUT = {"BBND": 0, "BNBD": 1, "TND": 2}
MSA_E2M1 = 5
FP4_FORMATS = {"mx": 0, "nv": 1}


class MsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class _SparseArgs(ctypes.Structure):
    """msa_sparse_attention_args of the C header."""
    _fields_ = [("value_cache", ctypes.c_void_p), ("selection", ctypes.c_void_p),
                ("k", ctypes.c_int32), ("sm_scale", ctypes.c_float)]


class _Args(ctypes.Structure):
    # field order and types follow msa_index_score_args in include/msa_index_score.h
    _fields_ = [
        ("query", ctypes.c_void_p), ("q_dtype", ctypes.c_int), ("T", ctypes.c_int64),
        ("H_q", ctypes.c_int32), ("D", ctypes.c_int32),
        ("key_cache", ctypes.c_void_p), ("k_dtype", ctypes.c_int), ("layout", ctypes.c_int),
        ("NP", ctypes.c_int64), ("P", ctypes.c_int32), ("H_kv", ctypes.c_int32),
        ("page_stride", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("B", ctypes.c_int32), ("MB", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.c_void_p), ("kv_len", ctypes.c_void_p),
        ("cu_seqlens_k", ctypes.c_void_p), ("start_loc", ctypes.c_void_p),
        ("scale", ctypes.c_void_p),
        ("sparse_mode", ctypes.c_int32), ("init_blocks", ctypes.c_int32),
        ("local_blocks", ctypes.c_int32), ("max_seqlen_q", ctypes.c_int32),
    ]


_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
            f"g.build()\"` (or block_score_gb300/_build.py); there is no CPU fallback")
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.POINTER(_Args)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.msa_abi_version.restype = ctypes.c_int32
    lib.msa_index_score_out_shape.argtypes = [P, ctypes.POINTER(ctypes.c_int64)]
    lib.msa_index_score_workspace_size.argtypes = [P, ctypes.POINTER(sz)]
    lib.msa_index_score.argtypes = [P, vp, vp, sz, vp]
    lib.msa_index_score_plan.argtypes = [P, vp, sz, vp]
    lib.msa_index_score_run.argtypes = [P, vp, vp, sz, vp]
    lib.msa_get_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
    lib.msa_index_score_noalloc.argtypes = [P, vp, vp]
    lib.msa_noalloc_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32), vp]
    lib.msa_block_topk.argtypes = [vp, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_int32, vp, vp]
    lib.msa_index_score_topk_workspace_size.argtypes = [P, ctypes.c_int32, ctypes.POINTER(sz)]
    lib.msa_index_score_topk.argtypes = [P, ctypes.c_int32, ctypes.c_int32, vp, vp, vp, sz, vp]
    lib.msa_index_score_fp4_workspace_size.argtypes = [P, ctypes.c_int32, ctypes.POINTER(sz)]
    lib.msa_index_score_fp4.argtypes = [P, ctypes.c_int32, vp, vp, vp, vp, sz, vp]
    lib.msa_index_score_fp4_plan.argtypes = [P, ctypes.c_int32, vp, vp, sz, vp]
    SA = ctypes.POINTER(_SparseArgs)
    lib.msa_sparse_attention_workspace_size.argtypes = [P, SA, ctypes.POINTER(sz)]
    lib.msa_sparse_attention.argtypes = [P, SA, vp, vp, vp, sz, vp]
    lib.msa_index_score_fp4_run.argtypes = [P, ctypes.c_int32, vp, vp, vp, sz, vp]
    lib.msa_set_watchdog.argtypes = [ctypes.c_uint64, ctypes.c_int32]
    lib.msa_set_watchdog.restype = ctypes.c_int
    lib.msa_status_string.restype = ctypes.c_char_p
    lib.msa_status_string.argtypes = [ctypes.c_int]
    lib.msa_last_error_message.restype = ctypes.c_char_p
    for name in ("msa_index_score_out_shape", "msa_index_score_workspace_size",
                 "msa_index_score", "msa_index_score_plan", "msa_index_score_run",
                 "msa_get_device_error", "msa_index_score_noalloc", "msa_noalloc_device_error",
                 "msa_block_topk", "msa_index_score_topk_workspace_size", "msa_index_score_topk",
                 "msa_index_score_fp4_workspace_size", "msa_index_score_fp4",
                 "msa_index_score_fp4_plan", "msa_index_score_fp4_run",
                 "msa_sparse_attention_workspace_size", "msa_sparse_attention"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status: int):
    if status == MSA_OK:
        return
    lib = load_library()
    msg = lib.msa_last_error_message().decode() or lib.msa_status_string(status).decode()
    exc = _STATUS_EXC.get(status)
    if exc is not None:
        raise exc(f"msa_index_score: {msg}")
    raise MsaError(status, f"msa_index_score: {lib.msa_status_string(status).decode()}: {msg}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _i32(t: Optional[torch.Tensor], name: str) -> Optional[torch.Tensor]:
    if t is None:
        return None
    if t.dtype != torch.int32:
        raise ValueError(f"{name} must be int32")
    return t.contiguous()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class _Call:
    """Marshalled arguments of one call (keeps the tensors alive)."""

    def __init__(self, query, key, start_loc, block_table, scale, actual_seq_qlen,
                 actual_seq_klen, layout_key, sparse_mode, init_blocks, local_blocks,
                 max_blocks, max_seqlen_q=None, fp4=None):
        layout = str(layout_key).upper()
        if layout not in _LAYOUT:
            raise ValueError(f"layout_key must be one of TND/BBND/BNBD, got {layout_key!r}")
        if query.dim() != 3:
            raise ValueError("query must be [T, H_q, D]")
        if layout == "BBND" and key.dim() == 3:
            key = key.unsqueeze(2)                     # [NP, P, D] -> [NP, P, 1, D]
        query = query.contiguous()
        if layout == "TND":
            if key.dim() != 3:
                raise ValueError("TND key must be [T2, H_kv, D]")
            if not key.is_contiguous():
                raise ValueError("TND key must be contiguous")
            NP, H_kv, D = key.shape
            P = 128
            page_stride = H_kv * D
        else:
            if key.dim() != 4:
                raise ValueError("paged key must be 4-D")
            if layout == "BBND":
                NP, P, H_kv, D = key.shape
                inner = (H_kv * D, D, 1)
            else:
                NP, H_kv, P, D = key.shape
                inner = (P * D, D, 1)
            # dim0 may be strided (pages with gaps); the inner axes must be compact
            # (axes of size 1 do not take part in addressing)
            for ax, want in zip(range(1, 4), inner):
                if key.shape[ax] != 1 and key.stride(ax) != want:
                    raise ValueError("paged key: only dim0 may be non-contiguous")
            page_stride = key.stride(0)
        self.query, self.key = query, key
        self.cu_q = _i32(actual_seq_qlen, "actual_seq_qlen")
        if self.cu_q is None:
            raise ValueError("actual_seq_qlen (cu_seqlens_q, [B+1]) is required")
        B = self.cu_q.shape[0] - 1
        klen = _i32(actual_seq_klen, "actual_seq_klen")
        if klen is None:
            raise ValueError("actual_seq_klen is required")
        self.start_loc = _i32(start_loc, "start_loc")
        self.scale = None if scale is None else scale.contiguous()
        if self.scale is not None and self.scale.dtype != torch.float32:
            raise ValueError("scale must be float32")
        # the kernels dereference every array on the query's device
        for name, t in (("key", key), ("start_loc", self.start_loc), ("block_table", block_table),
                        ("scale", self.scale), ("actual_seq_qlen", self.cu_q),
                        ("actual_seq_klen", klen)):
            if t is not None and t.device != query.device:
                raise ValueError(f"{name} is on {t.device}, the query on {query.device}: "
                                 "all arrays must be on one device")
        if layout == "TND":
            self.block_table, self.kv_len, self.cu_k = None, None, klen
            if max_blocks is None:
                lens = (klen[1:] - klen[:-1]).to(torch.int64)
                nb = int(((lens + P - 1) // P).max().item()) if B > 0 else 1
                max_blocks = max(1, nb)
            MB = int(max_blocks)
        else:
            if block_table is None:
                raise ValueError("block_table is required for paged layouts")
            self.block_table = _i32(block_table, "block_table")
            self.kv_len, self.cu_k = klen, None
            MB = int(self.block_table.shape[1])
        a = _Args()
        if fp4 is not None and (query.dtype != torch.uint8 or key.dtype != torch.uint8):
            raise ValueError("FP4 query and key are uint8 tensors of packed E2M1 codes")
        a.query = _ptr(query)
        a.q_dtype = MSA_E2M1 if fp4 is not None else _DT.get(query.dtype, -1)
        a.T = int(query.shape[0])
        a.H_q = int(query.shape[1])
        a.D = int(query.shape[2]) * (2 if fp4 is not None else 1)   # FP4: two codes per byte
        a.key_cache = _ptr(key)
        a.k_dtype = MSA_E2M1 if fp4 is not None else _DT.get(key.dtype, -1)
        a.layout = _LAYOUT[layout]
        a.NP = int(NP)
        a.P = int(P)
        a.H_kv = int(H_kv)
        a.page_stride = int(page_stride)
        a.block_table = _ptr(self.block_table)
        a.B = int(B)
        a.MB = int(MB)
        a.cu_seqlens_q = _ptr(self.cu_q)
        a.kv_len = _ptr(self.kv_len)
        a.cu_seqlens_k = _ptr(self.cu_k)
        a.start_loc = _ptr(self.start_loc)
        a.scale = _ptr(self.scale)
        a.sparse_mode = int(sparse_mode)
        a.init_blocks = int(init_blocks)
        a.local_blocks = int(local_blocks)
        a.max_seqlen_q = 0 if max_seqlen_q is None else int(max_seqlen_q)
        self.args = a
        self.device = query.device

    def out_shape(self) -> Tuple[int, int, int]:
        shape = (ctypes.c_int64 * 3)()
        _check(load_library().msa_index_score_out_shape(ctypes.byref(self.args), shape))
        return tuple(int(x) for x in shape)

    def workspace_bytes(self) -> int:
        n = ctypes.c_size_t()
        _check(load_library().msa_index_score_workspace_size(ctypes.byref(self.args),
                                                             ctypes.byref(n)))
        return int(n.value)


def _prepare(query, key, start_loc, block_table, scale, actual_seq_qlen, actual_seq_klen,
             layout_key, sparse_mode, init_blocks, local_blocks, max_blocks,
             max_seqlen_q=None, fp4=None) -> _Call:
    return _Call(query, key, start_loc, block_table, scale, actual_seq_qlen, actual_seq_klen,
                 layout_key, sparse_mode, init_blocks, local_blocks, max_blocks, max_seqlen_q,
                 fp4)


def msa_index_score(query: torch.Tensor, key: torch.Tensor, start_loc: torch.Tensor, *,
                    block_table: Optional[torch.Tensor] = None,
                    scale: Optional[torch.Tensor] = None,
                    actual_seq_qlen: Optional[torch.Tensor] = None,
                    actual_seq_klen: Optional[torch.Tensor] = None,
                    layout_key: str = "BBND", sparse_mode: int = 3, init_blocks: int = 0,
                    local_blocks: int = 1, max_blocks: Optional[int] = None,
                    max_seqlen_q: Optional[int] = None,
                    out: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Block scores ``[H_q, T, RoundUp(MB, 16)]`` fp32 on the query's device.

    ``actual_seq_qlen`` is the [B+1] prefix sum of query lengths;
    ``actual_seq_klen`` is [B] kv lengths for BBND/BNBD and the [B+1] prefix
    sum for TND.  ``max_blocks`` is MB for TND (computed from actual_seq_klen
    when omitted, which reads it on the host).  ``max_seqlen_q`` is an optional
    host-known bound on every request's query length (an addition of this
    library: with int8 keys and short requests only, it saves a kernel launch).
    """
    c = _prepare(query, key, start_loc, block_table, scale, actual_seq_qlen, actual_seq_klen,
                 layout_key, sparse_mode, init_blocks, local_blocks, max_blocks, max_seqlen_q)
    if not query.is_cuda:
        raise ValueError("msa_index_score runs on CUDA tensors only")
    shape = c.out_shape()
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=query.device)
    elif tuple(out.shape) != shape or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous float32 tensor of shape {shape}")
    ws_bytes = c.workspace_bytes()
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=query.device)
    elif workspace.numel() * workspace.element_size() < ws_bytes:
        raise ValueError(f"workspace needs {ws_bytes} bytes")
    _check(load_library().msa_index_score(ctypes.byref(c.args), out.data_ptr(),
                                          workspace.data_ptr(), ws_bytes,
                                          _stream_handle(stream)))
    return out


def msa_index_score_noalloc(prepared: "Prepared", out: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """Same scores as ``msa_index_score`` without a caller workspace.

    For callers that cannot allocate device memory on their hot path: the
    library keeps the plan scratch in a fixed array of its own (at most 1024
    requests).  Calls that overlap on the GPU share that array and race, so
    keep them on one stream.  ``out`` defaults to ``prepared.out``.
    """
    shape = tuple(prepared.shape)
    out = prepared.out if out is None else out
    if (tuple(out.shape) != shape or out.dtype != torch.float32 or not out.is_contiguous()
            or not out.is_cuda):
        raise ValueError(f"out must be a contiguous float32 CUDA tensor of shape {shape}")
    _check(load_library().msa_index_score_noalloc(ctypes.byref(prepared.call.args),
                                                  out.data_ptr(), _stream_handle(stream)))
    return out


def noalloc_device_error(stream=None) -> int:
    """Device error bits left by the last ``msa_index_score_noalloc`` call on
    the current device (synchronises ``stream``; 0 = clean)."""
    bits = ctypes.c_int32(0)
    _check(load_library().msa_noalloc_device_error(ctypes.byref(bits), _stream_handle(stream)))
    return int(bits.value)


def msa_block_topk(score: torch.Tensor, k: int = 16, MB: Optional[int] = None,
                   out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Top-k blocks of every score row: int32 ``[T, H, k]``, block indices ascending, -1 tail.

    ``score`` is a contiguous fp32 CUDA tensor ``[H, T, MBp]`` (msa_index_score's
    output); ``MB`` is the number of valid columns (default: all ``MBp``).
    """
    if not score.is_cuda or score.dtype != torch.float32 or score.dim() != 3:
        raise ValueError("score must be a float32 CUDA tensor [H, T, MBp]")
    score = score.contiguous()
    H, T, MBp = score.shape
    MB = MBp if MB is None else int(MB)
    shape = (T, H, int(k))
    if out is None:
        out = torch.empty(shape, dtype=torch.int32, device=score.device)
    elif tuple(out.shape) != shape or out.dtype != torch.int32 or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous int32 tensor of shape {shape}")
    _check(load_library().msa_block_topk(score.data_ptr(), H, T, MBp, MB, int(k), out.data_ptr(),
                                         _stream_handle(stream)))
    return out


def msa_index_score_out_shape(query, key, start_loc, **kw) -> Tuple[int, int, int]:
    kw = dict(kw)
    return _prepare(query, key, start_loc, kw.pop("block_table", None), kw.pop("scale", None),
                    kw.pop("actual_seq_qlen", None), kw.pop("actual_seq_klen", None),
                    kw.pop("layout_key", "BBND"), kw.pop("sparse_mode", 3),
                    kw.pop("init_blocks", 0), kw.pop("local_blocks", 1),
                    kw.pop("max_blocks", None)).out_shape()


def msa_index_score_workspace_size(query, key, start_loc, **kw) -> int:
    kw = dict(kw)
    return _prepare(query, key, start_loc, kw.pop("block_table", None), kw.pop("scale", None),
                    kw.pop("actual_seq_qlen", None), kw.pop("actual_seq_klen", None),
                    kw.pop("layout_key", "BBND"), kw.pop("sparse_mode", 3),
                    kw.pop("init_blocks", 0), kw.pop("local_blocks", 1),
                    kw.pop("max_blocks", None)).workspace_bytes()


class Prepared:
    """Arguments marshalled once, for repeated plan/run calls (benchmarks).

    FP4 inputs: ``fp4="mx"`` or ``"nv"`` with uint8 ``query`` / ``key`` of
    packed E2M1 codes and the group scale bytes ``q_scale`` / ``k_scale``
    (see ``msa_index_score_fp4`` in the C header); the call then goes through
    the FP4 entry point."""

    def __init__(self, query, key, start_loc, **kw):
        kw = dict(kw)
        fp4 = kw.pop("fp4", None)
        q_scale, k_scale = kw.pop("q_scale", None), kw.pop("k_scale", None)
        if fp4 is not None and fp4 not in FP4_FORMATS:
            raise ValueError(f"fp4 must be one of {sorted(FP4_FORMATS)}")
        self.call = _prepare(query, key, start_loc, kw.pop("block_table", None),
                             kw.pop("scale", None), kw.pop("actual_seq_qlen", None),
                             kw.pop("actual_seq_klen", None), kw.pop("layout_key", "BBND"),
                             kw.pop("sparse_mode", 3), kw.pop("init_blocks", 0),
                             kw.pop("local_blocks", 1), kw.pop("max_blocks", None),
                             kw.pop("max_seqlen_q", None), fp4)
        if kw:
            raise TypeError(f"unknown arguments {sorted(kw)}")
        self.fp4 = fp4
        if fp4 is not None:
            if q_scale is None or k_scale is None:
                raise ValueError("FP4 inputs need q_scale and k_scale")
            if q_scale.dtype != torch.uint8 or k_scale.dtype != torch.uint8:
                raise ValueError("q_scale and k_scale are uint8 scale bytes")
            if q_scale.device != query.device or k_scale.device != query.device:
                raise ValueError("q_scale and k_scale must be on the query's device")
            self.q_scale, self.k_scale = q_scale.contiguous(), k_scale.contiguous()
        self.shape = self.call.out_shape()
        if fp4 is not None:
            n = ctypes.c_size_t()
            _check(load_library().msa_index_score_fp4_workspace_size(
                ctypes.byref(self.call.args), FP4_FORMATS[fp4], ctypes.byref(n)))
            self.ws_bytes = int(n.value)
        else:
            self.ws_bytes = self.call.workspace_bytes()
        dev = query.device
        self.out = torch.empty(self.shape, dtype=torch.float32, device=dev)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)

    def __call__(self, stream=None) -> torch.Tensor:
        if self.fp4 is not None:
            _check(load_library().msa_index_score_fp4(
                ctypes.byref(self.call.args), FP4_FORMATS[self.fp4], self.q_scale.data_ptr(),
                self.k_scale.data_ptr(), self.out.data_ptr(), self.workspace.data_ptr(),
                self.ws_bytes, _stream_handle(stream)))
            return self.out
        _check(load_library().msa_index_score(ctypes.byref(self.call.args), self.out.data_ptr(),
                                              self.workspace.data_ptr(), self.ws_bytes,
                                              _stream_handle(stream)))
        return self.out

    def plan(self, stream=None):
        if self.fp4 is not None:
            _check(load_library().msa_index_score_fp4_plan(
                ctypes.byref(self.call.args), FP4_FORMATS[self.fp4], self.q_scale.data_ptr(),
                self.workspace.data_ptr(), self.ws_bytes, _stream_handle(stream)))
            return
        _check(load_library().msa_index_score_plan(ctypes.byref(self.call.args),
                                                   self.workspace.data_ptr(), self.ws_bytes,
                                                   _stream_handle(stream)))

    def run(self, stream=None) -> torch.Tensor:
        if self.fp4 is not None:
            _check(load_library().msa_index_score_fp4_run(
                ctypes.byref(self.call.args), FP4_FORMATS[self.fp4], self.k_scale.data_ptr(),
                self.out.data_ptr(), self.workspace.data_ptr(), self.ws_bytes,
                _stream_handle(stream)))
            return self.out
        _check(load_library().msa_index_score_run(ctypes.byref(self.call.args),
                                                  self.out.data_ptr(), self.workspace.data_ptr(),
                                                  self.ws_bytes, _stream_handle(stream)))
        return self.out

    def device_error(self, stream=None) -> int:
        return msa_get_device_error(self.workspace, stream)

    def select_workspace_bytes(self, k: int) -> int:
        n = ctypes.c_size_t()
        _check(load_library().msa_index_score_topk_workspace_size(ctypes.byref(self.call.args),
                                                                  int(k), ctypes.byref(n)))
        return int(n.value)

    def topk(self, k: int = 16, local_slot: bool = True, scores: bool = True,
             indices: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
             stream=None) -> torch.Tensor:
        """Scores (into ``self.out`` when ``scores``) and the fused per-GQA-group
        selection: int32 ``[T, H_kv, k]``, ascending block indices, -1 tail.

        ``local_slot``: each query token's own block always takes a slot.
        ``workspace`` (optional) is reused across calls when given; it must hold
        ``select_workspace_bytes(k)`` bytes."""
        T, H_kv = int(self.call.args.T), int(self.call.args.H_kv)
        shape = (T, H_kv, int(k))
        if indices is None:
            indices = torch.empty(shape, dtype=torch.int32, device=self.out.device)
        elif tuple(indices.shape) != shape or indices.dtype != torch.int32 or not indices.is_contiguous():
            raise ValueError(f"indices must be a contiguous int32 tensor of shape {shape}")
        nbytes = self.select_workspace_bytes(k)
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.out.device)
        elif workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace needs {nbytes} bytes")
        self.select_workspace = workspace
        _check(load_library().msa_index_score_topk(
            ctypes.byref(self.call.args), int(k), 1 if local_slot else 0,
            self.out.data_ptr() if scores else None, indices.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(stream)))
        return indices

    def sparse_attention(self, value: torch.Tensor, selection: torch.Tensor,
                         sm_scale: float = 0.0, out: Optional[torch.Tensor] = None,
                         lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                         stream=None):
        """The sparse main branch over the selected blocks (see
        ``msa_sparse_attention`` in the C header): this object's query and key
        cache are the main branch's; ``value`` has the key cache's layout,
        shape, dtype and strides; ``selection`` is int32 ``[T, H_kv, k]``.
        Returns ``(out [T, H_q, D] fp32, lse [T, H_q] fp32)``."""
        key = self.call.key
        T, H_q = int(self.call.args.T), int(self.call.args.H_q)
        H_kv, D = int(self.call.args.H_kv), int(self.call.args.D)
        # every array the kernels index must have the shape they index it with
        if (selection.dtype != torch.int32 or selection.dim() != 3 or not selection.is_contiguous()
                or tuple(selection.shape[:2]) != (T, H_kv)):
            raise ValueError(f"selection must be a contiguous int32 tensor [T, H_kv, k] = "
                             f"[{T}, {H_kv}, k]")
        for name, t, shape in (("out", out, (T, H_q, D)), ("lse", lse, (T, H_q))):
            if t is not None and (tuple(t.shape) != shape or t.dtype != torch.float32
                                  or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous float32 tensor of shape {shape}")
        if (tuple(value.shape) != tuple(key.shape) or value.stride() != key.stride()
                or value.dtype != key.dtype or not value.is_cuda):
            raise ValueError("value must match the key cache's shape, strides and dtype")
        for name, t in (("selection", selection), ("out", out), ("lse", lse)):
            if t is not None and t.device != value.device:
                raise ValueError(f"{name} must be on the value cache's device {value.device}")
        sa = _SparseArgs()
        sa.value_cache = value.data_ptr()
        sa.selection = selection.data_ptr()
        sa.k = int(selection.shape[2])
        sa.sm_scale = float(sm_scale)
        n = ctypes.c_size_t()
        _check(load_library().msa_sparse_attention_workspace_size(
            ctypes.byref(self.call.args), ctypes.byref(sa), ctypes.byref(n)))
        if workspace is None or workspace.numel() * workspace.element_size() < n.value:
            workspace = torch.empty(n.value, dtype=torch.uint8, device=value.device)
        self.sparse_workspace = workspace
        if out is None:
            out = torch.empty((T, H_q, D), dtype=torch.float32, device=value.device)
        if lse is None:
            lse = torch.empty((T, H_q), dtype=torch.float32, device=value.device)
        _check(load_library().msa_sparse_attention(
            ctypes.byref(self.call.args), ctypes.byref(sa), out.data_ptr(), lse.data_ptr(),
            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            _stream_handle(stream)))
        return out, lse

    def sparse_device_error(self, stream=None) -> int:
        """Device error bits of the last ``sparse_attention`` call."""
        return msa_get_device_error(self.sparse_workspace, stream)

    def select_device_error(self, stream=None) -> int:
        """Device error bits of the last ``topk`` call (its workspace holds them)."""
        return msa_get_device_error(self.select_workspace, stream)


def msa_index_score_plan(prepared: Prepared, stream=None):
    prepared.plan(stream)


def msa_index_score_run(prepared: Prepared, stream=None) -> torch.Tensor:
    return prepared.run(stream)


def msa_get_device_error(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return the device error bits of the last call."""
    v = ctypes.c_int32()
    _check(load_library().msa_get_device_error(workspace.data_ptr(), ctypes.byref(v),
                                               _stream_handle(stream)))
    return int(v.value)


def from_case(case, device, max_seqlen_q: Optional[int] = None) -> Prepared:
    """Move a synthetic case (``synth.MsaCase``) to ``device`` and marshal it.

    ``max_seqlen_q`` is passed through as the host-side length bound (None: not
    given)."""
    def mv(t):
        return None if t is None else t.to(device)
    key = case.key
    if case.layout != "TND" and not key.is_contiguous():
        # keep the dim0 gap: move the backing storage, then view it the same way
        base = key
        while base._base is not None:
            base = base._base
        base_dev = base.to(device)
        key_dev = torch.as_strided(base_dev, key.shape, key.stride(), key.storage_offset())
    else:
        key_dev = key.to(device)
    klen = case.cu_seqlens_k if case.layout == "TND" else case.kv_len
    fp4 = {}
    if getattr(case, "fp4", None):
        fp4 = dict(fp4=case.fp4, q_scale=mv(case.q_scale), k_scale=mv(case.k_scale))
    return Prepared(case.query.to(device), key_dev, mv(case.start_loc), **fp4,
                    block_table=mv(case.block_table), scale=mv(case.scale),
                    actual_seq_qlen=mv(case.cu_seqlens_q), actual_seq_klen=mv(klen),
                    layout_key=case.layout, sparse_mode=case.sparse_mode,
                    init_blocks=case.init_blocks, local_blocks=case.local_blocks,
                    max_blocks=case.MB if case.layout == "TND" else None,
                    max_seqlen_q=max_seqlen_q)
