"""Python binding of libattn.so (argument marshalling only).

Every step of the attention path runs in the library's CUDA kernels; this
module converts torch tensors into the pointers, sizes and cache
descriptors that the C ABI (include/attn_decode.h) takes, and turns
non-zero status codes into exceptions.  PyTorch supplies device memory
(including the split-K workspace) and the current stream.  There is no CPU
fallback: if libattn.so has not been built, importing the library fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_WORKSPACE = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_DEVICE = 5
ATTN_MAX_PARTITIONS = 1024
ATTN_PARTITIONS_BALANCED = -1   # the balanced MLA split (planner request; num_partitions 0)
ATTN_PARTITIONS_TILE_PAIR = -2  # the tile path with two Q tiles per CTA pair

_STATUS_NAMES = {
    ATTN_ERR_INVALID_ARG: "ATTN_ERR_INVALID_ARG",
    ATTN_ERR_UNSUPPORTED: "ATTN_ERR_UNSUPPORTED",
    ATTN_ERR_WORKSPACE: "ATTN_ERR_WORKSPACE",
    ATTN_ERR_CUDA: "ATTN_ERR_CUDA",
    ATTN_ERR_DEVICE: "ATTN_ERR_DEVICE",
}


class AttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {_STATUS_NAMES.get(status, status)}")
        self.status = status


class attn_kv_t(ctypes.Structure):
    _fields_ = [
        ("base", ctypes.c_void_p),
        ("page_stride", ctypes.c_int64),
        ("token_stride", ctypes.c_int64),
        ("head_stride", ctypes.c_int64),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("page_table", ctypes.c_void_p),
        ("max_pages", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


_c = ctypes
_SIGNATURES = {
    "attn_plan_partitions": [_c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,
                             _c.c_int, _c.c_int, _c.c_int, _c.POINTER(_c.c_int),
                             _c.POINTER(_c.c_size_t)],
    "attn_decode": [_c.c_void_p, _c.POINTER(attn_kv_t), _c.POINTER(attn_kv_t), _c.c_void_p,
                    _c.c_void_p, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,
                    _c.c_int, _c.c_float, _c.c_void_p, _c.c_int, _c.c_int, _c.c_void_p,
                    _c.c_size_t, _c.c_void_p, _c.c_void_p, _c.c_void_p],
    "attn_mla_decode": [_c.c_void_p, _c.POINTER(attn_kv_t), _c.c_void_p, _c.c_int, _c.c_int,
                        _c.c_int, _c.c_int, _c.c_int, _c.c_float, _c.c_void_p, _c.c_int,
                        _c.c_void_p, _c.c_size_t, _c.c_void_p, _c.c_void_p, _c.c_void_p],
    "attn_mla_decode_rows": [_c.c_void_p, _c.POINTER(attn_kv_t), _c.c_void_p, _c.c_void_p,
                             _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,
                             _c.c_float, _c.c_void_p, _c.c_int, _c.c_int, _c.c_void_p,
                             _c.c_size_t, _c.c_void_p, _c.c_void_p, _c.c_void_p],
    "attn_mla_decode_sparse": [_c.c_void_p, _c.POINTER(attn_kv_t), _c.c_void_p, _c.c_int,
                               _c.c_void_p, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_float,
                               _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_size_t, _c.c_void_p,
                               _c.c_void_p, _c.c_void_p],
    "attn_splitk_reduce": [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_int, _c.c_int,
                           _c.c_int, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p],
    "attn_device_error_flags": [_c.POINTER(_c.c_uint), _c.c_int],
    "attn_selftest_wait_timeout": [_c.c_void_p],
    "attn_decode_noalloc": [_c.c_void_p, _c.POINTER(attn_kv_t), _c.POINTER(attn_kv_t),
                            _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_int, _c.c_int, _c.c_int,
                            _c.c_int, _c.c_int, _c.c_int, _c.c_float, _c.c_void_p, _c.c_int,
                            _c.c_int, _c.c_void_p, _c.c_void_p, _c.c_void_p],
}

_lib = None


def lib():
    """The loaded libattn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "split_flash_decoding_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, argtypes in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = argtypes
            fn.restype = ctypes.c_int
        _lib = handle
    return _lib


def _check(fn: str, status: int):
    if status != ATTN_OK:
        raise AttnError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


# ---------------------------------------------------------------------------
# cache descriptors
# ---------------------------------------------------------------------------

def kv_descriptor(cache: torch.Tensor, page_table: Optional[torch.Tensor] = None) -> attn_kv_t:
    """Describe a bf16 cache tensor for the C ABI.

    Paged: cache [num_pages, page_size, num_kv_heads, dim] with page_table
    int32 [batch, max_pages].  Contiguous: cache [batch, capacity,
    num_kv_heads, dim] and page_table None.  The last dimension must be
    contiguous; other strides are taken from the tensor.
    """
    if cache.dtype != torch.bfloat16:
        raise TypeError("cache must be bf16")
    if cache.dim() != 4 or cache.stride(3) != 1:
        raise ValueError("cache must be 4-D with contiguous channels")
    d = attn_kv_t()
    d.base = cache.data_ptr()
    d.page_stride = cache.stride(0)
    d.token_stride = cache.stride(1)
    d.head_stride = cache.stride(2)
    d.page_size = cache.shape[1]
    d.num_pages = cache.shape[0]
    if page_table is not None:
        if page_table.dtype != torch.int32 or page_table.dim() != 2 or not page_table.is_contiguous():
            raise ValueError("page_table must be a contiguous int32 [batch, max_pages] tensor")
        d.page_table = page_table.data_ptr()
        d.max_pages = page_table.shape[1]
    else:
        d.page_table = None
        d.max_pages = 0
    d.reserved = 0
    return d


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def attn_plan_partitions(batch: int, num_q_rows: int, num_q_heads: int, num_kv_heads: int,
                         head_dim_v: int, max_kv_len: int, requested: int = 0,
                         num_sms: int = 0, max_q_len: int = 1):
    """Returns (num_partitions, workspace_bytes).  max_q_len (rows of the
    longest sequence) lets the library route a multi-row GQA call: the
    few-row fold keeps split-K, longer row runs get (1, 0)."""
    P = ctypes.c_int(0)
    ws = ctypes.c_size_t(0)
    _check("attn_plan_partitions",
           lib().attn_plan_partitions(num_sms, batch, num_q_rows, max_q_len, num_q_heads,
                                      num_kv_heads, head_dim_v, max_kv_len, requested,
                                      ctypes.byref(P), ctypes.byref(ws)))
    return P.value, ws.value


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]):
    if nbytes == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                kv_len: torch.Tensor, *, group: int, scale: float, max_kv_len: int,
                page_table: Optional[torch.Tensor] = None, sink: Optional[torch.Tensor] = None,
                q_row_offsets: Optional[torch.Tensor] = None, max_q_len: int = 1,
                causal: bool = False, num_partitions: int = 0,
                workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                lse: Optional[torch.Tensor] = None, return_lse: bool = True, stream=None):
    """Attention of q rows against a KV cache through attn_decode.

    q bf16 [rows, num_q_heads, head_dim] (rows = batch for single-token
    decode, else q_row_offsets[-1]); caches as for kv_descriptor; kv_len
    int32/uint32 [batch] on the device; q_row_offsets int32 [batch + 1] on
    the device or None; sink fp32 [num_q_heads] or None.  num_partitions 0
    plans automatically.  The library's planner routes the call (a few rows
    per sequence keep split-K on the decode kernel; longer row runs take the
    tile kernel, which is not split) and sizes the workspace.  Returns
    (out, lse).
    """
    rows, hq, d = q.shape
    batch = kv_len.shape[0]
    if out is None:
        out = torch.empty((rows, hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((rows, hq), dtype=torch.float32, device=q.device)
    P, ws_bytes = attn_plan_partitions(batch, rows, hq, hq // group, d, max_kv_len,
                                       num_partitions, max_q_len=max_q_len)
    ws, ws_size = _workspace(ws_bytes, q.device, workspace)
    kd = kv_descriptor(k_cache, page_table)
    vd = kv_descriptor(v_cache, page_table)
    _check("attn_decode",
           lib().attn_decode(q.data_ptr(), ctypes.byref(kd), ctypes.byref(vd), kv_len.data_ptr(),
                             _ptr(q_row_offsets), batch, rows, hq, group, d, max_q_len,
                             max_kv_len, scale, _ptr(sink), 1 if causal else 0, P, _ptr(ws),
                             ws_size, out.data_ptr(), _ptr(lse), _stream_handle(stream)))
    return out, lse


def attn_mla_decode(q: torch.Tensor, kv_cache: torch.Tensor, kv_len: torch.Tensor, *,
                    scale: float, max_kv_len: int, dim_v: int = 512,
                    page_table: Optional[torch.Tensor] = None,
                    sink: Optional[torch.Tensor] = None, num_partitions: int = 0,
                    workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                    lse: Optional[torch.Tensor] = None, return_lse: bool = True, stream=None):
    """MLA decode through attn_mla_decode: q bf16 [batch, num_q_heads, 576],
    one-head cache [pages, page_size, 1, 576]; V = K[..., :dim_v].
    num_partitions: 0 = the planner's choice, > 0 = that many key slices per
    row, ATTN_PARTITIONS_BALANCED = the balanced split (as for the _rows and
    _sparse variants)."""
    batch, hq, dqk = q.shape
    if out is None:
        out = torch.empty((batch, hq, dim_v), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((batch, hq), dtype=torch.float32, device=q.device)
    P, ws_bytes = attn_plan_partitions(batch, batch, hq, 1, dim_v, max_kv_len, num_partitions)
    ws, ws_size = _workspace(ws_bytes, q.device, workspace)
    kd = kv_descriptor(kv_cache, page_table)
    _check("attn_mla_decode",
           lib().attn_mla_decode(q.data_ptr(), ctypes.byref(kd), kv_len.data_ptr(), batch, hq, dqk,
                                 dim_v, max_kv_len, scale, _ptr(sink), P, _ptr(ws), ws_size,
                                 out.data_ptr(), _ptr(lse), _stream_handle(stream)))
    return out, lse


def attn_mla_decode_rows(q: torch.Tensor, kv_cache: torch.Tensor, kv_len: torch.Tensor,
                         q_row_offsets: torch.Tensor, *, scale: float, max_kv_len: int,
                         causal: bool = True, dim_v: int = 512,
                         page_table: Optional[torch.Tensor] = None,
                         sink: Optional[torch.Tensor] = None, num_partitions: int = 0,
                         workspace: Optional[torch.Tensor] = None,
                         out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                         return_lse: bool = True, stream=None):
    """MLA decode of several query rows per sequence (draft tokens) through
    attn_mla_decode_rows: q bf16 [rows, 128, 576]; q_row_offsets int32
    [batch + 1] on the device; row i of n sees keys j <= L - n + i when
    causal."""
    rows, hq, dqk = q.shape
    batch = kv_len.shape[0]
    if q_row_offsets.shape[0] != batch + 1:
        raise ValueError("q_row_offsets must have batch + 1 entries")
    if out is None:
        out = torch.empty((rows, hq, dim_v), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((rows, hq), dtype=torch.float32, device=q.device)
    P, ws_bytes = attn_plan_partitions(batch, rows, hq, 1, dim_v, max_kv_len, num_partitions)
    ws, ws_size = _workspace(ws_bytes, q.device, workspace)
    kd = kv_descriptor(kv_cache, page_table)
    _check("attn_mla_decode_rows",
           lib().attn_mla_decode_rows(q.data_ptr(), ctypes.byref(kd), kv_len.data_ptr(),
                                      q_row_offsets.data_ptr(), batch, rows, hq, dqk, dim_v,
                                      max_kv_len, scale, _ptr(sink), 1 if causal else 0, P,
                                      _ptr(ws), ws_size, out.data_ptr(), _ptr(lse),
                                      _stream_handle(stream)))
    return out, lse


def attn_mla_decode_sparse(q: torch.Tensor, kv_cache: torch.Tensor, indices: torch.Tensor,
                           topk_lengths: torch.Tensor, *, scale: float, dim_v: int = 512,
                           sink: Optional[torch.Tensor] = None, num_partitions: int = 0,
                           workspace: Optional[torch.Tensor] = None,
                           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                           return_lse: bool = True, stream=None):
    """Sparse top-k MLA decode through attn_mla_decode_sparse: q bf16
    [batch, num_q_heads, 576]; kv_cache [num_pages, page_size, 1, 576] read as
    rows (row r = slot r % page_size of page r // page_size); indices int32
    [batch, indices_stride] naming each sequence's rows; topk_lengths int32
    [batch] valid entries per row of indices."""
    batch, hq, dqk = q.shape
    if indices.dtype != torch.int32 or indices.dim() != 2 or not indices.is_contiguous():
        raise ValueError("indices must be a contiguous int32 [batch, indices_stride] tensor")
    if indices.shape[0] != batch or topk_lengths.shape[0] != batch:
        raise ValueError("indices and topk_lengths need one row per sequence")
    stride = indices.shape[1]
    if out is None:
        out = torch.empty((batch, hq, dim_v), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((batch, hq), dtype=torch.float32, device=q.device)
    P, ws_bytes = attn_plan_partitions(batch, batch, hq, 1, dim_v, stride, num_partitions)
    ws, ws_size = _workspace(ws_bytes, q.device, workspace)
    kd = kv_descriptor(kv_cache)
    _check("attn_mla_decode_sparse",
           lib().attn_mla_decode_sparse(q.data_ptr(), ctypes.byref(kd), indices.data_ptr(), stride,
                                        topk_lengths.data_ptr(), batch, hq, dqk, dim_v, scale,
                                        _ptr(sink), P, _ptr(ws), ws_size, out.data_ptr(),
                                        _ptr(lse), _stream_handle(stream)))
    return out, lse


def attn_splitk_reduce(ws_o: torch.Tensor, ws_m: torch.Tensor, ws_l: torch.Tensor, *,
                       sink: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                       lse: Optional[torch.Tensor] = None, stream=None):
    """Merge fp32 partials ws_o [P, rows, Hq, dv], ws_m / ws_l [P, rows, Hq]."""
    P, rows, hq, dv = ws_o.shape
    for t in (ws_o, ws_m, ws_l):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("partials must be contiguous fp32")
    if out is None:
        out = torch.empty((rows, hq, dv), dtype=torch.bfloat16, device=ws_o.device)
    if lse is None:
        lse = torch.empty((rows, hq), dtype=torch.float32, device=ws_o.device)
    _check("attn_splitk_reduce",
           lib().attn_splitk_reduce(ws_o.data_ptr(), ws_m.data_ptr(), ws_l.data_ptr(), P, rows,
                                    hq, dv, _ptr(sink), out.data_ptr(), _ptr(lse),
                                    _stream_handle(stream)))
    return out, lse


def attn_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                        kv_len: torch.Tensor, *, group: int, scale: float, max_kv_len: int,
                        page_table: Optional[torch.Tensor] = None,
                        sink: Optional[torch.Tensor] = None,
                        q_row_offsets: Optional[torch.Tensor] = None, max_q_len: int = 1,
                        causal: bool = False, num_partitions: int = 0,
                        out: torch.Tensor, lse: Optional[torch.Tensor] = None, stream=None):
    """attn_decode whose split-K scratch is the library's fixed device array,
    for callers that cannot allocate: the caller passes only inputs and
    outputs (out must be preallocated), and the call allocates nothing."""
    rows, hq, d = q.shape
    batch = kv_len.shape[0]
    kd = kv_descriptor(k_cache, page_table)
    vd = kv_descriptor(v_cache, page_table)
    _check("attn_decode_noalloc",
           lib().attn_decode_noalloc(q.data_ptr(), ctypes.byref(kd), ctypes.byref(vd),
                                     kv_len.data_ptr(), _ptr(q_row_offsets), batch, rows, hq,
                                     group, d, max_q_len, max_kv_len, scale, _ptr(sink),
                                     1 if causal else 0, num_partitions, out.data_ptr(),
                                     _ptr(lse), _stream_handle(stream)))
    return out, lse


def attn_selftest_wait_timeout(stream=None) -> None:
    """Failure-path check: one kernel whose bounded wait on a barrier nothing
    arrives on gives up after its time limit and sets bit 0 of the device
    error word (read it with attn_device_error_flags)."""
    _check("attn_selftest_wait_timeout", lib().attn_selftest_wait_timeout(_stream_handle(stream)))


def attn_device_error_flags(clear: bool = True) -> int:
    flags = ctypes.c_uint(0)
    _check("attn_device_error_flags", lib().attn_device_error_flags(ctypes.byref(flags),
                                                                    1 if clear else 0))
    return flags.value
