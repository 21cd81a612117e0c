"""fp64 CPU attention oracle (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product package never imports it, and this package never imports the
product package: the two share nothing but the seeded input generators in
``split_flash_decoding_gb300.workloads``, which hold none of the method's
arithmetic.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, pthreads); this
module compiles it with gcc and marshals numpy arrays into it.  The
definition it implements is written out at the top of ``attn_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_objs")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile attn_oracle.c (or another source, for the planted-mistake
    tests) into a shared library with gcc, -O2, pthreads."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    # -ffp-contract=off: every product and sum is rounded as written.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class _KV(ctypes.Structure):
    _fields_ = [
        ("base", ctypes.c_void_p),
        ("page_stride", ctypes.c_int64),
        ("token_stride", ctypes.c_int64),
        ("head_stride", ctypes.c_int64),
        ("page_size", ctypes.c_int32),
        ("_pad", ctypes.c_int32),
        ("page_table", ctypes.c_void_p),
        ("max_pages", ctypes.c_int64),
        ("indices", ctypes.c_void_p),
        ("indices_stride", ctypes.c_int64),
    ]


class _Problem(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p),
        ("k", ctypes.POINTER(_KV)),
        ("v", ctypes.POINTER(_KV)),
        ("kv_len", ctypes.c_void_p),
        ("q_row_offsets", ctypes.c_void_p),
        ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("dim_qk", ctypes.c_int32),
        ("dim_v", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("sink", ctypes.c_void_p),
    ]


def _open(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention.argtypes = [
        ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_partials.restype = ctypes.c_int
    lib.oracle_partials.argtypes = [
        ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    if hasattr(lib, "oracle_spread"):
        lib.oracle_spread.restype = ctypes.c_int
        lib.oracle_spread.argtypes = [
            ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    return lib


def use_library(path):
    """Swap the compiled oracle (used by the planted-mistake tests); returns
    the previous handle so it can be restored with ``restore_library``."""
    global _lib
    with _lock:
        prev = _lib
        _lib = _open(path)
    return prev


def restore_library(prev):
    global _lib
    with _lock:
        _lib = prev


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _open(_LIB_PATH)
    return _lib


def _bits(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> contiguous uint16 bit pattern array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype != torch.bfloat16:
                raise TypeError(f"oracle expects bf16 tensors, got {x.dtype}")
            x = x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
            return x
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x)
    if x.dtype != np.uint16:
        raise TypeError("oracle expects bf16 bit patterns as uint16")
    return np.ascontiguousarray(x)


def _i32(x):
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x).astype(np.int32))


def _f64(x):
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().double().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


class KV:
    """A K or V cache operand for the oracle.

    ``data`` is a bf16 tensor (or uint16 bit array) whose element
    ``page * page_stride + slot * token_stride + head * head_stride + c`` is
    channel c of the token in slot ``slot`` of page ``page``.  With
    ``page_table`` None, page = sequence index and slot = token index.
    With ``indices`` [batch, indices_stride] (sparse top-k), token t of
    sequence b is physical row r = indices[b, t], slot r % page_size of page
    r // page_size; ``num_rows`` bounds r.
    """

    def __init__(self, data, page_stride, token_stride, head_stride, page_size,
                 page_table=None, channel_offset=0, indices=None, num_rows=None):
        self.data = _bits(data).reshape(-1)
        self.page_stride = int(page_stride)
        self.token_stride = int(token_stride)
        self.head_stride = int(head_stride)
        self.page_size = int(page_size)
        self.page_table = _i32(page_table)
        self.channel_offset = int(channel_offset)
        self.indices = _i32(indices)
        if self.indices is not None:
            if self.page_table is not None:
                raise ValueError("a sparse operand has indices instead of a page table")
            if self.indices.ndim != 2:
                raise ValueError("indices must be [batch, indices_stride]")
            if num_rows is None:
                raise ValueError("a sparse operand needs num_rows")
        self.num_rows = None if num_rows is None else int(num_rows)

    @classmethod
    def paged(cls, cache, page_table):
        """cache [num_pages, page_size, num_kv_heads, dim], page_table [B, max_pages]."""
        n, ps, hk, d = cache.shape
        return cls(cache, ps * hk * d, hk * d, d, ps, page_table)

    @classmethod
    def sparse(cls, cache, indices):
        """cache [num_pages, page_size, num_kv_heads, dim] read as
        num_pages * page_size physical rows; indices int [batch, stride]."""
        n, ps, hk, d = cache.shape
        return cls(cache, ps * hk * d, hk * d, d, ps, None, indices=indices, num_rows=n * ps)

    def check_rows(self, kv_len):
        """Every index a sequence uses (the first kv_len[b]) names a row."""
        if self.indices is None:
            return
        for b, L in enumerate(kv_len):
            if L > self.indices.shape[1]:
                raise ValueError(f"sequence {b}: {L} keys but indices_stride "
                                 f"{self.indices.shape[1]}")
            r = self.indices[b, :L]
            if L and (r.min() < 0 or r.max() >= self.num_rows):
                raise ValueError(f"sequence {b}: index outside [0, {self.num_rows})")

    @classmethod
    def contiguous(cls, cache):
        """cache [B, capacity, num_kv_heads, dim]; sequence b is page b."""
        b, cap, hk, d = cache.shape
        return cls(cache, cap * hk * d, hk * d, d, cap, None)

    def _struct(self):
        pt = self.page_table
        s = _KV()
        s.base = self.data.ctypes.data + 2 * self.channel_offset
        s.page_stride = self.page_stride
        s.token_stride = self.token_stride
        s.head_stride = self.head_stride
        s.page_size = self.page_size
        s.page_table = pt.ctypes.data if pt is not None else None
        s.max_pages = pt.shape[1] if pt is not None else 0
        s.indices = self.indices.ctypes.data if self.indices is not None else None
        s.indices_stride = self.indices.shape[1] if self.indices is not None else 0
        return s


def _problem(q, k: KV, v: KV, kv_len, q_row_offsets, group, scale, sink, causal, dim_v):
    qb = _bits(q)
    kvl = _i32(kv_len)
    offs = _i32(q_row_offsets)
    snk = _f64(sink)
    if qb.ndim != 3:
        raise ValueError("q must be [rows, num_q_heads, dim_qk]")
    rows, hq, dqk = qb.shape
    batch = kvl.shape[0]
    if offs is None and rows != batch:
        raise ValueError("without q_row_offsets q must have one row per sequence")
    if offs is not None and (offs.shape[0] != batch + 1 or offs[-1] != rows):
        raise ValueError("q_row_offsets must be [batch+1] ending at the row count")
    if hq % group:
        raise ValueError("num_q_heads must be a multiple of group")
    k.check_rows(kvl)
    v.check_rows(kvl)
    ks, vs = k._struct(), v._struct()
    pr = _Problem()
    pr.q = qb.ctypes.data
    pr.k = ctypes.pointer(ks)
    pr.v = ctypes.pointer(vs)
    pr.kv_len = kvl.ctypes.data
    pr.q_row_offsets = offs.ctypes.data if offs is not None else None
    pr.batch = batch
    pr.num_q_heads = hq
    pr.group = int(group)
    pr.dim_qk = dqk
    pr.dim_v = int(dim_v)
    pr.causal = 1 if causal else 0
    pr.scale = float(scale)
    pr.sink = snk.ctypes.data if snk is not None else None
    keep = (qb, kvl, offs, snk, ks, vs, k, v)
    return pr, rows, hq, keep


def attention(q, k: KV, v: KV, kv_len, *, group, scale, dim_v=None, sink=None,
              causal=False, q_row_offsets=None, sample=None, threads=None):
    """Exact softmax attention in fp64.

    q: bf16 [rows, num_q_heads, dim_qk]; kv_len: [batch] keys per sequence.
    scale: the fp32 scale as the GPU sees it (pass float(np.float32(s))).
    sink: per-q-head logits [num_q_heads] (fp32 values) or None.
    sample: optional (rows, heads) integer arrays; only those pairs are
    computed and the result is out [n, dim_v], lse [n].
    Returns (out, lse) as float64 arrays: out [rows, num_q_heads, dim_v],
    lse [rows, num_q_heads] natural-log units.
    """
    lib = _load()
    if dim_v is None:
        dim_v = int(np.asarray(_bits(q)).shape[-1])
    pr, rows, hq, keep = _problem(q, k, v, kv_len, q_row_offsets, group, scale, sink,
                                  causal, dim_v)
    nthreads = threads or os.cpu_count() or 1
    if sample is not None:
        srows = np.ascontiguousarray(np.asarray(sample[0], dtype=np.int64))
        sheads = np.ascontiguousarray(np.asarray(sample[1], dtype=np.int32))
        n = srows.shape[0]
        out = np.zeros((n, dim_v), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        st = lib.oracle_attention(ctypes.byref(pr), srows.ctypes.data, sheads.ctypes.data, n,
                                  out.ctypes.data, lse.ctypes.data, nthreads)
    else:
        out = np.zeros((rows, hq, dim_v), dtype=np.float64)
        lse = np.zeros((rows, hq), dtype=np.float64)
        st = lib.oracle_attention(ctypes.byref(pr), None, None, 0,
                                  out.ctypes.data, lse.ctypes.data, nthreads)
    del keep
    if st != 0:
        raise RuntimeError(f"oracle_attention failed with status {st}")
    return out, lse


def partials(q, k: KV, v: KV, kv_len, bounds, *, group, scale, dim_v=None,
             causal=False, q_row_offsets=None, threads=None):
    """Per-partition (O_p unnormalised, m_p, l_p) for key slices
    [bounds[p], bounds[p+1]) of every (row, head), in fp64.

    Returns ws_o [P, rows, Hq, dim_v], ws_m [P, rows, Hq], ws_l [P, rows, Hq].
    """
    lib = _load()
    if dim_v is None:
        dim_v = int(np.asarray(_bits(q)).shape[-1])
    pr, rows, hq, keep = _problem(q, k, v, kv_len, q_row_offsets, group, scale, None,
                                  causal, dim_v)
    b = np.ascontiguousarray(np.asarray(bounds, dtype=np.int64))
    nparts = b.shape[0] - 1
    ws_o = np.zeros((nparts, rows, hq, dim_v), dtype=np.float64)
    ws_m = np.zeros((nparts, rows, hq), dtype=np.float64)
    ws_l = np.zeros((nparts, rows, hq), dtype=np.float64)
    st = lib.oracle_partials(ctypes.byref(pr), b.ctypes.data, nparts, ws_o.ctypes.data,
                             ws_m.ctypes.data, ws_l.ctypes.data,
                             threads or os.cpu_count() or 1)
    del keep
    if st != 0:
        raise RuntimeError(f"oracle_partials failed with status {st}")
    return ws_o, ws_m, ws_l


def spread(q, k: KV, v: KV, kv_len, *, group, scale, dim_v=None, sink=None, causal=False,
           q_row_offsets=None, sample=None, threads=None):
    """Error-bound statistics of the exact result (not part of the attention
    definition): with the exact weights w_j = exp(s_j - M) / Z over the visible
    keys (Z includes the sink),

        sd[c] = sqrt(sum_j w_j (V[j, c] - out[c])^2),  am[c] = sum_j w_j |V[j, c]|,

    and per (row, head) the visible key count, max_j scale * sum_c |q[c] K[j, c]|
    and max_j |s_j|.  sample as for attention (default: every (row, head)).
    Returns (sd, am, stats): sd and am shaped like attention's out, stats
    [..., 3] = (nvis, sabs, smax).
    """
    lib = _load()
    if dim_v is None:
        dim_v = int(np.asarray(_bits(q)).shape[-1])
    pr, rows, hq, keep = _problem(q, k, v, kv_len, q_row_offsets, group, scale, sink,
                                  causal, dim_v)
    if sample is None:
        srows = np.repeat(np.arange(rows, dtype=np.int64), hq)
        sheads = np.tile(np.arange(hq, dtype=np.int32), rows)
        shape = (rows, hq)
    else:
        srows = np.ascontiguousarray(np.asarray(sample[0], dtype=np.int64))
        sheads = np.ascontiguousarray(np.asarray(sample[1], dtype=np.int32))
        shape = (srows.shape[0],)
    n = srows.shape[0]
    sd = np.zeros((n, dim_v), dtype=np.float64)
    am = np.zeros((n, dim_v), dtype=np.float64)
    stats = np.zeros((n, 3), dtype=np.float64)
    st = lib.oracle_spread(ctypes.byref(pr), srows.ctypes.data, sheads.ctypes.data, n,
                           sd.ctypes.data, am.ctypes.data, stats.ctypes.data,
                           threads or os.cpu_count() or 1)
    del keep
    if st != 0:
        raise RuntimeError(f"oracle_spread failed with status {st}")
    return sd.reshape(shape + (dim_v,)), am.reshape(shape + (dim_v,)), stats.reshape(shape + (3,))
