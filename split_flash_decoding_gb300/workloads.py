"""Seeded synthetic inputs shaped like the decode-attention workloads.

This module only draws random numbers and lays them out; it computes no part
of attention.  Both the CUDA path's tests/benchmark and the fp64 oracle
consume what it produces, so it must stay free of the method's arithmetic.

Layouts produced (all bf16 unless noted):

* q            [rows, num_q_heads, dim_qk]; rows = batch for single-token
               decode, else q_row_offsets[-1] (ragged, one block of rows per
               sequence).
* paged cache  [num_pages, page_size, num_kv_heads, dim] with a page table
               int32 [batch, max_pages]: token t of sequence b lives in slot
               t % page_size of page page_table[b, t // page_size].  Pages are
               handed out from a seeded random permutation of the pool.
* contiguous   [batch, capacity, num_kv_heads, dim]: sequence b is "page" b.
* kv_len       int32 [batch], q_row_offsets int32 [batch + 1] or None,
               sink fp32 [num_q_heads] or None.
* sparse top-k a one-head row pool [num_pages, page_size, 1, dim] read as
               rows (row r = slot r % page_size of page r // page_size), an
               index list int32 [batch, indices_stride] of the rows each
               sequence attends to (-1 past its count) and kv_len = the
               per-sequence counts.

Values are N(0, 1) drawn in fp32 from a torch.Generator seeded per workload,
then rounded to bf16; lengths and the page permutation come from a CPU
generator so they are identical on every device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch


@dataclass
class Workload:
    name: str
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: Optional[torch.Tensor]      # None: V is K[..., :dim_v] (MLA)
    page_table: Optional[torch.Tensor]   # None: contiguous layout
    page_size: int
    kv_len: torch.Tensor                 # int32 [batch], on the data device
    kv_len_host: list                    # python ints
    q_row_offsets: Optional[torch.Tensor]
    q_row_offsets_host: Optional[list]
    group: int
    dim_v: int
    scale: float                         # exactly representable in fp32
    sink: Optional[torch.Tensor]
    causal: bool
    indices: Optional[torch.Tensor] = None   # sparse top-k rows [batch, stride], else None

    @property
    def batch(self) -> int:
        return len(self.kv_len_host)

    @property
    def num_q_heads(self) -> int:
        return self.q.shape[1]

    @property
    def num_kv_heads(self) -> int:
        return self.num_q_heads // self.group

    @property
    def dim_qk(self) -> int:
        return self.q.shape[2]

    @property
    def rows(self) -> int:
        return self.q.shape[0]

    @property
    def max_kv_len(self) -> int:
        return max(self.kv_len_host) if self.kv_len_host else 0

    @property
    def max_q_len(self) -> int:
        if self.q_row_offsets_host is None:
            return 1
        o = self.q_row_offsets_host
        return max((o[i + 1] - o[i] for i in range(len(o) - 1)), default=0)

    @property
    def is_mla(self) -> bool:
        return self.v_cache is None

    def to(self, device) -> "Workload":
        mv = lambda t: None if t is None else t.to(device)
        return replace(self, q=mv(self.q), k_cache=mv(self.k_cache), v_cache=mv(self.v_cache),
                       page_table=mv(self.page_table), kv_len=mv(self.kv_len),
                       q_row_offsets=mv(self.q_row_offsets), sink=mv(self.sink),
                       indices=mv(self.indices))


def fp32(x: float) -> float:
    """Round a python float to the nearest fp32 value."""
    return float(torch.tensor(x, dtype=torch.float32).item())


def _randn_bf16(shape, gen, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_workload(name: str, *, batch: int, num_q_heads: int, num_kv_heads: int, dim_qk: int,
                  kv_lens, page_size: Optional[int], seed: int, device="cpu",
                  dim_v: Optional[int] = None, mla: bool = False, sink: bool = False,
                  q_lens=None, causal: bool = False, scale: Optional[float] = None,
                  capacity: Optional[int] = None) -> Workload:
    """Build one seeded workload.

    kv_lens: keys per sequence (python ints).  page_size None gives the
    contiguous layout [batch, capacity, Hkv, dim] (capacity defaults to
    max(kv_lens), at least 1).  mla=True stores only K (one KV head) and
    V is read as K[..., :dim_v].  q_lens: query rows per sequence (None: one).
    """
    device = torch.device(device)
    kv_lens = [int(x) for x in kv_lens]
    assert len(kv_lens) == batch
    dim_v = dim_qk if dim_v is None else dim_v
    if scale is None:
        scale = 1.0 / math.sqrt(dim_qk)
    scale = fp32(scale)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    cpu_gen = torch.Generator()
    cpu_gen.manual_seed(seed + 7919)

    rows = batch if q_lens is None else int(sum(q_lens))
    q = _randn_bf16((rows, num_q_heads, dim_qk), gen, device)

    if page_size is None:
        cap = capacity if capacity is not None else max(max(kv_lens, default=1), 1)
        k_cache = _randn_bf16((batch, cap, num_kv_heads, dim_qk), gen, device)
        v_cache = None if mla else _randn_bf16((batch, cap, num_kv_heads, dim_v), gen, device)
        page_table = None
        ps = cap
    else:
        ps = int(page_size)
        pages_per_seq = [max(1, -(-L // ps)) for L in kv_lens]
        total = sum(pages_per_seq)
        max_pages = max(pages_per_seq, default=1)
        perm = torch.randperm(total, generator=cpu_gen)
        pt = torch.zeros((batch, max_pages), dtype=torch.int32)
        pos = 0
        for b, n in enumerate(pages_per_seq):
            pt[b, :n] = perm[pos:pos + n].to(torch.int32)
            pos += n
        k_cache = _randn_bf16((total, ps, num_kv_heads, dim_qk), gen, device)
        v_cache = None if mla else _randn_bf16((total, ps, num_kv_heads, dim_v), gen, device)
        page_table = pt.to(device)

    kv_len = torch.tensor(kv_lens, dtype=torch.int32, device=device)
    offs = offs_host = None
    if q_lens is not None:
        offs_host = [0]
        for n in q_lens:
            offs_host.append(offs_host[-1] + int(n))
        offs = torch.tensor(offs_host, dtype=torch.int32, device=device)
    sk = None
    if sink:
        sk = torch.randn((num_q_heads,), generator=gen, device=device, dtype=torch.float32)
    return Workload(name=name, q=q, k_cache=k_cache, v_cache=v_cache, page_table=page_table,
                    page_size=ps, kv_len=kv_len, kv_len_host=kv_lens, q_row_offsets=offs,
                    q_row_offsets_host=offs_host, group=num_q_heads // num_kv_heads,
                    dim_v=dim_v, scale=scale, sink=sk, causal=causal)


def make_sparse_mla_workload(name: str, *, ctx_lens, topk: int, page_size: int, seed: int,
                             device="cpu", num_q_heads: int = 128, dim_qk: int = 576,
                             dim_v: int = 512, sink: bool = False,
                             scale: Optional[float] = None,
                             replace_rows: bool = False) -> Workload:
    """Sparse top-k MLA decode: sequence b has a context of ctx_lens[b] tokens
    in a paged one-head pool (random page permutation, as make_workload) and
    attends to min(topk, ctx_lens[b]) of them, a seeded random choice in
    random order (replace_rows: drawn with repetition).  Each chosen token t
    is named by its physical row page_table[b, t // page_size] * page_size +
    t % page_size; the page table itself is not part of the workload."""
    ctx = [int(x) for x in ctx_lens]
    batch = len(ctx)
    base = make_workload(name, batch=batch, num_q_heads=num_q_heads, num_kv_heads=1,
                         dim_qk=dim_qk, dim_v=dim_v, mla=True, kv_lens=ctx,
                         page_size=page_size, seed=seed, device=device, sink=sink, scale=scale)
    g = torch.Generator()
    g.manual_seed(seed + 104729)
    counts = [min(int(topk), c) for c in ctx]
    stride = max(max(counts, default=0), 1)
    idx = torch.full((batch, stride), -1, dtype=torch.int64)
    pt = base.page_table.cpu().long()
    for b, (c, n) in enumerate(zip(ctx, counts)):
        if n == 0:
            continue
        if replace_rows:
            t = torch.randint(0, c, (n,), generator=g)
        else:
            t = torch.randperm(c, generator=g)[:n]
        idx[b, :n] = pt[b, t // page_size] * page_size + t % page_size
    dev = torch.device(device)
    return replace(base, page_table=None, kv_len=torch.tensor(counts, dtype=torch.int32,
                                                                 device=dev),
                   kv_len_host=counts, indices=idx.to(torch.int32).to(dev))


def deepseek_v32_sparse_mla_decode(device="cpu", seed: int = 7, batch: int = 128,
                                   topk: int = 2048) -> Workload:
    """DeepSeek-V3.2-shaped sparse MLA decode: batch 128, 128 q heads, one KV
    head of depth 576, V = K[:, :512], contexts uniform in [1024, 32768] in a
    page-64 pool, top-2048 rows per sequence (all rows when the context is
    shorter), scale 1/sqrt(192)."""
    ctx = _uniform_ints(1024, 32768, batch, seed)
    return make_sparse_mla_workload(f"deepseek_v32_sparse_mla_decode_b{batch}_top{topk}_h128_d576",
                                    ctx_lens=ctx, topk=topk, page_size=64, seed=seed,
                                    device=device, scale=1.0 / math.sqrt(192.0))


def contiguous_copy(w: Workload, capacity: Optional[int] = None) -> Workload:
    """The same logical K/V laid out contiguously ([batch, capacity, Hkv, d]).

    Token t of sequence b is copied from its page slot; slots past kv_len are
    zero.  Used to check that the paged and contiguous layouts give the same
    result.
    """
    if w.page_table is None:
        return w
    cap = capacity if capacity is not None else max(w.max_kv_len, 1)
    pt = w.page_table.long()
    ps = w.page_size

    def gather(cache):
        if cache is None:
            return None
        out = torch.zeros((w.batch, cap) + tuple(cache.shape[2:]), dtype=cache.dtype,
                          device=cache.device)
        for b, L in enumerate(w.kv_len_host):
            if L == 0:
                continue
            t = torch.arange(L, device=cache.device)
            pages = pt[b, t // ps]
            out[b, :L] = cache[pages, t % ps]
        return out

    return replace(w, k_cache=gather(w.k_cache), v_cache=gather(w.v_cache), page_table=None,
                   page_size=cap)


# ---------------------------------------------------------------------------
# The five standard workloads.
# ---------------------------------------------------------------------------

def _uniform_ints(lo: int, hi: int, n: int, seed: int):
    g = torch.Generator()
    g.manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def tiny_decode(device="cpu", seed: int = 1) -> Workload:
    """batch 2, 4 q heads on 1 KV head (group 4), head_dim 64, contiguous
    cache with 37 and 100 keys, scale 1/8, no sinks."""
    return make_workload("tiny_decode_b2_h4kv1_d64", batch=2, num_q_heads=4, num_kv_heads=1,
                         dim_qk=64, kv_lens=[37, 100], page_size=None, seed=seed, device=device,
                         scale=1.0 / 8.0)


def llama3_8b_decode(device="cpu", seed: int = 2, batch: int = 64) -> Workload:
    """Llama-3-8B-shaped GQA decode: batch 64, 32 q / 8 KV heads, head_dim 128,
    ragged lengths uniform in [512, 8192], paged (page 128, random page
    permutation), scale 1/sqrt(128)."""
    lens = _uniform_ints(512, 8192, batch, seed)
    return make_workload(f"llama3_8b_gqa_decode_b{batch}_h32kv8_d128_paged128", batch=batch,
                         num_q_heads=32, num_kv_heads=8, dim_qk=128, kv_lens=lens,
                         page_size=128, seed=seed, device=device)


def long_context_decode(device="cpu", seed: int = 3, kv_len: int = 131072) -> Workload:
    """Single-sequence long-context decode: 32 q / 8 KV heads, head_dim 128,
    131072 keys, paged (page 128), per-q-head sink logits ~ N(0, 1)."""
    return make_workload(f"long_context_decode_b1_L{kv_len}_h32kv8_d128_sinks", batch=1,
                         num_q_heads=32, num_kv_heads=8, dim_qk=128, kv_lens=[kv_len],
                         page_size=128, seed=seed, device=device, sink=True)


def deepseek_v3_mla_decode(device="cpu", seed: int = 4, batch: int = 32) -> Workload:
    """DeepSeek-V3-shaped MLA decode: batch 32, 128 q heads, one KV head of
    depth 576 (512 latent + 64 rope), V = K[:, :512], lengths uniform in
    [1024, 32768], paged (page 64), scale 1/sqrt(192)."""
    lens = _uniform_ints(1024, 32768, batch, seed)
    return make_workload(f"deepseek_v3_mla_decode_b{batch}_h128_d576_paged64", batch=batch,
                         num_q_heads=128, num_kv_heads=1, dim_qk=576, dim_v=512, mla=True,
                         kv_lens=lens, page_size=64, seed=seed, device=device,
                         scale=1.0 / math.sqrt(192.0))


def deepseek_v3_mtp_decode(device="cpu", seed: int = 8, batch: int = 32,
                           q_len: int = 2) -> Workload:
    """DeepSeek-V3-shaped MLA decode with multi-token prediction: every
    sequence carries q_len query rows (the current token and q_len - 1 draft
    tokens), causal (row i of n sees keys j <= L - n + i); batch 32, 128 q
    heads, one KV head of depth 576, V = K[:, :512], lengths uniform in
    [1024, 32768], paged (page 64), scale 1/sqrt(192)."""
    lens = _uniform_ints(1024, 32768, batch, seed)
    return make_workload(f"deepseek_v3_mtp{q_len}_mla_decode_b{batch}_h128_d576_paged64",
                         batch=batch, num_q_heads=128, num_kv_heads=1, dim_qk=576, dim_v=512,
                         mla=True, kv_lens=lens, page_size=64, seed=seed, device=device,
                         q_lens=[q_len] * batch, causal=True, scale=1.0 / math.sqrt(192.0))


def few_token_decode(device="cpu", seed: int = 6, batch: int = 64, max_q_len: int = 4) -> Workload:
    """Few-token decode on the Llama-3-8B shapes: batch 64, 32 q / 8 KV heads,
    head_dim 128, paged (page 128), cache lengths uniform in [512, 8192], and
    1..max_q_len query rows per sequence (draft tokens being verified),
    causal (row i of n sees keys j <= L - n + i)."""
    g = torch.Generator()
    g.manual_seed(seed)
    q_lens = [int(x) for x in torch.randint(1, max_q_len + 1, (batch,), generator=g)]
    kv_lens = _uniform_ints(512, 8192, batch, seed)
    return make_workload(f"few_token_decode_b{batch}_q{max_q_len}_h32kv8_d128_paged128",
                         batch=batch, num_q_heads=32, num_kv_heads=8, dim_qk=128,
                         kv_lens=kv_lens, page_size=128, seed=seed, device=device,
                         q_lens=q_lens, causal=True)


def mixed_prefill_decode(device="cpu", seed: int = 5) -> Workload:
    """Ragged mixed prefill + decode: 16 sequences, eight with one query row
    and eight with q_len uniform in [512, 4096]; cached prefix uniform in
    [0, 8192]; causal; 32 q / 8 KV heads, head_dim 128, paged (page 128)."""
    g = torch.Generator()
    g.manual_seed(seed)
    prefill = [int(x) for x in torch.randint(512, 4097, (8,), generator=g)]
    prefix = [int(x) for x in torch.randint(0, 8193, (16,), generator=g)]
    q_lens = [1] * 8 + prefill
    perm = torch.randperm(16, generator=g).tolist()
    q_lens = [q_lens[i] for i in perm]
    kv_lens = [p + n for p, n in zip(prefix, q_lens)]
    return make_workload("mixed_prefill_decode_16seq_h32kv8_d128_causal", batch=16,
                         num_q_heads=32, num_kv_heads=8, dim_qk=128, kv_lens=kv_lens,
                         page_size=128, seed=seed, device=device, q_lens=q_lens, causal=True)
