"""Seeded random sweep of the configuration space against the fp64 oracle:
every entry point over random shapes, group sizes, page sizes (or the
contiguous layout), partition counts (workspace, on-chip, and for MLA the
balanced split), sinks, query rows per sequence, causal or not, with ragged,
empty and sub-tile lengths."""
import math
import random

import pytest
import torch

from split_flash_decoding_gb300 import workloads as W
from tests.helpers import assert_close, oracle_result

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def attn():
    from split_flash_decoding_gb300 import build
    build.build()
    from split_flash_decoding_gb300 import attn as a
    a.attn_device_error_flags(clear=True)
    yield a
    assert a.attn_device_error_flags(clear=True) == 0


def random_lengths(rng, batch, hi):
    pick = [0, 1, 2, 63, 64, 65, 127, 128, 129]
    return [rng.choice(pick) if rng.random() < 0.3 else rng.randint(1, hi) for _ in range(batch)]


@pytest.mark.parametrize("case", range(64))
def test_gqa_decode_random_configs(attn, case):
    rng = random.Random(1000 + case)
    d = rng.choice([64, 128, 128, 128])
    group = rng.choice([1, 2, 4, 8])
    hkv = rng.choice([1, 2, 4, 8])
    batch = rng.randint(1, 7)
    lens = random_lengths(rng, batch, 3000)
    page = rng.choice([None, 8, 16, 32, 64, 128, 256])
    sink = rng.random() < 0.4
    # a few rows per sequence only on the tensor-core path (rows x group <= 16)
    max_rows = 16 // group if d == 128 else 1
    q_lens = None
    causal = False
    if max_rows > 1 and rng.random() < 0.4:
        q_lens = [rng.randint(1, max_rows) for _ in range(batch)]
        lens = [max(L, n) if rng.random() < 0.8 else L for L, n in zip(lens, q_lens)]
        causal = rng.random() < 0.7
    P = rng.choice([0, 1, 2, 3, 4, 5, 9])
    w = W.make_workload("fuzz", batch=batch, num_q_heads=hkv * group, num_kv_heads=hkv, dim_qk=d,
                        kv_lens=lens, page_size=page, seed=2000 + case, device=DEV, sink=sink,
                        q_lens=q_lens, causal=causal)
    out, lse = attn.attn_decode(w.q, w.k_cache, w.v_cache, w.kv_len, group=group, scale=w.scale,
                                max_kv_len=max(1, w.max_kv_len), page_table=w.page_table,
                                sink=w.sink, q_row_offsets=w.q_row_offsets,
                                max_q_len=w.max_q_len, causal=causal, num_partitions=P)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l,
                 f"case {case}: d={d} g={group} hkv={hkv} lens={lens} page={page} P={P} "
                 f"rows={q_lens} causal={causal} sink={sink}")


@pytest.mark.parametrize("case", range(16))
def test_mla_random_configs(attn, case):
    rng = random.Random(3000 + case)
    batch = rng.randint(1, 5)
    lens = random_lengths(rng, batch, 5000)
    page = rng.choice([None, 8, 16, 64, 128])
    sink = rng.random() < 0.4
    P = rng.choice([-1, 0, 1, 2, 3, 7])   # -1: the balanced split
    rows = rng.random() < 0.5
    q_lens = [rng.randint(1, 3) for _ in range(batch)] if rows else None
    causal = rows and rng.random() < 0.7
    w = W.make_workload("fuzz_mla", batch=batch, num_q_heads=128, num_kv_heads=1, dim_qk=576,
                        dim_v=512, mla=True, kv_lens=lens, page_size=page, seed=4000 + case,
                        device=DEV, sink=sink, scale=1.0 / math.sqrt(192.0), q_lens=q_lens,
                        causal=causal)
    if rows:
        out, lse = attn.attn_mla_decode_rows(w.q, w.k_cache, w.kv_len, w.q_row_offsets,
                                             scale=w.scale, max_kv_len=max(1, w.max_kv_len),
                                             causal=causal, page_table=w.page_table,
                                             sink=w.sink, num_partitions=P)
    else:
        out, lse = attn.attn_mla_decode(w.q, w.k_cache, w.kv_len, scale=w.scale,
                                        max_kv_len=max(1, w.max_kv_len),
                                        page_table=w.page_table, sink=w.sink, num_partitions=P)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l,
                 f"mla case {case}: lens={lens} page={page} P={P} rows={q_lens} causal={causal}")


@pytest.mark.parametrize("case", range(12))
def test_sparse_mla_random_configs(attn, case):
    rng = random.Random(5000 + case)
    batch = rng.randint(1, 5)
    ctx = [rng.randint(0, 4000) for _ in range(batch)]
    topk = rng.choice([1, 17, 64, 300, 1024])
    page = rng.choice([1, 16, 64])
    P = rng.choice([-1, 0, 1, 2, 5])   # -1: the balanced split
    w = W.make_sparse_mla_workload("fuzz_sparse", ctx_lens=ctx, topk=topk, page_size=page,
                                   seed=6000 + case, device=DEV, sink=rng.random() < 0.4,
                                   scale=1.0 / math.sqrt(192.0),
                                   replace_rows=rng.random() < 0.3)
    out, lse = attn.attn_mla_decode_sparse(w.q, w.k_cache, w.indices, w.kv_len, scale=w.scale,
                                           sink=w.sink, num_partitions=P)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, f"sparse case {case}: ctx={ctx} topk={topk} P={P}")
