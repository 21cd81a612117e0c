"""GPU parity of the GQA split-K decode path (attn_decode, attn_splitk_reduce)
against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
from split_flash_decoding_gb300 import workloads as W
from tests.helpers import assert_close, assert_pair, bits_equal, oracle_result

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    from split_flash_decoding_gb300 import build
    build.build()
    from split_flash_decoding_gb300 import attn as a
    a.attn_device_error_flags(clear=True)
    yield a
    assert a.attn_device_error_flags(clear=True) == 0


DEV = "cuda:0"


def run(attn, w, P=0, sink="workload", **kw):
    s = w.sink if sink == "workload" else sink
    out, lse = attn.attn_decode(w.q, w.k_cache, w.v_cache, w.kv_len, group=w.group,
                                scale=w.scale, max_kv_len=w.max_kv_len,
                                page_table=w.page_table, sink=s, num_partitions=P, **kw)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("P", [1, 3])
def test_tiny_decode_matches_oracle(attn, P):
    w = W.tiny_decode(device=DEV)
    out, lse = run(attn, w, P)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, f"tiny P={P}")


@pytest.mark.parametrize("d,hq,hkv", [(64, 4, 1), (128, 8, 8), (128, 8, 4), (128, 32, 8),
                                      (64, 16, 2), (128, 16, 2)])
@pytest.mark.parametrize("P", [1, 2, 5])
def test_shapes_and_groups(attn, d, hq, hkv, P):
    lens = [1, 31, 32, 33, 200, 517]
    w = W.make_workload("t", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, dim_qk=d,
                        kv_lens=lens, page_size=64, seed=100 + d + hq + hkv, device=DEV)
    out, lse = run(attn, w, P)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, f"d={d} hq={hq} hkv={hkv} P={P}")


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128, 256])
def test_paged_equals_contiguous_bitwise(attn, page_size):
    lens = [1, 7, 64, 100, 255, 256, 1000]
    w = W.make_workload("t", batch=len(lens), num_q_heads=32, num_kv_heads=8, dim_qk=128,
                        kv_lens=lens, page_size=page_size, seed=7, device=DEV)
    c = W.contiguous_copy(w)
    for P in (1, 4):
        o1, l1 = run(attn, w, P)
        o2, l2 = run(attn, c, P)
        assert bits_equal(o1, o2) and bits_equal(l1, l2), f"page {page_size} P={P}"
    ref_o, ref_l = oracle_result(w)
    assert_close(o1, l1, ref_o, ref_l, f"page {page_size}")


def test_split_k_matches_single_partition(attn):
    lens = [3000, 4097, 129, 8192]
    w = W.make_workload("t", batch=4, num_q_heads=32, num_kv_heads=8, dim_qk=128,
                        kv_lens=lens, page_size=128, seed=8, device=DEV)
    o1, l1 = run(attn, w, 1)
    ref_o, ref_l = oracle_result(w)
    assert_close(o1, l1, ref_o, ref_l, "P=1")
    for P in (2, 7, 16, 64, 256):
        oP, lP = run(attn, w, P)
        assert_pair(oP, lP, o1, l1, ref_o, ref_l, f"P={P} vs P=1")


def test_empty_and_tiny_sequences(attn):
    lens = [0, 1, 2, 0, 33]
    w = W.make_workload("t", batch=5, num_q_heads=8, num_kv_heads=2, dim_qk=128,
                        kv_lens=lens, page_size=16, seed=9, device=DEV)
    for P in (1, 3):
        out, lse = run(attn, w, P)
        ref_o, ref_l = oracle_result(w)
        assert_close(out, lse, ref_o, ref_l, f"P={P}")
        assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_sinks(attn):
    lens = [50, 700, 0, 4000]
    w = W.make_workload("t", batch=4, num_q_heads=16, num_kv_heads=4, dim_qk=128,
                        kv_lens=lens, page_size=64, seed=10, device=DEV, sink=True)
    no_sink = torch.full((16,), -math.inf, dtype=torch.float32, device=DEV)
    for P in (1, 5):
        out, lse = run(attn, w, P)
        ref_o, ref_l = oracle_result(w)
        assert_close(out, lse, ref_o, ref_l, f"sinks P={P}")
        o_inf, l_inf = run(attn, w, P, sink=no_sink)
        o_none, l_none = run(attn, w, P, sink=None)
        assert bits_equal(o_inf, o_none) and bits_equal(l_inf, l_none), f"-inf sink P={P}"


def test_splitk_reduce_merges_oracle_partials(attn):
    lens = [300, 77]
    w = W.make_workload("t", batch=2, num_q_heads=8, num_kv_heads=2, dim_qk=128,
                        kv_lens=lens, page_size=32, seed=11, device=DEV, sink=True)
    from tests.helpers import oracle_kv
    k, v = oracle_kv(w, w.k_cache), oracle_kv(w, w.v_cache)
    bounds = [0, 64, 65, 200, 290, 400, 500]          # includes empty slices
    wo, wm, wl = oracle.partials(w.q.cpu(), k, v, w.kv_len.cpu(), bounds, group=w.group,
                                 scale=w.scale)
    t = lambda a: torch.tensor(a, dtype=torch.float32, device=DEV).contiguous()
    out, lse = attn.attn_splitk_reduce(t(wo), t(wm), t(wl), sink=w.sink)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, "reduce of oracle partials")


def test_graph_capture_replays_with_new_lengths(attn):
    lens = [900, 40, 2048]
    w = W.make_workload("t", batch=3, num_q_heads=32, num_kv_heads=8, dim_qk=128,
                        kv_lens=lens, page_size=128, seed=12, device=DEV)
    P, ws_bytes = attn.attn_plan_partitions(3, 3, 32, 8, 128, 2048, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    out = torch.empty(3, 32, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(3, 32, dtype=torch.float32, device=DEV)
    kv_len = w.kv_len.clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        attn.attn_decode(w.q, w.k_cache, w.v_cache, kv_len, group=4, scale=w.scale,
                         max_kv_len=2048, page_table=w.page_table, num_partitions=P,
                         workspace=ws, out=out, lse=lse)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        attn.attn_decode(w.q, w.k_cache, w.v_cache, kv_len, group=4, scale=w.scale,
                         max_kv_len=2048, page_table=w.page_table, num_partitions=P,
                         workspace=ws, out=out, lse=lse, stream=s)
    for new in ([900, 40, 2048], [1, 2047, 513]):
        kv_len.copy_(torch.tensor(new, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        w2 = W.make_workload("t", batch=3, num_q_heads=32, num_kv_heads=8, dim_qk=128,
                             kv_lens=lens, page_size=128, seed=12, device=DEV)
        w2.kv_len_host = new
        w2.kv_len = kv_len
        ref_o, ref_l = oracle_result(w2)
        assert_close(out, lse, ref_o, ref_l, f"graph replay {new}")


@pytest.mark.parametrize("P", [2, 4])
def test_small_split_merged_on_chip(attn, P):
    """2 or 4 partitions on the tensor cores: a cluster of P CTAs splits each
    (sequence, KV head) and merges on chip.  Lengths below one tile per CTA
    leave some CTAs of a cluster without keys; sinks; every group size."""
    for hq, hkv, seed in ((32, 8, 61), (16, 16, 62), (64, 8, 63)):
        w = W.make_workload("t", batch=6, num_q_heads=hq, num_kv_heads=hkv, dim_qk=128,
                            kv_lens=[1, 100, 129, 513, 5000, 0], page_size=64, seed=seed,
                            device=DEV, sink=True)
        out, lse = run(attn, w, P)
        ref_o, ref_l = oracle_result(w)
        assert_close(out, lse, ref_o, ref_l, f"on-chip merge P={P} hq={hq} hkv={hkv}")
        o1, l1 = run(attn, w, 1)
        assert_pair(out, lse, o1, l1, ref_o, ref_l, f"on-chip merge P={P} vs P=1")


def test_llama3_8b_full_size_merged_on_chip(attn):
    w = W.llama3_8b_decode(device=DEV)
    ref_o, ref_l = oracle_result(w)
    for P in (2, 4):
        out, lse = run(attn, w, P)
        assert_close(out, lse, ref_o, ref_l, f"llama3-8b on-chip P={P}")


def test_maximum_batch(attn):
    """The decode kernel's largest batch (2048 sequences, one item table entry
    each) with ragged short lengths, empty sequences included."""
    g = torch.Generator().manual_seed(71)
    lens = [int(x) for x in torch.randint(0, 300, (2048,), generator=g)]
    w = W.make_workload("t", batch=2048, num_q_heads=32, num_kv_heads=8, dim_qk=128,
                        kv_lens=lens, page_size=32, seed=71, device=DEV)
    ref_o, ref_l = oracle_result(w)
    for P in (0, 3):
        out, lse = run(attn, w, P)
        assert_close(out, lse, ref_o, ref_l, f"batch 2048 P={P}")


def test_maximum_partitions(attn):
    """ATTN_MAX_PARTITIONS slices of one tile each over one long sequence:
    the wide reduce merges 1024 partials per (row, head)."""
    w = W.make_workload("t", batch=1, num_q_heads=32, num_kv_heads=8, dim_qk=128,
                        kv_lens=[131072], page_size=128, seed=72, device=DEV, sink=True)
    out, lse = run(attn, w, attn.ATTN_MAX_PARTITIONS)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, "P=1024")


def test_llama3_8b_decode_full_size(attn):
    """The Llama-3-8B-shaped decode batch at full size, auto split-K, against
    the oracle on every (sequence, head)."""
    w = W.llama3_8b_decode(device=DEV)
    out, lse = run(attn, w, 0)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, "llama3-8b auto P")
    o1, l1 = run(attn, w, 1)
    assert_close(o1, l1, ref_o, ref_l, "llama3-8b P=1")


@pytest.mark.parametrize("P", [0, 16, 37, 148])
def test_long_context_with_sinks(attn, P):
    w = W.long_context_decode(device=DEV)
    out, lse = run(attn, w, P)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, f"long context P={P}")


def test_bad_page_entries_are_flagged_not_followed(attn):
    lens = [100, 100]
    w = W.make_workload("t", batch=2, num_q_heads=8, num_kv_heads=2, dim_qk=128,
                        kv_lens=lens, page_size=32, seed=13, device=DEV)
    attn.attn_device_error_flags(clear=True)
    bad = w.page_table.clone()
    bad[1, 2] = w.k_cache.shape[0] + 5          # past the pool
    bad[0, 0] = -3
    attn.attn_decode(w.q, w.k_cache, w.v_cache, w.kv_len, group=4, scale=w.scale,
                     max_kv_len=100, page_table=bad, num_partitions=2)
    flags = attn.attn_device_error_flags(clear=True)
    assert flags & 2, f"bad page not flagged: {flags:#x}"


def test_length_above_plan_is_flagged(attn):
    w = W.make_workload("t", batch=1, num_q_heads=8, num_kv_heads=2, dim_qk=128,
                        kv_lens=[300], page_size=64, seed=14, device=DEV)
    attn.attn_device_error_flags(clear=True)
    out, lse = attn.attn_decode(w.q, w.k_cache, w.v_cache, w.kv_len, group=4, scale=w.scale,
                                max_kv_len=100, page_table=w.page_table, num_partitions=2)
    flags = attn.attn_device_error_flags(clear=True)
    assert flags & 4, f"over-long kv_len not flagged: {flags:#x}"
