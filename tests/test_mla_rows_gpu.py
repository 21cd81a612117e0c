"""GPU parity of multi-row MLA decode (attn_mla_decode_rows: the current
token plus draft tokens per sequence, causal) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

from split_flash_decoding_gb300 import workloads as W
from tests.helpers import assert_close, assert_consistent, bits_equal, oracle_result, full_rows_sample

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SCALE = 1.0 / math.sqrt(192.0)


@pytest.fixture(scope="module")
def attn():
    from split_flash_decoding_gb300 import build
    build.build()
    from split_flash_decoding_gb300 import attn as a
    a.attn_device_error_flags(clear=True)
    yield a
    assert a.attn_device_error_flags(clear=True) == 0


def rows_workload(lens, q_lens, page_size=64, seed=0, sink=False, causal=True):
    return W.make_workload("mla_rows", batch=len(lens), num_q_heads=128, num_kv_heads=1,
                           dim_qk=576, dim_v=512, mla=True, kv_lens=lens, page_size=page_size,
                           seed=seed, device=DEV, sink=sink, scale=SCALE, q_lens=q_lens,
                           causal=causal)


def run(attn, w, P=0, sink="workload"):
    s = w.sink if sink == "workload" else sink
    out, lse = attn.attn_mla_decode_rows(w.q, w.k_cache, w.kv_len, w.q_row_offsets,
                                         scale=w.scale, max_kv_len=w.max_kv_len,
                                         causal=w.causal, page_table=w.page_table, sink=s,
                                         num_partitions=P)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("P", [0, 1, 2, 5])
def test_mla_rows_small_matches_oracle(attn, P):
    # rows per sequence 1..4; short sequences leave early rows with no key
    w = rows_workload([1, 2, 63, 64, 65, 700, 3], [4, 2, 3, 1, 2, 4, 4], seed=41)
    out, lse = run(attn, w, P)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, f"mla rows P={P}")


def test_mla_rows_non_causal(attn):
    w = rows_workload([130, 1000, 5], [3, 2, 4], seed=42, causal=False)
    for P in (1, 3):
        out, lse = run(attn, w, P)
        ref_o, ref_l = oracle_result(w)
        assert_close(out, lse, ref_o, ref_l, f"mla rows non-causal P={P}")


def test_one_row_per_sequence_equals_single_token_call_bitwise(attn):
    w = rows_workload([5, 130, 1000, 4096], [1, 1, 1, 1], seed=43)
    for P in (0, 1, 3):
        o1, l1 = run(attn, w, P)
        o2, l2 = attn.attn_mla_decode(w.q, w.k_cache, w.kv_len, scale=w.scale,
                                      max_kv_len=w.max_kv_len, page_table=w.page_table,
                                      num_partitions=P)
        torch.cuda.synchronize()
        assert bits_equal(o1, o2) and bits_equal(l1, l2), f"P={P}"


@pytest.mark.parametrize("page_size", [16, 128])
def test_mla_rows_paged_equals_contiguous_bitwise(attn, page_size):
    w = rows_workload([300, 77, 2000], [2, 4, 3], page_size=page_size, seed=44)
    c = W.contiguous_copy(w)
    for P in (1, 4):
        o1, l1 = run(attn, w, P)
        o2, l2 = run(attn, c, P)
        assert bits_equal(o1, o2) and bits_equal(l1, l2), f"page {page_size} P={P}"


def test_mla_rows_sinks_and_empty(attn):
    w = rows_workload([0, 300, 2], [2, 3, 4], seed=45, sink=True)
    no_sink = torch.full((128,), -math.inf, dtype=torch.float32, device=DEV)
    for P in (0, 1, 4):
        out, lse = run(attn, w, P)
        ref_o, ref_l = oracle_result(w)
        assert_close(out, lse, ref_o, ref_l, f"mla rows sinks P={P}")
        o_inf, l_inf = run(attn, w, P, sink=no_sink)
        o_none, l_none = run(attn, w, P, sink=None)
        assert bits_equal(o_inf, o_none) and bits_equal(l_inf, l_none)


def test_mla_rows_split_k_matches_single_partition(attn):
    w = rows_workload([4096, 1500, 64, 9000], [2, 2, 4, 3], seed=46)
    ref_o, ref_l = oracle_result(w)
    o1, l1 = run(attn, w, 1)
    assert_close(o1, l1, ref_o, ref_l, "mla rows P=1")
    for P in (2, 9, 40):
        oP, lP = run(attn, w, P)
        assert_close(oP, lP, ref_o, ref_l, f"mla rows P={P}")


def test_deepseek_v3_mtp_full_size_sampled(attn):
    """The DeepSeek-V3-shaped batch with one draft token per sequence at full
    size and the automatic split (the launch the benchmark times); the oracle
    checks 8 heads of every query row, and P=1 vs auto P every output."""
    w = W.deepseek_v3_mtp_decode(device=DEV)
    out, lse = run(attn, w, 0)
    row_len = [w.kv_len_host[b] for b in range(w.batch)
               for _ in range(w.q_row_offsets_host[b + 1] - w.q_row_offsets_host[b])]
    rows, heads = full_rows_sample(row_len, w.num_q_heads, 4, seed=2)
    ref_o, ref_l = oracle_result(w, sample=(rows, heads))
    ri, hi = torch.as_tensor(rows, device=DEV), torch.as_tensor(heads, device=DEV)
    assert_close(out[ri, hi], lse[ri, hi], ref_o, ref_l, "deepseek-v3 mtp sampled")
    o1, l1 = run(attn, w, 1)
    assert_consistent(out, lse, o1, l1, float(ref_o.eps.max()),
                      "deepseek-v3 mtp auto P vs P=1")
