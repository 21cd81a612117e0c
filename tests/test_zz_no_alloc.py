"""attn_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (e.g. an engine plugin held to a memory plan fixed at
start-up, or a C program with no allocator).  Its split-K scratch is a fixed
array inside the library, so the caller hands over only inputs and outputs.

Checked through the C ABI on two calls in a row against attn_decode (which
takes a caller-allocated workspace) and against the fp64 oracle, for
single-token decode and for draft rows folded onto the split-K decode kernel
(where the caller's partition count must be honoured, not dropped).

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import pytest
import torch

from split_flash_decoding_gb300 import workloads as W
from tests.helpers import assert_close, assert_pair, bits_equal, oracle_result

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


def kw(w, P):
    return dict(group=w.group, scale=w.scale, max_kv_len=w.max_kv_len,
                page_table=w.page_table, sink=w.sink, q_row_offsets=w.q_row_offsets,
                max_q_len=w.max_q_len, causal=w.causal, num_partitions=P)


def with_workspace(attn, w, P):
    out, lse = attn.attn_decode(w.q, w.k_cache, w.v_cache, w.kv_len, **kw(w, P))
    torch.cuda.synchronize()
    return out, lse


def no_alloc(attn, w, P):
    out = torch.empty((w.rows, w.num_q_heads, w.dim_v), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((w.rows, w.num_q_heads), dtype=torch.float32, device=DEV)
    attn.attn_decode_noalloc(w.q, w.k_cache, w.v_cache, w.kv_len, out=out, lse=lse,
                             **kw(w, P))
    torch.cuda.synchronize()
    return out, lse


def test_no_alloc_matches_attn_decode_on_two_calls_in_a_row(attn):
    first = W.make_workload("na1", batch=8, num_q_heads=32, num_kv_heads=8, dim_qk=128,
                            kv_lens=[700, 8000, 1, 4097, 2048, 33, 6000, 512], page_size=128,
                            seed=41, device=DEV, sink=True)
    second = W.make_workload("na2", batch=3, num_q_heads=16, num_kv_heads=4, dim_qk=128,
                             kv_lens=[300, 2500, 90], page_size=64, seed=42, device=DEV)
    for w, P in ((first, 16), (second, 0)):
        ref_o, ref_l = oracle_result(w)
        o_ws, l_ws = with_workspace(attn, w, P)
        out, lse = no_alloc(attn, w, P)
        # the same plan, the same kernels: the same bits as attn_decode
        assert bits_equal(out, o_ws) and bits_equal(lse, l_ws), f"{w.name} P={P}"
        assert_close(out, lse, ref_o, ref_l, f"{w.name} P={P} against the oracle")


def test_no_alloc_draft_rows_keep_the_callers_split(attn):
    """Draft rows (1-4 per sequence, group 4) fold onto the split-K decode
    kernel: P = 3 goes through the scratch array (P = 1 would write no
    partial), P = 2 merges on chip; both against the oracle and P = 1."""
    w = W.make_workload("na4", batch=5, num_q_heads=32, num_kv_heads=8, dim_qk=128,
                        kv_lens=[900, 3000, 5, 2049, 130], q_lens=[2, 4, 1, 3, 4],
                        page_size=64, seed=44, device=DEV, causal=True, sink=True)
    ref_o, ref_l = oracle_result(w)
    o1, l1 = no_alloc(attn, w, 1)
    for P in (3, 2, 0):
        o_ws, l_ws = with_workspace(attn, w, P)
        out, lse = no_alloc(attn, w, P)
        assert bits_equal(out, o_ws) and bits_equal(lse, l_ws), f"draft rows P={P}"
        assert_pair(out, lse, o1, l1, ref_o, ref_l, f"draft rows P={P} vs P=1")


def test_no_alloc_rejects_a_workspace_beyond_its_fixed_scratch(attn):
    w = W.make_workload("na3", batch=64, num_q_heads=32, num_kv_heads=8, dim_qk=128,
                        kv_lens=[64] * 64, page_size=64, seed=43, device=DEV)
    # 64 partitions x 64 rows x 32 heads x 128 channels x 4 B = 64 MiB > 32 MiB
    with pytest.raises(attn.AttnError) as e:
        no_alloc(attn, w, 64)
    assert e.value.status == attn.ATTN_ERR_WORKSPACE
