"""attn_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (e.g. an engine plugin held to a fixed memory plan).
Its split-K scratch is a fixed array inside the library, so the caller hands
over only inputs and outputs.  Checked against attn_decode (which takes a
caller-allocated workspace) on two calls in a row, through the C ABI.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import pytest
import torch

from split_flash_decoding_gb300 import workloads as W
from tests.helpers import assert_close

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


def reference(attn, w, P):
    out, lse = attn.attn_decode(w.q, w.k_cache, w.v_cache, w.kv_len, group=w.group,
                                scale=w.scale, max_kv_len=w.max_kv_len,
                                page_table=w.page_table, sink=w.sink, num_partitions=P)
    torch.cuda.synchronize()
    return out, lse


def no_alloc(attn, w, P):
    out = torch.empty((w.rows, w.num_q_heads, w.dim_v), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((w.rows, w.num_q_heads), dtype=torch.float32, device=DEV)
    attn.attn_decode_noalloc(w.q, w.k_cache, w.v_cache, w.kv_len, group=w.group,
                             scale=w.scale, max_kv_len=w.max_kv_len, page_table=w.page_table,
                             sink=w.sink, num_partitions=P, out=out, lse=lse)
    torch.cuda.synchronize()
    return out, lse


def test_no_alloc_matches_attn_decode_on_two_calls_in_a_row(attn):
    first = W.make_workload("na1", batch=8, num_q_heads=32, num_kv_heads=8, dim_qk=128,
                            kv_lens=[700, 8000, 1, 4097, 2048, 33, 6000, 512], page_size=128,
                            seed=41, device=DEV, sink=True)
    second = W.make_workload("na2", batch=3, num_q_heads=16, num_kv_heads=4, dim_qk=128,
                             kv_lens=[300, 2500, 90], page_size=64, seed=42, device=DEV)
    for w, P in ((first, 16), (second, 0)):
        ref_o, ref_l = reference(attn, w, P)
        out, lse = no_alloc(attn, w, P)
        assert_close(out, lse, ref_o.float().cpu().numpy(), ref_l.cpu().double().numpy(),
                     f"{w.name} P={P}")


def test_no_alloc_rejects_a_workspace_beyond_its_fixed_scratch(attn):
    w = W.make_workload("na3", batch=64, num_q_heads=32, num_kv_heads=8, dim_qk=128,
                        kv_lens=[64] * 64, page_size=64, seed=43, device=DEV)
    # 64 partitions x 64 rows x 32 heads x 128 channels x 4 B = 64 MiB > 32 MiB
    with pytest.raises(attn.AttnError) as e:
        no_alloc(attn, w, 64)
    assert e.value.status == attn.ATTN_ERR_WORKSPACE
