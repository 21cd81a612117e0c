"""GPU parity of sparse top-k MLA decode (attn_mla_decode_sparse) against the
fp64 oracle: each sequence attends only to the cache rows its index list
names (one KV head, K depth 576, V = K[:, :512], 128 heads)."""
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


def sparse_workload(ctx, topk, page_size=64, seed=0, sink=False, replace_rows=False):
    return W.make_sparse_mla_workload("sparse", ctx_lens=ctx, topk=topk, page_size=page_size,
                                      seed=seed, device=DEV, sink=sink, scale=SCALE,
                                      replace_rows=replace_rows)


def run(attn, w, P=0, sink="workload", cache=None, indices=None, topk=None):
    s = w.sink if sink == "workload" else sink
    out, lse = attn.attn_mla_decode_sparse(
        w.q, w.k_cache if cache is None else cache, w.indices if indices is None else indices,
        w.kv_len if topk is None else topk, scale=w.scale, sink=s, num_partitions=P)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("P", [0, 1, 2, 5])
def test_sparse_small_matches_oracle(attn, P):
    w = sparse_workload([1, 70, 700, 3000, 64, 301], topk=300, seed=31)
    out, lse = run(attn, w, P)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, f"sparse P={P}")


def test_sparse_repeated_rows(attn):
    """Rows drawn with repetition: a row named twice counts twice."""
    w = sparse_workload([50, 400, 2000], topk=513, seed=32, replace_rows=True)
    assert any(len(set(w.indices[b, :n].tolist())) < n for b, n in enumerate(w.kv_len_host))
    for P in (0, 1, 3):
        out, lse = run(attn, w, P)
        ref_o, ref_l = oracle_result(w)
        assert_close(out, lse, ref_o, ref_l, f"sparse repeated P={P}")


def test_sparse_row_mapping_is_layout_independent_bitwise(attn):
    """The same pool viewed with page sizes 64, 16 and 1 names the same rows,
    so the results agree bit for bit."""
    w = sparse_workload([900, 2500, 130], topk=640, seed=33)
    n, ps = w.k_cache.shape[:2]
    for P in (0, 1, 4):
        o64, l64 = run(attn, w, P)
        for new_ps in (16, 1):
            view = w.k_cache.view(n * ps // new_ps, new_ps, 1, 576)
            o, l = run(attn, w, P, cache=view)
            assert bits_equal(o, o64) and bits_equal(l, l64), f"page {new_ps} P={P}"
    ref_o, ref_l = oracle_result(w)
    assert_close(o64, l64, ref_o, ref_l, "sparse layouts")


def test_sparse_identity_indices_equal_dense_paged_bitwise(attn):
    """Indices naming tokens 0..L-1 in order reproduce the dense paged MLA
    call bit for bit (same slices, same tile contents)."""
    lens = [5, 130, 1000, 64]
    w = W.make_workload("mla", batch=4, num_q_heads=128, num_kv_heads=1, dim_qk=576, dim_v=512,
                        mla=True, kv_lens=lens, page_size=64, seed=34, device=DEV, scale=SCALE)
    pt = w.page_table.cpu().long()
    idx = torch.full((4, max(lens)), -1, dtype=torch.int64)
    for b, L in enumerate(lens):
        t = torch.arange(L)
        idx[b, :L] = pt[b, t // 64] * 64 + t % 64
    idx = idx.to(torch.int32).to(DEV)
    for P in (0, 1, 3):
        od, ld = attn.attn_mla_decode(w.q, w.k_cache, w.kv_len, scale=w.scale,
                                      max_kv_len=max(lens), page_table=w.page_table,
                                      num_partitions=P)
        os_, ls = attn.attn_mla_decode_sparse(w.q, w.k_cache, idx, w.kv_len, scale=w.scale,
                                              num_partitions=P)
        torch.cuda.synchronize()
        assert bits_equal(od, os_) and bits_equal(ld, ls), f"P={P}"


def test_sparse_sinks_and_empty(attn):
    w = sparse_workload([0, 300, 2000, 7], topk=1024, seed=35, sink=True)
    assert w.kv_len_host[0] == 0
    no_sink = torch.full((128,), -math.inf, dtype=torch.float32, device=DEV)
    for P in (0, 1, 4):
        out, lse = run(attn, w, P)
        ref_o, ref_l = oracle_result(w)
        assert_close(out, lse, ref_o, ref_l, f"sparse sinks P={P}")
        o_inf, l_inf = run(attn, w, P, sink=no_sink)
        o_none, l_none = run(attn, w, P, sink=None)
        assert bits_equal(o_inf, o_none) and bits_equal(l_inf, l_none)
    # all sequences empty: out = 0, lse = -inf without sinks
    zero = torch.zeros(4, dtype=torch.int32, device=DEV)
    out, lse = run(attn, w, 2, sink=None, topk=zero)
    assert torch.count_nonzero(out.float()) == 0
    assert bool(torch.isneginf(lse).all())


def test_sparse_split_k_matches_single_partition(attn):
    w = sparse_workload([4096, 1500, 64, 9000], topk=2048, seed=36)
    ref_o, ref_l = oracle_result(w)
    o1, l1 = run(attn, w, 1)
    assert_close(o1, l1, ref_o, ref_l, "sparse P=1")
    for P in (2, 9, 32):
        oP, lP = run(attn, w, P)
        assert_close(oP, lP, ref_o, ref_l, f"sparse P={P}")


def test_sparse_single_key_and_unit_stride(attn):
    """indices_stride 1, one key per sequence: out is that row's V exactly up
    to bf16 rounding and lse is its score."""
    w = sparse_workload([40, 1, 900], topk=1, seed=39)
    assert w.indices.shape[1] == 1
    for P in (1, 2):
        out, lse = run(attn, w, P)
        ref_o, ref_l = oracle_result(w)
        assert_close(out, lse, ref_o, ref_l, f"sparse top-1 P={P}")


def test_sparse_entries_past_topk_are_not_read(attn):
    """Entries past topk_lengths[b] may hold anything, out-of-range rows
    included: they are never read and set no error bit."""
    w = sparse_workload([800, 3000], topk=1000, seed=37)
    o1, l1 = run(attn, w, 2)
    junk = w.indices.clone()
    n0 = w.kv_len_host[0]
    junk[0, n0:] = 2 ** 31 - 1
    o2, l2 = run(attn, w, 2, indices=junk)
    assert bits_equal(o1, o2) and bits_equal(l1, l2)
    assert attn.attn_device_error_flags(clear=True) == 0


def test_sparse_bad_index_and_length_set_error_bits(attn):
    """An index outside the pool is not read and sets bit 1; a count above
    indices_stride (or below 0) is clamped and sets bit 2."""
    w = sparse_workload([500, 600], topk=256, seed=38)
    rows = w.k_cache.shape[0] * w.k_cache.shape[1]
    BAL = attn.ATTN_PARTITIONS_BALANCED   # the first cluster checks the counts there
    for P1, P2 in ((1, 2), (BAL, BAL)):
        bad = w.indices.clone()
        bad[1, 5] = rows
        run(attn, w, P1, indices=bad)
        assert attn.attn_device_error_flags(clear=True) == 2
        bad[1, 5] = -3
        run(attn, w, P2, indices=bad)
        assert attn.attn_device_error_flags(clear=True) == 2
        too_long = torch.tensor([256, 300], dtype=torch.int32, device=DEV)
        run(attn, w, P2, topk=too_long)
        assert attn.attn_device_error_flags(clear=True) == 4
        negative = torch.tensor([-1, 10], dtype=torch.int32, device=DEV)
        run(attn, w, P1, topk=negative)
        assert attn.attn_device_error_flags(clear=True) == 4
        # the context is still usable and correct afterwards
        out, lse = run(attn, w, P2)
        ref_o, ref_l = oracle_result(w)
        assert_close(out, lse, ref_o, ref_l, f"sparse after errors, P={P2}")


def test_deepseek_v32_sparse_full_size_sampled(attn):
    """The DeepSeek-V3.2-shaped batch at full size with the automatic split
    (the launch the benchmark times); the oracle checks 8 heads of every
    sequence, and P=1 vs auto P is checked on every output."""
    w = W.deepseek_v32_sparse_mla_decode(device=DEV)
    out, lse = run(attn, w, 0)
    rows, heads = full_rows_sample(w.kv_len_host, w.num_q_heads, 4, seed=3)
    ref_o, ref_l = oracle_result(w, sample=(rows, heads))
    ri, hi = torch.as_tensor(rows, device=DEV), torch.as_tensor(heads, device=DEV)
    assert_close(out[ri, hi], lse[ri, hi], ref_o, ref_l, "deepseek-v3.2 sparse sampled")
    o1, l1 = run(attn, w, 1)
    assert_consistent(out, lse, o1, l1, float(ref_o.eps.max()),
                      "deepseek-v3.2 sparse auto P vs P=1")


def test_graph_capture_replays_with_new_index_lists(attn):
    """One captured sparse call replayed with other index lists and counts
    (lists swapped between sequences, shortened, one emptied)."""
    w = sparse_workload([900, 2500, 130, 3000], topk=640, seed=36)
    stride = w.indices.shape[1]
    P, ws_bytes = attn.attn_plan_partitions(4, 4, 128, 1, 512, stride, 0)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=DEV)
    out = torch.empty(4, 128, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(4, 128, dtype=torch.float32, device=DEV)
    idx = w.indices.clone()
    cnt = w.kv_len.clone()
    s = torch.cuda.Stream()

    def call():
        attn.attn_mla_decode_sparse(w.q, w.k_cache, idx, cnt, scale=w.scale, num_partitions=P,
                                    workspace=ws, out=out, lse=lse, stream=s)

    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    swapped = w.indices.clone()
    swapped[0], swapped[3] = w.indices[3].clone(), w.indices[0].clone()
    for new_idx, new_cnt in ((w.indices, list(w.kv_len_host)), (swapped, [640, 1, 0, 300])):
        idx.copy_(new_idx)
        cnt.copy_(torch.tensor(new_cnt, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        w2 = sparse_workload([900, 2500, 130, 3000], topk=640, seed=36)
        w2.indices = idx
        w2.kv_len = cnt
        w2.kv_len_host = new_cnt
        ref_o, ref_l = oracle_result(w2)
        assert_close(out, lse, ref_o, ref_l, f"sparse graph replay {new_cnt}")
