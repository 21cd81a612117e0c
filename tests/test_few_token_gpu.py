"""GPU parity of few-token decode (a handful of query rows per sequence,
e.g. draft tokens being verified) on the split-K tensor-core decode path:
the rows of a sequence fold onto the MMA's N side next to the group's heads,
so max_q_len * group <= 16 keeps the split-K decode kernel.  Checked against
the fp64 oracle, for P > 1 against P = 1, and paged against contiguous."""
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


def few_workload(q_lens, kv_lens, hq=32, hkv=8, page_size=128, seed=0, causal=True,
                 sink=False):
    return W.make_workload("few", batch=len(q_lens), num_q_heads=hq, num_kv_heads=hkv,
                           dim_qk=128, kv_lens=kv_lens, page_size=page_size, seed=seed,
                           device=DEV, q_lens=q_lens, causal=causal, sink=sink)


def run(attn, w, P, k=None, v=None, page_table="workload"):
    pt = w.page_table if page_table == "workload" else page_table
    out, lse = attn.attn_decode(w.q, w.k_cache if k is None else k,
                                w.v_cache if v is None else v, w.kv_len, group=w.group,
                                scale=w.scale, max_kv_len=w.max_kv_len, page_table=pt,
                                sink=w.sink, q_row_offsets=w.q_row_offsets,
                                max_q_len=w.max_q_len, causal=w.causal, num_partitions=P)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("P", [0, 1, 5])
def test_few_token_matches_oracle(attn, causal, P):
    w = few_workload([1, 2, 3, 4, 2, 1], [700, 130, 1, 2500, 4, 129], seed=61, causal=causal)
    out, lse = run(attn, w, P)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, f"few causal={causal} P={P}")


@pytest.mark.parametrize("hq,hkv,n", [(32, 4, 2), (16, 8, 8), (8, 8, 16), (32, 16, 8)])
def test_groups_and_row_counts(attn, hq, hkv, n):
    q_lens = [n, 1, max(1, n // 2), n]
    w = few_workload(q_lens, [300, 1000, 50, 129], hq=hq, hkv=hkv, seed=62)
    out, lse = run(attn, w, 3)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, f"few hq={hq} hkv={hkv} n={n}")


def test_rows_without_keys_and_empty_sequences(attn):
    # L = 1 with three causal rows: rows 0 and 1 see no key (out 0, lse -inf);
    # a sequence with no rows and one with no keys sit in between.
    w = few_workload([3, 0, 2, 4], [1, 500, 0, 260], seed=63)
    out, lse = run(attn, w, 2)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, "few edge rows")


def test_sinks(attn):
    w = few_workload([2, 4, 1], [400, 90, 1500], seed=64, sink=True)
    out, lse = run(attn, w, 4)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, "few sinks")


def test_split_matches_unsplit(attn):
    w = few_workload([4, 3, 2, 1, 4], [3000, 1500, 7000, 200, 5000], seed=65)
    o1, l1 = run(attn, w, 1)
    ref_o, ref_l = oracle_result(w)
    for P in (2, 4, 7, 16):
        o, l = run(attn, w, P)
        assert_pair(o, l, o1, l1, ref_o, ref_l, f"few P={P} vs P=1")


@pytest.mark.parametrize("page_size", [16, 64, 128])
def test_paged_equals_contiguous_bitwise(attn, page_size):
    w = few_workload([2, 4, 1, 3], [900, 129, 2048, 77], page_size=page_size, seed=66)
    c = W.contiguous_copy(w)
    o_p, l_p = run(attn, w, 6)
    o_c, l_c = run(attn, w, 6, k=c.k_cache, v=c.v_cache, page_table=None)
    assert bits_equal(o_p, o_c) and bits_equal(l_p, l_c)


def test_long_context_two_rows(attn):
    w = few_workload([2, 2], [65536, 40000], seed=67, sink=True)
    out, lse = run(attn, w, 0)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, "few long context")


def test_workload_full_size_sampled(attn):
    w = W.few_token_decode(device=DEV)
    out, lse = run(attn, w, 0)
    offs = w.q_row_offsets.cpu().tolist()
    rows = [offs[b] + (offs[b + 1] - offs[b] - 1) for b in range(0, w.batch, 5)]
    heads = [(7 * i) % w.num_q_heads for i in range(len(rows))]
    ref_o, ref_l = oracle_result(w, sample=(rows, heads))
    ri = torch.tensor(rows)
    hi = torch.tensor(heads)
    assert_close(out[ri, hi], lse[ri, hi], ref_o, ref_l, "few-token workload sampled")


def test_graph_capture_replays_with_new_lengths(attn):
    """Draft rows on the balanced split: one captured call replayed with other
    cache lengths (the rows per sequence fixed by the captured offsets)."""
    q_lens, lens = [1, 4, 2, 3], [700, 2500, 130, 64]
    w = few_workload(q_lens, lens, seed=69, sink=True)
    P, ws_bytes = attn.attn_plan_partitions(4, w.rows, 32, 8, 128, 2500, 0, max_q_len=4)
    assert P == attn.ATTN_PARTITIONS_BALANCED
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    out = torch.empty(w.rows, 32, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(w.rows, 32, dtype=torch.float32, device=DEV)
    kv_len = w.kv_len.clone()
    s = torch.cuda.Stream()

    def call():
        attn.attn_decode(w.q, w.k_cache, w.v_cache, kv_len, group=4, scale=w.scale,
                         max_kv_len=2500, page_table=w.page_table, sink=w.sink,
                         q_row_offsets=w.q_row_offsets, max_q_len=4, causal=True,
                         num_partitions=P, workspace=ws, out=out, lse=lse, stream=s)

    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for new in ([700, 2500, 130, 64], [4, 1999, 128, 3]):
        kv_len.copy_(torch.tensor(new, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        w2 = few_workload(q_lens, lens, seed=69, sink=True)
        w2.kv_len_host = new
        w2.kv_len = kv_len
        ref_o, ref_l = oracle_result(w2)
        assert_close(out, lse, ref_o, ref_l, f"few-token graph replay {new}")
