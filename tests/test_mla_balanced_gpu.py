"""GPU parity of the balanced MLA split (num_partitions 0, requested from the
planner as ATTN_PARTITIONS_BALANCED) against the fp64 oracle.  The key tiles of every query row, concatenated, are dealt out in
equal contiguous ranges to one wave of two-CTA clusters; a cluster walks the
rows its range meets, and rows cut by a range boundary are merged by the
reduce from consecutive workspace slots."""
import math
import random

import numpy as np
import pytest
import torch

from split_flash_decoding_gb300 import workloads as W
from tests.helpers import assert_close, assert_consistent, bits_equal, oracle_result

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


def mla_workload(lens, page_size=64, seed=0, sink=False, q_lens=None, causal=False):
    return W.make_workload("mla_balanced", batch=len(lens), num_q_heads=128, num_kv_heads=1,
                           dim_qk=576, dim_v=512, mla=True, kv_lens=lens, page_size=page_size,
                           seed=seed, device=DEV, sink=sink, scale=SCALE, q_lens=q_lens,
                           causal=causal)


def run(attn, w, P, kv_len=None, max_kv_len=None, sink="workload"):
    s = w.sink if sink == "workload" else sink
    kvl = w.kv_len if kv_len is None else kv_len
    mkl = max(1, w.max_kv_len) if max_kv_len is None else max_kv_len
    if w.q_row_offsets is not None:
        out, lse = attn.attn_mla_decode_rows(w.q, w.k_cache, kvl, w.q_row_offsets, scale=w.scale,
                                             max_kv_len=mkl, causal=w.causal,
                                             page_table=w.page_table, sink=s, num_partitions=P)
    else:
        out, lse = attn.attn_mla_decode(w.q, w.k_cache, kvl, scale=w.scale, max_kv_len=mkl,
                                        page_table=w.page_table, sink=s, num_partitions=P)
    torch.cuda.synchronize()
    return out, lse


def sampled_check(attn, w, out, lse, heads_per_row, seed, what):
    rng = np.random.default_rng(seed)
    n = out.shape[0]
    rows = np.repeat(np.arange(n), heads_per_row)
    heads = np.concatenate([rng.choice(128, heads_per_row, replace=False) for _ in range(n)])
    ref_o, ref_l = oracle_result(w, sample=(rows, heads))
    ri, hi = torch.as_tensor(rows, device=DEV), torch.as_tensor(heads, device=DEV)
    assert_close(out[ri, hi], lse[ri, hi], ref_o, ref_l, what)
    return float(ref_o.eps.max())


def test_balanced_many_rows_per_cluster(attn):
    """300 rows of 0..700 keys (a few long ones): every cluster walks several
    rows, some rows are empty, some are cut by one or two range ends."""
    rng = random.Random(71)
    lens = [rng.choice([0, 1, 63, 64, 65, 129]) if rng.random() < 0.3 else rng.randint(1, 700)
            for _ in range(300)]
    lens[17], lens[200] = 9000, 5000
    w = mla_workload(lens, seed=71, sink=True)
    out, lse = run(attn, w, attn.ATTN_PARTITIONS_BALANCED)
    eps = sampled_check(attn, w, out, lse, 4, 1, "balanced many rows")
    o1, l1 = run(attn, w, 1)
    assert_consistent(out, lse, o1, l1, eps, "balanced vs P=1, many rows")


def test_balanced_one_long_row_spans_every_cluster(attn):
    """One row of 40000 keys: each cluster takes ~1/76 of it and the reduce
    merges one partial per cluster."""
    w = mla_workload([40000], seed=72)
    out, lse = run(attn, w, attn.ATTN_PARTITIONS_BALANCED)
    eps = sampled_check(attn, w, out, lse, 16, 2, "balanced one long row")
    o1, l1 = run(attn, w, 1)
    assert_consistent(out, lse, o1, l1, eps, "balanced vs P=1, one row")


@pytest.mark.parametrize("sink", [False, True])
def test_balanced_fewer_tiles_than_clusters(attn, sink):
    """Four tiles in all: most clusters have nothing to do, a two-tile row is
    split across two clusters, the empty row is written by the reduce."""
    w = mla_workload([100, 30, 0, 1], seed=73, sink=sink)
    out, lse = run(attn, w, attn.ATTN_PARTITIONS_BALANCED)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, f"balanced few tiles sink={sink}")
    if not sink:
        assert torch.count_nonzero(out[2].float()) == 0
        assert bool(torch.isneginf(lse[2]).all())


def test_balanced_all_rows_empty(attn):
    w = mla_workload([0, 0, 0], seed=74, sink=True)
    out, lse = run(attn, w, attn.ATTN_PARTITIONS_BALANCED)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, "balanced all empty, sinks")
    out, lse = run(attn, w, attn.ATTN_PARTITIONS_BALANCED, sink=None)
    assert torch.count_nonzero(out.float()) == 0
    assert bool(torch.isneginf(lse).all())


@pytest.mark.parametrize("page_size", [8, 128])
def test_balanced_paged_equals_contiguous_bitwise(attn, page_size):
    w = mla_workload([5, 130, 1000, 77, 4000, 64], page_size=page_size, seed=75)
    c = W.contiguous_copy(w)
    o1, l1 = run(attn, w, attn.ATTN_PARTITIONS_BALANCED)
    o2, l2 = run(attn, c, 0)
    assert bits_equal(o1, o2) and bits_equal(l1, l2)
    ref_o, ref_l = oracle_result(w)
    assert_close(o1, l1, ref_o, ref_l, f"balanced page {page_size}")


def test_balanced_rows_causal(attn):
    """Several causal query rows per sequence: each row has its own visible
    length, so the rows of one sequence carry different tile counts."""
    lens = [1, 2, 63, 64, 65, 700, 3, 3000, 129]
    q_lens = [4, 2, 3, 1, 2, 4, 4, 3, 2]
    w = mla_workload(lens, seed=76, q_lens=q_lens, causal=True, sink=True)
    out, lse = run(attn, w, attn.ATTN_PARTITIONS_BALANCED)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, "balanced causal rows")


def test_balanced_length_over_max_is_clamped_and_reported(attn):
    """kv_len above max_kv_len reads max_kv_len keys and sets bit 2."""
    w = mla_workload([3000, 500, 2500], seed=77)
    out, lse = run(attn, w, attn.ATTN_PARTITIONS_BALANCED, max_kv_len=2048)
    assert attn.attn_device_error_flags(clear=True) == 4
    clamped = torch.clamp(w.kv_len, max=2048)
    o2, l2 = run(attn, w, attn.ATTN_PARTITIONS_BALANCED, kv_len=clamped, max_kv_len=2048)
    assert attn.attn_device_error_flags(clear=True) == 0
    assert bits_equal(out, o2) and bits_equal(lse, l2)


def test_balanced_repeated_calls_reuse_workspace(attn):
    """Back-to-back calls with one workspace and different lengths: each
    call's plan replaces the last one's (the balanced workspace depends on
    the row count only)."""
    rng = random.Random(78)
    BAL = attn.ATTN_PARTITIONS_BALANCED
    P, ws_bytes = attn.attn_plan_partitions(6, 6, 128, 1, 512, 6000, BAL)
    assert P == 0
    assert attn.attn_plan_partitions(6, 6, 128, 1, 512, 600, 0) == (P, ws_bytes)
    assert attn.attn_plan_partitions(6, 6, 128, 1, 512, 60, BAL) == (P, ws_bytes)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    for i in range(3):
        lens = [rng.randint(0, 6000) for _ in range(6)]
        w = mla_workload(lens, seed=80 + i)
        out, lse = attn.attn_mla_decode(w.q, w.k_cache, w.kv_len, scale=w.scale,
                                        max_kv_len=w.max_kv_len, page_table=w.page_table,
                                        num_partitions=BAL, workspace=ws)
        torch.cuda.synchronize()
        eps = sampled_check(attn, w, out, lse, 8, 20 + i, f"call {i}")
        o1, l1 = run(attn, w, 1)
        assert_consistent(out, lse, o1, l1, eps, f"call {i} vs P=1")


@pytest.mark.parametrize("rows_per_seq", [1, 2])
def test_balanced_plan_over_many_sequences(attn, rows_per_seq):
    """More sequences than the 32 lanes of the warp that finds a cluster's
    range: each lane sums a chunk of sequences before the warp scan, and
    the lane holding a range end walks its chunk's rows.  Forced balanced
    split (the planner would not split rows this short)."""
    rng = random.Random(90 + rows_per_seq)
    batch = 1500 if rows_per_seq == 1 else 1100
    lens = [rng.choice([0, 1, 64, 65]) if rng.random() < 0.2 else rng.randint(1, 300)
            for _ in range(batch)]
    q_lens = None if rows_per_seq == 1 else [rng.randint(1, 3) for _ in range(batch)]
    if q_lens is not None:
        lens = [max(L, n) for L, n in zip(lens, q_lens)]
    w = mla_workload(lens, seed=95 + rows_per_seq, q_lens=q_lens, causal=q_lens is not None,
                     sink=True)
    out, lse = run(attn, w, attn.ATTN_PARTITIONS_BALANCED)
    eps = sampled_check(attn, w, out, lse, 1, 3, f"balanced, {batch} sequences")
    o1, l1 = run(attn, w, 1)
    assert_consistent(out, lse, o1, l1, eps, f"balanced vs P=1, {batch} sequences")


def test_bad_page_sets_error_bit_and_context_survives(attn):
    """A page-table entry outside the pool is not read and sets bit 1, under
    the balanced split and unsplit; the next call is correct."""
    w = mla_workload([700, 300, 1500], seed=79)
    bad = w.page_table.clone()
    bad[2, 3] = w.k_cache.shape[0]          # one past the last page
    for P in (attn.ATTN_PARTITIONS_BALANCED, 1):
        attn.attn_mla_decode(w.q, w.k_cache, w.kv_len, scale=w.scale, max_kv_len=w.max_kv_len,
                             page_table=bad, num_partitions=P)
        torch.cuda.synchronize()
        assert attn.attn_device_error_flags(clear=True) == 2
    out, lse = run(attn, w, attn.ATTN_PARTITIONS_BALANCED)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, "balanced after a bad page")


def test_graph_capture_replays_with_new_lengths(attn):
    """The balanced split is planned on the device from kv_len, so one
    captured call (decode, reduce) serves any lengths up to the planned
    maximum: replayed with other lengths, including an empty row."""
    lens = [3000, 64, 1500, 700]
    w = mla_workload(lens, seed=90)
    P, ws_bytes = attn.attn_plan_partitions(4, 4, 128, 1, 512, 3000, 0)
    assert P == 0
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    out = torch.empty(4, 128, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(4, 128, dtype=torch.float32, device=DEV)
    kv_len = w.kv_len.clone()
    s = torch.cuda.Stream()

    def call():
        attn.attn_mla_decode(w.q, w.k_cache, kv_len, scale=w.scale, max_kv_len=3000,
                             page_table=w.page_table, num_partitions=P, workspace=ws, out=out,
                             lse=lse, stream=s)

    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for new in ([3000, 64, 1500, 700], [1, 2999, 65, 0]):
        kv_len.copy_(torch.tensor(new, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        w2 = mla_workload(lens, seed=90)
        w2.kv_len_host = new
        w2.kv_len = kv_len
        ref_o, ref_l = oracle_result(w2)
        assert_close(out, lse, ref_o, ref_l, f"mla graph replay {new}")
