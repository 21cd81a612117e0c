"""GPU parity of the balanced split of the tensor-core GQA decode kernel
(attn_decode with num_partitions ATTN_PARTITIONS_BALANCED, the automatic
choice for at most eight (sequence, KV head) units per SM): the 128-key
tiles of every unit, concatenated, are dealt out in equal contiguous ranges
to one CTA per SM; units a range end cuts leave partials that the split-K
reduce merges through a slot table.  Against the fp64 oracle, against one
partition, and paged against contiguous bit for bit."""
import numpy as np
import pytest
import torch

from split_flash_decoding_gb300 import workloads as W
from tests.helpers import (assert_close, assert_consistent, assert_pair, bits_equal,
                           full_rows_sample, oracle_result)

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


def run(attn, w, P, **kw):
    out, lse = attn.attn_decode(w.q, w.k_cache, w.v_cache, w.kv_len, group=w.group,
                                scale=w.scale, max_kv_len=kw.pop("max_kv_len", w.max_kv_len),
                                page_table=w.page_table, sink=w.sink,
                                q_row_offsets=w.q_row_offsets, max_q_len=w.max_q_len,
                                causal=w.causal, num_partitions=P, **kw)
    torch.cuda.synchronize()
    return out, lse


def workload(lens, q_lens=None, hq=32, hkv=8, page_size=64, seed=0, sink=False):
    return W.make_workload("bal", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, dim_qk=128,
                           kv_lens=lens, page_size=page_size, seed=seed, device=DEV,
                           q_lens=q_lens, causal=q_lens is not None, sink=sink)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 16), (64, 8), (8, 4)])
def test_balanced_matches_oracle_and_one_partition(attn, hq, hkv):
    """Ragged lengths with empty, one-key, one-tile and tile-boundary units:
    every CTA's range cuts some units and holds others whole."""
    rng = np.random.default_rng(hq + hkv)
    lens = [0, 1, 127, 128, 129, 3000] + rng.integers(1, 9000, size=10).tolist()
    w = workload(lens, hq=hq, hkv=hkv, seed=200 + hq, sink=True)
    BAL = attn.ATTN_PARTITIONS_BALANCED
    assert attn.attn_plan_partitions(w.batch, w.rows, hq, hkv, 128, w.max_kv_len, 0)[0] == BAL
    ob, lb = run(attn, w, BAL)
    o1, l1 = run(attn, w, 1)
    ref_o, ref_l = oracle_result(w)
    assert_pair(ob, lb, o1, l1, ref_o, ref_l, f"balanced hq={hq} hkv={hkv}")
    oa, la = run(attn, w, 0)                 # the automatic choice is this split
    assert bits_equal(oa, ob) and bits_equal(la, lb)


@pytest.mark.parametrize("causal", [True, False])
def test_balanced_draft_rows(attn, causal):
    """Draft rows folded onto the kernel's 16 columns (1-4 rows, group 4):
    a unit's partial holds every row of its sequence."""
    q_lens = [1, 2, 3, 4, 4, 1, 2, 3, 4, 1, 3, 2]
    lens = [700, 130, 4, 2500, 9000, 1, 4096, 4097, 128, 0, 6000, 3]
    lens = [max(L, n) for L, n in zip(lens, q_lens)]
    w = W.make_workload("bal_rows", batch=len(lens), num_q_heads=32, num_kv_heads=8,
                        dim_qk=128, kv_lens=lens, page_size=128, seed=211, device=DEV,
                        q_lens=q_lens, causal=causal, sink=True)
    ob, lb = run(attn, w, attn.ATTN_PARTITIONS_BALANCED)
    o1, l1 = run(attn, w, 1)
    ref_o, ref_l = oracle_result(w)
    assert_pair(ob, lb, o1, l1, ref_o, ref_l, f"balanced draft rows causal={causal}")


@pytest.mark.parametrize("page_size", [8, 64, 256])
def test_balanced_paged_equals_contiguous_bitwise(attn, page_size):
    w = workload([1000, 17, 5000, 3, 2049, 128], page_size=page_size, seed=212)
    c = W.contiguous_copy(w)
    BAL = attn.ATTN_PARTITIONS_BALANCED
    o1, l1 = run(attn, w, BAL)
    o2, l2 = run(attn, c, BAL)
    assert bits_equal(o1, o2) and bits_equal(l1, l2)
    ref_o, ref_l = oracle_result(w)
    assert_close(o1, l1, ref_o, ref_l, f"balanced page {page_size}")


def test_balanced_fewer_tiles_than_ctas(attn):
    """Eleven tiles in all: most CTAs have none, some units are split over
    two CTAs, the empty unit is written by the CTA holding its virtual tile."""
    w = workload([300, 0, 130, 1], hq=8, hkv=2, seed=213, sink=True)
    ob, lb = run(attn, w, attn.ATTN_PARTITIONS_BALANCED)
    ref_o, ref_l = oracle_result(w)
    assert_close(ob, lb, ref_o, ref_l, "balanced few tiles")


def test_balanced_more_units_than_ctas(attn):
    """The split on request with 2400 units on the SMs: every CTA walks many
    whole units and cuts at most two."""
    rng = np.random.default_rng(214)
    lens = rng.integers(1, 4000, size=300).tolist()
    w = workload(lens, seed=214)
    ob, lb = run(attn, w, attn.ATTN_PARTITIONS_BALANCED)
    rows, heads = full_rows_sample(w.kv_len_host, w.num_q_heads, 4, seed=5)
    ref_o, ref_l = oracle_result(w, sample=(rows, heads))
    ri, hi = torch.as_tensor(rows, device=DEV), torch.as_tensor(heads, device=DEV)
    assert_close(ob[ri, hi], lb[ri, hi], ref_o, ref_l, "balanced 300 sequences sampled")
    o1, l1 = run(attn, w, 1)
    assert_consistent(ob, lb, o1, l1, float(ref_o.eps.max()), "balanced 300 vs P=1")


def test_balanced_one_long_sequence(attn):
    """One sequence of 131072 keys and sinks (the long-context shape): each
    CTA takes about 1/152 of every KV head's tiles."""
    w = W.long_context_decode(device=DEV)
    BAL = attn.ATTN_PARTITIONS_BALANCED
    assert attn.attn_plan_partitions(1, 1, 32, 8, 128, w.max_kv_len, 0)[0] == BAL
    ob, lb = run(attn, w, BAL)
    ref_o, ref_l = oracle_result(w)
    assert_close(ob, lb, ref_o, ref_l, "balanced long context")


def test_balanced_clamps_a_length_above_max_kv_len(attn):
    """A kv_len above the planned max_kv_len (rounded up to whole tiles) is
    clamped to it and reported (bit 2)."""
    w = workload([500, 300], seed=215)
    out, lse = run(attn, w, attn.ATTN_PARTITIONS_BALANCED, max_kv_len=200)
    assert attn.attn_device_error_flags(clear=True) == 4
    # two tiles of keys were used: the oracle over the first 256 keys
    w.kv_len.copy_(torch.tensor([256, 256], dtype=w.kv_len.dtype, device=DEV))
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, "balanced clamped")
