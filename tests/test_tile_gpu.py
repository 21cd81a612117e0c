"""GPU parity of the tensor-core tile path (attn_decode with several query
rows per sequence: ragged prefill mixed with decode, causal) against the
fp64 oracle, for both tile kernels: one 128-row Q tile per CTA
(num_partitions 1, and the automatic choice) and two adjacent Q tiles per
CTA pair sharing each K/V tile (ATTN_PARTITIONS_TILE_PAIR)."""
import math

import numpy as np
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


def tile_workload(q_lens, prefix, hq=8, hkv=2, page_size=16, seed=0, causal=True, sink=False,
                  scale=None):
    kv_lens = [p + n for p, n in zip(prefix, q_lens)]
    return W.make_workload("tile", batch=len(q_lens), num_q_heads=hq, num_kv_heads=hkv,
                           dim_qk=128, kv_lens=kv_lens, page_size=page_size, seed=seed,
                           device=DEV, q_lens=q_lens, causal=causal, sink=sink, scale=scale)


def grow_keys(w, per_token):
    """Scale the K row of logical token t of every sequence by 1 + t * per_token
    (through the page table), so scores grow along the sequence."""
    ps = w.k_cache.shape[1]
    flat = w.k_cache.view(-1, w.k_cache.shape[2], w.k_cache.shape[3])
    pt = w.page_table.cpu()
    for b, L in enumerate(w.kv_len_host):
        t = torch.arange(L)
        rows = (pt[b, t // ps].long() * ps + t % ps).to(DEV)
        f = (1.0 + t.float() * per_token).to(DEV)[:, None, None]
        flat[rows] = (flat[rows].float() * f).to(torch.bfloat16)


# num_partitions on the tile path: 1 = one Q tile per CTA, -2 =
# ATTN_PARTITIONS_TILE_PAIR, two Q tiles per CTA pair
KERNELS = pytest.mark.parametrize("kern", [1, -2], ids=["one_tile", "tile_pair"])


def run(attn, w, sink="workload", kern=1):
    s = w.sink if sink == "workload" else sink
    out, lse = attn.attn_decode(w.q, w.k_cache, w.v_cache, w.kv_len, group=w.group,
                                scale=w.scale, max_kv_len=w.max_kv_len,
                                page_table=w.page_table, sink=s,
                                q_row_offsets=w.q_row_offsets, max_q_len=w.max_q_len,
                                causal=w.causal, num_partitions=kern)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("causal", [True, False])
@KERNELS
def test_mixed_rows_match_oracle(attn, causal, kern):
    w = tile_workload([1, 5, 40, 130, 1], [0, 20, 100, 7, 300], seed=31, causal=causal)
    out, lse = run(attn, w, kern=kern)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, f"tile causal={causal}")


@pytest.mark.parametrize("scale", [4.0, 0.7, -0.3])
@KERNELS
def test_scores_far_above_the_reference(attn, scale, kern):
    """Keys whose scores grow along the sequence and large (or negative)
    scales: later tiles hold keys tens to hundreds of base-2 units above the
    running maximum of earlier ones, so the maximum is raised and O rescaled
    many times per row."""
    w = tile_workload([1, 37, 300, 129], [0, 500, 60, 900], seed=35, scale=scale, sink=True)
    grow_keys(w, 1.0 / 64)
    out, lse = run(attn, w, kern=kern)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, f"tile growing keys scale={scale}")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 4), (32, 4)])
@KERNELS
def test_groups(attn, hq, hkv, kern):
    w = tile_workload([3, 70, 129], [10, 0, 200], hq=hq, hkv=hkv, seed=32)
    out, lse = run(attn, w, kern=kern)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, f"tile hq={hq} hkv={hkv}")


@pytest.mark.parametrize("page_size", [16, 64, 128, 256])
@KERNELS
def test_tile_paged_equals_contiguous_bitwise(attn, page_size, kern):
    w = tile_workload([33, 1, 300], [90, 500, 0], page_size=page_size, seed=33)
    c = W.contiguous_copy(w)
    o1, l1 = run(attn, w, kern=kern)
    o2, l2 = run(attn, c, kern=kern)
    assert bits_equal(o1, o2) and bits_equal(l1, l2)
    ref_o, ref_l = oracle_result(w)
    assert_close(o1, l1, ref_o, ref_l, f"tile page {page_size}")


@KERNELS
def test_tile_sinks(attn, kern):
    w = tile_workload([17, 1, 64], [5, 40, 0], seed=34, sink=True)
    out, lse = run(attn, w, kern=kern)
    ref_o, ref_l = oracle_result(w)
    assert_close(out, lse, ref_o, ref_l, "tile sinks")
    no_sink = torch.full((w.num_q_heads,), -math.inf, dtype=torch.float32, device=DEV)
    o1, l1 = run(attn, w, sink=no_sink, kern=kern)
    o2, l2 = run(attn, w, sink=None, kern=kern)
    assert bits_equal(o1, o2) and bits_equal(l1, l2)


@KERNELS
def test_mixed_prefill_decode_full_size_sampled(attn, kern):
    """The 16-sequence mixed batch at full size; the oracle checks 1024
    sampled (row, head) pairs covering every sequence, first and last rows
    included."""
    w = W.mixed_prefill_decode(device=DEV)
    out, lse = run(attn, w, kern=kern)
    offs = w.q_row_offsets_host
    rng = np.random.default_rng(5)
    rows, heads = [], []
    for b in range(w.batch):
        lo, hi = offs[b], offs[b + 1]
        pick = {lo, hi - 1} | set(rng.integers(lo, hi, size=min(62, hi - lo)).tolist())
        for r in sorted(pick):
            rows.append(r)
            heads.append(int(rng.integers(0, w.num_q_heads)))
    rows, heads = np.array(rows), np.array(heads)
    ref_o, ref_l = oracle_result(w, sample=(rows, heads))
    ri, hi_ = torch.as_tensor(rows, device=DEV), torch.as_tensor(heads, device=DEV)
    assert_close(out[ri, hi_], lse[ri, hi_], ref_o, ref_l, "mixed full size sampled")


@pytest.mark.parametrize("q_lens,prefix", [
    ([65, 1, 200], [10, 700, 0]),          # odd tile counts: the last pair has one tile
    ([96, 33, 500], [0, 3000, 40]),        # pair boundaries, lengths that leave a K half empty
    ([5, 1, 20], [900, 10, 70]),           # no sequence spans two tiles: half of each pair idle
])
def test_pair_and_one_tile_kernels_agree(attn, q_lens, prefix):
    """The two tile kernels on one problem: each against the oracle, and the
    pair within two roundings of the one-tile result."""
    w = tile_workload(q_lens, prefix, page_size=64, seed=36, sink=True)
    o1, l1 = run(attn, w, kern=1)
    o2, l2 = run(attn, w, kern=attn.ATTN_PARTITIONS_TILE_PAIR)
    o0, l0 = run(attn, w, kern=0)          # the automatic choice: one tile per CTA
    assert bits_equal(o0, o1) and bits_equal(l0, l1)
    ref_o, ref_l = oracle_result(w)
    assert_pair(o2, l2, o1, l1, ref_o, ref_l, f"pair vs one tile {q_lens}")


@KERNELS
def test_graph_capture_replays_with_new_prefixes(attn, kern):
    """One captured tile call replayed with other cached prefixes (the rows
    per sequence fixed by the captured offsets, causal alignment following
    the new lengths)."""
    q_lens, prefix = [300, 1, 140, 7], [200, 900, 0, 260]
    w = tile_workload(q_lens, prefix, seed=95, sink=True)
    out = torch.empty(w.rows, w.num_q_heads, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(w.rows, w.num_q_heads, dtype=torch.float32, device=DEV)
    kv_len = w.kv_len.clone()
    s = torch.cuda.Stream()

    def call():
        attn.attn_decode(w.q, w.k_cache, w.v_cache, kv_len, group=w.group, scale=w.scale,
                         max_kv_len=w.max_kv_len, page_table=w.page_table, sink=w.sink,
                         q_row_offsets=w.q_row_offsets, max_q_len=w.max_q_len, causal=True,
                         num_partitions=kern, out=out, lse=lse, stream=s)

    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for new_prefix in (prefix, [17, 0, 500, 1]):
        new = [p + n for p, n in zip(new_prefix, q_lens)]
        kv_len.copy_(torch.tensor(new, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        w2 = tile_workload(q_lens, prefix, seed=95, sink=True)
        w2.kv_len_host = new
        w2.kv_len = kv_len
        ref_o, ref_l = oracle_result(w2)
        assert_close(out, lse, ref_o, ref_l, f"tile graph replay {new_prefix} kern={kern}")
