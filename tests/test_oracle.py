"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: a closed
form, an invariant of softmax attention, brute force through a library
routine (torch's fp64 scaled_dot_product_attention on CPU), or the
hand-derived values in tests/golden/.  Together they are chosen so that a
dropped term, a wrong sign, a wrong head or page index, or a transposed
operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from split_flash_decoding_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def logical_problem(seed, batch, hq, hkv, d, lens, dv=None, q_lens=None):
    """Logical (unpaged) random problem: q [rows, hq, d], K [B, cap, hkv, d]."""
    g = torch.Generator().manual_seed(seed)
    dv = d if dv is None else dv
    rows = batch if q_lens is None else sum(q_lens)
    cap = max(max(lens), 1)
    q = torch.randn(rows, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(batch, cap, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(batch, cap, hkv, dv, generator=g).to(torch.bfloat16)
    return q, k, v


def sdpa_reference(q, k, v, lens, group, scale, q_lens=None, causal=False, sink=None):
    """Brute force via torch's fp64 SDPA, one sequence at a time.

    GQA is expanded with repeat_interleave (query head h uses KV head
    h // group); a sink becomes one extra key per query head whose score is
    exactly the sink logit and whose value is zero.
    """
    batch = len(lens)
    q_lens = [1] * batch if q_lens is None else q_lens
    hq = q.shape[1]
    dv = v.shape[-1]
    outs, lses = [], []
    row = 0
    for b in range(batch):
        n, L = q_lens[b], lens[b]
        qb = q[row:row + n].double().permute(1, 0, 2)            # [hq, n, d]
        kb = k[b, :L].double().permute(1, 0, 2).repeat_interleave(group, 0)  # [hq, L, d]
        vb = v[b, :L].double().permute(1, 0, 2).repeat_interleave(group, 0)
        mask = torch.ones(n, L, dtype=torch.bool)
        if causal:
            i = torch.arange(n)[:, None]
            j = torch.arange(L)[None, :]
            mask = j <= (L - n + i)
        mask = mask[None].expand(hq, n, L)
        s = torch.einsum("hnd,hld->hnl", qb, kb) * scale
        if sink is not None:
            # extra key with score == sink[h] and zero value
            t = torch.as_tensor(sink, dtype=torch.float64)
            unit = qb / (qb * qb).sum(-1, keepdim=True)          # q . unit = 1
            k_extra = unit * (t[:, None, None] / scale)           # per (h, n)
            kb_ext = torch.cat([kb[:, None].expand(hq, n, L, kb.shape[-1]),
                                k_extra[:, :, None, :]], 2)       # [hq, n, L+1, d]
            vb_ext = torch.cat([vb[:, None].expand(hq, n, L, dv),
                                torch.zeros(hq, n, 1, dv, dtype=torch.float64)], 2)
            m_ext = torch.cat([mask, torch.ones(hq, n, 1, dtype=torch.bool)], 2)
            o = torch.empty(hq, n, dv, dtype=torch.float64)
            for h in range(hq):
                for i in range(n):
                    o[h, i] = F.scaled_dot_product_attention(
                        qb[h, i][None, None], kb_ext[h, i][None], vb_ext[h, i][None],
                        attn_mask=m_ext[h, i][None, None], scale=scale)[0, 0]
            s_ext = torch.cat([s, t[:, None, None].expand(hq, n, 1)], 2)
            s_ext = s_ext.masked_fill(~m_ext, -math.inf)
            lse = torch.logsumexp(s_ext, -1)
        else:
            if L == 0:
                o = torch.zeros(hq, n, dv, dtype=torch.float64)
                lse = torch.full((hq, n), -math.inf, dtype=torch.float64)
            else:
                o = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, scale=scale)
                lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), -1)
        outs.append(o.permute(1, 0, 2))
        lses.append(lse.permute(1, 0))
        row += n
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


def to_paged(k, lens, page_size, seed):
    """Scatter a logical cache [B, cap, hkv, d] into pages, written with
    explicit loops (independent of the oracle's page arithmetic)."""
    batch = k.shape[0]
    npages = [max(1, -(-L // page_size)) for L in lens]
    total = sum(npages)
    perm = np.random.default_rng(seed).permutation(total)
    pool = torch.zeros((total, page_size) + tuple(k.shape[2:]), dtype=k.dtype)
    table = np.zeros((batch, max(npages)), dtype=np.int32)
    pos = 0
    for b in range(batch):
        for pi in range(npages[b]):
            page = int(perm[pos]); pos += 1
            table[b, pi] = page
            for slot in range(page_size):
                t = pi * page_size + slot
                if t < lens[b]:
                    pool[page, slot] = k[b, t]
    return pool, table


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def test_golden_worked_examples():
    with open(os.path.join(GOLDEN, "two_keys.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q = bf16([c["q"]])                       # [1, 1, d]
        k = bf16([c["k"]])[:, :, None, :]          # [1, L, 1, d]
        v = bf16([c["v"]])[:, :, None, :]
        L = k.shape[1]
        sink = None if c["sink"] is None else [W.fp32(c["sink"])]
        out, lse = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), [L],
                                    group=1, scale=W.fp32(c["scale"]), sink=sink)
        np.testing.assert_allclose(out[0, 0], c["out"], rtol=0, atol=1e-6, err_msg=c["name"])
        assert abs(lse[0, 0] - c["lse"]) < 1e-6, c["name"]


def test_single_key_returns_v_and_its_score():
    q, k, v = logical_problem(11, 3, 8, 2, 64, [1, 1, 1])
    scale = W.fp32(0.125)
    out, lse = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), [1, 1, 1],
                                group=4, scale=scale)
    for b in range(3):
        for h in range(8):
            kh = h // 4
            assert np.array_equal(out[b, h], v[b, 0, kh].double().numpy())
            s0 = scale * float(np.dot(q[b, h].double().numpy(), k[b, 0, kh].double().numpy()))
            assert abs(lse[b, h] - s0) <= 1e-12 * max(1.0, abs(s0))


def test_identical_keys_give_mean_of_v():
    lens = [5, 17, 64]
    q, k, v = logical_problem(12, 3, 4, 1, 32, lens)
    k[:] = k[:, :1]                              # every key equals key 0
    scale = W.fp32(0.3)
    out, lse = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), lens,
                                group=4, scale=scale)
    for b, L in enumerate(lens):
        mean_v = v[b, :L, 0].double().numpy().mean(0)
        for h in range(4):
            np.testing.assert_allclose(out[b, h], mean_v, rtol=0, atol=1e-13)
            s = scale * float(np.dot(q[b, h].double().numpy(), k[b, 0, 0].double().numpy()))
            assert abs(lse[b, h] - (s + math.log(L))) <= 1e-12 * max(1.0, abs(s))


def test_empty_sequence():
    q, k, v = logical_problem(13, 2, 4, 2, 16, [0, 3])
    out, lse = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), [0, 3],
                                group=2, scale=0.25)
    assert np.all(out[0] == 0.0) and np.all(np.isneginf(lse[0]))
    sink = [0.5, -1.0, 2.0, 0.0]
    out, lse = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), [0, 3],
                                group=2, scale=0.25, sink=sink)
    assert np.all(out[0] == 0.0)
    np.testing.assert_array_equal(lse[0], sink)


# --------------------------------------------------------------------------
# brute force through the library routine
# --------------------------------------------------------------------------

@pytest.mark.parametrize("hq,hkv,d,lens", [
    (4, 1, 64, [37, 100]),
    (8, 2, 32, [1, 7, 33]),
    (6, 3, 16, [64, 5]),
    (4, 4, 24, [9]),
])
def test_matches_fp64_sdpa(hq, hkv, d, lens):
    q, k, v = logical_problem(20 + d, len(lens), hq, hkv, d, lens)
    scale = W.fp32(1.0 / math.sqrt(d))
    out, lse = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), lens,
                                group=hq // hkv, scale=scale)
    ref_o, ref_l = sdpa_reference(q, k, v, lens, hq // hkv, scale)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12, atol=1e-12)


def test_causal_ragged_matches_fp64_sdpa():
    lens = [12, 40, 9]
    q_lens = [3, 1, 9]
    q, k, v = logical_problem(31, 3, 4, 2, 32, lens, q_lens=q_lens)
    offs = np.cumsum([0] + q_lens)
    scale = W.fp32(0.2)
    out, lse = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), lens,
                                group=2, scale=scale, causal=True, q_row_offsets=offs)
    ref_o, ref_l = sdpa_reference(q, k, v, lens, 2, scale, q_lens=q_lens, causal=True)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12, atol=1e-12)


def test_sink_is_an_extra_key_with_zero_value():
    lens = [21, 4]
    q, k, v = logical_problem(41, 2, 4, 2, 16, lens)
    scale = W.fp32(0.25)
    sink = [W.fp32(x) for x in (0.7, -2.0, 3.5, 0.0)]
    out, lse = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), lens,
                                group=2, scale=scale, sink=sink)
    ref_o, ref_l = sdpa_reference(q, k, v, lens, 2, scale, sink=sink)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12, atol=1e-12)


def test_sink_minus_infinity_is_a_no_op():
    lens = [50, 3]
    q, k, v = logical_problem(42, 2, 8, 2, 32, lens)
    kk, vv = oracle.KV.contiguous(k), oracle.KV.contiguous(v)
    o0, l0 = oracle.attention(q, kk, vv, lens, group=4, scale=0.17)
    o1, l1 = oracle.attention(q, kk, vv, lens, group=4, scale=0.17, sink=[-math.inf] * 8)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def test_paged_layout_equals_contiguous_bitwise():
    lens = [130, 7, 64, 129]
    q, k, v = logical_problem(51, 4, 8, 2, 32, lens)
    kp, table = to_paged(k, lens, 16, seed=1)
    vp, table_v = to_paged(v, lens, 16, seed=1)
    assert np.array_equal(table, table_v)
    oc, lc = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), lens,
                              group=4, scale=0.2)
    op, lp = oracle.attention(q, oracle.KV.paged(kp, table), oracle.KV.paged(vp, table), lens,
                              group=4, scale=0.2)
    assert np.array_equal(oc, op) and np.array_equal(lc, lp)
    # a different head mapping would change the answer
    ok_, _ = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), lens,
                              group=4, scale=0.2)
    assert np.array_equal(ok_, oc)


def test_key_permutation_invariance():
    lens = [77]
    q, k, v = logical_problem(52, 1, 4, 1, 32, lens)
    perm = torch.randperm(77, generator=torch.Generator().manual_seed(3))
    k2, v2 = k.clone(), v.clone()
    k2[0, :77] = k[0, perm]
    v2[0, :77] = v[0, perm]
    o1, l1 = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), lens,
                              group=4, scale=0.3)
    o2, l2 = oracle.attention(q, oracle.KV.contiguous(k2), oracle.KV.contiguous(v2), lens,
                              group=4, scale=0.3)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)


def test_output_is_a_convex_combination_of_values():
    lens = [200, 31]
    q, k, v = logical_problem(53, 2, 4, 2, 16, lens)
    out, _ = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), lens,
                              group=2, scale=0.9)
    for b, L in enumerate(lens):
        for h in range(4):
            vb = v[b, :L, h // 2].double().numpy()
            assert np.all(out[b, h] >= vb.min(0) - 1e-12)
            assert np.all(out[b, h] <= vb.max(0) + 1e-12)


def test_causal_row_equals_decode_over_truncated_cache():
    lens = [30]
    q_lens = [6]
    q, k, v = logical_problem(54, 1, 4, 2, 16, lens, q_lens=q_lens)
    out, lse = oracle.attention(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v), lens,
                                group=2, scale=0.3, causal=True, q_row_offsets=[0, 6])
    for i in range(6):
        Li = 30 - 6 + i + 1
        o1, l1 = oracle.attention(q[i:i + 1], oracle.KV.contiguous(k), oracle.KV.contiguous(v),
                                  [Li], group=2, scale=0.3)
        assert np.array_equal(out[i], o1[0]) and np.array_equal(lse[i], l1[0])


def test_mla_v_is_a_prefix_of_k():
    lens = [19, 70]
    g = torch.Generator().manual_seed(55)
    q = torch.randn(2, 16, 72, generator=g).to(torch.bfloat16)
    k = torch.randn(2, 70, 1, 72, generator=g).to(torch.bfloat16)
    v_copy = k[..., :64].contiguous()
    kk = oracle.KV.contiguous(k)
    o_alias, l_alias = oracle.attention(q, kk, kk, lens, group=16, scale=0.1, dim_v=64)
    o_copy, l_copy = oracle.attention(q, kk, oracle.KV.contiguous(v_copy), lens, group=16,
                                      scale=0.1, dim_v=64)
    assert np.array_equal(o_alias, o_copy) and np.array_equal(l_alias, l_copy)
    ref_o, ref_l = sdpa_reference(q, k, v_copy, lens, 16, 0.1)
    np.testing.assert_allclose(o_alias, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_alias, ref_l, rtol=1e-12, atol=1e-12)


def test_sampled_rows_equal_full_result():
    lens = [40, 90, 3]
    q, k, v = logical_problem(56, 3, 8, 2, 32, lens)
    kk, vv = oracle.KV.contiguous(k), oracle.KV.contiguous(v)
    out, lse = oracle.attention(q, kk, vv, lens, group=4, scale=0.2)
    rows = [2, 0, 1, 1]
    heads = [7, 3, 0, 5]
    so, sl = oracle.attention(q, kk, vv, lens, group=4, scale=0.2, sample=(rows, heads))
    for i, (r, h) in enumerate(zip(rows, heads)):
        assert np.array_equal(so[i], out[r, h]) and sl[i] == lse[r, h]


# --------------------------------------------------------------------------
# split-K partial statistics
# --------------------------------------------------------------------------

def test_partials_single_partition_normalises_to_the_result():
    lens = [33, 80]
    q, k, v = logical_problem(61, 2, 4, 1, 32, lens)
    kk, vv = oracle.KV.contiguous(k), oracle.KV.contiguous(v)
    out, lse = oracle.attention(q, kk, vv, lens, group=4, scale=0.2)
    wo, wm, wl = oracle.partials(q, kk, vv, lens, [0, 10_000], group=4, scale=0.2)
    np.testing.assert_allclose(wo[0] / wl[0][..., None], out, rtol=0, atol=1e-14)
    np.testing.assert_allclose(wm[0] + np.log(wl[0]), lse, rtol=1e-14, atol=1e-14)


def test_partials_of_single_keys_are_the_keys():
    lens = [4]
    q, k, v = logical_problem(62, 1, 2, 1, 16, lens)
    kk, vv = oracle.KV.contiguous(k), oracle.KV.contiguous(v)
    wo, wm, wl = oracle.partials(q, kk, vv, lens, [0, 1, 2, 3, 4, 5], group=2, scale=0.5)
    for j in range(4):
        for h in range(2):
            s = 0.5 * float(np.dot(q[0, h].double().numpy(), k[0, j, 0].double().numpy()))
            assert abs(wm[j, 0, h] - s) < 1e-13
            assert wl[j, 0, h] == 1.0
            assert np.array_equal(wo[j, 0, h], v[0, j, 0].double().numpy())
    # the slice past the end is empty
    assert np.isneginf(wm[4]).all() and (wl[4] == 0).all() and (wo[4] == 0).all()


def test_partials_merge_to_the_unsplit_result():
    """log-sum-exp merge of any key split reproduces the unsplit answer."""
    lens = [100, 57]
    q, k, v = logical_problem(63, 2, 4, 2, 16, lens)
    kk, vv = oracle.KV.contiguous(k), oracle.KV.contiguous(v)
    out, lse = oracle.attention(q, kk, vv, lens, group=2, scale=0.3)
    bounds = [0, 13, 14, 60, 61, 100, 120]
    wo, wm, wl = oracle.partials(q, kk, vv, lens, bounds, group=2, scale=0.3)
    M = wm.max(0)
    w = np.where(np.isneginf(wm), 0.0, np.exp(wm - M))
    Z = (w * wl).sum(0)
    merged = (w[..., None] * wo).sum(0) / Z[..., None]
    np.testing.assert_allclose(merged, out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(M + np.log(Z), lse, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# sparse top-k (indices name the physical rows each sequence attends to)
# --------------------------------------------------------------------------

def sparse_problem(seed, batch, hq, d, num_pages, page_size, topk, replace=False):
    """q [batch, hq, d], a one-head row pool [num_pages, page_size, 1, d] and
    index lists int32 [batch, max(topk)]; entries past topk[b] are -1."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(batch, hq, d, generator=g).to(torch.bfloat16)
    pool = torch.randn(num_pages, page_size, 1, d, generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(seed)
    idx = np.full((batch, max(max(topk), 1)), -1, dtype=np.int32)
    for b, L in enumerate(topk):
        idx[b, :L] = rng.choice(num_pages * page_size, L, replace=replace)
    return q, pool, idx


def gather_rows(pool, idx, topk):
    """Logical cache [batch, max(topk), 1, d] holding the named rows in
    order, copied with explicit loops from (page, slot) = divmod(row, page_size)."""
    ps = pool.shape[1]
    out = torch.zeros((idx.shape[0], max(max(topk), 1), 1, pool.shape[-1]), dtype=pool.dtype)
    for b, L in enumerate(topk):
        for t in range(L):
            page, slot = divmod(int(idx[b, t]), ps)
            out[b, t] = pool[page, slot]
    return out


@pytest.mark.parametrize("replace", [False, True])
def test_sparse_equals_sdpa_over_gathered_rows(replace):
    topk = [37, 0, 64, 5]
    q, pool, idx = sparse_problem(61, 4, 8, 40, num_pages=12, page_size=16, topk=topk,
                                  replace=replace)
    kv = oracle.KV.sparse(pool, idx)
    out, lse = oracle.attention(q, kv, kv, topk, group=8, scale=0.15, dim_v=32)
    k = gather_rows(pool, idx, topk)
    ref_o, ref_l = sdpa_reference(q, k, k[..., :32], topk, 8, 0.15)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12, atol=1e-12)


def test_sparse_identity_indices_equal_paged_bitwise():
    lens = [70, 3, 33]
    q, k, _ = logical_problem(62, 3, 4, 1, 24, lens)
    pool, table = to_paged(k, lens, 8, seed=4)
    idx = np.full((3, 70), -1, dtype=np.int32)
    for b, L in enumerate(lens):
        for t in range(L):
            idx[b, t] = table[b, t // 8] * 8 + t % 8
    kp = oracle.KV.paged(pool, table)
    ks = oracle.KV.sparse(pool, idx)
    o1, l1 = oracle.attention(q, kp, kp, lens, group=4, scale=0.3, dim_v=16)
    o2, l2 = oracle.attention(q, ks, ks, lens, group=4, scale=0.3, dim_v=16)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_sparse_ignores_indices_past_topk():
    topk = [10, 25]
    q, pool, idx = sparse_problem(63, 2, 4, 16, num_pages=4, page_size=32, topk=topk)
    kv = oracle.KV.sparse(pool, idx)
    o1, l1 = oracle.attention(q, kv, kv, topk, group=4, scale=0.5)
    idx2 = idx.copy()
    idx2[0, 10:] = np.arange(15) + 3          # valid rows, but past topk[0]
    kv2 = oracle.KV.sparse(pool, idx2)
    o2, l2 = oracle.attention(q, kv2, kv2, topk, group=4, scale=0.5)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_sparse_identical_selected_rows_closed_form():
    # every selected row equals x: uniform weights, out = x[:dv], lse = s + ln L
    topk = [9]
    q, pool, idx = sparse_problem(64, 1, 2, 16, num_pages=3, page_size=8, topk=topk)
    x = torch.randn(16, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    for r in idx[0, :9]:
        pool[int(r) // 8, int(r) % 8, 0] = x
    kv = oracle.KV.sparse(pool, idx)
    out, lse = oracle.attention(q, kv, kv, topk, group=2, scale=0.25, dim_v=12)
    xd = x.double().numpy()
    for h in range(2):
        assert np.array_equal(out[0, h], xd[:12])
        s = 0.25 * float(np.dot(q[0, h].double().numpy(), xd))
        np.testing.assert_allclose(lse[0, h], s + math.log(9), rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# the standard workload generators
# --------------------------------------------------------------------------

def test_tiny_workload_matches_sdpa():
    w = W.tiny_decode()
    kk = oracle.KV.contiguous(w.k_cache)
    vv = oracle.KV.contiguous(w.v_cache)
    out, lse = oracle.attention(w.q, kk, vv, w.kv_len, group=w.group, scale=w.scale)
    ref_o, ref_l = sdpa_reference(w.q, w.k_cache, w.v_cache, w.kv_len_host, w.group, w.scale)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12, atol=1e-12)


def test_workload_paged_and_contiguous_copies_agree():
    w = W.make_workload("t", batch=3, num_q_heads=4, num_kv_heads=2, dim_qk=32,
                        kv_lens=[70, 1, 129], page_size=32, seed=9)
    c = W.contiguous_copy(w)
    o1, l1 = oracle.attention(w.q, oracle.KV.paged(w.k_cache, w.page_table),
                              oracle.KV.paged(w.v_cache, w.page_table), w.kv_len,
                              group=2, scale=w.scale)
    o2, l2 = oracle.attention(c.q, oracle.KV.contiguous(c.k_cache),
                              oracle.KV.contiguous(c.v_cache), c.kv_len, group=2, scale=w.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_workload_generators_are_seeded():
    a = W.llama3_8b_decode(batch=4)
    b = W.llama3_8b_decode(batch=4)
    assert a.kv_len_host == b.kv_len_host
    assert torch.equal(a.page_table, b.page_table)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert all(512 <= L <= 8192 for L in a.kv_len_host)


def test_sparse_workload_names_rows_of_the_pool():
    w = W.make_sparse_mla_workload("s", ctx_lens=[0, 5, 300, 1000], topk=256, page_size=16,
                                   seed=3, dim_qk=32, dim_v=16, num_q_heads=4)
    rows = w.k_cache.shape[0] * w.k_cache.shape[1]
    assert w.kv_len_host == [0, 5, 256, 256]
    assert w.indices.shape == (4, 256) and w.page_table is None
    for b, n in enumerate(w.kv_len_host):
        r = w.indices[b, :n]
        assert bool(((r >= 0) & (r < rows)).all())
        assert len(set(r.tolist())) == n                  # drawn without repetition
        assert bool((w.indices[b, n:] == -1).all())
    again = W.make_sparse_mla_workload("s", ctx_lens=[0, 5, 300, 1000], topk=256, page_size=16,
                                       seed=3, dim_qk=32, dim_v=16, num_q_heads=4)
    assert torch.equal(w.indices, again.indices)


# ---------------------------------------------------------------------------
# oracle.spread: the error-bound statistics of the exact result
# ---------------------------------------------------------------------------

def _onehot_problem(a, v_rows, scale, hq=1, d=8, dv=4):
    """One sequence whose key j is a_j e_0 and q = e_0, so s_j = scale * a_j
    exactly; V rows given.  Returns (q, K, V) as bf16 tensors."""
    L = len(a)
    q = torch.zeros(1, hq, d)
    q[0, :, 0] = 1.0
    k = torch.zeros(1, L, 1, d)
    k[0, :, 0, 0] = torch.tensor(a, dtype=torch.float32)
    v = torch.tensor(v_rows, dtype=torch.float32).reshape(1, L, 1, dv)
    return bf16(q), bf16(k), bf16(v)


def _spread(q, k, v, lens, group, scale, **kw):
    return oracle.spread(q, oracle.KV.contiguous(k), oracle.KV.contiguous(v),
                         torch.tensor(lens, dtype=torch.int32), group=group, scale=scale,
                         dim_v=v.shape[-1], **kw)


def test_spread_single_key_is_zero():
    q, k, v = _onehot_problem([3.0], [[1.5, -2.0, 0.25, 4.0]], 0.5)
    sd, am, st = _spread(q, k, v, [1], 1, 0.5)
    assert np.all(sd[0, 0] == 0.0)
    assert np.allclose(am[0, 0], [1.5, 2.0, 0.25, 4.0], rtol=0, atol=1e-15)
    assert st[0, 0, 0] == 1 and st[0, 0, 1] == 1.5 and st[0, 0, 2] == 1.5


def test_spread_two_keys_closed_form():
    """Two weights w and 1 - w: the spread of a two-point distribution is
    sqrt(w (1 - w)) |v0 - v1|."""
    v_rows = [[1.0, -2.0, 0.5, 3.0], [-1.0, 2.0, 0.5, -0.75]]
    q, k, v = _onehot_problem([2.0, 0.0], v_rows, 0.5)
    sd, am, st = _spread(q, k, v, [2], 1, 0.5)
    w0 = 1.0 / (1.0 + math.exp(-1.0))           # scores 1 and 0
    v0, v1 = np.array(v_rows[0]), np.array(v_rows[1])
    assert np.allclose(sd[0, 0], math.sqrt(w0 * (1 - w0)) * np.abs(v0 - v1), rtol=1e-13, atol=0)
    assert np.allclose(am[0, 0], w0 * np.abs(v0) + (1 - w0) * np.abs(v1), rtol=1e-13)
    assert st[0, 0, 0] == 2 and st[0, 0, 2] == 1.0


def test_spread_one_key_and_a_sink_closed_form():
    """One key of weight w beside a sink (a zero value): out = w v, and the
    spread of the key around it is sqrt(w) (1 - w) |v|."""
    q, k, v = _onehot_problem([1.0], [[2.0, -1.0, 0.5, 3.0]], 1.0)
    sink = torch.tensor([0.25])
    sd, am, st = _spread(q, k, v, [1], 1, 1.0, sink=sink)
    w = 1.0 / (1.0 + math.exp(0.25 - 1.0))
    vv = np.array([2.0, 1.0, 0.5, 3.0])
    assert np.allclose(sd[0, 0], math.sqrt(w) * (1 - w) * vv, rtol=1e-13)
    assert np.allclose(am[0, 0], w * vv, rtol=1e-13)


def test_spread_identical_keys_is_population_std():
    """Equal scores: the weights are uniform, so sd is numpy's population
    standard deviation of V over the keys and am the mean of |V|."""
    g = torch.Generator().manual_seed(5)
    L, d = 37, 16
    q = bf16(torch.randn(1, 2, d, generator=g))
    k = bf16(torch.randn(1, 1, 1, d, generator=g)).expand(1, L, 1, d).contiguous()
    v = bf16(torch.randn(1, L, 1, 8, generator=g))
    sd, am, _ = _spread(q, k, v, [L], 2, 0.3)
    vv = v[0, :, 0].double().numpy()
    for h in range(2):
        assert np.allclose(sd[0, h], vv.std(axis=0), rtol=1e-12)
        assert np.allclose(am[0, h], np.abs(vv).mean(axis=0), rtol=1e-12)


@pytest.mark.parametrize("with_sink", [False, True])
def test_spread_equals_the_second_moment_through_attention(with_sink):
    """sd^2 = E_w[v^2] - out^2 (2 - sum w): the second moment taken by the
    (separately pinned) attention function with V squared, on a paged GQA
    cache with causal multi-row sequences.  V holds multiples of 1/8 below 2
    in magnitude, so V^2 and |V| are exact in bf16."""
    g = torch.Generator().manual_seed(9)
    lens, q_lens, hq, hkv, d = [40, 3, 130], [2, 3, 1], 8, 2, 16
    q, k, _ = logical_problem(9, 3, hq, hkv, d, lens, q_lens=q_lens)
    v = bf16(torch.randint(-15, 16, (3, max(lens), hkv, 8), generator=g).float() / 8)
    offs = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32)
    kvl = torch.tensor(lens, dtype=torch.int32)
    pk, table = to_paged(k, lens, 16, 3)
    pv, _ = to_paged(v, lens, 16, 3)
    K = oracle.KV.paged(pk, torch.tensor(table))
    sink = torch.randn(hq, generator=g) if with_sink else None
    kw = dict(group=hq // hkv, scale=0.25, dim_v=8, sink=sink, causal=True, q_row_offsets=offs)
    out, lse = oracle.attention(q, K, oracle.KV.paged(pv, torch.tensor(table)), kvl, **kw)
    m2, _ = oracle.attention(q, K, oracle.KV.paged(bf16(pv.float() ** 2), torch.tensor(table)),
                             kvl, **kw)
    ab, _ = oracle.attention(q, K, oracle.KV.paged(bf16(pv.float().abs()), torch.tensor(table)),
                             kvl, **kw)
    sd, am, st = oracle.spread(q, K, oracle.KV.paged(pv, torch.tensor(table)), kvl, **kw)
    wsum = (np.ones_like(lse) if sink is None
            else 1.0 - np.exp(sink.double().numpy()[None, :] - lse))
    var = m2 - out ** 2 * (2.0 - wsum)[..., None]
    assert np.allclose(sd ** 2, np.maximum(var, 0.0), rtol=1e-10, atol=1e-13)
    assert np.allclose(am, ab, rtol=1e-12, atol=1e-15)
    # visible keys: rows 0-1 of sequence 0 see 39 and 40; sequence 1's three
    # rows see 1, 2, 3; sequence 2's row sees 130
    assert st[:, 0, 0].tolist() == [39, 40, 1, 2, 3, 130]


def test_spread_translation_invariant():
    """Shifting every value by a constant shifts out by it and leaves the
    spread unchanged (no sink)."""
    g = torch.Generator().manual_seed(13)
    q, k, _ = logical_problem(13, 2, 4, 1, 16, [50, 9])
    v = bf16(torch.randint(-12, 13, (2, 50, 1, 8), generator=g).float() / 8)
    a = _spread(q, k, v, [50, 9], 4, 0.25)[0]
    b = _spread(q, k, bf16(v.float() + 1.0), [50, 9], 4, 0.25)[0]
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)
    assert np.any(a > 0.1)
