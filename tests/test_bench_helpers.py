"""bench.py's accounting on CPU: algorithmic bytes and FLOPs per workload
kind, the roofline bound, and the oracle's CPU-baseline sample."""
import math

import pytest
import torch

import bench
from split_flash_decoding_gb300 import workloads as W


def test_gqa_bytes_count_k_and_v_per_kv_head():
    w = W.make_workload("t", batch=2, num_q_heads=8, num_kv_heads=2, dim_qk=64,
                        kv_lens=[10, 30], page_size=16, seed=1)
    kv = 40 * 2 * (64 + 64) * 2
    qo = 2 * 8 * 64 * 2 * 2 + 2 * 8 * 4
    assert bench.algorithmic_bytes(w) == kv + qo
    assert bench.algorithmic_flops(w) == 40 * 8 * 2 * (64 + 64)


def test_mla_bytes_count_k_once_and_sparse_indices():
    w = W.make_workload("m", batch=1, num_q_heads=4, num_kv_heads=1, dim_qk=48, dim_v=32,
                        mla=True, kv_lens=[20], page_size=8, seed=2)
    assert bench.algorithmic_bytes(w) == 20 * 48 * 2 + 4 * 48 * 2 + 4 * 32 * 2 + 4 * 4
    s = W.make_sparse_mla_workload("s", ctx_lens=[50, 9], topk=16, page_size=8, seed=3,
                                   dim_qk=48, dim_v=32, num_q_heads=4)
    keys = 16 + 9
    assert bench.algorithmic_bytes(s) == keys * (48 * 2 + 4) + 2 * 4 * (48 * 2 + 32 * 2 + 4)


def test_causal_rows_count_visible_pairs_only():
    w = W.make_workload("c", batch=2, num_q_heads=2, num_kv_heads=1, dim_qk=16,
                        kv_lens=[5, 3], page_size=4, seed=4, q_lens=[3, 4], causal=True)
    # sequence 0: rows see 3, 4, 5 keys; sequence 1: 0, 1, 2, 3
    assert bench.visible_pairs(w) == 12 + 6


def test_roofline_bound_follows_the_ridge():
    ridge = 1892.1e12 / 6775.9e9
    assert bench.roofline_bound(4.0 * 1e9, 1e9, 1892.1, 6775.9) == "hbm"          # GQA decode
    assert bench.roofline_bound(238.0 * 1e9, 1e9, 1892.1, 6775.9) == "hbm"        # MLA, 1 row
    assert bench.roofline_bound(476.0 * 1e9, 1e9, 1892.1, 6775.9) == "tensor"     # MLA, 2 rows
    assert math.isclose(ridge, 279.2, rel_tol=1e-3)


def test_oracle_sample_covers_every_row_of_a_sequence():
    w = W.make_workload("r", batch=3, num_q_heads=4, num_kv_heads=1, dim_qk=32,
                        kv_lens=[10, 20, 30], page_size=8, seed=5, q_lens=[1, 3, 2],
                        causal=True)
    dt, nbytes, threads = bench.oracle_sample_time(w, w.k_cache, w.v_cache, [1, 2], threads=1)
    per_key = 1 * (32 + 32) * 2
    rows = 3 + 2
    assert nbytes == (20 + 30) * per_key + rows * 4 * (32 * 2 + 32 * 2 + 4)
    assert threads == 1 and dt >= 0.0
