"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, validates arguments on the host (no launch), and the
partition planner follows its stated formulas."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def attn():
    from split_flash_decoding_gb300 import build
    build.build()
    from split_flash_decoding_gb300 import attn as a
    return a


def declared_functions():
    names = set()
    for f in os.listdir(HEADER_DIR):
        if f.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"^\s*int\s+(attn_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("attn_decode", "attn_mla_decode", "attn_splitk_reduce",
                     "attn_plan_partitions"):
        assert required in names


def test_library_exports_every_declared_symbol(attn):
    handle = ctypes.CDLL(attn.LIB_PATH)
    for name in declared_functions():
        assert hasattr(handle, name), name
    assert set(declared_functions()) <= set(attn._SIGNATURES)


def test_struct_layout_matches_header(attn):
    # attn_kv_t: pointer, 3 x int64, 2 x int32, pointer, 2 x int32
    assert ctypes.sizeof(attn.attn_kv_t) == 56
    assert attn.attn_kv_t.page_table.offset == 40


def kv(attn, **over):
    d = attn.attn_kv_t()
    d.base = 0x10000
    d.page_stride = 128 * 8 * 128
    d.token_stride = 8 * 128
    d.head_stride = 128
    d.page_size = 128
    d.num_pages = 10
    d.page_table = 0x20000
    d.max_pages = 4
    d.reserved = 0
    for k, v in over.items():
        setattr(d, k, v)
    return d


def call_decode(attn, k=None, v=None, **over):
    args = dict(q=0x30000, kv_len=0x40000, offs=None, batch=2, rows=None, hq=32, group=4,
                d=128, max_q_len=1, max_kv_len=500, scale=0.088, sink=None, causal=0, P=1,
                ws=None, ws_bytes=0, out=0x50000, lse=None)
    args.update(over)
    if args["rows"] is None:
        args["rows"] = args["batch"]
    k = k or kv(attn)
    v = v or kv(attn)
    return attn.lib().attn_decode(args["q"], ctypes.byref(k), ctypes.byref(v), args["kv_len"],
                                  args["offs"], args["batch"], args["rows"], args["hq"],
                                  args["group"], args["d"], args["max_q_len"],
                                  args["max_kv_len"], args["scale"], args["sink"],
                                  args["causal"], args["P"], args["ws"], args["ws_bytes"],
                                  args["out"], args["lse"], None)


def test_decode_rejects_bad_arguments_before_launch(attn):
    E = attn
    assert call_decode(attn, q=None) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, out=None) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, kv_len=None) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, hq=30, group=4) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, group=0) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, hq=48, group=16) == E.ATTN_ERR_UNSUPPORTED
    assert call_decode(attn, d=96) == E.ATTN_ERR_UNSUPPORTED
    assert call_decode(attn, P=-3) == E.ATTN_ERR_INVALID_ARG
    # the balanced split (-1) runs on the tensor-core decode kernel only
    assert call_decode(attn, d=64, P=E.ATTN_PARTITIONS_BALANCED) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, P=E.ATTN_MAX_PARTITIONS + 1) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, scale=float("nan")) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, max_kv_len=-1) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, q=0x30008) == E.ATTN_ERR_INVALID_ARG          # misaligned
    assert call_decode(attn, k=kv(attn, base=0)) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, k=kv(attn, base=0x10008)) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, k=kv(attn, reserved=1)) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, k=kv(attn, token_stride=1020)) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, k=kv(attn, page_size=96)) == E.ATTN_ERR_UNSUPPORTED
    assert call_decode(attn, k=kv(attn, page_size=4)) == E.ATTN_ERR_UNSUPPORTED
    assert call_decode(attn, k=kv(attn, max_pages=3)) == E.ATTN_ERR_INVALID_ARG  # 500 > 3*128
    assert call_decode(attn, k=kv(attn, page_table=None, page_size=400, num_pages=2)) \
        == E.ATTN_ERR_INVALID_ARG                                             # capacity < 500
    assert call_decode(attn, k=kv(attn, page_table=None, page_size=512, num_pages=1)) \
        == E.ATTN_ERR_INVALID_ARG                                             # fewer seqs
    # K and V must share one page-table layout
    assert call_decode(attn, v=kv(attn, page_table=0x20100)) == E.ATTN_ERR_UNSUPPORTED
    # split-K through the workspace needs a large enough, aligned one
    assert call_decode(attn, P=3) == E.ATTN_ERR_WORKSPACE
    assert call_decode(attn, P=3, ws=0x60000, ws_bytes=16) == E.ATTN_ERR_WORKSPACE
    P, need = attn.attn_plan_partitions(2, 2, 32, 8, 128, 500, 3, num_sms=152)
    assert call_decode(attn, P=3, ws=0x60010, ws_bytes=need) == E.ATTN_ERR_WORKSPACE
    # rows must match the batch without row offsets; multi-row needs offsets
    assert call_decode(attn, rows=3) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, max_q_len=4) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, max_q_len=0) == E.ATTN_ERR_INVALID_ARG
    # the multi-row tile path does not split K
    assert call_decode(attn, offs=0x70000, rows=40, max_q_len=30, P=2) == E.ATTN_ERR_UNSUPPORTED
    # the decode kernel's item table holds at most 2048 sequences
    assert call_decode(attn, batch=2049) == E.ATTN_ERR_UNSUPPORTED
    # an empty batch is a no-op
    assert call_decode(attn, batch=0, q=None, out=None) == E.ATTN_OK


def call_sparse(attn, k=None, **over):
    args = dict(q=0x30000, idx=0x80000, stride=2048, topk=0x40000, batch=2, hq=128, dqk=576,
                dv=512, scale=0.07, sink=None, P=1, ws=None, ws_bytes=0, out=0x50000, lse=None)
    args.update(over)
    k = k or kv(attn, page_table=None, page_stride=64 * 576, token_stride=576, head_stride=576,
                page_size=64, num_pages=100)
    return attn.lib().attn_mla_decode_sparse(args["q"], ctypes.byref(k), args["idx"],
                                             args["stride"], args["topk"], args["batch"],
                                             args["hq"], args["dqk"], args["dv"], args["scale"],
                                             args["sink"], args["P"], args["ws"],
                                             args["ws_bytes"], args["out"], args["lse"], None)


def test_sparse_mla_rejects_bad_arguments_before_launch(attn):
    E = attn
    rows = dict(page_table=None, page_stride=64 * 576, token_stride=576, head_stride=576,
                page_size=64, num_pages=100)
    assert call_sparse(attn, q=None) == E.ATTN_ERR_INVALID_ARG
    assert call_sparse(attn, out=None) == E.ATTN_ERR_INVALID_ARG
    assert call_sparse(attn, topk=None) == E.ATTN_ERR_INVALID_ARG
    assert call_sparse(attn, idx=None) == E.ATTN_ERR_INVALID_ARG       # stride > 0 needs indices
    assert call_sparse(attn, idx=0x80002) == E.ATTN_ERR_INVALID_ARG    # misaligned int32
    assert call_sparse(attn, stride=-1) == E.ATTN_ERR_INVALID_ARG
    assert call_sparse(attn, hq=64) == E.ATTN_ERR_UNSUPPORTED
    assert call_sparse(attn, dqk=512) == E.ATTN_ERR_UNSUPPORTED
    assert call_sparse(attn, P=-1) == E.ATTN_ERR_INVALID_ARG
    assert call_sparse(attn, P=1025) == E.ATTN_ERR_INVALID_ARG
    # P = 0 (the balanced split) needs a workspace
    assert call_sparse(attn, P=0) == E.ATTN_ERR_WORKSPACE
    assert call_sparse(attn, scale=float("nan")) == E.ATTN_ERR_INVALID_ARG
    # the indices replace the page table; row strides keep the 16-byte rule
    assert call_sparse(attn, k=kv(attn, **dict(rows, page_table=0x20000))) \
        == E.ATTN_ERR_INVALID_ARG
    assert call_sparse(attn, k=kv(attn, **dict(rows, token_stride=580))) \
        == E.ATTN_ERR_INVALID_ARG
    assert call_sparse(attn, k=kv(attn, **dict(rows, page_size=0))) == E.ATTN_ERR_INVALID_ARG
    # rows must sit at one stride: padded pages are not a row array
    assert call_sparse(attn, k=kv(attn, **dict(rows, page_stride=65 * 576))) \
        == E.ATTN_ERR_UNSUPPORTED
    assert call_sparse(attn, k=kv(attn, **dict(rows, base=0x10008))) == E.ATTN_ERR_INVALID_ARG
    # split-K needs a large enough workspace
    assert call_sparse(attn, P=4) == E.ATTN_ERR_WORKSPACE
    # an empty batch is a no-op
    assert call_sparse(attn, batch=0, q=None, out=None, topk=None) == E.ATTN_OK


def test_mla_rows_rejects_bad_arguments_before_launch(attn):
    E = attn
    k = kv(attn, page_stride=64 * 576, token_stride=576, head_stride=576, page_size=64,
           num_pages=100, max_pages=40)

    def call(**over):
        a = dict(q=0x30000, kvl=0x40000, offs=0x48000, batch=2, rows=5, hq=128, dqk=576, dv=512,
                 maxkv=2000, scale=0.07, sink=None, causal=1, P=1, ws=None, ws_bytes=0,
                 out=0x50000, lse=None)
        a.update(over)
        return attn.lib().attn_mla_decode_rows(a["q"], ctypes.byref(k), a["kvl"], a["offs"],
                                               a["batch"], a["rows"], a["hq"], a["dqk"], a["dv"],
                                               a["maxkv"], a["scale"], a["sink"], a["causal"],
                                               a["P"], a["ws"], a["ws_bytes"], a["out"],
                                               a["lse"], None)
    assert call(offs=None) == E.ATTN_ERR_INVALID_ARG
    assert call(rows=-1) == E.ATTN_ERR_INVALID_ARG
    assert call(q=None) == E.ATTN_ERR_INVALID_ARG
    assert call(hq=64) == E.ATTN_ERR_UNSUPPORTED
    assert call(rows=70000) == E.ATTN_ERR_UNSUPPORTED
    assert call(P=3) == E.ATTN_ERR_WORKSPACE
    assert call(rows=0, q=None, out=None) == E.ATTN_OK


def test_reduce_rejects_bad_arguments(attn):
    L = attn.lib()
    f = L.attn_splitk_reduce
    assert f(0x1000, 0x2000, 0x3000, 0, 4, 8, 128, None, 0x4000, None, None) == attn.ATTN_ERR_INVALID_ARG
    assert f(0x1000, 0x2000, 0x3000, 2, 4, 8, 130, None, 0x4000, None, None) == attn.ATTN_ERR_INVALID_ARG
    assert f(None, 0x2000, 0x3000, 2, 4, 8, 128, None, 0x4000, None, None) == attn.ATTN_ERR_INVALID_ARG
    assert f(0x1000, 0x2000, 0x3000, 2, 0, 8, 128, None, None, None, None) == attn.ATTN_OK


def test_planner_formulas(attn):
    # explicit request is honoured verbatim
    for req in (1, 3, 7, 148, 1024):
        P, ws = attn.attn_plan_partitions(64, 64, 32, 8, 128, 8192, req, num_sms=152)
        assert P == req
        n = req * 64 * 32
        align = lambda x: (x + 255) // 256 * 256
        expect = 0 if req == 1 else align(n * 128 * 4) + 2 * align(n * 4)
        assert ws == expect
    align = lambda x: (x + 255) // 256 * 256
    # 2 or 4 partitions on the tensor-core path merge on chip: no workspace
    for req in (2, 4):
        assert attn.attn_plan_partitions(64, 64, 32, 8, 128, 8192, req, num_sms=152)[1] == 0
        P, ws = attn.attn_plan_partitions(64, 64, 32, 16, 64, 8192, req, num_sms=152)
        assert ws > 0                                 # head_dim 64 keeps the workspace
    # automatic GQA (head_dim 128: one CTA per SM; head_dim 64: two): with
    # head_dim 128 and at most eight (sequence, KV head) units per SM, the
    # balanced split; otherwise (and for head_dim 64: fewer units than CTAs
    # -> one wave of slices) >= 4 items per CTA at full length and slices of
    # <= ~1024 keys
    BAL = attn.ATTN_PARTITIONS_BALANCED
    P, _ = attn.attn_plan_partitions(200, 200, 32, 8, 128, 8192, 0, num_sms=152)
    assert P == 8                                     # 1600 units: slices of <= 1024 keys
    for batch, rows, hkv, max_len in ((1, 1, 8, 131072), (16, 16, 8, 8192), (37, 37, 8, 5000),
                                      (64, 64, 8, 8192), (152, 152, 8, 8192)):
        P, ws = attn.attn_plan_partitions(batch, rows, 8 * hkv // 2, hkv, 128, max_len, 0,
                                          num_sms=152)
        slots = 152 + batch * hkv
        assert P == BAL
        assert ws == align(slots * 16 * 128 * 4) + 2 * align(slots * 16 * 4) + align(batch * hkv * 8)
    # the rule's edge: 8 units per SM exactly is balanced, one sequence more is not
    assert attn.attn_plan_partitions(152, 152, 32, 8, 128, 8192, 0, num_sms=152)[0] == BAL
    assert attn.attn_plan_partitions(153, 153, 32, 8, 128, 8192, 0, num_sms=152)[0] > 0
    assert attn.attn_plan_partitions(16, 16, 32, 8, 128, 8192, 0, num_sms=16)[0] == BAL
    assert attn.attn_plan_partitions(17, 17, 32, 8, 128, 8192, 0, num_sms=16)[0] > 0
    # one tile per unit cannot be balanced further: one slice
    assert attn.attn_plan_partitions(16, 16, 32, 8, 128, 128, 0, num_sms=152) == (1, 0)
    P, _ = attn.attn_plan_partitions(1, 1, 16, 8, 64, 131072, 0, num_sms=152)
    assert P == 38 and 8 * P == 2 * 152
    # automatic MLA (one KV head, 512 output channels): keys that need a
    # split at all take the balanced split (P = 0) over one wave of
    # num_sms / 2 two-CTA clusters; fp32 partials for clusters + rows slots,
    # then the reduce's per-row table of slots
    align = lambda x: (x + 255) // 256 * 256
    for sms, batch, rows, max_len in ((152, 32, 32, 32768), (152, 1, 1, 131072),
                                      (152, 4, 8, 2048), (16, 8, 8, 9000)):
        P, ws = attn.attn_plan_partitions(batch, rows, 128, 1, 512, max_len, 0, num_sms=sms)
        slots = sms // 2 + rows
        assert P == 0
        assert ws == (align(slots * 128 * 512 * 4) + 2 * align(slots * 128 * 4) +
                      align(rows * 8))
    # a wave of clusters or more with rows of <= ~4096 keys (a sparse top-k
    # span of 2048), or a single tile per row: no split at all
    assert attn.attn_plan_partitions(128, 128, 128, 1, 512, 2048, 0, num_sms=152) == (1, 0)
    assert attn.attn_plan_partitions(32, 64, 128, 1, 512, 64, 0, num_sms=16) == (1, 0)
    # the balanced split on request, whatever the lengths; MLA shapes only
    for max_len in (1, 64, 100000):
        P, ws = attn.attn_plan_partitions(3, 5, 128, 1, 512, max_len, attn.ATTN_PARTITIONS_BALANCED,
                                          num_sms=152)
        assert P == 0 and ws == (align(81 * 128 * 512 * 4) + 2 * align(81 * 128 * 4) +
                                 align(5 * 8))
    with pytest.raises(attn.AttnError):
        attn.attn_plan_partitions(64, 64, 16, 8, 64, 8192, attn.ATTN_PARTITIONS_BALANCED,
                                  num_sms=152)
    with pytest.raises(attn.AttnError):
        attn.attn_plan_partitions(3, 5, 128, 1, 512, 100, -3, num_sms=152)
    # an explicit MLA request is a fixed split into P slices per row
    P, ws = attn.attn_plan_partitions(32, 64, 128, 1, 512, 32768, 4, num_sms=152)
    assert P == 4 and ws == align(4 * 64 * 128 * 512 * 4) + 2 * align(4 * 64 * 128 * 4)
    P, _ = attn.attn_plan_partitions(1, 1, 32, 8, 128, 20, 0, num_sms=152)
    assert P == 1                                     # one tile of keys cannot split
    # a few query rows per sequence (the 16-column fold): the balanced split
    # up to 8 units per SM, long items beyond
    P, _ = attn.attn_plan_partitions(200, 500, 32, 8, 128, 8192, 0, num_sms=152, max_q_len=4)
    assert P == 1                                     # 1600 units, >= 2 per CTA
    P, _ = attn.attn_plan_partitions(64, 160, 32, 8, 128, 8192, 0, num_sms=152, max_q_len=4)
    assert P == BAL                                   # 512 units
    P, ws = attn.attn_plan_partitions(16, 40, 32, 8, 128, 8192, 0, num_sms=152, max_q_len=4)
    assert P == BAL and ws > 0                        # 128 units
    P, _ = attn.attn_plan_partitions(2, 8, 32, 8, 128, 8192, 0, num_sms=152, max_q_len=4)
    assert P == BAL                                   # 16 units
    # the balanced split on request: any head_dim-128 decode or few-row shape
    P, ws = attn.attn_plan_partitions(300, 300, 32, 8, 128, 4000, BAL, num_sms=152)
    assert P == BAL and ws == (align((152 + 2400) * 16 * 128 * 4) +
                               2 * align((152 + 2400) * 16 * 4) + align(2400 * 8))
    for args in ((4, 4, 16, 8, 64, 4000), (4, 40, 32, 8, 128, 4000)):   # head_dim 64; tile path
        with pytest.raises(attn.AttnError):
            attn.attn_plan_partitions(*args, BAL, num_sms=152,
                                      max_q_len=10 if args[1] > args[0] else 1)
    P, _ = attn.attn_plan_partitions(4, 4, 32, 8, 128, 0, 0, num_sms=152)
    assert P == 1
    # every CTA gets at least one slice of a full-length batch (head_dim 64:
    # two CTAs per SM); head_dim 128 deals the tiles out evenly instead
    for sms in (16, 64, 132, 152, 304):
        P, _ = attn.attn_plan_partitions(2, 2, 16, 8, 64, 65536, 0, num_sms=sms)
        assert 2 * 8 * P >= 2 * sms
        assert attn.attn_plan_partitions(2, 2, 32, 8, 128, 65536, 0, num_sms=sms)[0] == BAL
    with pytest.raises(attn.AttnError):
        attn.attn_plan_partitions(2, 2, 30, 8, 128, 100, 0, num_sms=152)
    with pytest.raises(attn.AttnError):
        attn.attn_plan_partitions(2, 2, 32, 8, 128, 100, attn.ATTN_MAX_PARTITIONS + 1,
                                  num_sms=152)


def test_planner_routes_multi_row_calls(attn):
    """The planner is the one place that routes a multi-row GQA call: the
    few-row fold (head_dim 128, max_q_len * group <= 16, batch <= 2048) keeps
    split-K on the decode kernel; longer row runs take the tile path, which
    does not split (P = 1, or the two-Q-tile request; no workspace; a larger
    request rejected)."""
    plan = attn.attn_plan_partitions
    # folded: a request is honoured verbatim, as for single rows
    for q_len, hq, hkv in ((4, 32, 8), (2, 64, 8), (16, 8, 8)):
        assert plan(4, 4 * q_len, hq, hkv, 128, 4096, 3, num_sms=152, max_q_len=q_len)[0] == 3
        assert plan(4, 4 * q_len, hq, hkv, 128, 4096, 2, num_sms=152,
                    max_q_len=q_len) == (2, 0)             # merged on chip
    # not folded: rows x group above 16, head_dim 64, or more than 2048 sequences
    for batch, q_len, hq, hkv, d in ((16, 4096, 32, 8, 128), (4, 5, 32, 8, 128),
                                     (4, 3, 64, 8, 128), (4, 2, 16, 8, 64),
                                     (2049, 2, 32, 8, 128)):
        for req in (0, 1):     # one Q tile per CTA
            assert plan(batch, batch * q_len, hq, hkv, d, 8192, req, num_sms=152,
                        max_q_len=q_len) == (1, 0)
        pair = attn.ATTN_PARTITIONS_TILE_PAIR
        assert plan(batch, batch * q_len, hq, hkv, d, 8192, pair, num_sms=152,
                    max_q_len=q_len) == (pair, 0)
        with pytest.raises(attn.AttnError) as e:
            plan(batch, batch * q_len, hq, hkv, d, 8192, 2, num_sms=152, max_q_len=q_len)
        assert e.value.status == attn.ATTN_ERR_UNSUPPORTED
    # the pair of Q tiles is a tile-path request only
    for batch, q_len, hq, hkv in ((4, 1, 32, 8), (4, 4, 32, 8), (4, 2, 128, 1)):
        with pytest.raises(attn.AttnError) as e:
            plan(batch, batch * q_len, hq, hkv, 512 if hkv == 1 else 128, 8192,
                 attn.ATTN_PARTITIONS_TILE_PAIR, num_sms=152, max_q_len=q_len)
        assert e.value.status == attn.ATTN_ERR_INVALID_ARG
    # MLA shapes ignore max_q_len (draft rows plan per query row)
    assert plan(32, 64, 128, 1, 512, 32768, 4, num_sms=152, max_q_len=2) == \
        plan(32, 64, 128, 1, 512, 32768, 4, num_sms=152, max_q_len=1)
    with pytest.raises(attn.AttnError) as e:
        plan(4, 4, 32, 8, 128, 100, 0, num_sms=152, max_q_len=0)
    assert e.value.status == attn.ATTN_ERR_INVALID_ARG


def call_noalloc(attn, k=None, v=None, **over):
    args = dict(q=0x30000, kv_len=0x40000, offs=None, batch=2, rows=None, hq=32, group=4,
                d=128, max_q_len=1, max_kv_len=500, scale=0.088, sink=None, causal=0, P=1,
                out=0x50000, lse=None)
    args.update(over)
    if args["rows"] is None:
        args["rows"] = args["batch"]
    k = k or kv(attn)
    v = v or kv(attn)
    return attn.lib().attn_decode_noalloc(args["q"], ctypes.byref(k), ctypes.byref(v),
                                          args["kv_len"], args["offs"], args["batch"],
                                          args["rows"], args["hq"], args["group"], args["d"],
                                          args["max_q_len"], args["max_kv_len"], args["scale"],
                                          args["sink"], args["causal"], args["P"], args["out"],
                                          args["lse"], None)


def test_noalloc_routes_and_rejects_as_attn_decode(attn):
    """attn_decode_noalloc plans through the same planner: a count attn_decode
    rejects is rejected here too, before anything is launched."""
    E = attn
    assert call_noalloc(attn, P=-1) == E.ATTN_ERR_INVALID_ARG
    assert call_noalloc(attn, P=E.ATTN_MAX_PARTITIONS + 1) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, P=E.ATTN_MAX_PARTITIONS + 1) == E.ATTN_ERR_INVALID_ARG
    # the pair of Q tiles only on the tile path
    pair = E.ATTN_PARTITIONS_TILE_PAIR
    assert call_decode(attn, P=pair) == E.ATTN_ERR_INVALID_ARG
    assert call_decode(attn, P=-3) == E.ATTN_ERR_INVALID_ARG
    # the tile kernel (rows x group above 16) does not split
    assert call_noalloc(attn, offs=0x70000, rows=40, max_q_len=30, P=2) == E.ATTN_ERR_UNSUPPORTED
    assert call_decode(attn, offs=0x70000, rows=40, max_q_len=30, P=2) == E.ATTN_ERR_UNSUPPORTED
    # 64 partitions x 64 rows x 32 heads x 128 channels x 4 B = 64 MiB > 32 MiB of scratch
    assert call_noalloc(attn, batch=64, P=64) == E.ATTN_ERR_WORKSPACE
    # argument checks of attn_decode still apply
    assert call_noalloc(attn, q=None) == E.ATTN_ERR_INVALID_ARG
    assert call_noalloc(attn, hq=30) == E.ATTN_ERR_INVALID_ARG


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "split_flash_decoding_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, flags=re.M), f
                assert "attn_oracle" not in text, f
