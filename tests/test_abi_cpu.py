"""C ABI checks that need no GPU: the library loads and exports every symbol
include/mcp.h declares; host-side validation; the slot-mapping builder against
the oracle (bit-exact); the work planner's coverage invariants."""

from __future__ import annotations

import ctypes
import math
import re
from pathlib import Path

import numpy as np
import pytest

import mixed_chunked_prefill_gb300 as mcp
import oracle
import synth
from mixed_chunked_prefill_gb300 import _capi
from plan_tools import desc_for, plan_host

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "mcp.h"


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from mixed_chunked_prefill_gb300 import build

    build.build()
    return mcp.load()


def header_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mcp_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = mcp.load()
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in mcp.h but not exported"
    assert set(names) == set(_capi.SIGNATURES), "binding signatures out of sync with mcp.h"


def test_status_strings_and_version():
    lib = mcp.load()
    for code, name in [(0, b"MCP_OK"), (1, b"MCP_ERR_INVALID_ARG"), (2, b"MCP_ERR_UNSUPPORTED"),
                       (3, b"MCP_ERR_WORKSPACE_TOO_SMALL"), (4, b"MCP_ERR_CUDA"),
                       (5, b"MCP_ERR_TIMEOUT"), (6, b"MCP_ERR_DEVICE_CHECK")]:
        assert lib.mcp_status_string(code) == name
    assert lib.mcp_status_string(99) == b"MCP_ERR_UNKNOWN"
    assert mcp.abi_version() == 1


# ---------------------------------------------------------------------------
# validation (returns before touching the device)
# ---------------------------------------------------------------------------

def _plan_status(desc, cu, sk, **kw):
    st, *_ = plan_host(desc, cu, sk, **kw)
    return st


def base_desc(**over):
    d = dict(num_seqs=3, total_q=1810, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
             max_pages_per_seq=625, num_pages=700, sm_scale=1 / math.sqrt(128))
    d.update(over)
    return mcp.make_desc(**d)


CU = [0, 1, 2, 1810]
SK = [121, 46, 10000]


def test_valid_worked_layout_plans():
    assert _plan_status(base_desc(), CU, SK) == _capi.MCP_OK


@pytest.mark.parametrize("over,cu,sk,code", [
    (dict(num_q_heads=30), CU, SK, _capi.MCP_ERR_INVALID_ARG),          # H_q % H_kv
    (dict(head_dim=80), CU, SK, _capi.MCP_ERR_UNSUPPORTED),
    (dict(page_size=4), CU, SK, _capi.MCP_ERR_UNSUPPORTED),
    (dict(page_size=48), CU, SK, _capi.MCP_ERR_UNSUPPORTED),
    (dict(page_size=128), CU, SK, _capi.MCP_ERR_UNSUPPORTED),
    (dict(num_pages=0), CU, SK, _capi.MCP_ERR_INVALID_ARG),
    (dict(max_pages_per_seq=100), CU, SK, _capi.MCP_ERR_INVALID_ARG),   # 10000 keys need 625 pages
    (dict(total_q=1811), CU, SK, _capi.MCP_ERR_INVALID_ARG),
    (dict(), [1, 1, 2, 1810], SK, _capi.MCP_ERR_INVALID_ARG),           # cu[0] != 0
    (dict(), [0, 2, 1, 1810], SK, _capi.MCP_ERR_INVALID_ARG),           # decreasing
    (dict(), CU, [121, 0, 10000], _capi.MCP_ERR_INVALID_ARG),           # Lq > Lk
    (dict(), CU, [121, 46, 1000], _capi.MCP_ERR_INVALID_ARG),           # chunk longer than its KV
    (dict(), CU, [121, -1, 10000], _capi.MCP_ERR_INVALID_ARG),
    (dict(sm_scale=float("nan")), CU, SK, _capi.MCP_ERR_INVALID_ARG),
    (dict(num_q_heads=1024, num_kv_heads=4), CU, SK, _capi.MCP_ERR_UNSUPPORTED),  # group > 128
])
def test_plan_rejects_bad_metadata(over, cu, sk, code):
    assert _plan_status(base_desc(**over), cu, sk) == code
    assert mcp.load().mcp_last_error() != b""


def test_plan_rejects_null_and_reserved_options():
    lib = mcp.load()
    cu = np.array(CU, dtype=np.int32)
    plan = mcp.Plan()
    d = base_desc()
    assert lib.mcp_mixed_attn_plan_host(None, cu.ctypes.data_as(ctypes.c_void_p), None, None,
                                        ctypes.byref(plan), None, 0) == _capi.MCP_ERR_INVALID_ARG
    assert lib.mcp_mixed_attn_plan_host(ctypes.byref(d), None, None, None, ctypes.byref(plan),
                                        None, 0) == _capi.MCP_ERR_INVALID_ARG
    opts = mcp.PlanOptions(152, 0, 0)
    opts.reserved[1] = 3
    sk = np.array(SK, dtype=np.int32)
    assert lib.mcp_mixed_attn_plan_host(ctypes.byref(d), cu.ctypes.data_as(ctypes.c_void_p),
                                        sk.ctypes.data_as(ctypes.c_void_p), ctypes.byref(opts),
                                        ctypes.byref(plan), None, 0) == _capi.MCP_ERR_INVALID_ARG


def test_plan_records_test_stall_and_rejects_other_values():
    """test_stall (failure-detection tests only) is 0 or 1 and travels in the
    plan to the forward call; it changes no work item."""
    opts = mcp.PlanOptions(152, 0, 0)
    st0, plan0, items0, _ = plan_host(base_desc(), CU, SK, opts=opts)
    opts.test_stall = 1
    st1, plan1, items1, _ = plan_host(base_desc(), CU, SK, opts=opts)
    assert st0 == st1 == 0
    assert plan0.test_stall == 0 and plan1.test_stall == 1
    assert np.array_equal(items0, items1)
    opts.test_stall = 2
    st2, *_ = plan_host(base_desc(), CU, SK, opts=opts)
    assert st2 == _capi.MCP_ERR_INVALID_ARG


def test_plan_host_buffer_too_small():
    lib = mcp.load()
    st, plan, _, _ = plan_host(base_desc(), CU, SK)
    assert st == 0
    cu = np.array(CU, dtype=np.int32)
    sk = np.array(SK, dtype=np.int32)
    buf = np.zeros(16, dtype=np.uint8)
    opts = mcp.PlanOptions(152, 0, 0)
    assert lib.mcp_mixed_attn_plan_host(
        ctypes.byref(base_desc()), cu.ctypes.data_as(ctypes.c_void_p),
        sk.ctypes.data_as(ctypes.c_void_p), ctypes.byref(opts), ctypes.byref(plan),
        buf.ctypes.data_as(ctypes.c_void_p), buf.size) == _capi.MCP_ERR_WORKSPACE_TOO_SMALL


def test_append_validation_before_launch():
    lib = mcp.load()
    assert lib.mcp_paged_kv_append(None, None, None, -1, 8, 128, 16, 10, None, None, None,
                                   None) == _capi.MCP_ERR_INVALID_ARG
    assert lib.mcp_paged_kv_append(None, None, None, 4, 8, 128, 16, 10, None, None, None,
                                   None) == _capi.MCP_ERR_INVALID_ARG
    assert lib.mcp_paged_kv_append(None, None, None, 4, 3, 5, 16, 10, None, None, None,
                                   None) == _capi.MCP_ERR_INVALID_ARG   # row not 16-byte multiple
    assert lib.mcp_paged_kv_append(None, None, None, 0, 8, 128, 16, 10, None, None, None,
                                   None) == _capi.MCP_OK               # nothing to do


def test_fwd_validation_before_launch():
    lib = mcp.load()
    bogus = mcp.Plan()
    assert lib.mcp_mixed_attn_fwd(ctypes.byref(bogus), *([None] * 9), 0, None) == \
        _capi.MCP_ERR_INVALID_ARG
    st, plan, _, _ = plan_host(base_desc(), CU, SK)
    assert lib.mcp_mixed_attn_fwd(ctypes.byref(plan), *([None] * 9), 0, None) == \
        _capi.MCP_ERR_INVALID_ARG
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check fails first
    assert lib.mcp_mixed_attn_fwd(ctypes.byref(plan), fake, fake, fake, fake, fake, fake, fake,
                                  None, fake, 16, None) == _capi.MCP_ERR_WORKSPACE_TOO_SMALL
    assert lib.mcp_merge_states(None, None, 0, 1, 1, 8, None, None, None) == \
        _capi.MCP_ERR_INVALID_ARG
    assert lib.mcp_check_device_errors(None, None) == _capi.MCP_ERR_INVALID_ARG


# ---------------------------------------------------------------------------
# slot mapping: the C builder equals the oracle, bit for bit
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", synth.CONFIG_NAMES)
def test_slot_mapping_matches_oracle(name):
    w = synth.make_workload(name)
    bt = w.block_tables()
    cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
    table = oracle.page_table_from_block_tables(bt, w.k_lens, w.page_size)
    expect = oracle.new_token_slots(table, cu, w.k_lens)
    got = mcp.build_slot_mapping(bt, cu, w.k_lens, w.page_size, w.num_pages)
    assert got.dtype == np.int64
    assert np.array_equal(got, expect)


def test_slot_mapping_history_layout_matches_oracle():
    # the same builder fills history positions (a step whose tokens are the history)
    w = synth.make_workload("balanced")
    bt = w.block_tables()
    hist = w.hist_lens
    cu_h, _, _, _ = oracle.segment_layout(hist, hist)
    table = oracle.page_table_from_block_tables(bt, w.k_lens, w.page_size)
    expect = oracle.new_token_slots(table, cu_h, hist)
    got = mcp.build_slot_mapping(bt, cu_h, hist, w.page_size, w.num_pages)
    assert np.array_equal(got, expect)


def test_slot_mapping_rejects_page_outside_pool():
    bt = np.array([[0, 1, 99]], dtype=np.int32)
    with pytest.raises(mcp.MCPError):
        mcp.build_slot_mapping(bt, [0, 3], [40], 16, 10)


def test_slot_mapping_rejects_shared_slots():
    """[L] 4.2 writes through atomics; the append here relies on distinct slots
    instead, so a step whose new tokens share a slot is refused on the host."""
    # two decodes whose last page is the same physical page 4, at the same offset
    bt = np.array([[0, 4], [1, 4]], dtype=np.int32)
    with pytest.raises(mcp.MCPError) as ei:
        mcp.build_slot_mapping(bt, [0, 1, 2], [20, 20], 16, 10)
    assert ei.value.status == _capi.MCP_ERR_INVALID_ARG
    assert b"two new tokens" in mcp.load().mcp_last_error()
    # the same page at different offsets is not a shared slot
    got = mcp.build_slot_mapping(bt, [0, 1, 2], [20, 21], 16, 10)
    assert got.tolist() == [4 * 16 + 3, 4 * 16 + 4]
    # a page repeated inside one row, both positions written this step
    bt1 = np.array([[3, 3]], dtype=np.int32)
    with pytest.raises(mcp.MCPError):
        mcp.build_slot_mapping(bt1, [0, 32], [32], 16, 10)


def test_checked_build_exports_the_same_abi_and_says_so():
    """The MCP_CHECKED variant (device-side duplicate-slot check in the append)
    builds, exports every declared symbol and reports its build flag; the
    default library does not."""
    from mixed_chunked_prefill_gb300 import build

    path = build.build(checked=True)
    lib = _capi.open_library(path)
    for n in header_functions():
        assert hasattr(lib, n), n
    assert lib.mcp_build_flags() == _capi.BUILD_CHECKED
    assert mcp.load().mcp_build_flags() == 0


# ---------------------------------------------------------------------------
# planner invariants
# ---------------------------------------------------------------------------

def check_plan_covers(w, items, comb, plan):
    """Every (segment, kv head, query token) row is covered by exactly one set
    of items whose KV ranges tile [0, visible end of the item's last token)."""
    G = w.num_q_heads // w.num_kv_heads
    cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
    assert plan.num_items == len(items)
    assert plan.num_decode_items + plan.num_prefill_items == len(items)
    assert (items["kind"] == 0).sum() == plan.num_decode_items
    cover = {}
    HG = 1
    while HG * 2 <= 8 and w.num_kv_heads % (HG * 2) == 0:
        HG *= 2
    for it in items:
        s = int(it["seg"])
        lq, lk = w.q_lens[s], w.k_lens[s]
        assert 0 <= it["q_begin"] and it["q_begin"] + it["q_count"] <= lq and it["q_count"] > 0
        assert 0 <= it["kv_begin"] < it["kv_end"] <= lk
        vis_end = lk - lq + it["q_begin"] + it["q_count"]
        assert it["kv_end"] <= vis_end
        if it["kind"] == 0:
            assert it["q_count"] * G <= 16 and it["kv_begin"] % 16 == 0
            assert it["q_begin"] == 0 and it["q_count"] == lq
            assert it["num_heads"] == HG and it["kv_head"] % HG == 0
        else:
            assert it["q_count"] * G <= 128 and it["kv_begin"] % 128 == 0
            # small segments take tiles only where the decode path is not built
            decode_built = w.head_dim <= 128 and w.page_size >= 8
            assert it["q_count"] * G > 16 or lq * G > 16 or not decode_built
            assert it["num_heads"] == 1
        for j in range(int(it["num_heads"])):
            h = int(it["kv_head"]) + j
            part = -1 if it["part_row"] < 0 else int(it["part_row"]) + j * int(it["part_head_stride"])
            key = (s, h, int(it["q_begin"]), int(it["q_count"]))
            cover.setdefault(key, []).append((int(it["kv_begin"]), int(it["kv_end"]), part))
    # each row group: KV ranges tile [0, vis_end)
    rows_seen = {}
    for (s, h, qb, qc), ranges in cover.items():
        ranges.sort()
        vis_end = w.k_lens[s] - w.q_lens[s] + qb + qc
        assert ranges[0][0] == 0 and ranges[-1][1] == vis_end
        for a, b in zip(ranges[:-1], ranges[1:]):
            assert a[1] == b[0]
        if len(ranges) == 1:
            assert ranges[0][2] == -1
        else:
            assert all(r[2] >= 0 for r in ranges)
        for t in range(qb, qb + qc):
            rows_seen[(s, h, t)] = rows_seen.get((s, h, t), 0) + 1
    for s in range(w.num_seqs):
        for h in range(w.num_kv_heads):
            for t in range(w.q_lens[s]):
                assert rows_seen.get((s, h, t), 0) == 1, (s, h, t)
    # combine entries match the split groups; partial rows never overlap
    split_groups = {k: v for k, v in cover.items() if len(v) > 1}
    assert len(comb) == len(split_groups) == plan.num_combine
    used = np.zeros(int(plan.partial_rows), dtype=np.int32)
    for e in comb:
        key = (int(e["seg"]), int(e["kv_head"]), int(e["q_begin"]), int(e["q_count"]))
        ranges = split_groups[key]
        assert e["num_splits"] == len(ranges) and e["rows"] == e["q_count"] * G
        parts = sorted(r[2] for r in ranges)
        assert parts == [int(e["part_row"]) + k * int(e["rows"]) for k in range(len(ranges))]
        used[e["part_row"]:e["part_row"] + e["num_splits"] * e["rows"]] += 1
    assert (used <= 1).all()
    # the combine kernel's flat row numbering: entries own consecutive row ranges
    if len(comb):
        starts = np.concatenate([[0], np.cumsum(comb["rows"])[:-1]])
        assert np.array_equal(comb["row_base"], starts)
    assert plan.combine_rows == int(comb["rows"].sum()) if len(comb) else plan.combine_rows == 0


@pytest.mark.parametrize("name", synth.CONFIG_NAMES)
def test_planner_covers_every_row_once(name):
    w = synth.make_workload(name)
    cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
    st, plan, items, comb = plan_host(desc_for(w), cu, w.k_lens)
    assert st == 0
    check_plan_covers(w, items, comb, plan)


@pytest.mark.parametrize("name", ["tiny", "worked", "balanced"])
@pytest.mark.parametrize("head_dim,page_size", [(256, None), (None, 1), (96, 8)])
def test_planner_covers_every_row_once_other_shapes(name, head_dim, page_size):
    """head_dim 256 and 1-token pages put decodes on tensor-core tiles;
    every (token, kv head) row is still covered exactly once."""
    w = synth.make_workload(name, head_dim=head_dim, page_size=page_size)
    cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
    for dsplit, psplit in [(0, 0), (16, 128)]:
        st, plan, items, comb = plan_host(desc_for(w), cu, w.k_lens, dsplit=dsplit, psplit=psplit)
        assert st == 0
        check_plan_covers(w, items, comb, plan)
        if w.head_dim == 256 or w.page_size == 1:
            assert plan.num_decode_items == 0


@pytest.mark.parametrize("dsplit,psplit", [(16, 128), (48, 256), (1024, 1024)])
def test_planner_forced_splits(dsplit, psplit):
    for name in ("tiny", "worked"):
        w = synth.make_workload(name)
        cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
        st, plan, items, comb = plan_host(desc_for(w), cu, w.k_lens, dsplit=dsplit, psplit=psplit)
        assert st == 0
        assert plan.decode_split_tokens == -(-dsplit // 16) * 16
        assert plan.prefill_split_tokens == -(-psplit // 128) * 128
        check_plan_covers(w, items, comb, plan)
        if psplit < 10000 or dsplit < 121:
            assert plan.num_combine > 0 or name == "tiny"


@pytest.mark.parametrize("name,dsplit,psplit", [("worked", 16, 256), ("balanced", 0, 0),
                                                ("balanced", 64, 1024), ("tiny", 16, 128)])
def test_combine_block_index(name, dsplit, psplit):
    """After the combine entries the plan stores, for every block of 8 merged
    rows, the entry that holds the block's first row; the lists region
    (off_part_o bytes) covers it."""
    lib = mcp.load()
    w = synth.make_workload(name)
    cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
    st, plan, items, comb = plan_host(desc_for(w), cu, w.k_lens, dsplit=dsplit, psplit=psplit)
    assert st == 0 and plan.num_combine > 0
    cu32 = np.ascontiguousarray(np.asarray(cu, dtype=np.int32))
    sk32 = np.ascontiguousarray(np.asarray(w.k_lens, dtype=np.int32))
    buf = np.zeros(int(plan.off_part_o), dtype=np.uint8)
    opts = mcp.PlanOptions(152, dsplit, psplit)
    assert lib.mcp_mixed_attn_plan_host(ctypes.byref(desc_for(w)), cu32.ctypes.data_as(ctypes.c_void_p),
                                        sk32.ctypes.data_as(ctypes.c_void_p), ctypes.byref(opts),
                                        ctypes.byref(plan), buf.ctypes.data_as(ctypes.c_void_p),
                                        buf.size) == 0
    nblocks = -(-int(plan.combine_rows) // 8)
    start = int(plan.off_combine) + int(plan.num_combine) * 32
    assert start + 4 * nblocks <= int(plan.off_part_o)
    idx = buf[start:start + 4 * nblocks].view("<i4")
    assert int(comb["row_base"][0]) == 0
    assert int(comb["row_base"][-1] + comb["rows"][-1]) == int(plan.combine_rows)
    for b, e in enumerate(idx):
        r = 8 * b
        assert 0 <= e < plan.num_combine
        assert comb["row_base"][e] <= r < comb["row_base"][e] + comb["rows"][e]


def test_planner_random_shapes():
    rng = np.random.Generator(np.random.PCG64(123))
    for trial in range(40):
        hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 3, 4, 8, 16]))
        S = int(rng.integers(1, 9))
        q, k = [], []
        for _ in range(S):
            lq = int(rng.choice([0, 1, 1, 2, 3, 17, 100, 300]))
            hist = int(rng.integers(0, 3000))
            q.append(lq)
            k.append(max(lq + hist, 1 if lq > 0 else 0))
        w = synth.make_workload_from_lengths("r", G * hkv, hkv, 128, 16, 0.1, q, k, 7 + trial)
        cu, _, _, _ = oracle.segment_layout(q, k)
        st, plan, items, comb = plan_host(desc_for(w), cu, k, num_sms=int(rng.integers(1, 200)),
                                          dsplit=int(rng.choice([0, 64, 512])),
                                          psplit=int(rng.choice([0, 256, 1024])))
        assert st == 0
        check_plan_covers(w, items, comb, plan)


def test_planner_balance_bound_big_configs():
    # greedy list scheduling of the planned order over 152 SMs stays close to the
    # lower bound max(total / SMs, longest item) under the planner's own cost units
    for name in ("decode-heavy", "long-context"):
        w = synth.make_workload(name)
        cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
        st, plan, items, comb = plan_host(desc_for(w), cu, w.k_lens)
        D = w.head_dim
        cost = np.where(items["kind"] == 0,
                        (items["kv_end"] - items["kv_begin"]) * 4.0 * D * items["num_heads"] / 45.0,
                        300.0 + np.ceil((items["kv_end"] - items["kv_begin"]) / 128)
                        * 4.0 * 128 * 128 * D / 6000.0)
        import heapq
        sms = [0.0] * 152
        heapq.heapify(sms)
        for c in cost:
            t = heapq.heappop(sms)
            heapq.heappush(sms, t + c)
        makespan = max(sms)
        lower = max(cost.sum() / 152, cost.max())
        assert makespan <= 1.1 * lower, (name, makespan / lower)


def test_kv_copy_pages_validation_before_launch():
    lib = mcp.load()
    p = ctypes.c_void_p(0x1000)
    # page_bytes not a multiple of 16, negative sizes, NULLs, misaligned pools
    assert lib.mcp_kv_copy_pages(p, p, 4, p, p, 4, 24, p, p, 1, None, None) == 1
    assert lib.mcp_kv_copy_pages(p, p, -1, p, p, 4, 32, p, p, 1, None, None) == 1
    assert lib.mcp_kv_copy_pages(None, p, 4, p, p, 4, 32, p, p, 1, None, None) == 1
    assert lib.mcp_kv_copy_pages(ctypes.c_void_p(0x1008), p, 4, p, p, 4, 32, p, p, 1, None,
                                 None) == 1
    assert lib.mcp_kv_copy_pages(None, None, 0, None, None, 0, 32, None, None, 0, None, None) == 0


@pytest.mark.parametrize("page_size", [8, 32, 64])
def test_other_page_sizes_plan_and_slot_mapping(page_size):
    """Pages of 8 / 32 / 64 tokens: the plan is the same as with 16-token pages
    (the kernels step over 16-token blocks), the slot mapping follows the oracle."""
    w16 = synth.make_workload("worked")
    w = synth.make_workload_from_lengths("p", w16.num_q_heads, w16.num_kv_heads, w16.head_dim,
                                         page_size, w16.sm_scale, w16.q_lens, w16.k_lens, 3)
    cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
    st, plan, items, comb = plan_host(desc_for(w), cu, w.k_lens)
    assert st == 0
    st16, plan16, items16, _ = plan_host(desc_for(w16), cu, w16.k_lens)
    assert plan.num_items == plan16.num_items
    assert np.array_equal(items, items16)
    bt = w.block_tables()
    table = oracle.page_table_from_block_tables(bt, w.k_lens, page_size)
    want = oracle.new_token_slots(table, cu, w.k_lens)
    got = mcp.build_slot_mapping(bt, cu, w.k_lens, page_size, w.num_pages)
    assert np.array_equal(got, want)


def test_varlen_fwd_validation_before_launch():
    lib = mcp.load()
    d = base_desc()
    cu = np.array([0, 1, 2, 1810], dtype=np.int32)
    sk = np.array([121, 46, 10000], dtype=np.int32)
    plan = mcp.Plan()
    opts = mcp.PlanOptions(152, 0, 0)  # no device query on the CPU
    assert lib.mcp_mixed_attn_plan(ctypes.byref(d), cu.ctypes.data_as(ctypes.c_void_p),
                                   sk.ctypes.data_as(ctypes.c_void_p), ctypes.byref(opts),
                                   ctypes.byref(plan), None, 0, None) == 0
    p = ctypes.c_void_p(0x1000)
    assert lib.mcp_mixed_attn_fwd_varlen(None, p, p, p, p, p, 10, p, None, p, 1 << 30, None) == 1
    assert lib.mcp_mixed_attn_fwd_varlen(ctypes.byref(plan), None, p, p, p, p, 10, p, None, p,
                                         1 << 30, None) == 1
    assert lib.mcp_mixed_attn_fwd_varlen(ctypes.byref(plan), p, p, p, p, p, -1, p, None, p,
                                         1 << 30, None) == 1
    # a plan for 32-token pages cannot drive the non-paged forward
    d32 = base_desc(page_size=32, max_pages_per_seq=313)
    plan32 = mcp.Plan()
    assert lib.mcp_mixed_attn_plan(ctypes.byref(d32), cu.ctypes.data_as(ctypes.c_void_p),
                                   sk.ctypes.data_as(ctypes.c_void_p), ctypes.byref(opts),
                                   ctypes.byref(plan32), None, 0, None) == 0
    assert lib.mcp_mixed_attn_fwd_varlen(ctypes.byref(plan32), p, p, p, p, p, 10, p, None, p,
                                         1 << 30, None) == 1


def test_head_dim_96_plans_with_96_wide_partials():
    """head_dim 96 runs the D = 128 kernel on 96-wide tensors: the plan is the
    one for D = 128, and the split partials are 96 floats per row."""
    d96 = base_desc(head_dim=96, sm_scale=1 / math.sqrt(96))
    d128 = base_desc()
    st96, p96, items96, _ = plan_host(d96, CU, SK, dsplit=16, psplit=128)
    st128, p128, items128, _ = plan_host(d128, CU, SK, dsplit=16, psplit=128)
    assert st96 == 0 and st128 == 0
    assert p96.num_items == p128.num_items and np.array_equal(items96, items128)
    rows = p96.partial_rows
    assert rows > 0
    assert p96.off_part_lse - p96.off_part_o >= rows * 96 * 4
    assert p96.off_part_lse - p96.off_part_o < rows * 128 * 4


def test_head_dim_256_plans_without_decode_items():
    """The decode path is built up to head_dim 128: at 256 every segment,
    decodes included, becomes tensor-core tiles."""
    d = base_desc(head_dim=256, sm_scale=1 / 16.0)
    st, plan, items, _ = plan_host(d, CU, SK)
    assert st == 0
    assert plan.num_decode_items == 0
    assert plan.num_prefill_items == plan.num_items > 0
    kinds = items["kind"] if items.dtype.names else None
    if kinds is not None:
        assert (kinds == 1).all()


def test_page_size_1_plans_tiles_and_slot_mapping():
    """1-token pages: every segment becomes tensor-core tiles (the decode path
    is built for pages of 8 or more tokens); slots follow the oracle."""
    w16 = synth.make_workload("worked")
    w = synth.make_workload("worked", page_size=1)
    cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
    st, plan, items, _ = plan_host(desc_for(w), cu, w.k_lens)
    assert st == 0 and plan.num_decode_items == 0 and plan.num_prefill_items == plan.num_items
    st16, plan16, _, _ = plan_host(desc_for(w16), cu, w16.k_lens)
    assert plan.num_items == plan16.num_items - plan16.num_decode_items + 2 * w.num_kv_heads
    bt = w.block_tables()
    table = oracle.page_table_from_block_tables(bt, w.k_lens, 1)
    want = oracle.new_token_slots(table, cu, w.k_lens)
    got = mcp.build_slot_mapping(bt, cu, w.k_lens, 1, w.num_pages)
    assert np.array_equal(got, want)


def _exhaustive_chunk_split(q_lens, k_lens, hq, hkv, d, num_sms):
    """The split size an exhaustive list-scheduling search picks for a step of
    chunks only: the planner's cost model (per item ~5 us + ~0.75 us per
    128-key tile at D = 128, longest item first onto the least-loaded SM),
    every candidate from 65536 down to 2048 evaluated, ties within 2% to the
    larger split.  Returns (split, items of that split)."""
    import heapq

    G = hq // hkv
    TQ = 128 // G

    def cdiv(a, b):
        return -(-a // b)

    def even_split(length, cap, gran):
        k = max(1, cdiv(length, cap))
        sz = cdiv(cdiv(length, k), gran) * gran
        return cdiv(length, sz), sz

    vis = []
    for lq, lk in zip(q_lens, k_lens):
        assert lq * G > 16  # chunks only: no decode units
        for qb in range(0, lq, TQ):
            vis.append(lk - lq + qb + min(TQ, lq - qb))
    count = lambda ps: sum(even_split(v, ps, 128)[0] for v in vis) * hkv
    ps = 32768
    while count(ps) < 2 * num_sms and ps > 2048:
        ps //= 2
    tile_ns, item_ns = 750.0 * d / 128.0, 5000.0

    def makespan(cand):
        cost = []
        for v in vis:
            n, sz = even_split(v, cand, 128)
            for k in range(n):
                c = item_ns + cdiv(min(sz, v - k * sz), 128) * tile_ns
                cost += [c] * hkv
        cost.sort(reverse=True)
        load = [0.0] * num_sms
        for c in cost:
            heapq.heapreplace(load, load[0] + c)
        return max(load)

    best, best_t = ps, makespan(ps)
    cand = 65536
    while cand >= 2048:
        t = makespan(cand)
        if t < best_t * 0.98 or (t <= best_t * 1.02 and cand > best):
            best_t = min(best_t, t)
            best = cand
        cand //= 2
    return best, count(best)


@pytest.mark.parametrize("seed", range(40))
def test_pruned_split_search_matches_exhaustive(seed):
    """The planner evaluates only distinct split candidates and none past
    sixteen items per SM; on chunk-only steps it picks what the exhaustive
    search picks whenever that choice is within sixteen items per SM."""
    rng = np.random.Generator(np.random.PCG64(5000 + seed))
    num_sms = int(rng.choice([152, 148, 132, 100]))
    hq, hkv = [(32, 8), (64, 8), (16, 16), (32, 4)][seed % 4]
    nseg = int(rng.integers(1, 4))
    q_lens = [int(x) for x in rng.integers(64, 2048, size=nseg)]
    k_lens = [q + int(h) for q, h in zip(q_lens, rng.integers(0, 40000, size=nseg))]
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    mp = max(-(-k // 16) for k in k_lens)
    d = mcp.make_desc(nseg, int(cu[-1]), hq, hkv, 128, 16, mp, mp * nseg + 1, 1 / math.sqrt(128))
    st, plan, _, _ = plan_host(d, cu, k_lens, num_sms=num_sms)
    assert st == 0
    want, items = _exhaustive_chunk_split(q_lens, k_lens, hq, hkv, 128, num_sms)
    if items <= 16 * num_sms:
        assert plan.prefill_split_tokens == want, (q_lens, k_lens, num_sms, want)
