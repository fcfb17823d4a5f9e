"""Test helpers: run the host planner through the C ABI and decode its lists."""

from __future__ import annotations

import ctypes

import numpy as np

import mixed_chunked_prefill_gb300 as mcp
from mixed_chunked_prefill_gb300 import _capi

ITEM = np.dtype([("seg", "<i4"), ("kv_head", "<i2"), ("kind", "i1"), ("num_heads", "i1"),
                 ("q_begin", "<i4"), ("q_count", "<i4"), ("kv_begin", "<i4"), ("kv_end", "<i4"),
                 ("part_row", "<i4"), ("part_head_stride", "<i4")])
COMB = np.dtype([("seg", "<i4"), ("kv_head", "<i4"), ("q_begin", "<i4"), ("q_count", "<i4"),
                 ("num_splits", "<i4"), ("part_row", "<i4"), ("rows", "<i4"), ("row_base", "<i4")])


def desc_for(w):
    return mcp.make_desc(w.num_seqs, w.total_q, w.num_q_heads, w.num_kv_heads, w.head_dim,
                         w.page_size, w.max_pages_per_seq, w.num_pages, w.sm_scale)


def plan_host(desc, cu, sk, num_sms=152, dsplit=0, psplit=0, opts=None):
    """(status, plan, items, combine) from mcp_mixed_attn_plan_host (``opts``
    replaces num_sms / dsplit / psplit when given)."""
    lib = mcp.load()
    cu = np.ascontiguousarray(np.asarray(cu, dtype=np.int32))
    sk = np.ascontiguousarray(np.asarray(sk, dtype=np.int32))
    if opts is None:
        opts = mcp.PlanOptions(num_sms, dsplit, psplit)
    plan = mcp.Plan()
    st = lib.mcp_mixed_attn_plan_host(ctypes.byref(desc), cu.ctypes.data_as(ctypes.c_void_p),
                                      sk.ctypes.data_as(ctypes.c_void_p), ctypes.byref(opts),
                                      ctypes.byref(plan), None, 0)
    if st != _capi.MCP_OK:
        return st, None, None, None
    buf = np.zeros(max(1, int(plan.off_part_o)), dtype=np.uint8)
    st = lib.mcp_mixed_attn_plan_host(ctypes.byref(desc), cu.ctypes.data_as(ctypes.c_void_p),
                                      sk.ctypes.data_as(ctypes.c_void_p), ctypes.byref(opts),
                                      ctypes.byref(plan), buf.ctypes.data_as(ctypes.c_void_p),
                                      buf.size)
    assert st == _capi.MCP_OK
    items = buf[:plan.num_items * 32].view(ITEM).copy()
    comb = buf[plan.off_combine:plan.off_combine + plan.num_combine * 32].view(COMB).copy()
    return st, plan, items, comb


def plan_rows_host(desc, cu, sk, rows, num_sms=152, dsplit=0, psplit=0):
    """(status, plan, items, combine) from mcp_mixed_attn_plan_rows_host."""
    lib = mcp.load()
    cu = np.ascontiguousarray(np.asarray(cu, dtype=np.int32))
    sk = np.ascontiguousarray(np.asarray(sk, dtype=np.int32))
    rw = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    opts = mcp.PlanOptions(num_sms, dsplit, psplit)
    plan = mcp.Plan()
    args = (ctypes.byref(desc), cu.ctypes.data_as(ctypes.c_void_p),
            sk.ctypes.data_as(ctypes.c_void_p), rw.ctypes.data_as(ctypes.c_void_p), int(rw.size),
            ctypes.byref(opts), ctypes.byref(plan))
    st = lib.mcp_mixed_attn_plan_rows_host(*args, None, 0)
    if st != _capi.MCP_OK:
        return st, None, None, None
    buf = np.zeros(max(1, int(plan.off_part_o)), dtype=np.uint8)
    st = lib.mcp_mixed_attn_plan_rows_host(*args, buf.ctypes.data_as(ctypes.c_void_p), buf.size)
    assert st == _capi.MCP_OK
    items = buf[:plan.num_items * 32].view(ITEM).copy()
    comb = buf[plan.off_combine:plan.off_combine + plan.num_combine * 32].view(COMB).copy()
    return st, plan, items, comb
