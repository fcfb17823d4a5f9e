"""Sampled rows on the host: logits_indices and the rows-only planner.

[W] wangyu.me "大语言模型推理优化（二）：Chunked Prefill", section
"采样：只有该出字的请求才出字": logits are computed at the last position of
every segment, logits_indices = query_start_loc[1:] - 1.
"""

from __future__ import annotations

import numpy as np
import pytest

import mixed_chunked_prefill_gb300 as mcp
import oracle
import synth
from plan_tools import desc_for, plan_rows_host


def test_logits_indices_worked_layout():
    # the page's worked layout: query_start_loc = [0, 1, 2, 1810]
    assert mcp.build_logits_indices([0, 1, 2, 1810]).tolist() == [0, 1, 1809]
    # only the decodes sample when the chunk does not finish its prompt
    assert mcp.build_logits_indices([0, 1, 2, 1810], [1, 1, 0]).tolist() == [0, 1]


def test_logits_indices_random_against_definition():
    rng = np.random.Generator(np.random.PCG64(31))
    for _ in range(50):
        S = int(rng.integers(1, 20))
        lq = rng.choice([0, 1, 1, 2, 5, 300], size=S)
        cu = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
        mask = rng.integers(0, 2, size=S).astype(np.uint8)
        want = [int(cu[s + 1] - 1) for s in range(S) if lq[s] > 0]
        assert mcp.build_logits_indices(cu).tolist() == want
        want_m = [int(cu[s + 1] - 1) for s in range(S) if lq[s] > 0 and mask[s]]
        assert mcp.build_logits_indices(cu, mask).tolist() == want_m


def check_rows_plan(w, rows, items, comb, plan):
    """Every listed token is covered, for every kv head, by items whose KV
    ranges tile [0, visible end of that token); no other token is covered."""
    G = w.num_q_heads // w.num_kv_heads
    cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
    listed = set(int(r) for r in rows)
    cover = {}
    for it in items:
        s = int(it["seg"])
        hist = w.k_lens[s] - w.q_lens[s]
        qb, qc = int(it["q_begin"]), int(it["q_count"])
        assert qc > 0 and qb + qc <= w.q_lens[s]
        assert it["kv_end"] <= hist + qb + qc
        if it["kind"] == 0:
            assert qc * G <= 16
        for j in range(int(it["num_heads"])):
            h = int(it["kv_head"]) + j
            cover.setdefault((s, h, qb, qc), []).append((int(it["kv_begin"]), int(it["kv_end"])))
    seen = {}
    for (s, h, qb, qc), ranges in cover.items():
        ranges.sort()
        hist = w.k_lens[s] - w.q_lens[s]
        assert ranges[0][0] == 0 and ranges[-1][1] == hist + qb + qc
        for a, b in zip(ranges[:-1], ranges[1:]):
            assert a[1] == b[0]
        for t in range(qb, qb + qc):
            seen[(int(cu[s]) + t, h)] = seen.get((int(cu[s]) + t, h), 0) + 1
    for t in listed:
        for h in range(w.num_kv_heads):
            assert seen.get((t, h), 0) == 1, (t, h)
    assert all(t in listed for t, _ in seen)
    assert plan.num_combine == len(comb)


@pytest.mark.parametrize("name", ["tiny", "worked", "balanced"])
def test_rows_plan_logits_indices(name):
    w = synth.make_workload(name)
    cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
    rows = mcp.build_logits_indices(cu)
    st, plan, items, comb = plan_rows_host(desc_for(w), cu, w.k_lens, rows)
    assert st == 0
    check_rows_plan(w, rows, items, comb, plan)
    # one token per segment: every item is on the decode path (G <= 16 here)
    assert (items["kind"] == 0).all()


def test_rows_plan_random_subsets_and_splits():
    rng = np.random.Generator(np.random.PCG64(9))
    for trial in range(30):
        hkv = int(rng.choice([1, 2, 8]))
        G = int(rng.choice([1, 4, 8, 32]))
        S = int(rng.integers(1, 6))
        q = [int(rng.choice([0, 1, 3, 40, 300])) for _ in range(S)]
        k = [qq + int(rng.integers(0, 5000)) for qq in q]
        k = [max(kk, 1) if qq > 0 else kk for qq, kk in zip(q, k)]
        w = synth.make_workload_from_lengths("r", G * hkv, hkv, 128, 16, 0.1, q, k, trial)
        cu, _, _, _ = oracle.segment_layout(q, k)
        T = int(cu[-1])
        if T == 0:
            continue
        n = int(rng.integers(1, T + 1))
        rows = np.sort(rng.choice(T, size=n, replace=False)).astype(np.int32)
        st, plan, items, comb = plan_rows_host(desc_for(w), cu, k, rows,
                                               num_sms=int(rng.integers(1, 200)),
                                               dsplit=int(rng.choice([0, 64, 512])),
                                               psplit=int(rng.choice([0, 256])))
        assert st == 0
        check_rows_plan(w, rows, items, comb, plan)


@pytest.mark.parametrize("rows,code", [([2, 1], 1), ([0, 0], 1), ([-1], 1), ([1810], 1), ([], 0)])
def test_rows_plan_validation(rows, code):
    w = synth.make_workload("worked")
    cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
    st, plan, items, comb = plan_rows_host(desc_for(w), cu, w.k_lens, rows)
    assert st == code
    if code == 0:
        assert plan.num_items == 0
