"""The chunked-prefill scheduler (step builder), on the host.

[W] wangyu.me "大语言模型推理优化（二）：Chunked Prefill": sections "Token 预算：
max_num_batched_tokens", "调度器：running 优先，waiting 填充", "采样", and the
A/B/C example (chunk size 2048, a 10000-token prompt cut into 5 chunks while
A and B decode).  [X] m.xxqk.cn "动态批处理中的抢占与优先级调度": a 4096-token
prompt under a 512-token budget takes 8 iterations and produces its first
token in the 8th; priority admission; preemption by recompute or swap.
"""

from __future__ import annotations

import numpy as np
import pytest

import mixed_chunked_prefill_gb300 as mcp
from mixed_chunked_prefill_gb300.sched import Scheduler

P = 16


def test_budget_example_4096_prompt_512_budget():
    s = Scheduler(512, 1000, 300)
    s.add_request(7, 4096, 2)
    for it in range(8):
        p = s.schedule()
        assert p.q_lens.tolist() == [512]
        assert p.seqlens_k.tolist() == [512 * (it + 1)]
        assert p.sample_mask.tolist() == ([1] if it == 7 else [0])
        s.finish_step()
    p = s.schedule()  # the first sampled token goes through as a decode
    assert p.q_lens.tolist() == [1] and p.seqlens_k.tolist() == [4097]
    assert p.logits_indices.tolist() == [0]
    assert s.finish_step().tolist() == [7]
    assert s.stats()["free_pages"] == 1000


def test_abc_example_chunk_size_2048():
    # chunk size as a per-prefill cap; A and B decode in every step
    s = Scheduler(8192, 4000, 1000, long_prefill_token_threshold=2048)
    s.add_request(0, 8, 100)   # A
    s.add_request(1, 8, 100)   # B
    s.add_request(2, 10000, 1)  # C
    chunks = []
    for it in range(5):
        p = s.schedule()
        ids = p.request_ids.tolist()
        assert ids[:2] == [0, 1]  # A and B first: running before (and in) admission order
        assert p.q_lens[:2].tolist() == ([8, 8] if it == 0 else [1, 1])
        assert p.sample_mask[:2].tolist() == [1, 1]
        chunks.append(int(p.q_lens[2]))
        assert p.sample_mask[2] == (1 if it == 4 else 0)
        s.finish_step()
    assert chunks == [2048, 2048, 2048, 2048, 1808]


def run_random_traffic(s, reqs, steps, check_step=None):
    """Drive the scheduler; mirror every request's state from the plans and
    check the invariants the pages fix."""
    B, T_cap, thr, S_cap, pool = s._cfg
    P = s._page
    state = {r: dict(prompt=pl, tokens=pl, computed=0, generated=0, max_new=mn, pages=[])
             for r, (pl, mn, pr) in reqs.items()}
    done = set()
    for step in range(steps):
        p = s.schedule()
        if check_step:
            check_step(step, p)
        assert p.total_q <= B and p.num_seqs <= S_cap
        assert len(set(p.request_ids.tolist())) == p.num_seqs
        # preemption resets (recompute) or keeps (swap) computed tokens: read from the plan
        used = []
        for i, rid in enumerate(p.request_ids.tolist()):
            st = state[rid]
            lq = int(p.q_lens[i])
            lk = int(p.seqlens_k[i])
            assert lq >= 1
            if thr > 0 and lq > 1:
                assert lq <= thr
            start = lk - lq
            if start != st["computed"]:
                # only a recompute restarts from zero
                assert start == 0, (rid, start, st["computed"])
                st["prompt"] = st["tokens"]
                st["computed"] = 0
            assert lk <= st["tokens"]
            row = p.block_tables[i]
            npg = -(-lk // P)
            assert (row[:npg] >= 0).all() and (row[npg:] == -1).all()
            used.extend(row[:npg].tolist())
            want_sample = lk >= st["prompt"] and lk == st["tokens"]
            assert bool(p.sample_mask[i]) == want_sample
        assert len(used) == len(set(used)), "a page held by two requests in one step"
        assert all(0 <= u < pool for u in used)
        cu = p.cu_seqlens_q
        assert p.logits_indices.tolist() == [int(cu[i + 1] - 1) for i in range(p.num_seqs)
                                             if p.sample_mask[i]]
        fin = s.finish_step().tolist()
        for i, rid in enumerate(p.request_ids.tolist()):
            st = state[rid]
            st["computed"] = int(p.seqlens_k[i])
            if p.sample_mask[i]:
                st["generated"] += 1
                if st["generated"] < st["max_new"]:
                    st["tokens"] += 1
        for rid in fin:
            assert state[rid]["generated"] == state[rid]["max_new"]
            done.add(rid)
        if len(done) == len(reqs):
            break
    return done, state


class Sched(Scheduler):
    def __init__(self, budget, pages, mp, thr=0, seqs=256, swap=False, host=0, page_size=P):
        super().__init__(budget, pages, mp, page_size=page_size, max_num_seqs=seqs,
                         long_prefill_token_threshold=thr, preempt_swap=swap,
                         num_host_pages=host)
        self._cfg = (budget, mp * page_size, thr, seqs, pages)
        self._page = page_size


@pytest.mark.parametrize("swap", [False, True])
def test_random_traffic_invariants_and_completion(swap):
    rng = np.random.Generator(np.random.PCG64(12 + swap))
    reqs = {}
    s = Sched(256, 60, 40, thr=96, seqs=12, swap=swap, host=200)
    for rid in range(25):
        pl, mn, pr = int(rng.integers(1, 300)), int(rng.integers(1, 40)), int(rng.integers(0, 3))
        reqs[rid] = (pl, mn, pr)
        s.add_request(rid, pl, mn, pr)
    done, _ = run_random_traffic(s, reqs, 3000)
    assert done == set(reqs), f"unfinished: {set(reqs) - done}"
    st = s.stats()
    assert st["free_pages"] == 60 and st["finished"] == 25
    assert st["waiting"] == st["running"] == st["swapped"] == 0


def test_recompute_preemption_restarts_the_victim():
    s = Sched(512, 8, 8)  # 128 tokens of KV in total
    s.add_request(0, 60, 40)
    s.add_request(1, 60, 40)
    saw = []

    def check(step, p):
        if p.preempted.size:
            saw.append((step, p.preempted.tolist()))
    done, _ = run_random_traffic(s, {0: (60, 40, 0), 1: (60, 40, 0)}, 500, check)
    assert done == {0, 1}
    assert saw and saw[0][1] == [1]  # the later arrival goes first


def test_swap_preemption_moves_pages_out_and_back():
    s = Sched(512, 8, 8, swap=True, host=16)
    s.add_request(0, 60, 40)
    s.add_request(1, 60, 40)
    events = []

    def check(step, p):
        if p.swap_out.size:
            events.append(("out", step, p.swap_out.copy()))
        if p.swap_in.size:
            events.append(("in", step, p.swap_in.copy()))
    done, _ = run_random_traffic(s, {0: (60, 40, 0), 1: (60, 40, 0)}, 500, check)
    assert done == {0, 1}
    kinds = [e[0] for e in events]
    assert "out" in kinds and "in" in kinds and kinds.index("out") < kinds.index("in")
    out = next(e for e in events if e[0] == "out")[2]
    back = next(e for e in events if e[0] == "in")[2]
    assert sorted(out[:, 1].tolist()) == sorted(back[:, 0].tolist())  # the same host pages return


def test_priority_admission():
    s = Scheduler(100, 1000, 100)
    s.add_request(1, 100, 1, priority=0)
    s.add_request(2, 100, 1, priority=5)
    p = s.schedule()
    assert p.request_ids.tolist() == [2]


@pytest.mark.parametrize("kw,code", [
    (dict(max_num_batched_tokens=0), 1), (dict(max_num_seqs=0), 1), (dict(num_pages=0), 1),
    (dict(long_prefill_token_threshold=-1), 1), (dict(preempt_swap=2), 1),
])
def test_config_validation(kw, code):
    import ctypes

    from mixed_chunked_prefill_gb300 import _capi

    base = dict(max_num_batched_tokens=16, long_prefill_token_threshold=0, max_num_seqs=4,
                num_pages=8, page_size=16, max_pages_per_seq=4, preempt_swap=0,
                num_host_pages=0)
    base.update(kw)
    cfg = _capi.SchedConfig(*base.values(), (ctypes.c_int32 * 4)())
    h = ctypes.c_void_p()
    assert mcp.load().mcp_sched_create(ctypes.byref(cfg), ctypes.byref(h)) == code


def test_request_validation():
    s = Scheduler(64, 8, 4)
    with pytest.raises(mcp.MCPError):
        s.add_request(1, 60, 10)  # 70 tokens > 4 pages of 16
    s.add_request(2, 10, 1)
    with pytest.raises(mcp.MCPError):
        s.add_request(2, 5, 1)  # duplicate live id
    with pytest.raises(mcp.MCPError):
        s.add_request(3, 0, 1)


@pytest.mark.parametrize("page_size", [1, 8, 64])
@pytest.mark.parametrize("swap", [False, True])
def test_random_traffic_other_page_sizes(page_size, swap):
    """The same traffic with 1-, 8- and 64-token pages (the pool holds the
    same number of tokens): page-aligned block tables, no page shared, every
    request finishes and every page comes back."""
    rng = np.random.Generator(np.random.PCG64(40 + swap))
    pages, mp, host = 60 * P // page_size, 40 * P // page_size, 200 * P // page_size
    s = Sched(256, pages, mp, thr=96, seqs=12, swap=swap, host=host, page_size=page_size)
    reqs = {}
    for rid in range(25):
        pl, mn, pr = int(rng.integers(1, 300)), int(rng.integers(1, 40)), int(rng.integers(0, 3))
        reqs[rid] = (pl, mn, pr)
        s.add_request(rid, pl, mn, pr)
    done, _ = run_random_traffic(s, reqs, 3000)
    assert done == set(reqs), f"unfinished: {set(reqs) - done}"
    st = s.stats()
    assert st["free_pages"] == pages and st["finished"] == 25
