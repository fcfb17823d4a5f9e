"""GPU: requests served through many steps -- step builder, swap of preempted
sequences, pipelined host step -- against the oracle.

[W] wangyu.me "大语言模型推理优化（二）：Chunked Prefill": prompts are cut into
chunks under a token budget and mixed with decodes; every step appends
through the slot mapping, then attends ("输入组装").  [X] m.xxqk.cn: a pool too
small for all requests forces preemption (recompute, or swap to host memory
and back).  Each token's q/k/v depend only on (request, position), so
recomputed or re-chunked tokens are the same tokens; every step's output and
LSE are checked against the float64 oracle run on a page store that mirrors
the swaps and appends.
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import synth
from gpu_harness import ATOL, LSE_TOL, RMS_TOL
from harness import rel_rms

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

H_Q, H_KV, D = 8, 2, 128


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from mixed_chunked_prefill_gb300 import build

    build.build()
    import mixed_chunked_prefill_gb300 as mcp

    return mcp.load()


@pytest.mark.parametrize("swap,P", [(False, 16), (True, 16), (True, 32), (False, 8)])
def test_serving_loop_matches_oracle(swap, P):
    from mixed_chunked_prefill_gb300.serve import ServeLoop

    rng = np.random.Generator(np.random.PCG64(77 + swap))
    num_pages, mp = 40 * 16 // P, 40 * 16 // P
    scale = 1.0 / math.sqrt(D)
    loop = ServeLoop(H_Q, H_KV, D, num_pages, scale, max_num_batched_tokens=128,
                     max_pages_per_seq=mp, max_num_seqs=8, long_prefill_token_threshold=64,
                     preempt_swap=swap, num_host_pages=80, page_size=P)
    nreq = 8
    for r in range(nreq):
        loop.add_request(r, int(rng.integers(20, 300)), int(rng.integers(3, 20)),
                         int(rng.integers(0, 3)))

    def token_fn(plan):
        rid, pos = loop.positions(plan)
        return tuple(synth.token_values(rid, pos, h, D, tag).pin_memory()
                     for h, tag in ((H_Q, 0), (H_KV, 1), (H_KV, 2)))

    store = oracle.PagedKVStore(P, H_KV, D)
    host_cells = {}
    results, expected = [], []
    finished, preemptions, swaps = set(), 0, 0
    for _ in range(400):
        res = loop.step(token_fn)
        if res is None:
            break
        plan = res.plan
        preemptions += plan.preempted.size
        # mirror the swaps in the oracle's page store, then append and attend
        # (a sequence's last page may be partly filled: move the cells that exist)
        for dpage, hpage in plan.swap_out:
            swaps += 1
            for off in range(P):
                cell = store.cells.pop((int(dpage), off), None)
                if cell is not None:
                    host_cells[(int(hpage), off)] = cell
        for hpage, dpage in plan.swap_in:
            for off in range(P):
                store.cells.pop((int(dpage), off), None)
                cell = host_cells.pop((int(hpage), off), None)
                if cell is not None:
                    store.cells[(int(dpage), off)] = cell
        table = oracle.page_table_from_block_tables(plan.block_tables, plan.seqlens_k, P)
        rid, pos = loop.positions(plan)
        q = synth.token_values(rid, pos, H_Q, D, 0)
        k = synth.token_values(rid, pos, H_KV, D, 1)
        v = synth.token_values(rid, pos, H_KV, D, 2)
        oracle.append(store, oracle.new_token_slots(table, plan.cu_seqlens_q, plan.seqlens_k),
                      synth.bf16_bits(k), synth.bf16_bits(v))
        expected.append(oracle.mixed_attention(oracle.bf16_bits_to_f64(synth.bf16_bits(q)), store,
                                               table, plan.cu_seqlens_q, plan.seqlens_k, H_KV,
                                               scale))
        results.append(res)
        finished |= set(res.finished.tolist())
        if len(finished) == nreq:
            break
    assert len(finished) == nreq, f"unfinished: {set(range(nreq)) - finished}"
    assert preemptions > 0, "the pool was meant to force preemption"
    if swap:
        assert swaps > 0
    worst = 0.0
    for i, (res, (ref_o, ref_l)) in enumerate(zip(results, expected)):
        loop.wait(res)
        got = res.out.float().numpy()
        assert np.isfinite(got).all(), f"step {i}: non-finite output"
        err = float(np.abs(got - ref_o).max())
        rr = rel_rms(got, ref_o)
        lerr = float(np.abs(res.lse.numpy() - ref_l).max())
        worst = max(worst, err)
        assert err <= ATOL and rr <= RMS_TOL and lerr <= LSE_TOL, (i, err, rr, lerr)
    print(f"{len(results)} steps, {preemptions} preemptions, {swaps} pages swapped, "
          f"worst max|err| {worst:.3g}")
    loop.close()
