"""Failure detection on the GPU without a fault: the fused kernel's bounded
waits.

Every mbarrier wait in the fused kernel gives up after a time bound; the CTA
then records MCP_DEVERR_TIMEOUT, every role leaves its loop, the copies and
MMAs it did issue are drained, TMEM is freed and no output row is written.
A plan built with ``test_stall = 1`` makes that happen on purpose and safely:
its tensor-core items never issue their Q-tile load (so nothing is in flight
for the wait that runs out) and every wait is bounded at about 1 ms.  The
host then reads MCP_ERR_TIMEOUT from the error word, the context stays usable,
and the next ordinary step on the same workspace matches the oracle.
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import synth
from gpu_harness import OracleStep, compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from mixed_chunked_prefill_gb300 import build

    build.build()
    import mixed_chunked_prefill_gb300 as mcp

    return mcp.load()


def _setup(w, t):
    from mixed_chunked_prefill_gb300.step import write_history

    td = {k: v.cuda() for k, v in t.items()}
    shape = (w.num_pages, w.page_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    write_history(w.block_tables(), w.hist_lens, td["k_hist"], td["v_hist"], kc, vc, w.page_size)
    return td, kc, vc


@pytest.mark.parametrize("lens", [([300], [1000]), ([1, 1, 200], [121, 46, 900])],
                         ids=["chunk-only", "decodes+chunk"])
def test_bounded_wait_runs_out_reports_timeout_and_recovers(lens):
    import mixed_chunked_prefill_gb300 as mcp
    from mixed_chunked_prefill_gb300.step import MixedStep

    q_lens, k_lens = lens
    w = synth.make_workload_from_lengths("stall", 8, 2, 128, 16, 1 / math.sqrt(128), q_lens,
                                         k_lens, 31)
    t = w.tensors("cpu")
    ref = OracleStep(w, t)
    ref.do_append()
    ref_out, ref_lse = ref.attention()
    td, kc, vc = _setup(w, t)
    cu = np.concatenate([[0], np.cumsum(w.q_lens)]).astype(np.int32)
    # whole KV ranges (no split, so no combine over partials that were never written)
    stall = mcp.PlanOptions(0, 1 << 20, 1 << 20)
    stall.test_stall = 1
    step = MixedStep(w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size, w.num_pages,
                     w.sm_scale, cu, w.k_lens, w.block_tables(), options=stall)
    assert step.plan.test_stall == 1 and step.plan.num_combine == 0
    assert step.plan.num_prefill_items > 0
    out = torch.full_like(td["q"], float("nan"))
    lse = torch.full((w.total_q, w.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
    step.run(td["q"], td["k_new"], td["v_new"], kc, vc, out, lse)
    with pytest.raises(mcp.MCPError) as ei:
        step.check()
    assert ei.value.status == 5  # MCP_ERR_TIMEOUT
    torch.cuda.synchronize()  # the context still answers
    # no row of an aborted (tensor-core) item was written; decode items ran normally
    chunk_rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in range(w.num_seqs)
                                 if w.q_lens[s] > 1])
    dec_rows = np.array([cu[s] for s in range(w.num_seqs) if w.q_lens[s] == 1], dtype=np.int64)
    o = out.float().cpu().numpy()
    assert np.isnan(o[chunk_rows]).all()
    assert np.isnan(lse.cpu().numpy()[chunk_rows]).all()
    if dec_rows.size:
        compare(w, out, lse, ref_out, ref_lse, rows=dec_rows, label="decodes beside the stall")
    # the next ordinary step on the same workspace (append already done)
    step.plan = mcp.mixed_attn_plan(step.desc, cu, w.k_lens, mcp.PlanOptions(0, 0, 0),
                                    step.workspace)
    step.error_word = mcp.workspace_error_word(step.plan, step.workspace)
    assert step.plan.test_stall == 0
    out2 = torch.full_like(td["q"], float("nan"))
    lse2 = torch.full_like(lse, float("nan"))
    step.attention(td["q"], kc, vc, out2, lse2)
    step.check()
    compare(w, out2, lse2, ref_out, ref_lse, label="after the stall")
