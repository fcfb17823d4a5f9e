"""GPU: attention for listed rows only (logits_indices in the last layer) and
the row gather, against the oracle.

[W] wangyu.me "大语言模型推理优化（二）：Chunked Prefill", section
"采样：只有该出字的请求才出字".  Listed rows must equal the oracle's rows of the
full step; rows not listed must stay untouched (the output is NaN-filled).
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import synth
from gpu_harness import ATOL, LSE_TOL, RMS_TOL
from harness import OracleStep, rel_rms

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


def rows_step(w, rows, options=None):
    import mixed_chunked_prefill_gb300 as mcp
    from mixed_chunked_prefill_gb300.step import MixedStep, write_history

    t = w.tensors("cpu")
    td = {k: v.cuda() for k, v in t.items()}
    shape = (w.num_pages, w.page_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    bt = w.block_tables()
    write_history(bt, w.hist_lens, td["k_hist"], td["v_hist"], kc, vc, w.page_size)
    cu = np.concatenate([[0], np.cumsum(w.q_lens)]).astype(np.int32)
    step = MixedStep(w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size, w.num_pages,
                     w.sm_scale, cu, w.k_lens, bt, options=options, rows=rows)
    out = torch.full_like(td["q"], float("nan"))
    lse = torch.full((w.total_q, w.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
    step.run(td["q"], td["k_new"], td["v_new"], kc, vc, out, lse)
    step.check()
    torch.cuda.synchronize()
    ref = OracleStep(w, t)
    ref.do_append()
    ref_o, ref_l = ref.attention(tokens=[int(r) for r in rows])
    return out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, step


def check(rows, got, gl, ref_o, ref_l, label):
    rows = np.asarray(rows)
    g = got[rows]
    assert np.isfinite(g).all(), f"{label}: non-finite listed row"
    assert float(np.abs(g - ref_o[rows]).max()) <= ATOL, label
    assert rel_rms(g, ref_o[rows]) <= RMS_TOL, label
    assert float(np.abs(gl[rows] - ref_l[rows]).max()) <= LSE_TOL, label
    others = np.setdiff1d(np.arange(got.shape[0]), rows)
    assert np.isnan(got[others]).all(), f"{label}: an unlisted row was written"
    assert np.isnan(gl[others]).all(), f"{label}: an unlisted lse was written"


@pytest.mark.parametrize("name", ["tiny", "worked", "balanced"])
def test_logits_rows_match_oracle(name):
    import mixed_chunked_prefill_gb300 as mcp

    w = synth.make_workload(name)
    cu = np.concatenate([[0], np.cumsum(w.q_lens)]).astype(np.int32)
    rows = mcp.build_logits_indices(cu)
    got, gl, ref_o, ref_l, step = rows_step(w, rows)
    check(rows, got, gl, ref_o, ref_l, name)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 1), (4, 4)])
def test_random_row_subsets_with_splits(hq, hkv):
    import mixed_chunked_prefill_gb300 as mcp

    rng = np.random.Generator(np.random.PCG64(hq * 100 + hkv))
    q, k = [1, 40, 3, 130, 1], [700, 300, 43, 900, 17]
    w = synth.make_workload_from_lengths("rows", hq, hkv, 128, 16, 1 / math.sqrt(128), q, k, 5)
    T = sum(q)
    rows = np.sort(rng.choice(T, size=60, replace=False)).astype(np.int32)
    rows = np.union1d(rows, np.arange(44, 50)).astype(np.int32)  # a run of consecutive tokens
    for opts in (None, mcp.PlanOptions(0, 16, 128)):
        got, gl, ref_o, ref_l, step = rows_step(w, rows, opts)
        if opts is not None:
            assert step.plan.num_combine > 0
        check(rows, got, gl, ref_o, ref_l, f"{hq}/{hkv}/{'split' if opts else 'whole'}")


def test_gather_rows_bit_exact_and_range_check():
    import mixed_chunked_prefill_gb300 as mcp

    g = torch.Generator().manual_seed(3)
    src = torch.randn((300, 32, 128), generator=g).to(torch.bfloat16).cuda()
    rows = torch.tensor([5, 0, 299, 17, 17, 150], dtype=torch.int32, device="cuda")
    dst = torch.full((6, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    mcp.gather_rows(src, rows, dst)
    torch.cuda.synchronize()
    assert torch.equal(dst.view(torch.int16), src[rows.long()].view(torch.int16))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([1, 300, -1, 2], dtype=torch.int32, device="cuda")
    dst2 = torch.full((4, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    mcp.gather_rows(src, bad, dst2, err)
    torch.cuda.synchronize()
    assert torch.equal(dst2[0], src[1]) and torch.equal(dst2[3], src[2])
    assert (dst2[1:3].float() == 0).all()
    with pytest.raises(mcp.MCPError) as ei:
        mcp.check_device_errors(err.data_ptr())
    assert ei.value.status == 6
