"""GPU: the non-paged varlen forward ([W] wangyu.me "大语言模型推理优化（二）：
Chunked Prefill", section "Flash Attention 的 varlen 接口": packed K/V with
cu_seqlens_k, right-aligned causal) against the oracle.  Segment starts in
the packed K/V are not multiples of 16, so 16-token blocks straddle segments.
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import synth
from gpu_harness import compare, per_segment_rel_rms
from harness import OracleStep

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


def packed_kv(w, t):
    """Per segment: its history rows, then this step's new rows."""
    cu = np.concatenate([[0], np.cumsum(w.q_lens)])
    hcu = np.concatenate([[0], np.cumsum(w.hist_lens)])
    ks, vs = [], []
    for s in range(w.num_seqs):
        ks += [t["k_hist"][hcu[s]:hcu[s + 1]], t["k_new"][cu[s]:cu[s + 1]]]
        vs += [t["v_hist"][hcu[s]:hcu[s + 1]], t["v_new"][cu[s]:cu[s + 1]]]
    cu_k = np.concatenate([[0], np.cumsum(w.k_lens)]).astype(np.int32)
    return torch.cat(ks), torch.cat(vs), cu, cu_k


def run_varlen(w, options=None):
    import mixed_chunked_prefill_gb300 as mcp

    t = w.tensors("cpu")
    k, v, cu, cu_k = packed_kv(w, t)
    q = t["q"].cuda()
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.total_q, w.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
    mcp.mixed_attn_varlen(q, k.cuda(), v.cuda(), cu, cu_k, w.sm_scale, out, lse, options)
    torch.cuda.synchronize()
    ref = OracleStep(w, t)
    ref.do_append()
    ref_o, ref_l = ref.attention()
    compare(w, out, lse, ref_o, ref_l, label=w.name)
    assert max(per_segment_rel_rms(w, out, ref_o)) <= 1e-2


@pytest.mark.parametrize("name", ["tiny", "worked", "balanced"])
def test_varlen_workloads(name):
    run_varlen(synth.make_workload(name))


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (16, 1, 128), (6, 2, 64), (4, 4, 64)])
def test_varlen_unaligned_segments_and_splits(hq, hkv, d):
    import mixed_chunked_prefill_gb300 as mcp

    q = [1, 40, 3, 130, 0, 1, 77]
    k = [17, 45, 300, 380, 9, 1, 77]
    w = synth.make_workload_from_lengths("varlen", hq, hkv, d, 16, 1 / math.sqrt(d), q, k, 8)
    run_varlen(w)
    run_varlen(w, mcp.PlanOptions(0, 16, 128))
