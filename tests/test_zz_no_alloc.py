"""The workspace-free forward (mcp_mixed_attn_fwd_noalloc) against the
workspace entry point.

Some callers cannot allocate device memory when they run a step (their
framework's memory pool owns every device allocation, or the server must not
grow its footprint after start-up); for them the library keeps the step's
scratch in a fixed 16 MiB device array.  This file is named so that pytest
collects it last; it is self-contained, so it passes alone in a fresh process
and after the other tests.
"""

from __future__ import annotations

import ctypes
import math

import numpy as np
import pytest

import synth
from gpu_harness import ATOL, RMS_TOL, LSE_TOL, gpu_step
from harness import rel_rms

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


def _call_noalloc(lib, step, q, kc, vc, out, lse, options):
    """One call through the C ABI (ctypes), on the current stream."""
    import mixed_chunked_prefill_gb300 as mcp

    ew = ctypes.c_void_p()
    st = lib.mcp_mixed_attn_fwd_noalloc(
        ctypes.byref(step.desc), step.cu_h.ctypes.data_as(ctypes.c_void_p),
        step.sk_h.ctypes.data_as(ctypes.c_void_p),
        ctypes.byref(options) if options is not None else None,
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()),
        ctypes.c_void_p(vc.data_ptr()), ctypes.c_void_p(step.bt_d.data_ptr()),
        ctypes.c_void_p(step.cu_d.data_ptr()), ctypes.c_void_p(step.sk_d.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), ctypes.byref(ew),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.mcp_last_error()
    mcp.check_device_errors(ew.value)
    return ew.value


@pytest.mark.parametrize("name,dsplit,psplit", [("tiny", 0, 0), ("tiny", 16, 128),
                                                ("worked", 0, 0), ("worked", 16, 0)])
def test_noalloc_matches_workspace_entry_point(library, name, dsplit, psplit):
    import mixed_chunked_prefill_gb300 as mcp

    w = synth.make_workload(name)
    t = w.tensors("cpu")
    options = mcp.PlanOptions(0, dsplit, psplit)
    # the existing entry point (caller-provided workspace)
    ref_out, ref_lse, kc, vc, step = gpu_step(w, t, options=options)
    q = t["q"].cuda()
    addrs = set()
    for call in range(2):  # two calls in a row share (and reuse) the scratch
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.total_q, w.num_q_heads), float("nan"), dtype=torch.float32,
                         device="cuda")
        addrs.add(_call_noalloc(library, step, q, kc, vc, out, lse, options))
        torch.cuda.synchronize()
        a = out.float().cpu().numpy()
        b = ref_out.float().cpu().numpy()
        assert np.isfinite(a).all()
        assert float(np.abs(a - b).max()) <= ATOL, (name, call)
        assert rel_rms(a, b) <= RMS_TOL, (name, call)
        assert float((lse - ref_lse).abs().max()) <= LSE_TOL, (name, call)
    assert len(addrs) == 1  # the same fixed scratch every call


def test_noalloc_rejects_steps_beyond_the_fixed_scratch(library):
    import mixed_chunked_prefill_gb300 as mcp

    # the long-context step's plan needs ~142 MiB of split partials
    w = synth.make_workload("long-context")
    cu = np.concatenate([[0], np.cumsum(w.q_lens)]).astype(np.int32)
    sk = np.asarray(w.k_lens, dtype=np.int32)
    desc = mcp.make_desc(w.num_seqs, w.total_q, w.num_q_heads, w.num_kv_heads, w.head_dim,
                         w.page_size, w.max_pages_per_seq, w.num_pages, 1 / math.sqrt(128))
    st = library.mcp_mixed_attn_fwd_noalloc(
        ctypes.byref(desc), cu.ctypes.data_as(ctypes.c_void_p), sk.ctypes.data_as(ctypes.c_void_p),
        None, *([None] * 8), None, None)
    assert st == 3  # MCP_ERR_WORKSPACE_TOO_SMALL, before anything is launched
    assert b"fixed scratch" in library.mcp_last_error()
