"""The workspace-free forward (mcp_mixed_attn_fwd_noalloc) against the oracle
and against the workspace entry point.

Some callers cannot allocate device memory when they run a step (their
framework's memory pool owns every device allocation, or the server must not
grow its footprint after start-up); for them the library keeps the step's
scratch in a fixed 16 MiB device array.  Every call goes through the C ABI
(ctypes).  This file is named so that pytest collects it last; it is
self-contained, so it passes alone in a fresh process and after the other
tests.
"""

from __future__ import annotations

import ctypes
import math

import numpy as np
import pytest

import synth
from gpu_harness import ATOL, LSE_TOL, RMS_TOL, OracleStep, compare, gpu_step
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


def _call_noalloc(lib, step, q, kc, vc, out, lse, options, bt=None):
    """One call through the C ABI on the current stream; returns (status,
    error-word address)."""
    ew = ctypes.c_void_p()
    st = lib.mcp_mixed_attn_fwd_noalloc(
        ctypes.byref(step.desc), step.cu_h.ctypes.data_as(ctypes.c_void_p),
        step.sk_h.ctypes.data_as(ctypes.c_void_p),
        ctypes.byref(options) if options is not None else None,
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()),
        ctypes.c_void_p(vc.data_ptr()),
        ctypes.c_void_p((bt if bt is not None else step.bt_d).data_ptr()),
        ctypes.c_void_p(step.cu_d.data_ptr()), ctypes.c_void_p(step.sk_d.data_ptr()),
        ctypes.c_void_p(out.data_ptr() if out is not None else 0),
        ctypes.c_void_p(lse.data_ptr()), ctypes.byref(ew),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, ew.value


class _DeviceBytes:
    """A raw device address seen as a uint8 array (for reading the scratch)."""

    def __init__(self, ptr, nbytes):
        self.__cuda_array_interface__ = {"shape": (int(nbytes),), "typestr": "|u1",
                                         "data": (int(ptr), False), "version": 3}


def _read_device(ptr, nbytes):
    return torch.as_tensor(_DeviceBytes(ptr, nbytes), device="cuda").clone().cpu().numpy()


class Case:
    """One workload: the oracle's result, the workspace entry point's result
    and the device inputs the no-alloc call reuses."""

    def __init__(self, name, dsplit=0, psplit=0):
        import mixed_chunked_prefill_gb300 as mcp

        self.w = synth.make_workload(name)
        t = self.w.tensors("cpu")
        self.options = mcp.PlanOptions(0, dsplit, psplit)
        ref = OracleStep(self.w, t)
        ref.do_append()
        self.ref_out, self.ref_lse = ref.attention()
        # the existing entry point (caller-provided workspace)
        self.ws_out, self.ws_lse, self.kc, self.vc, self.step = gpu_step(self.w, t,
                                                                          options=self.options)
        self.q = t["q"].cuda()

    def run(self, lib, bt=None):
        import mixed_chunked_prefill_gb300 as mcp

        out = torch.full_like(self.q, float("nan"))
        lse = torch.full((self.w.total_q, self.w.num_q_heads), float("nan"), dtype=torch.float32,
                         device="cuda")
        st, ew = _call_noalloc(lib, self.step, self.q, self.kc, self.vc, out, lse, self.options,
                               bt)
        assert st == 0, lib.mcp_last_error()
        return out, lse, ew

    def check(self, out, lse, label):
        torch.cuda.synchronize()
        # against the oracle, with the tolerances of every parity test
        compare(self.w, out, lse, self.ref_out, self.ref_lse, label=label)
        # and against the workspace entry point on the same inputs
        a = out.float().cpu().numpy()
        b = self.ws_out.float().cpu().numpy()
        assert float(np.abs(a - b).max()) <= ATOL, label
        assert rel_rms(a, b) <= RMS_TOL, label
        assert float((lse - self.ws_lse).abs().max()) <= LSE_TOL, label


@pytest.mark.parametrize("name,dsplit,psplit", [("tiny", 0, 0), ("tiny", 16, 128),
                                                ("worked", 0, 0), ("worked", 16, 0)])
def test_noalloc_matches_oracle_and_workspace_entry_point(library, name, dsplit, psplit):
    import mixed_chunked_prefill_gb300 as mcp

    c = Case(name, dsplit, psplit)
    addrs = set()
    for call in range(2):  # two calls in a row share (and reuse) the scratch
        out, lse, ew = c.run(library)
        mcp.check_device_errors(ew)
        addrs.add(ew)
        c.check(out, lse, f"{name}/{dsplit}/{psplit}/call{call}")
    assert len(addrs) == 1  # the same fixed scratch (and plan) every call


def test_noalloc_alternating_plans_reuse_the_scratch(library):
    """Steps with different plans (other offsets for the partials and the error
    word) in turn on one stream: each reads only what its own call wrote,
    whatever an earlier, larger call left in the array."""
    import mixed_chunked_prefill_gb300 as mcp

    big = Case("worked", 16, 0)      # many split partials
    small = Case("tiny", 16, 128)    # a different, smaller layout
    words = {}
    for i, c in enumerate([big, small, big, small]):
        out, lse, ew = c.run(library)
        mcp.check_device_errors(ew)
        words.setdefault(c.w.name, set()).add(ew)
        c.check(out, lse, f"{c.w.name}/call{i}")
    assert words[big.w.name] != words[small.w.name]  # the error word moved with the plan


def test_noalloc_reports_out_of_range_pages_through_its_error_word(library):
    """A block-table entry outside the page pool is skipped (zero fill) and
    reported through the returned error word, not as a fault."""
    import mixed_chunked_prefill_gb300 as mcp

    c = Case("tiny")
    bad = c.step.bt_d.clone()
    bad[0, 0] = c.w.num_pages + 5  # first page of the first decode
    out, lse, ew = c.run(library, bt=bad)
    with pytest.raises(mcp.MCPError) as ei:
        mcp.check_device_errors(ew)
    assert ei.value.status == 6  # MCP_ERR_DEVICE_CHECK
    # the error word was cleared by the check; a good call right after is clean
    out, lse, ew = c.run(library)
    mcp.check_device_errors(ew)
    c.check(out, lse, "after-range-error")


def test_noalloc_argument_errors_leave_the_scratch_untouched(library):
    """A NULL output is an argument error: returned before anything is
    enqueued, so the scratch still holds the previous call's work lists."""
    import mixed_chunked_prefill_gb300 as mcp

    first = Case("worked")
    out, lse, ew = first.run(library)
    mcp.check_device_errors(ew)
    plan = first.step.plan
    base = ew - int(plan.off_error)
    before = _read_device(base, int(plan.off_part_o))
    other = Case("tiny", 16, 128)  # would upload a different work list
    torch.cuda.synchronize()
    lse = torch.empty((other.w.total_q, other.w.num_q_heads), dtype=torch.float32, device="cuda")
    st, ew2 = _call_noalloc(library, other.step, other.q, other.kc, other.vc, None, lse,
                            other.options)
    assert st == 1  # MCP_ERR_INVALID_ARG
    assert ew2 is None  # no error word handed out
    torch.cuda.synchronize()
    after = _read_device(base, int(plan.off_part_o))
    assert np.array_equal(before, after)


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
