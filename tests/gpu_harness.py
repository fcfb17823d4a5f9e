"""GPU-side test glue: runs the CUDA library on a synthetic workload and the
oracle on the same inputs.  Test infrastructure only."""

from __future__ import annotations

import numpy as np

import oracle
import synth
from harness import OracleStep, rel_rms

ATOL = 2e-2       # max |err| on bf16 outputs
RMS_TOL = 1e-2    # relative RMS on bf16 outputs
LSE_TOL = 1e-2    # max |err| on the natural-log LSE


def gpu_step(w, t, options=None, fill=float("nan"), device="cuda", want_lse=True):
    """Run append + fused attention for workload ``w`` with tensors ``t`` (on
    any device); returns (out, lse, k_cache, v_cache, step) on the device."""
    import torch

    from mixed_chunked_prefill_gb300.step import MixedStep, write_history

    td = {k: v.to(device) for k, v in t.items()}
    shape = (w.num_pages, w.page_size, w.num_kv_heads, w.head_dim)
    k_cache = torch.full(shape, fill, dtype=torch.bfloat16, device=device)
    v_cache = torch.full(shape, fill, dtype=torch.bfloat16, device=device)
    bt = w.block_tables()
    write_history(bt, w.hist_lens, td["k_hist"], td["v_hist"], k_cache, v_cache, w.page_size)
    cu = np.concatenate([[0], np.cumsum(w.q_lens)]).astype(np.int32)
    step = MixedStep(w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size, w.num_pages,
                     w.sm_scale, cu, w.k_lens, bt, device=device, options=options)
    out = torch.full_like(td["q"], float("nan"))
    lse = (torch.full((w.total_q, w.num_q_heads), float("nan"), dtype=torch.float32, device=device)
           if want_lse else None)
    step.run(td["q"], td["k_new"], td["v_new"], k_cache, v_cache, out, lse)
    step.check()
    torch.cuda.synchronize()
    return out, lse, k_cache, v_cache, step


def compare(w, out, lse, ref_out, ref_lse, rows=None, label=""):
    """Element-wise check of GPU outputs against the oracle."""
    got = out.float().cpu().numpy()
    if rows is not None:
        got, ref_out = got[rows], ref_out[rows]
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    err = float(np.abs(got - ref_out).max()) if got.size else 0.0
    rr = rel_rms(got, ref_out) if got.size else 0.0
    assert err <= ATOL, f"{label}: max|err| {err:.4g} > {ATOL}"
    assert rr <= RMS_TOL, f"{label}: rel RMS {rr:.4g} > {RMS_TOL}"
    lerr = 0.0
    if lse is not None:
        gl = lse.cpu().numpy()
        rl = ref_lse
        if rows is not None:
            gl, rl = gl[rows], rl[rows]
        lerr = float(np.abs(gl - rl).max()) if gl.size else 0.0
        assert lerr <= LSE_TOL, f"{label}: lse max|err| {lerr:.4g}"
    return err, rr, lerr


def per_segment_rel_rms(w, out, ref_out):
    got = out.float().cpu().numpy()
    cu = np.concatenate([[0], np.cumsum(w.q_lens)])
    res = []
    for s in range(w.num_seqs):
        if w.q_lens[s]:
            res.append(rel_rms(got[cu[s]:cu[s + 1]], ref_out[cu[s]:cu[s + 1]]))
    return res


class SegmentKV:
    """The keys and values of each segment in position order, taken straight
    from the generated inputs: history positions 0 .. H_s - 1 (``k_hist``
    slice of segment s) followed by this step's tokens (its ``k_new`` rows,
    the last Lq_s positions; [W] "输入组装").

    It stands in for the oracle's dict page store (same ``gather`` call) on
    the full-size workloads, whose tens of GB of history are too large to
    hold as per-slot dict entries; the GPU's page translation is then checked
    against no page table at all.  Each segment is copied to the host and
    widened to float64 only while the oracle works on it."""

    def __init__(self, w, t):
        self.t = t
        self.cu = np.concatenate([[0], np.cumsum(w.q_lens)]).astype(np.int64)
        self.hcu = np.concatenate([[0], np.cumsum(w.hist_lens)]).astype(np.int64)

    def gather(self, table, s, length):
        import torch

        h0, h1 = int(self.hcu[s]), int(self.hcu[s + 1])
        q0, q1 = int(self.cu[s]), int(self.cu[s + 1])
        assert (h1 - h0) + (q1 - q0) == length
        out = []
        for hist, new in (("k_hist", "k_new"), ("v_hist", "v_new")):
            rows = torch.cat([self.t[hist][h0:h1], self.t[new][q0:q1]]).cpu()
            out.append(oracle.bf16_bits_to_f64(synth.bf16_bits(rows)))
        return out[0], out[1]


__all__ = ["SegmentKV", "gpu_step", "compare", "per_segment_rel_rms", "OracleStep", "oracle",
           "ATOL", "RMS_TOL", "LSE_TOL"]
