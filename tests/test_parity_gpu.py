"""GPU parity: the CUDA library against the CPU oracle on the same seeded inputs.

Append is bit-exact (every byte of both caches); attention outputs are bf16
with max |err| <= 2e-2 and relative RMS <= 1e-2 against the float64 oracle;
the LSE within 1e-2.  Caches start NaN-filled, so any read of an unused slot
or page shows up as a non-finite output.
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import synth
from gpu_harness import (
    OracleStep,
    compare,
    gpu_step,
    per_segment_rel_rms,
    sub_workload,
)

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


def opts(dsplit=0, psplit=0):
    import mixed_chunked_prefill_gb300 as mcp

    return mcp.PlanOptions(0, dsplit, psplit)


def full_parity(w, t=None, options=None, label=None, check_cache=True):
    t = t if t is not None else w.tensors("cpu")
    ref = OracleStep(w, t)
    ref.do_append()
    ref_out, ref_lse = ref.attention()
    out, lse, kc, vc, step = gpu_step(w, t, options=options)
    if check_cache:
        k_bits, v_bits = ref.cache_bits()
        assert np.array_equal(synth.bf16_bits(kc), k_bits), "k_cache not bit-exact"
        assert np.array_equal(synth.bf16_bits(vc), v_bits), "v_cache not bit-exact"
    res = compare(w, out, lse, ref_out, ref_lse, label=label or w.name)
    seg = per_segment_rel_rms(w, out, ref_out)
    assert max(seg) <= 1e-2, f"per-segment rel RMS {max(seg):.4g}"
    return res, step


# ---------------------------------------------------------------------------
# the workloads small enough for the oracle to run whole
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "worked", "balanced"])
def test_workload_parity(name):
    w = synth.make_workload(name)
    (err, rr, lerr), step = full_parity(w)
    print(f"{name}: max|err| {err:.3g} relRMS {rr:.3g} lse {lerr:.3g} items {step.plan.num_items}")


@pytest.mark.parametrize("name,dsplit,psplit", [("tiny", 16, 128), ("tiny", 48, 128),
                                                ("worked", 32, 256), ("worked", 1024, 2048),
                                                ("balanced", 512, 1024)])
def test_forced_splits_use_combine(name, dsplit, psplit):
    w = synth.make_workload(name)
    (err, rr, lerr), step = full_parity(w, options=opts(dsplit, psplit))
    assert step.plan.num_combine > 0


def test_shuffled_segment_order():
    w = synth.make_workload("balanced").shuffled(5)
    full_parity(w)


def test_peaky_scores_stress_rescale():
    w = synth.make_workload("worked")
    t = w.tensors("cpu")
    t["q"] = (t["q"].float() * 4).to(torch.bfloat16)
    full_parity(w, t, label="peaky")


def test_growing_scores_force_lazy_rescale():
    # later keys score higher, so the running max keeps growing across tiles
    w = synth.make_workload_from_lengths("ramp", 8, 2, 128, 16, 1 / math.sqrt(128),
                                         [1, 200, 1], [3000, 1700, 700], 99)
    t = w.tensors("cpu")
    ramp_h = torch.linspace(0, 3, w.total_hist).view(-1, 1, 1)
    t["k_hist"] = (t["k_hist"].float() + ramp_h * t["q"].float().mean(0, keepdim=True)[:, :2].mean(1, keepdim=True)).to(torch.bfloat16)
    t["q"] = (t["q"].float() * 3).to(torch.bfloat16)
    full_parity(w, t, label="ramp")
    full_parity(w, t, options=opts(64, 256), label="ramp-split")


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

EDGE = {
    # decode contexts at and around page boundaries, Lk = 1
    "decode-edges": ([1] * 8, [1, 2, 15, 16, 17, 31, 32, 33]),
    # chunks without history (Lq == Lk), including partial tiles
    "no-history": ([1, 33, 128, 129, 300], [1, 33, 128, 129, 300]),
    # chunks starting mid-page and mid-tile
    "mid-page": ([40, 77, 130], [45, 77 + 133, 130 + 250]),
    # empty segments between others
    "empty-segments": ([0, 1, 0, 50, 0], [10, 20, 5, 90, 1]),
    # multi-token segments that stay on the decode path (Lq * G <= 16 with G = 4)
    "spec-decode": ([2, 3, 4, 5], [40, 41, 300, 301]),
}


@pytest.mark.parametrize("case", sorted(EDGE))
@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (4, 4, 64), (16, 1, 128), (6, 2, 64),
                                      (32, 8, 96), (12, 3, 96), (16, 4, 256), (8, 8, 256)])
def test_edge_cases(case, hq, hkv, d):
    q, k = EDGE[case]
    w = synth.make_workload_from_lengths(case, hq, hkv, d, 16, 1 / math.sqrt(d), q, k, 1234)
    full_parity(w, label=f"{case}/{hq}/{hkv}/{d}")
    full_parity(w, options=opts(16, 128), label=f"{case}/{hq}/{hkv}/{d}/split")


def test_many_decodes_single_chunk_gqa8():
    rng = np.random.Generator(np.random.PCG64(8))
    dec = [int(x) for x in rng.integers(1, 3000, size=40)]
    w = synth.make_workload_from_lengths("dec-gqa8", 64, 8, 128, 16, 1 / math.sqrt(128),
                                         [1] * 40 + [64], dec + [64 + 1000], 77)
    full_parity(w)


def test_append_skips_negative_slots_and_flags_out_of_range():
    import mixed_chunked_prefill_gb300 as mcp

    P, H, D, pages = 16, 2, 64, 8
    kc = torch.zeros((pages, P, H, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.randn((4, H, D), device="cuda").to(torch.bfloat16)
    v = torch.randn((4, H, D), device="cuda").to(torch.bfloat16)
    slots = torch.tensor([3, -1, pages * P + 5, 17], dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mcp.paged_kv_append(k, v, slots, kc, vc, err)
    torch.cuda.synchronize()
    flat_k = kc.view(-1, H, D)
    assert torch.equal(flat_k[3], k[0]) and torch.equal(flat_k[17], k[3])
    assert int((flat_k != 0).any(dim=(1, 2)).sum()) == 2  # nothing else written
    with pytest.raises(mcp.MCPError) as ei:
        mcp.check_device_errors(err.data_ptr())
    assert ei.value.status == 6


def test_merge_states_matches_oracle():
    import mixed_chunked_prefill_gb300 as mcp
    import oracle

    g = torch.Generator().manual_seed(5)
    n, R, H, D = 3, 7, 4, 128
    o = torch.randn((n, R, H, D), generator=g)
    lse = torch.randn((n, R, H), generator=g) * 3
    lse[1, 2, 1] = -math.inf
    out = torch.empty((R, H, D), dtype=torch.bfloat16, device="cuda")
    lo = torch.empty((R, H), dtype=torch.float32, device="cuda")
    mcp.merge_states(o.cuda(), lse.cuda(), out, lo)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.merge_states(o.double().numpy(), lse.double().numpy())
    assert np.abs(out.float().cpu().numpy() - ref_o).max() <= 2e-2
    assert np.abs(lo.cpu().numpy() - ref_l).max() <= 1e-4


# ---------------------------------------------------------------------------
# full-size workloads: sampled rows, in the launch configuration bench.py times
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["decode-heavy", "long-context"])
def test_full_size_sampled_rows(name):
    w = synth.make_workload(name)
    t = w.tensors("cuda")
    out, lse, kc, vc, step = gpu_step(w, t, fill=0.0)
    del kc, vc
    # sample: the shortest and longest decode, plus the chunk
    dec = [s for s in range(w.num_seqs) if w.q_lens[s] == 1]
    chunk = [s for s in range(w.num_seqs) if w.q_lens[s] > 1]
    segs = [min(dec, key=lambda s: w.k_lens[s]), max(dec, key=lambda s: w.k_lens[s])] + chunk
    sub, ts = sub_workload(w, t, segs)
    del t
    ref = OracleStep(sub, ts)
    ref.do_append()
    cu_sub = np.concatenate([[0], np.cumsum(sub.q_lens)])
    lq_chunk = sub.q_lens[-1]
    local = [0, 1] + [int(cu_sub[-2] + i) for i in (0, 1, lq_chunk // 2, lq_chunk - 2, lq_chunk - 1)]
    ref_out, ref_lse = ref.attention(tokens=local)
    cu_full = np.concatenate([[0], np.cumsum(w.q_lens)])
    full_rows = []
    for r in local:
        si = int(np.searchsorted(cu_sub, r, side="right") - 1)
        full_rows.append(int(cu_full[segs[si]] + (r - cu_sub[si])))
    got = out[full_rows].float().cpu().numpy()
    gl = lse[full_rows].cpu().numpy()
    want = ref_out[local]
    assert np.isfinite(got).all()
    err = float(np.abs(got - want).max())
    from harness import rel_rms

    rr = rel_rms(got, want)
    lerr = float(np.abs(gl - ref_lse[local]).max())
    print(f"{name}: sampled rows {full_rows}: max|err| {err:.3g} relRMS {rr:.3g} lse {lerr:.3g}")
    assert err <= 2e-2 and rr <= 1e-2 and lerr <= 1e-2
    assert torch.isfinite(out).all()


# ---------------------------------------------------------------------------
# cache pages of 8, 32 and 64 tokens (the kernels step over 16-token blocks,
# loaded as one 16-token box, or as two 8-token boxes from 8-token pages)
# ---------------------------------------------------------------------------

BIG_PAGE_CASES = {
    "decode-edges": ([1] * 13, [1, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65]),
    "mid-page": ([40, 77, 130], [45, 77 + 133, 130 + 250]),
    "mixed": ([1, 1, 300, 2], [121, 46, 2000, 700]),
}


@pytest.mark.parametrize("page_size", [1, 8, 32, 64])
@pytest.mark.parametrize("case", sorted(BIG_PAGE_CASES))
def test_other_page_sizes(case, page_size):
    q, k = BIG_PAGE_CASES[case]
    w = synth.make_workload_from_lengths(f"{case}-p{page_size}", 32, 8, 128, page_size,
                                         1 / math.sqrt(128), q, k, 4321)
    full_parity(w, label=f"{case}/p{page_size}")
    full_parity(w, options=opts(16, 128), label=f"{case}/p{page_size}/split")


@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 64), (6, 2, 64), (16, 1, 128), (32, 8, 96),
                                      (16, 4, 256)])
def test_page8_head_shapes(hq, hkv, d):
    """8-token pages with D = 64 (one 64-column panel), D = 96 (one box per
    panel) and other head groups."""
    q, k = BIG_PAGE_CASES["mixed"]
    w = synth.make_workload_from_lengths(f"p8-{hq}-{hkv}-{d}", hq, hkv, d, 8, 1 / math.sqrt(d),
                                         q, k, 99)
    full_parity(w, label=f"p8/{hq}/{hkv}/{d}")
    full_parity(w, options=opts(16, 128), label=f"p8/{hq}/{hkv}/{d}/split")


@pytest.mark.parametrize("page_size", [16, 64])
def test_head_dim_256_mixed_step(page_size):
    """head_dim 256: 64-key tiles and every segment (decodes included) on the
    tensor-core path; several tiles per item, a ragged tail and splits."""
    q = [1, 1, 3, 300, 1]
    k = [121, 4000, 700, 300 + 2500, 65]
    w = synth.make_workload_from_lengths(f"d256-p{page_size}", 16, 4, 256, page_size,
                                         1 / math.sqrt(256), q, k, 256)
    full_parity(w, label=f"d256/p{page_size}")
    full_parity(w, options=opts(16, 128), label=f"d256/p{page_size}/split")


@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 64), (32, 8, 96), (16, 4, 256), (16, 1, 128)])
def test_page1_head_shapes(hq, hkv, d):
    """1-token pages: K/V rows gathered with cp.async, every segment on
    tensor-core tiles; other head dims and head groups."""
    q, k = BIG_PAGE_CASES["mixed"]
    w = synth.make_workload_from_lengths(f"p1-{hq}-{hkv}-{d}", hq, hkv, d, 1, 1 / math.sqrt(d),
                                         q, k, 11)
    full_parity(w, label=f"p1/{hq}/{hkv}/{d}")
    full_parity(w, options=opts(16, 128), label=f"p1/{hq}/{hkv}/{d}/split")
