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
    SegmentKV,
    compare,
    gpu_step,
    per_segment_rel_rms,
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


def test_checked_build_flags_duplicate_slots_on_the_device():
    """The MCP_CHECKED library compares every pair of append slots on the
    device and reports a shared slot; distinct slots pass clean, and the
    default library skips the check."""
    import ctypes

    import mixed_chunked_prefill_gb300 as mcp
    from mixed_chunked_prefill_gb300 import _capi, build

    lib = _capi.open_library(build.build(checked=True))
    assert lib.mcp_build_flags() == _capi.BUILD_CHECKED
    P, H, D, pages, T = 16, 2, 64, 256, 3000  # three 1024-slot windows
    kc = torch.zeros((pages, P, H, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    g = torch.Generator(device="cuda").manual_seed(2)
    k = torch.randn((T, H, D), device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn((T, H, D), device="cuda", generator=g).to(torch.bfloat16)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def append(library, slots):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = library.mcp_paged_kv_append(
            ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
            ctypes.c_void_p(slots.data_ptr()), T, H, D, P, pages, ctypes.c_void_p(kc.data_ptr()),
            ctypes.c_void_p(vc.data_ptr()), ctypes.c_void_p(err.data_ptr()), stream)
        assert st == 0
        torch.cuda.synchronize()
        return int(err.item())

    perm = torch.randperm(pages * P, generator=torch.Generator().manual_seed(3))[:T]
    distinct = perm.to(torch.int64).cuda()
    assert append(lib, distinct) == 0
    assert torch.equal(kc.view(-1, H, D)[distinct], k)  # the checked build still appends
    for a, b in [(0, 1), (5, 2999), (1500, 2100)]:  # inside one window and across windows
        dup = distinct.clone()
        dup[b] = dup[a]
        bits = append(lib, dup)
        assert bits == mcp.DEVERR_SLOT_DUP, (a, b, bits)
        padded = dup.clone()
        padded[a] = padded[b] = -1  # padding tokens (slot < 0) never collide
        assert append(lib, padded) == 0
    assert append(mcp.load(), dup) == 0  # the default build does not look


@pytest.mark.parametrize("name,dsplit,psplit", [("tiny", 16, 128), ("worked", 16, 0),
                                                ("balanced", 0, 0)])
def test_outputs_and_workspace_stay_in_bounds(name, dsplit, psplit):
    """Canary bytes before and after the output, the LSE and the workspace
    come back bit-identical: the fused kernel and the combine write only the
    step's rows and the plan's workspace bytes."""
    import mixed_chunked_prefill_gb300 as mcp
    from mixed_chunked_prefill_gb300.step import MixedStep, write_history

    w = synth.make_workload(name)
    t = w.tensors("cpu")
    ref = OracleStep(w, t)
    ref.do_append()
    ref_out, ref_lse = ref.attention()
    td = {k: v.cuda() for k, v in t.items()}
    shape = (w.num_pages, w.page_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    write_history(w.block_tables(), w.hist_lens, td["k_hist"], td["v_hist"], kc, vc, w.page_size)
    cu = np.concatenate([[0], np.cumsum(w.q_lens)]).astype(np.int32)
    opts = mcp.PlanOptions(0, dsplit, psplit)
    step = MixedStep(w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size, w.num_pages,
                     w.sm_scale, cu, w.k_lens, w.block_tables(), options=opts)
    step.append(td["k_new"], td["v_new"], kc, vc)
    guard = 4096  # bytes on each side (a multiple of 256 keeps every buffer aligned)
    sizing = mcp.mixed_attn_plan(step.desc, cu, w.k_lens, opts)
    ws_big = torch.full((int(sizing.workspace_bytes) + 2 * guard,), 0xA5, dtype=torch.uint8,
                        device="cuda")
    ws = ws_big[guard:guard + int(sizing.workspace_bytes)]
    plan = mcp.mixed_attn_plan(step.desc, cu, w.k_lens, opts, ws)
    n_out = w.total_q * w.num_q_heads * w.head_dim
    ge = guard // 2
    out_big = torch.full((n_out + 2 * ge,), -7.0, dtype=torch.bfloat16, device="cuda")
    out_big[ge:ge + n_out] = float("nan")
    out = out_big[ge:ge + n_out].view(w.total_q, w.num_q_heads, w.head_dim)
    gl = guard // 4
    n_lse = w.total_q * w.num_q_heads
    lse_big = torch.full((n_lse + 2 * gl,), -3.0, dtype=torch.float32, device="cuda")
    lse = lse_big[gl:gl + n_lse].view(w.total_q, w.num_q_heads)
    before_ws = ws_big.clone()
    mcp.mixed_attn_fwd(plan, td["q"], kc, vc, step.bt_d, step.cu_d, step.sk_d, out, lse, ws)
    mcp.check_device_errors(mcp.workspace_error_word(plan, ws))
    torch.cuda.synchronize()
    assert torch.equal(ws_big[:guard], before_ws[:guard])
    assert torch.equal(ws_big[-guard:], before_ws[-guard:])
    assert bool((out_big[:ge] == -7.0).all()) and bool((out_big[-ge:] == -7.0).all())
    assert bool((lse_big[:gl] == -3.0).all()) and bool((lse_big[-gl:] == -3.0).all())
    compare(w, out, lse, ref_out, ref_lse, label=f"canary/{name}")


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
# full-size workloads: every row, in the launch configuration bench.py times
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["decode-heavy", "long-context"])
def test_full_size_every_row(name):
    """Every query row of every head of the two largest workloads ([W] "Flash
    Attention 的 varlen 接口": each segment sees only its own KV,
    right-aligned), with the default plan bench.py times.  Unused slots and
    spare pages hold NaN, so a read outside a segment's KV shows up.  The
    oracle reads each segment's keys in position order from the generated
    inputs (SegmentKV) instead of its dict page store; this step's new
    tokens are also checked bit-exact in their cache slots."""
    import oracle

    w = synth.make_workload(name)
    t = w.tensors("cuda")
    out, lse, kc, vc, step = gpu_step(w, t)
    # the append: each new token's K/V rows, bit-exact, at the oracle's slots
    bt = w.block_tables()
    cu, _, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
    table = oracle.page_table_from_block_tables(bt, w.k_lens, w.page_size)
    slots = torch.from_numpy(oracle.new_token_slots(table, cu, w.k_lens)).cuda()
    H, D = w.num_kv_heads, w.head_dim
    assert torch.equal(kc.view(-1, H, D)[slots].view(torch.int16), t["k_new"].view(torch.int16))
    assert torch.equal(vc.view(-1, H, D)[slots].view(torch.int16), t["v_new"].view(torch.int16))
    del kc, vc
    q = oracle.bf16_bits_to_f64(synth.bf16_bits(t["q"]))
    ref_out, ref_lse = oracle.mixed_attention(q, SegmentKV(w, t), None, cu, w.k_lens,
                                              w.num_kv_heads, w.sm_scale)
    err, rr, lerr = compare(w, out, lse, ref_out, ref_lse, label=name)
    seg = per_segment_rel_rms(w, out, ref_out)
    print(f"{name}: {w.total_q} rows x {w.num_q_heads} heads: max|err| {err:.3g} "
          f"relRMS {rr:.3g} (worst segment {max(seg):.3g}) lse {lerr:.3g} "
          f"items {step.plan.num_items}")
    assert max(seg) <= 1e-2, f"per-segment rel RMS {max(seg):.4g}"


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
