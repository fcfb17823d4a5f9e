"""GPU: KV page copies between pools (swap-out / swap-in of a preempted
sequence, [X] m.xxqk.cn "动态批处理中的抢占与优先级调度", section "Prefill 算力
霸占与抢占策略演进").

A sequence's pages go out to a page-locked host pool (bit-exact), its device
pages are poisoned, and it comes back into different free pages with a
remapped block table: attention must equal the oracle's (the method is
invariant to which physical pages hold a sequence's KV, [L] 4.1).
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import synth
from gpu_harness import compare
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


def test_swap_out_and_back_into_other_pages():
    import mixed_chunked_prefill_gb300 as mcp
    from mixed_chunked_prefill_gb300.step import MixedStep, write_history

    # decodes plus a chunk; the pool has room for one more copy of the longest sequence
    q, k = [1, 1, 200, 1], [900, 77, 1300, 2048]
    w = synth.make_workload_from_lengths("swap", 16, 4, 128, 16, 1 / math.sqrt(128), q, k, 21)
    victim = 3
    n_v = w.pages_of(victim)
    extra = n_v + 2
    t = w.tensors("cpu")
    td = {n: v.cuda() for n, v in t.items()}
    bt = w.block_tables()
    pages = w.num_pages + extra
    shape = (pages, w.page_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    write_history(bt, w.hist_lens, td["k_hist"], td["v_hist"], kc, vc, w.page_size)
    cu = np.concatenate([[0], np.cumsum(w.q_lens)]).astype(np.int32)
    step = MixedStep(w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size, pages, w.sm_scale,
                     cu, w.k_lens, bt)
    step.append(td["k_new"], td["v_new"], kc, vc)
    torch.cuda.synchronize()
    before_k, before_v = kc.clone(), vc.clone()

    # swap the victim out: its pages -> host pool slots 0 .. n_v-1
    host_k = torch.zeros((n_v + 1,) + shape[1:], dtype=torch.bfloat16).pin_memory()
    host_v = torch.zeros_like(host_k).pin_memory()
    src = torch.from_numpy(bt[victim, :n_v].copy()).cuda()
    slots = torch.arange(n_v, dtype=torch.int32, device="cuda")
    mcp.kv_copy_pages(kc, vc, host_k, host_v, src, slots)
    torch.cuda.synchronize()
    assert torch.equal(host_k[:n_v].view(torch.int16), before_k[src.long()].cpu().view(torch.int16))
    assert torch.equal(host_v[:n_v].view(torch.int16), before_v[src.long()].cpu().view(torch.int16))
    # its device pages are reused by someone else meanwhile
    kc[src.long()] = float("nan")
    vc[src.long()] = float("nan")
    # swap in to the spare pages, in a shuffled order
    rng = np.random.Generator(np.random.PCG64(5))
    new_pages = (w.num_pages + rng.permutation(extra)[:n_v]).astype(np.int32)
    mcp.kv_copy_pages(host_k, host_v, kc, vc, slots, torch.from_numpy(new_pages).cuda())
    torch.cuda.synchronize()
    assert torch.equal(kc[torch.from_numpy(new_pages).long()].view(torch.int16),
                       before_k[src.long()].view(torch.int16))
    bt2 = bt.copy()
    bt2[victim, :n_v] = new_pages
    # attention over the remapped block table equals the oracle's over the original one
    step2 = MixedStep(w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size, pages, w.sm_scale,
                      cu, w.k_lens, bt2)
    out = torch.full_like(td["q"], float("nan"))
    lse = torch.full((w.total_q, w.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
    step2.attention(td["q"], kc, vc, out, lse)
    step2.check()
    ref = OracleStep(w, t)
    ref.do_append()
    ref_o, ref_l = ref.attention()
    compare(w, out, lse, ref_o, ref_l, label="swapped")


def test_copy_within_device_pool_and_range_check():
    import mixed_chunked_prefill_gb300 as mcp

    g = torch.Generator().manual_seed(8)
    kc = torch.randn((40, 16, 2, 64), generator=g).to(torch.bfloat16).cuda()
    vc = torch.randn((40, 16, 2, 64), generator=g).to(torch.bfloat16).cuda()
    k0, v0 = kc.clone(), vc.clone()
    src = torch.tensor([3, 7, 11], dtype=torch.int32, device="cuda")
    dst = torch.tensor([30, 31, 20], dtype=torch.int32, device="cuda")
    mcp.kv_copy_pages(kc, vc, kc, vc, src, dst)
    torch.cuda.synchronize()
    for s_, d_ in ((3, 30), (7, 31), (11, 20)):
        assert torch.equal(kc[d_].view(torch.int16), k0[s_].view(torch.int16))
        assert torch.equal(vc[d_].view(torch.int16), v0[s_].view(torch.int16))
    untouched = [i for i in range(40) if i not in (30, 31, 20)]
    assert torch.equal(kc[untouched].view(torch.int16), k0[untouched].view(torch.int16))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mcp.kv_copy_pages(kc, vc, kc, vc, torch.tensor([1, 40], dtype=torch.int32, device="cuda"),
                      torch.tensor([2, 5], dtype=torch.int32, device="cuda"), err)
    torch.cuda.synchronize()
    assert torch.equal(kc[2].view(torch.int16), k0[1].view(torch.int16))
    assert torch.equal(kc[5].view(torch.int16), k0[5].view(torch.int16))  # skipped
    with pytest.raises(mcp.MCPError) as ei:
        mcp.check_device_errors(err.data_ptr())
    assert ei.value.status == 6
