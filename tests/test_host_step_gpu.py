"""GPU: several serving steps through the pipelined host step against the
oracle.

A prompt is prefilled in chunks across steps while other sequences decode, one
sequence finishes and another joins ([W] "组装长序列" and "输入组装": every step
appends its tokens through the slot mapping, then attends over each
segment's own paged KV).  Steps are enqueued back to back (two in flight) and
only then waited for, so each step must see exactly the K/V the steps before
it appended.  Outputs and LSE of every step are compared with the float64
oracle, the final caches bit for bit.
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

H_Q, H_KV, D, P = 8, 2, 128, 16

# per step: list of (sequence, tokens this step); a sequence's KV length after a
# step is its history plus everything it has appended so far
SCHEDULE = [
    [("B", 1), ("D", 1), ("A", 256)],
    [("D", 1), ("B", 1), ("A", 256)],
    [("B", 1), ("D", 1), ("A", 88), ("C", 40)],
    [("C", 1), ("B", 1), ("A", 1)],
    [("A", 1), ("B", 1), ("C", 1)],
    [("B", 1), ("C", 3), ("A", 2)],  # the last one: short speculative-style segments
]
HISTORY = {"A": 0, "B": 300, "C": 0, "D": 1000}


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from mixed_chunked_prefill_gb300 import build

    build.build()
    import mixed_chunked_prefill_gb300 as mcp

    return mcp.load()


def test_pipelined_steps_match_oracle():
    from mixed_chunked_prefill_gb300.step import HostStep

    rng = np.random.Generator(np.random.PCG64(4242))
    final = dict(HISTORY)
    for step in SCHEDULE:
        for s, n in step:
            final[s] += n
    seqs = sorted(final)
    pages_of = {s: -(-final[s] // P) for s in seqs}
    mp = max(pages_of.values())
    num_pages = sum(pages_of.values()) + 3
    perm = rng.permutation(num_pages).astype(np.int32)
    table, off = {}, 0
    for s in seqs:
        table[s] = perm[off:off + pages_of[s]]
        off += pages_of[s]
    scale = 1.0 / math.sqrt(D)

    def bt_rows(names):
        bt = np.full((len(names), mp), -1, dtype=np.int32)
        for i, s in enumerate(names):
            bt[i, :pages_of[s]] = table[s]
        return bt

    dev = torch.device("cuda")
    kc = torch.full((num_pages, P, H_KV, D), float("nan"), dtype=torch.bfloat16, device=dev)
    vc = torch.full_like(kc, float("nan"))
    store = oracle.PagedKVStore(P, H_KV, D)
    gen = torch.Generator().manual_seed(77)

    def rand(*shape):
        return torch.randn(shape, generator=gen).to(torch.bfloat16)

    # histories: written by the library's append, mirrored into the oracle store
    import mixed_chunked_prefill_gb300 as mcp

    hist_names = [s for s in seqs if HISTORY[s] > 0]
    hl = [HISTORY[s] for s in hist_names]
    cu_h = np.concatenate([[0], np.cumsum(hl)]).astype(np.int32)
    bt_h = bt_rows(hist_names)
    slots_h = mcp.build_slot_mapping(bt_h, cu_h, hl, P, num_pages)
    kh, vh = rand(int(cu_h[-1]), H_KV, D), rand(int(cu_h[-1]), H_KV, D)
    mcp.paged_kv_append(kh.to(dev), vh.to(dev), torch.from_numpy(slots_h).to(dev), kc, vc)
    tab_h = oracle.page_table_from_block_tables(bt_h, hl, P)
    oracle.append(store, oracle.new_token_slots(tab_h, cu_h, hl), synth.bf16_bits(kh),
                  synth.bf16_bits(vh))
    torch.cuda.synchronize()

    hs = HostStep(H_Q, H_KV, D, P, num_pages, scale, max_tokens=400, max_seqs=8,
                  max_pages_per_seq=mp, device=dev, workspace_bytes=16 << 20,
                  list_bytes=1 << 20)
    length = dict(HISTORY)
    tickets, expect, outs = [], [], []
    for step in SCHEDULE:
        names = [s for s, _ in step]
        q_lens = [n for _, n in step]
        for s, n in step:
            length[s] += n
        k_lens = [length[s] for s in names]
        cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
        T = int(cu[-1])
        bt = bt_rows(names)
        q, kn, vn = rand(T, H_Q, D), rand(T, H_KV, D), rand(T, H_KV, D)
        # oracle: append this step's tokens, then attend
        tab = oracle.page_table_from_block_tables(bt, k_lens, P)
        oracle.append(store, oracle.new_token_slots(tab, cu, k_lens), synth.bf16_bits(kn),
                      synth.bf16_bits(vn))
        ref_o, ref_l = oracle.mixed_attention(oracle.bf16_bits_to_f64(synth.bf16_bits(q)), store,
                                              tab, cu, k_lens, H_KV, scale)
        expect.append((ref_o, ref_l))
        out_h = torch.full((T, H_Q, D), float("nan"), dtype=torch.bfloat16).pin_memory()
        lse_h = torch.full((T, H_Q), float("nan"), dtype=torch.float32).pin_memory()
        qh, kh_, vh_ = q.pin_memory(), kn.pin_memory(), vn.pin_memory()
        outs.append((out_h, lse_h, qh, kh_, vh_))
        tickets.append(hs.run(qh, kh_, vh_, cu, k_lens, bt, kc, vc, out_h, lse_h))
    for t, (ref_o, ref_l), (out_h, lse_h, *_) in zip(tickets, expect, outs):
        hs.wait(t)
        got = out_h.float().numpy()
        assert np.isfinite(got).all(), f"step {t}: non-finite output"
        err = float(np.abs(got - ref_o).max())
        rr = rel_rms(got, ref_o)
        lerr = float(np.abs(lse_h.numpy() - ref_l).max())
        print(f"step {t}: max|err| {err:.3g} relRMS {rr:.3g} lse {lerr:.3g}")
        assert err <= ATOL and rr <= RMS_TOL and lerr <= LSE_TOL
    hs.close()
    k_bits, v_bits = store.materialize(num_pages, 0x7FC0)
    assert np.array_equal(synth.bf16_bits(kc), k_bits), "k_cache not bit-exact"
    assert np.array_equal(synth.bf16_bits(vc), v_bits), "v_cache not bit-exact"


def test_metadata_error_enqueues_nothing():
    """A block-table page outside the pool is rejected on the host; the object
    stays usable."""
    import mixed_chunked_prefill_gb300 as mcp
    from mixed_chunked_prefill_gb300.step import HostStep

    dev = torch.device("cuda")
    kc = torch.zeros((8, P, H_KV, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    hs = HostStep(H_Q, H_KV, D, P, 8, 0.1, max_tokens=4, max_seqs=2, max_pages_per_seq=2,
                  device=dev, workspace_bytes=1 << 20, list_bytes=1 << 16)
    q = torch.zeros((1, H_Q, D), dtype=torch.bfloat16).pin_memory()
    kv = torch.zeros((1, H_KV, D), dtype=torch.bfloat16).pin_memory()
    out = torch.empty_like(q).pin_memory()
    with pytest.raises(mcp.MCPError) as ei:
        hs.run(q, kv, kv, [0, 1], [1], [[9]], kc, vc, out)
    assert ei.value.status == 1
    hs(q, kv, kv, [0, 1], [1], [[3]], kc, vc, out)  # a valid step still runs
    assert torch.equal(out.float(), torch.zeros_like(out).float())
    hs.close()
