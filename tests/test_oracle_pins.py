"""Pins for the CPU oracle (no GPU).

Each check ties the oracle to something other than itself: arrays the pages
print, library routines (torch SDPA with a lower-right causal bias and grouped
heads, torch.logsumexp), closed forms, and brute force on tiny inputs.  The
mutation tests at the end plant plausible mistakes in the oracle and show that
some pin fails.
"""

from __future__ import annotations

import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

import oracle
import synth
from harness import OracleStep
from oracle import mixed_attn_ref as ref

GOLDEN = Path(__file__).parent / "golden"


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def tiny_workload(q_lens, k_lens, hq=4, hkv=2, d=8, p=4, seed=7, scale=None):
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    return synth.make_workload_from_lengths("pin", hq, hkv, d, p, scale, q_lens, k_lens, seed)


def run_oracle(w, tensors=None):
    t = tensors if tensors is not None else w.tensors("cpu")
    st = OracleStep(w, t)
    st.do_append()
    out, lse = st.attention()
    return st, t, out, lse


def logical_kv(w, t, s):
    """Segment s's K, V in position order, float64 [Lk, H_kv, D], straight from
    the generator (history then this step's tokens) -- no page table involved."""
    hist = w.hist_lens
    h0 = sum(hist[:s])
    q0 = sum(w.q_lens[:s])
    k = torch.cat([t["k_hist"][h0:h0 + hist[s]], t["k_new"][q0:q0 + w.q_lens[s]]]).double()
    v = torch.cat([t["v_hist"][h0:h0 + hist[s]], t["v_new"][q0:q0 + w.q_lens[s]]]).double()
    return k, v


def sdpa_segment(w, t, s):
    """torch SDPA of segment s with a lower-right causal bias and grouped heads."""
    k, v = logical_kv(w, t, s)
    q0 = sum(w.q_lens[:s])
    q = t["q"][q0:q0 + w.q_lens[s]].double()
    lq, lk = q.shape[0], k.shape[0]
    qh, kh, vh = q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None], v.permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(qh, kh, vh, attn_mask=causal_lower_right(lq, lk),
                                       scale=w.sm_scale, enable_gqa=True)
    return o[0].permute(1, 0, 2).numpy()


# ---------------------------------------------------------------------------
# layout values printed on the pages
# ---------------------------------------------------------------------------

def test_worked_layout_arrays():
    g = json.loads((GOLDEN / "worked_layout.json").read_text())
    cu_q, cu_k, mq, mk = oracle.segment_layout(g["q_lens"], g["k_lens"])
    assert cu_q == g["cu_seqlens_q"]
    assert cu_k == g["cu_seqlens_k"]
    assert mq == g["max_seqlen_q"] and mk == g["max_seqlen_k"]


def test_worked_layout_visibility_counts():
    g = json.loads((GOLDEN / "worked_layout.json").read_text())
    vis = g["visible"]
    lq, lk = g["q_lens"], g["k_lens"]
    assert oracle.visible_keys(0, lq[0], lk[0]) == vis["decode_A"]
    assert oracle.visible_keys(0, lq[1], lk[1]) == vis["decode_B"]
    assert oracle.visible_keys(0, lq[2], lk[2]) == vis["chunk_C_first"]
    # the i-th chunk token (1-based) sees the history plus chunk tokens 1..i
    for i1 in (1, 2, 17, 1000, 1808):
        assert oracle.visible_keys(i1 - 1, lq[2], lk[2]) == vis["chunk_C_history"] + i1


def test_lpnh_packed_layout():
    g = json.loads((GOLDEN / "lpnh_packed_layout.json").read_text())
    cu_q, _, _, _ = oracle.segment_layout(g["q_lens"], g["q_lens"])
    assert cu_q == g["cu_seqlens"]


def test_worked_workload_matches_page_layout():
    w = synth.make_workload("worked")
    g = json.loads((GOLDEN / "worked_layout.json").read_text())
    cu_q, cu_k, _, _ = oracle.segment_layout(w.q_lens, w.k_lens)
    assert cu_q == g["cu_seqlens_q"] and cu_k == g["cu_seqlens_k"]


# ---------------------------------------------------------------------------
# attention against library routines
# ---------------------------------------------------------------------------

MIXED = ([1, 3, 5, 1, 2, 4], [7, 3, 13, 1, 9, 4])  # decodes, a no-history chunk, chunks with history


def check_segments_match_sdpa(w):
    st, t, out, lse = run_oracle(w)
    for s in range(w.num_seqs):
        ref_o = sdpa_segment(w, t, s)
        got = out[st.cu_q[s]:st.cu_q[s + 1]]
        np.testing.assert_allclose(got, ref_o, rtol=1e-12, atol=1e-12)


def test_segments_match_sdpa_lower_right_gqa():
    check_segments_match_sdpa(tiny_workload(*MIXED))


def test_segments_match_sdpa_mha_and_wide_groups():
    check_segments_match_sdpa(tiny_workload(*MIXED, hq=3, hkv=3, d=16, p=16, seed=11))
    check_segments_match_sdpa(tiny_workload(*MIXED, hq=8, hkv=1, d=4, p=2, seed=12))


def test_decode_rows_equal_unmasked_softmax_attention():
    # a one-token segment sees its whole context: plain SDPA with no mask
    w = tiny_workload([1, 1, 1], [1, 6, 23], seed=3)
    st, t, out, _ = run_oracle(w)
    for s in range(w.num_seqs):
        k, v = logical_kv(w, t, s)
        q = t["q"][st.cu_q[s]:st.cu_q[s] + 1].double()
        o = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None],
                                           v.permute(1, 0, 2)[None], scale=w.sm_scale,
                                           enable_gqa=True)[0].permute(1, 0, 2).numpy()
        np.testing.assert_allclose(out[st.cu_q[s]:st.cu_q[s] + 1], o, rtol=1e-12, atol=1e-12)


def test_no_history_segment_is_standard_causal():
    # Lq = Lk: the right-aligned mask is ordinary causal self-attention
    w = tiny_workload([6], [6], seed=5)
    st, t, out, _ = run_oracle(w)
    k, v = logical_kv(w, t, 0)
    q = t["q"].double()
    o = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None],
                                       v.permute(1, 0, 2)[None], is_causal=True,
                                       scale=w.sm_scale, enable_gqa=True)[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, o.numpy(), rtol=1e-12, atol=1e-12)


def test_lse_matches_logsumexp_of_sdpa_scores():
    w = tiny_workload(*MIXED, seed=21)
    st, t, out, lse = run_oracle(w)
    for s in range(w.num_seqs):
        k, v = logical_kv(w, t, s)
        q = t["q"][st.cu_q[s]:st.cu_q[s + 1]].double()
        lq, lk = q.shape[0], k.shape[0]
        keep = causal_lower_right(lq, lk)._materialize()
        krep = k.repeat_interleave(w.num_q_heads // w.num_kv_heads, dim=1)
        scores = torch.einsum("qhd,khd->hqk", q, krep) * w.sm_scale
        scores = scores.masked_fill(~keep[None], -math.inf)
        expect = torch.logsumexp(scores, dim=-1).T.numpy()
        np.testing.assert_allclose(lse[st.cu_q[s]:st.cu_q[s + 1]], expect, rtol=1e-12, atol=1e-12)


def test_lse_closed_form_exact_scores():
    # q = a e0, k_j = b_j e0: s_j = a b_j scale exactly; lse over visible keys by hand
    w = tiny_workload([2], [5], hq=1, hkv=1, d=4, p=2, seed=1, scale=0.5)
    b = [1.0, -2.0, 0.5, 3.0, -1.0]
    a = 2.0
    q = torch.zeros(2, 1, 4, dtype=torch.bfloat16)
    q[:, 0, 0] = a
    kh = torch.zeros(3, 1, 4, dtype=torch.bfloat16)
    kn = torch.zeros(2, 1, 4, dtype=torch.bfloat16)
    for j in range(3):
        kh[j, 0, 0] = b[j]
    for j in range(2):
        kn[j, 0, 0] = b[3 + j]
    t = {"q": q, "k_hist": kh, "k_new": kn, "v_hist": torch.ones(3, 1, 4, dtype=torch.bfloat16),
         "v_new": torch.ones(2, 1, 4, dtype=torch.bfloat16)}
    _, _, out, lse = run_oracle(w, t)
    for i in range(2):
        n = 3 + i + 1
        expect = math.log(sum(math.exp(a * b[j] * 0.5) for j in range(n)))
        assert abs(lse[i, 0] - expect) < 1e-12
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# chunked prefill equals one-shot prefill
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("splits", [[13], [6, 7], [3, 5, 5], [1, 1, 4, 2, 1, 1, 1, 2]])
def test_chunked_prefill_equals_one_shot(splits):
    L = sum(splits)
    hq, hkv, d, p = 4, 2, 8, 4
    g = torch.Generator().manual_seed(99)
    q = torch.randn(L, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(L, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(L, hkv, d, generator=g).to(torch.bfloat16)
    scale = 1 / math.sqrt(d)
    # one sequence, pages in a shuffled order
    n_pages = -(-L // p) + 2
    perm = np.random.Generator(np.random.PCG64(5)).permutation(n_pages)
    table = oracle.PageTable(p)
    for lp in range(-(-L // p)):
        table.map(0, lp, int(perm[lp]))
    store = oracle.PagedKVStore(p, hkv, d)
    outs = []
    done = 0
    for n in splits:
        cu = [0, n]
        lk = [done + n]
        slots = oracle.new_token_slots(table, cu, lk)
        oracle.append(store, slots, synth.bf16_bits(k[done:done + n]), synth.bf16_bits(v[done:done + n]))
        qb = oracle.bf16_bits_to_f64(synth.bf16_bits(q[done:done + n]))
        o, _ = oracle.mixed_attention(qb, store, table, cu, lk, hkv, scale)
        outs.append(o)
        done += n
    got = np.concatenate(outs)
    expect = F.scaled_dot_product_attention(q.double().permute(1, 0, 2)[None],
                                            k.double().permute(1, 0, 2)[None],
                                            v.double().permute(1, 0, 2)[None], is_causal=True,
                                            scale=scale, enable_gqa=True)[0].permute(1, 0, 2)
    np.testing.assert_allclose(got, expect.numpy(), rtol=1e-10, atol=1e-10)


# ---------------------------------------------------------------------------
# brute force: which keys change which rows
# ---------------------------------------------------------------------------

def test_visibility_by_perturbation():
    # worded rule: a query sees all history positions and the chunk tokens up to itself
    w = tiny_workload([1, 4], [5, 7], hq=2, hkv=1, d=4, p=4, seed=17)
    st, t, base, _ = run_oracle(w)
    for s in range(w.num_seqs):
        lq, lk = w.q_lens[s], w.k_lens[s]
        hist = lk - lq
        for j in range(lk):
            st2 = OracleStep(w, t)
            st2.do_append()
            kb, vb = st2.store.read(st2.table, s, j)
            vb = oracle.f64_to_bf16_bits(oracle.bf16_bits_to_f64(vb) + 4.0)
            st2.store.write_slot(st2.table.slot(s, j), kb, vb)
            out2, _ = st2.attention()
            for i in range(lq):
                tok = st.cu_q[s] + i
                changed = not np.array_equal(out2[tok], base[tok])
                expected_visible = j < hist or (j - hist) <= i
                assert changed == expected_visible, (s, i, j)
            for s2 in range(w.num_seqs):  # other segments are untouched
                if s2 != s:
                    sl = slice(st.cu_q[s2], st.cu_q[s2 + 1])
                    assert np.array_equal(out2[sl], base[sl])


# ---------------------------------------------------------------------------
# closed forms and invariants
# ---------------------------------------------------------------------------

def test_constant_values_give_that_value():
    w = tiny_workload(*MIXED, seed=31)
    t = w.tensors("cpu")
    c = torch.linspace(-3, 3, w.head_dim).to(torch.bfloat16)
    t["v_hist"] = c.expand_as(t["v_hist"]).clone()
    t["v_new"] = c.expand_as(t["v_new"]).clone()
    _, _, out, _ = run_oracle(w, t)
    np.testing.assert_allclose(out, np.broadcast_to(c.double().numpy(), out.shape), rtol=0, atol=1e-13)


def test_zero_keys_give_mean_of_visible_values():
    w = tiny_workload(*MIXED, seed=32)
    t = w.tensors("cpu")
    t["k_hist"].zero_()
    t["k_new"].zero_()
    st, _, out, lse = run_oracle(w, t)
    G = w.num_q_heads // w.num_kv_heads
    for s in range(w.num_seqs):
        _, v = logical_kv(w, t, s)
        csum = np.cumsum(v.numpy(), axis=0)
        lq, lk = w.q_lens[s], w.k_lens[s]
        for i in range(lq):
            n = (lk - lq) + i + 1
            for h in range(w.num_q_heads):
                np.testing.assert_allclose(out[st.cu_q[s] + i, h], csum[n - 1, h // G] / n,
                                           rtol=1e-12, atol=1e-13)
                assert abs(lse[st.cu_q[s] + i, h] - math.log(n)) < 1e-12


def test_page_permutation_invariance():
    w1 = tiny_workload(*MIXED, seed=41)
    t = w1.tensors("cpu")
    w2 = tiny_workload(*MIXED, seed=42)  # same lengths, another page permutation
    w2.seed = w1.seed
    assert not np.array_equal(w1.block_tables(), w2.block_tables())
    _, _, o1, l1 = run_oracle(w1, t)
    _, _, o2, l2 = run_oracle(w2, t)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_segment_independence():
    w = tiny_workload(*MIXED, seed=43)
    t = w.tensors("cpu")
    st, _, o1, _ = run_oracle(w, t)
    # perturb every K/V of segment 2 (history and new)
    t2 = {k: v.clone() for k, v in t.items()}
    h0 = sum(w.hist_lens[:2])
    t2["k_hist"][h0:h0 + w.hist_lens[2]] += 1
    t2["v_new"][st.cu_q[2]:st.cu_q[3]] -= 1
    _, _, o2, _ = run_oracle(w, t2)
    for s in range(w.num_seqs):
        sl = slice(st.cu_q[s], st.cu_q[s + 1])
        assert np.array_equal(o1[sl], o2[sl]) == (s != 2)


# ---------------------------------------------------------------------------
# merge of split states
# ---------------------------------------------------------------------------

def test_merge_states_equals_unsplit():
    g = torch.Generator().manual_seed(3)
    R, H, D, L = 3, 2, 8, 23
    q = torch.randn(H, R, D, generator=g, dtype=torch.float64)
    k = torch.randn(H, L, D, generator=g, dtype=torch.float64)
    v = torch.randn(H, L, D, generator=g, dtype=torch.float64)
    scale = 0.3
    cuts = [0, 5, 6, 17, 23]
    o_parts, l_parts = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o_parts.append(F.scaled_dot_product_attention(q, k[:, a:b], v[:, a:b], scale=scale).permute(1, 0, 2))
        l_parts.append(torch.logsumexp(q @ k[:, a:b].transpose(1, 2) * scale, -1).T)
    O, LSE = oracle.merge_states(torch.stack(o_parts).numpy(), torch.stack(l_parts).numpy())
    full = F.scaled_dot_product_attention(q, k, v, scale=scale).permute(1, 0, 2).numpy()
    full_lse = torch.logsumexp(q @ k.transpose(1, 2) * scale, -1).T.numpy()
    np.testing.assert_allclose(O, full, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(LSE, full_lse, rtol=1e-12, atol=1e-12)


def test_merge_states_identical_and_empty_parts():
    rng = np.random.Generator(np.random.PCG64(1))
    o = rng.standard_normal((4, 8))
    lse = rng.standard_normal(4)
    O, L = oracle.merge_states(np.stack([o, o, o]), np.stack([lse, lse, lse]))
    np.testing.assert_allclose(O, o, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(L, lse + math.log(3), rtol=1e-14, atol=1e-14)
    O2, L2 = oracle.merge_states(np.stack([o, np.full_like(o, np.nan)]),
                                 np.stack([lse, np.full_like(lse, -np.inf)]))
    np.testing.assert_allclose(O2, o, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(L2, lse, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------------------
# paged addressing and append
# ---------------------------------------------------------------------------

def check_slots_identity_pool():
    # pages handed out contiguously: slot = first_page * P + position
    P = 16
    q_lens, k_lens = [1, 1, 1808], [121, 46, 10000]
    first = [0, 8, 11]
    table = oracle.PageTable(P)
    for s, lk in enumerate(k_lens):
        for lp in range(-(-lk // P)):
            table.map(s, lp, first[s] + lp)
    cu_q, _, _, _ = oracle.segment_layout(q_lens, k_lens)
    slots = oracle.new_token_slots(table, cu_q, k_lens)
    expect = [first[0] * P + 120, first[1] * P + 45] + [first[2] * P + 8192 + i for i in range(1808)]
    assert list(slots) == expect


def test_slots_identity_pool():
    check_slots_identity_pool()


def test_slots_follow_block_table_pages():
    w = tiny_workload(*MIXED, p=4, seed=51)
    st = OracleStep(w, w.tensors("cpu"))
    bt = w.block_tables()
    for s in range(w.num_seqs):
        lq, lk = w.q_lens[s], w.k_lens[s]
        for i in range(lq):
            pos = lk - lq + i
            slot = int(st.slots[st.cu_q[s] + i])
            assert slot // 4 == bt[s][pos // 4]  # the page the block table names
            assert slot % 4 == pos % 4            # the offset inside it


def test_append_bit_exact_and_nothing_else():
    w = tiny_workload(*MIXED, seed=52)
    t = w.tensors("cpu")
    st = OracleStep(w, t)
    kc0, vc0 = st.cache_bits()
    slots = st.slots.copy()
    slots[2] = -1  # a skipped (padding) token
    oracle.append(st.store, slots, st.k_new_bits, st.v_new_bits)
    kc1, vc1 = st.cache_bits()
    P = w.page_size
    touched = np.zeros(kc0.shape[:2], dtype=bool)
    for tkn, slot in enumerate(slots):
        if slot < 0:
            continue
        assert np.array_equal(kc1[slot // P, slot % P], st.k_new_bits[tkn])
        assert np.array_equal(vc1[slot // P, slot % P], st.v_new_bits[tkn])
        touched[slot // P, slot % P] = True
    assert np.array_equal(kc1[~touched], kc0[~touched])
    assert np.array_equal(vc1[~touched], vc0[~touched])
    # the skipped token's slot still holds the fill
    s2 = int(st.slots[2])
    assert np.all(kc1[s2 // P, s2 % P] == 0x7FC0)


def test_bf16_roundtrip_helpers():
    x = torch.randn(1000, generator=torch.Generator().manual_seed(0)) * 100
    b = x.to(torch.bfloat16)
    bits = synth.bf16_bits(b)
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(bits), b.double().numpy())
    np.testing.assert_array_equal(oracle.f64_to_bf16_bits(x.double().numpy()), bits)


# ---------------------------------------------------------------------------
# planted mistakes: each must trip a pin
# ---------------------------------------------------------------------------

def test_planted_top_left_mask_is_caught(monkeypatch):
    monkeypatch.setattr(ref, "visible_keys", lambda i, lq, lk: int(i) + 1)
    with pytest.raises(AssertionError):
        check_segments_match_sdpa(tiny_workload(*MIXED))


def test_planted_off_by_one_mask_is_caught(monkeypatch):
    monkeypatch.setattr(ref, "visible_keys", lambda i, lq, lk: int(i) + (int(lk) - int(lq)))
    with pytest.raises(AssertionError):
        check_segments_match_sdpa(tiny_workload(*MIXED))


def test_planted_interleaved_gqa_is_caught(monkeypatch):
    monkeypatch.setattr(ref, "kv_head_of", lambda h, hq, hkv: int(h) % int(hkv))
    with pytest.raises(AssertionError):
        check_segments_match_sdpa(tiny_workload(*MIXED))


def test_planted_slot_formula_is_caught(monkeypatch):
    monkeypatch.setattr(ref.PageTable, "slot",
                        lambda self, seq, pos: self.physical_page(seq, pos) * self.page_size
                        + int(pos) // self.page_size)
    with pytest.raises(AssertionError):
        check_slots_identity_pool()


def test_planted_missing_scale_is_caught():
    w = tiny_workload(*MIXED)
    w_bad = tiny_workload(*MIXED)
    w_bad.sm_scale = 1.0
    st, t, out, _ = run_oracle(w_bad, w.tensors("cpu"))
    with pytest.raises(AssertionError):
        for s in range(w.num_seqs):
            np.testing.assert_allclose(out[st.cu_q[s]:st.cu_q[s + 1]], sdpa_segment(w, t, s),
                                       rtol=1e-12, atol=1e-12)


def test_worked_layout_rows_match_sdpa_at_full_size():
    # the page's worked layout at its real sizes, a sample of rows (the
    # oracle's row-subset mode is what full-size GPU parity samples with)
    w = synth.make_workload("worked")
    t = w.tensors("cpu")
    st = OracleStep(w, t)
    st.do_append()
    rows = [0, 1, 2, 3, 500, 1809]
    out, lse = st.attention(tokens=rows)
    for s in range(w.num_seqs):
        want = [r for r in rows if st.cu_q[s] <= r < st.cu_q[s + 1]]
        ref_o = sdpa_segment(w, t, s)
        for r in want:
            np.testing.assert_allclose(out[r], ref_o[r - st.cu_q[s]], rtol=1e-11, atol=1e-12)
    untouched = [r for r in range(w.total_q) if r not in rows]
    assert np.isnan(out[untouched]).all()
