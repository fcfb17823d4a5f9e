"""The seeded workload generator shared by the tests and the bench: the
named workloads keep their shapes, and the head_dim / page_size overrides
keep a workload's segments, heads and seed while changing only the shape."""

import math

import pytest

import synth


@pytest.mark.parametrize("name", synth.CONFIG_NAMES + synth.PROFILE_NAMES)
def test_named_workloads_are_deterministic(name):
    a = synth.make_workload(name)
    b = synth.make_workload(name)
    assert a.q_lens == b.q_lens and a.k_lens == b.k_lens and a.seed == b.seed
    assert (a.page_perm == b.page_perm).all()
    assert all(q <= k for q, k in zip(a.q_lens, a.k_lens))


@pytest.mark.parametrize("head_dim,page_size", [(96, None), (256, None), (None, 8), (64, 32)])
def test_overrides_change_only_the_shape(head_dim, page_size):
    base = synth.make_workload("worked")
    w = synth.make_workload("worked", head_dim=head_dim, page_size=page_size)
    assert w.q_lens == base.q_lens and w.k_lens == base.k_lens and w.seed == base.seed
    assert (w.num_q_heads, w.num_kv_heads) == (base.num_q_heads, base.num_kv_heads)
    d = head_dim or base.head_dim
    assert w.head_dim == d and w.page_size == (page_size or base.page_size)
    assert math.isclose(w.sm_scale, 1.0 / math.sqrt(d))
    # every segment still has the pages its keys need, plus spare pages
    need = sum(-(-k // w.page_size) for k in w.k_lens)
    assert len(w.page_perm) == need + w.spare_pages


def test_describe_names_the_overrides():
    assert synth.describe("worked") == synth.DESCRIPTIONS["worked"]
    text = synth.describe("worked", 256, 8)
    assert text.startswith(synth.DESCRIPTIONS["worked"]) and "head_dim 256" in text and "page 8" in text


def test_segment_kv_gathers_what_the_page_store_holds():
    """The full-size parity test reads each segment's keys through SegmentKV
    (position order straight from the inputs); on a workload the dict page
    store can hold, both give the same K/V, and the oracle's output over
    either is identical."""
    import numpy as np

    import oracle
    from gpu_harness import SegmentKV
    from harness import OracleStep

    w = synth.make_workload("balanced").shuffled(3)
    t = w.tensors("cpu")
    ref = OracleStep(w, t)
    ref.do_append()
    skv = SegmentKV(w, t)
    for s in range(w.num_seqs):
        K0, V0 = ref.store.gather(ref.table, s, w.k_lens[s])
        K1, V1 = skv.gather(None, s, w.k_lens[s])
        assert np.array_equal(K0, K1) and np.array_equal(V0, V1)
    toks = [0, 5, 29, 30, w.total_q - 1]
    a = ref.attention(tokens=toks)
    b = oracle.mixed_attention(ref.q, skv, None, ref.cu_q, w.k_lens, w.num_kv_heads, w.sm_scale,
                               tokens=toks)
    assert np.array_equal(a[0][toks], b[0][toks]) and np.array_equal(a[1][toks], b[1][toks])
