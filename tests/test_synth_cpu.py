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
