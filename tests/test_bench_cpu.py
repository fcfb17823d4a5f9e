"""bench.py bookkeeping that needs no GPU: the roofline numerators, the
profiled traffic lookup, the host details of the CPU baseline and the
oracle's segment sample of the big workloads."""

from __future__ import annotations

import bench
import synth


def test_algorithmic_bytes_and_flops_of_the_worked_layout():
    """The worked layout's numerators, written out from the definition: every
    KV position read once per kv head (K and V), Q read and O written once;
    tensor FLOPs = 4 * D * H_q * visible (query, key) pairs of the chunk."""
    w = synth.make_workload("worked")
    a = bench.algorithmic(w)
    D, Hq, Hkv = 128, 32, 8
    kv = (121 + 46 + 10000) * Hkv * D * 2 * 2
    qo = 1810 * Hq * D * 2
    assert a["kv_bytes"] == kv
    assert a["q_bytes"] == qo and a["o_bytes"] == qo
    assert a["fwd_bytes"] == kv + 2 * qo
    pairs = 1808 * 8192 + 1808 * 1809 // 2  # history fully visible + causal inside the chunk
    assert a["flops_tc"] == 4 * D * Hq * pairs
    assert abs(a["flops_tc"] - 2.695e11) < 1e9
    assert a["flops_dec"] == 4 * D * Hq * (121 + 46)  # the two decodes (off the tensor cores)
    assert a["append_bytes"] == 1810 * Hkv * D * 2 * 2 * 2


def test_sampled_rows_count_only_the_keys_they_see():
    w = synth.make_workload("worked")
    rows = [0, 1, 1809]  # logits_indices: the last token of each segment
    a = bench.algorithmic(w, rows)
    assert a["kv_bytes"] == (121 + 46 + 10000) * 8 * 128 * 4
    assert a["q_bytes"] == 3 * 32 * 128 * 2 and a["flops_tc"] == 0


def test_committed_profiles_match_the_kernel_source():
    """Every workload with a committed ncu summary reports its DRAM traffic:
    the summaries were taken on the current kernel source."""
    for name in synth.CONFIG_NAMES + synth.PROFILE_NAMES:
        t = bench.profiled_traffic(name)
        assert t is not None and t > 0, name
    # algorithmic bytes bound the traffic of the HBM-bound steps from below
    for name in ("decode-heavy", "long-context", "decode-32x16k"):
        w = synth.make_workload(name)
        assert bench.profiled_traffic(name) >= 0.9 * bench.algorithmic(w)["kv_bytes"], name


def test_host_details_of_the_cpu_baseline():
    h = bench.host_details()
    assert h["os_cpu_count"] >= 1 and h["machine"]
    assert h["affinity"] is None or 1 <= h["affinity"] <= h["os_cpu_count"]
    assert isinstance(h["blas_threads"], (int, str))
    assert "single-thread" in h["threading"]
    assert bench.oracle_cores() >= 1


def test_oracle_sample_of_a_big_workload_keeps_its_segments():
    """The CPU legs sample the big workloads by segment: the shortest and the
    longest decode plus the chunk, with their own lengths."""
    for name, chunk_q, chunk_k in (("long-context", 2048, 131072), ("decode-heavy", 512, 33280)):
        full = synth.make_workload(name)
        segs = bench.sample_segments(full)
        dec_k = [full.k_lens[s] for s in range(full.num_seqs) if full.q_lens[s] == 1]
        assert [full.q_lens[i] for i in segs] == [1, 1, chunk_q]
        assert [full.k_lens[i] for i in segs] == [min(dec_k), max(dec_k), chunk_k]
