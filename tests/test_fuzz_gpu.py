"""Randomised parity: seeded mixed steps against the oracle.

Each case draws a step the fixed tests do not spell out -- kv heads, group
size, head_dim, page size, and a mix of decode segments, speculative
multi-token segments, chunks with and without history, empty segments -- and
sometimes forces split KV ranges.  A second family takes large GQA groups
(6 to 128 query heads per kv head), speculative segments of up to 16 tokens
and histories up to 6000 keys.  Every row is compared with the oracle
([W] "Flash Attention 的 varlen 接口": each segment sees its own KV,
right-aligned), the caches bit-exact after the append, unused slots NaN.
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import synth
from test_parity_gpu import full_parity, opts

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


def random_step(seed):
    """(workload, plan options) of one seeded random mixed step."""
    rng = np.random.Generator(np.random.PCG64(9000 + seed))
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 3, 4, 8]))
    d = int(rng.choice([64, 96, 128, 128, 256]))
    page = int(rng.choice([1, 8, 16, 16, 16, 32, 64]))
    q_lens, k_lens = [], []
    for _ in range(int(rng.integers(1, 9))):
        kind = rng.choice(["decode", "decode", "spec", "chunk", "fresh", "empty"])
        hist = int(rng.integers(0, 3000))
        if kind == "decode":
            lq = 1
        elif kind == "spec":
            lq = int(rng.integers(2, 5))
        elif kind == "chunk":
            lq = int(rng.integers(2, 300))
        elif kind == "fresh":  # a prompt's first chunk: no history
            lq, hist = int(rng.integers(1, 300)), 0
        else:  # no token this step
            lq, hist = 0, int(rng.integers(1, 500))
        q_lens.append(lq)
        k_lens.append(lq + hist if lq + hist > 0 else 1)
    if sum(q_lens) == 0:
        q_lens[0], k_lens[0] = 1, k_lens[0] + 1
    w = synth.make_workload_from_lengths(f"fuzz{seed}", hkv * g, hkv, d, page, 1 / math.sqrt(d),
                                         q_lens, k_lens, 700 + seed)
    split = rng.random() < 0.4
    o = opts(int(rng.choice([16, 64, 256])), int(rng.choice([128, 256, 512]))) if split else None
    return w, o


@pytest.mark.parametrize("seed", range(48))
def test_random_mixed_step(seed):
    w, o = random_step(seed)
    label = (f"fuzz{seed}: H {w.num_q_heads}/{w.num_kv_heads} D {w.head_dim} P {w.page_size} "
             f"q {w.q_lens} k {w.k_lens} split {o is not None}")
    full_parity(w, options=o, label=label)


def random_wide_step(seed):
    """(workload, plan options) of one seeded random step with a large group."""
    rng = np.random.Generator(np.random.PCG64(50000 + seed))
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([6, 12, 16, 32, 64, 128]))
    while hkv * g > 256:
        g //= 2
    d = int(rng.choice([64, 96, 128, 256]))
    page = int(rng.choice([8, 16, 32, 64]))
    q_lens, k_lens = [], []
    for _ in range(int(rng.integers(1, 6))):
        kind = rng.choice(["decode", "spec", "chunk", "fresh"])
        hist = int(rng.integers(0, 6000))
        lq = {"decode": 1, "spec": int(rng.integers(2, 17)), "chunk": int(rng.integers(2, 200)),
              "fresh": int(rng.integers(1, 200))}[kind]
        if kind == "fresh":  # a prompt's first chunk: no history
            hist = 0
        q_lens.append(lq)
        k_lens.append(lq + hist)
    w = synth.make_workload_from_lengths(f"wide{seed}", hkv * g, hkv, d, page, 1 / math.sqrt(d),
                                         q_lens, k_lens, 900 + seed)
    o = opts(int(rng.choice([16, 64, 512])), int(rng.choice([128, 1024]))) if rng.random() < 0.5 else None
    return w, o


@pytest.mark.parametrize("seed", range(24))
def test_random_wide_step(seed):
    w, o = random_wide_step(seed)
    label = (f"wide{seed}: H {w.num_q_heads}/{w.num_kv_heads} D {w.head_dim} P {w.page_size} "
             f"q {w.q_lens} k {w.k_lens} split {o is not None}")
    full_parity(w, options=o, label=label)
