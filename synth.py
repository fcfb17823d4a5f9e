"""Seeded synthetic workloads for one mixed chunked-prefill + decode step.

Shared by the tests (for both the oracle and the CUDA path), ``bench.py`` and
``__graft_entry__.smoke()``.  It holds none of the step's arithmetic: it draws
segment lengths, hands out physical pages (a seeded random permutation of the
page pool, given to the segments in stream order) and draws N(0, 1) values
rounded to bf16.  Page addressing, append and attention live in the oracle and,
separately, in the CUDA library.

The five workloads mirror the shapes the chunked-prefill pages discuss: the
worked A/B/C layout of wangyu.me "大语言模型推理优化（二）：Chunked Prefill"
(section "组装长序列": two decodes with contexts 121 and 46 next to a 1808-token
chunk after 8192 history tokens), the 2 x 512 chunks + 30 decodes batch of
lpnh.cn "技术融合剖析…" (section 2.2), and decode-heavy / long-context mixes
with 16-token pages as in kwkr.cn's hybrid-kernel page.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20261202

# name -> (index, description).  The index offsets the seed.
CONFIG_NAMES = ["tiny", "worked", "balanced", "decode-heavy", "long-context"]
# small single-kind workloads for kernel profiles (larger than L2, a few GB at most)
PROFILE_NAMES = ["decode-32x16k", "chunk-512x16k"]

DESCRIPTIONS = {
    "tiny": "tiny mixed step: 4 q / 4 kv heads, head_dim 64, page 16; decodes ctx 121 and 46, "
            "a 64-token chunk after 192 history tokens",
    "worked": "worked-layout step: cu_seqlens_q=[0,1,2,1810], seqlens_k=[121,46,10000]; "
              "32 q / 8 kv heads, head_dim 128, page 16",
    "balanced": "balanced mix: 30 decodes ctx U[1024,8192] + 2 chunks of 512 after U[0,8192] "
                "history; 32 q / 8 kv heads, head_dim 128, page 16",
    "decode-heavy": "decode-heavy: 256 decodes ctx U[4096,32768] + one 512-token chunk after "
                    "32768 history; 64 q / 8 kv heads, head_dim 128, page 16",
    "long-context": "long-context: 64 decodes ctx U[65536,131072] + one 2048-token chunk after "
                    "126976 history; 32 q / 8 kv heads, head_dim 128, page 16",
    "decode-32x16k": "decode only: 32 decodes ctx 16384; 64 q / 8 kv heads, head_dim 128, page 16",
    "chunk-512x16k": "chunk only: one 512-token chunk after 16384 history; 32 q / 8 kv heads, "
                     "head_dim 128, page 16",
}


@dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    sm_scale: float
    q_lens: list
    k_lens: list
    seed: int
    spare_pages: int = 1
    page_perm: np.ndarray = field(default=None, repr=False)

    # -- sizes ---------------------------------------------------------------
    @property
    def num_seqs(self) -> int:
        return len(self.q_lens)

    @property
    def total_q(self) -> int:
        return int(sum(self.q_lens))

    @property
    def hist_lens(self) -> list:
        return [int(k) - int(q) for q, k in zip(self.q_lens, self.k_lens)]

    @property
    def total_hist(self) -> int:
        return int(sum(self.hist_lens))

    def pages_of(self, s: int) -> int:
        return -(-int(self.k_lens[s]) // self.page_size)

    @property
    def max_pages_per_seq(self) -> int:
        return max([self.pages_of(s) for s in range(self.num_seqs)] + [1])

    @property
    def num_pages(self) -> int:
        return int(len(self.page_perm))

    # -- page allocation (the caller's pool) ----------------------------------
    def block_tables(self) -> np.ndarray:
        """[num_seqs, max_pages_per_seq] int32; pages handed out in stream order
        from the seeded permutation; unused entries are -1."""
        bt = np.full((self.num_seqs, self.max_pages_per_seq), -1, dtype=np.int32)
        off = 0
        for s in range(self.num_seqs):
            n = self.pages_of(s)
            bt[s, :n] = self.page_perm[off:off + n]
            off += n
        return bt

    # -- values ----------------------------------------------------------------
    def tensors(self, device="cpu", parts=("q", "k_new", "v_new", "k_hist", "v_hist")):
        """bf16 torch tensors drawn N(0,1) (fp32, rounded to nearest-even bf16).

        q [T, H_q, D]; k_new, v_new [T, H_kv, D] (this step's tokens, stream
        order); k_hist, v_hist [sum of history lengths, H_kv, D] (each segment's
        history positions 0..Lk-Lq-1, segments in stream order).  Each part has
        its own generator stream, so asking for a subset gives the same values.
        The values depend on ``device`` (CPU and CUDA generators differ).
        """
        import torch

        H, Hk, D, T = self.num_q_heads, self.num_kv_heads, self.head_dim, self.total_q
        shapes = {
            "q": (T, H, D),
            "k_new": (T, Hk, D),
            "v_new": (T, Hk, D),
            "k_hist": (self.total_hist, Hk, D),
            "v_hist": (self.total_hist, Hk, D),
        }
        stream = {"q": 1, "k_new": 2, "v_new": 3, "k_hist": 4, "v_hist": 5}
        out = {}
        for p in parts:
            g = torch.Generator(device=device)
            g.manual_seed(self.seed * 16 + stream[p])
            out[p] = randn_bf16(shapes[p], g, device)
        return out

    def shuffled(self, seed: int) -> "Workload":
        """Same segments in a seeded random stream order (fresh page allocation)."""
        rng = np.random.Generator(np.random.PCG64(seed))
        order = rng.permutation(self.num_seqs)
        return make_workload_from_lengths(
            self.name + "-shuffled", self.num_q_heads, self.num_kv_heads, self.head_dim,
            self.page_size, self.sm_scale, [self.q_lens[i] for i in order],
            [self.k_lens[i] for i in order], seed)


def randn_bf16(shape, generator, device, chunk_elems=1 << 27):
    """N(0,1) fp32 draws rounded to bf16, produced in slabs along dim 0 so that
    multi-GB tensors never need a full fp32 copy."""
    import torch

    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if out.numel() == 0:
        return out
    row = max(1, out.numel() // max(1, shape[0]))
    step = max(1, chunk_elems // row)
    for r0 in range(0, shape[0], step):
        r1 = min(shape[0], r0 + step)
        out[r0:r1] = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=generator,
                                 device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_workload_from_lengths(name, num_q_heads, num_kv_heads, head_dim, page_size, sm_scale,
                               q_lens, k_lens, seed, spare_frac=0.01) -> Workload:
    """Workload with given segment lengths; the page pool is the pages the
    segments need plus ~1% spare pages, permuted with a seeded PCG64."""
    w = Workload(name, num_q_heads, num_kv_heads, head_dim, page_size, float(sm_scale),
                 [int(x) for x in q_lens], [int(x) for x in k_lens], int(seed))
    need = sum(w.pages_of(s) for s in range(w.num_seqs))
    spare = max(1, int(math.ceil(need * spare_frac)))
    rng = np.random.Generator(np.random.PCG64(seed))
    w.page_perm = rng.permutation(need + spare).astype(np.int32)
    w.spare_pages = spare
    return w


def make_workload(name: str, seed_offset: int = 0, head_dim: int | None = None,
                  page_size: int | None = None) -> Workload:
    """One of the named workloads, seeded with SEED_BASE + its index; with
    head_dim / page_size the same segments and heads at that head dim
    (sm_scale 1/sqrt(head_dim)) or page size."""
    w = _named_workload(name, seed_offset)
    if head_dim is None and page_size is None:
        return w
    d = int(head_dim or w.head_dim)
    P = int(page_size or w.page_size)
    return make_workload_from_lengths(f"{name}-d{d}-p{P}", w.num_q_heads, w.num_kv_heads, d, P,
                                      1.0 / math.sqrt(d), w.q_lens, w.k_lens, w.seed)


def describe(name: str, head_dim: int | None = None, page_size: int | None = None) -> str:
    """DESCRIPTIONS[name], with the head_dim / page_size overrides stated."""
    text = DESCRIPTIONS[name]
    over = []
    if head_dim is not None:
        over.append(f"head_dim {int(head_dim)}")
    if page_size is not None:
        over.append(f"page {int(page_size)}")
    return text + (" -- here with " + ", ".join(over) if over else "")


def _named_workload(name: str, seed_offset: int = 0) -> Workload:
    if name in PROFILE_NAMES:
        seed = SEED_BASE + 100 + PROFILE_NAMES.index(name) + seed_offset
        if name == "decode-32x16k":
            return make_workload_from_lengths(name, 64, 8, 128, 16, 1.0 / math.sqrt(128),
                                              [1] * 32, [16384] * 32, seed)
        return make_workload_from_lengths(name, 32, 8, 128, 16, 1.0 / math.sqrt(128),
                                          [512], [16384 + 512], seed)
    idx = CONFIG_NAMES.index(name)
    seed = SEED_BASE + idx + seed_offset
    rng = np.random.Generator(np.random.PCG64(seed))
    if name == "tiny":
        q, k = [1, 1, 64], [121, 46, 256]
        return make_workload_from_lengths(name, 4, 4, 64, 16, 1.0 / 8.0, q, k, seed)
    if name == "worked":
        q, k = [1, 1, 1808], [121, 46, 10000]
        return make_workload_from_lengths(name, 32, 8, 128, 16, 1.0 / math.sqrt(128), q, k, seed)
    if name == "balanced":
        dec = [int(rng.integers(1024, 8192 + 1)) for _ in range(30)]
        ch = [512 + int(rng.integers(0, 8192 + 1)) for _ in range(2)]
        q, k = [1] * 30 + [512, 512], dec + ch
        return make_workload_from_lengths(name, 32, 8, 128, 16, 1.0 / math.sqrt(128), q, k, seed)
    if name == "decode-heavy":
        dec = [int(rng.integers(4096, 32768 + 1)) for _ in range(256)]
        q, k = [1] * 256 + [512], dec + [33280]
        return make_workload_from_lengths(name, 64, 8, 128, 16, 1.0 / math.sqrt(128), q, k, seed)
    if name == "long-context":
        dec = [int(rng.integers(65536, 131072 + 1)) for _ in range(64)]
        q, k = [1] * 64 + [2048], dec + [131072]
        return make_workload_from_lengths(name, 32, 8, 128, 16, 1.0 / math.sqrt(128), q, k, seed)
    raise ValueError(f"unknown workload {name!r}")


def bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a bf16 torch tensor (CPU copy)."""
    import torch

    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def _splitmix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser (Steele, Lea, Flood 2014) on uint64 arrays."""
    x = (x + np.uint64(0x9E3779B97F4A7C15)) & np.uint64(0xFFFFFFFFFFFFFFFF)
    x = ((x ^ (x >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)) & np.uint64(0xFFFFFFFFFFFFFFFF)
    x = ((x ^ (x >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)) & np.uint64(0xFFFFFFFFFFFFFFFF)
    return x ^ (x >> np.uint64(31))


def token_values(request_ids, positions, heads: int, dim: int, tag: int):
    """Synthetic per-token rows for serving loops: a bf16 torch tensor
    [n, heads, dim] whose row i depends only on (request_ids[i], positions[i],
    tag) -- so a token recomputed after preemption, or cut into a different
    chunk, gets exactly the same values.  Values: uniform in [-2, 2) from a
    counter-based hash (SplitMix64), rounded to bf16."""
    import torch

    r = np.asarray(request_ids, dtype=np.uint64)[:, None, None]
    p = np.asarray(positions, dtype=np.uint64)[:, None, None]
    h = np.arange(heads, dtype=np.uint64)[None, :, None]
    d = np.arange(dim, dtype=np.uint64)[None, None, :]
    with np.errstate(over="ignore"):
        key = (((r * np.uint64(1000003) + p) * np.uint64(8191) + h) * np.uint64(1021) + d)
        key = key * np.uint64(16) + np.uint64(tag)
        bits = _splitmix64(key)
    u = (bits >> np.uint64(40)).astype(np.float64) / float(1 << 24)  # [0, 1)
    return torch.from_numpy((4.0 * u - 2.0).astype(np.float32)).to(torch.bfloat16)
