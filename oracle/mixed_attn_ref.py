"""Plain CPU oracle: one mixed (chunked-prefill + decode) paged-attention step.

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Nothing in the product
imports this module; it imports nothing from the product.

The oracle is the plain definition of what the step computes, written out with
NumPy in float64.  It does not replay any tiling, online softmax or split of the
key range: those are the fast method's ways of reaching the same numbers.

Pages cited (page title, then section):

* [W] wangyu.me, "大语言模型推理优化（二）：Chunked Prefill"
* [L] lpnh.cn, "技术融合剖析：Chunked Prefill如何借助FlashAttention/FlashInfer实现混合批次推理"
* [K] kwkr.cn, the hybrid-batch Chunked Prefill page with the Triton mixed kernel

What each function follows:

* ``segment_layout``  -- [W] "记录 KV Cache 的长度": cu_seqlens_q / cu_seqlens_k
  are exclusive prefix sums of the per-segment query and KV lengths; the KV
  length counts the token(s) computed in this step.
* ``PageTable`` / ``PagedKVStore`` -- [L] section 4.1 (a per-request
  logical-to-physical block table held in a dict) and [K] "混合批次计算图与内存访问
  不对称性" (KV pages scattered across physical memory).
* ``new_token_slots`` / ``append`` -- [W] "输入组装": the new K/V are written into
  the paged cache through slot_mapping before attention runs; [L] section 4.2
  (physical address translation through the block table, scattered writes).
* ``visible_keys`` -- [W] "Flash Attention 的 varlen 接口": the query segment is
  right-aligned to the end of its KV segment, so query i of a segment with Lq
  queries and Lk keys sees keys 0 .. i + (Lk - Lq).
* ``kv_head_of`` -- grouped-query mapping: not on the pages ([K]'s kernel is
  multi-head only).  Reading taken: q head h uses kv head h // (H_q / H_kv),
  which is [K]'s multi-head indexing when H_q == H_kv.
* ``mixed_attention`` -- [W] "Flash Attention 的 varlen 接口": the i-th query
  segment attends only to the i-th KV segment; softmax(q k^T * scale + mask) v.
  The log-sum-exp it also returns is max_j s_ij + ln sum_j exp(s_ij - max).
* ``merge_states`` -- not on the pages; it is the plain identity for combining
  softmax-attention results over disjoint key sets, used by split-KV.

Every function here is pinned by tests/test_oracle_pins.py against something
other than itself (values the pages print, library routines, closed forms,
brute force); none is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# bf16 values: the step's tensors are bf16; the oracle widens them exactly.
# ---------------------------------------------------------------------------


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float values to bf16, nearest-even, returned as uint16 bit patterns.

    Used only to express expected bf16 outputs in tests; NaN maps to the
    canonical quiet NaN 0x7FC0.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    rounded = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return np.where(np.isnan(f), np.uint16(0x7FC0), rounded)


# ---------------------------------------------------------------------------
# Segment layout  ([W] "记录 KV Cache 的长度")
# ---------------------------------------------------------------------------


def segment_layout(q_lens, k_lens):
    """Return (cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k).

    q_lens[s] is the number of tokens segment s computes in this step; k_lens[s]
    is the number of KV positions it sees, history plus this step's tokens.
    """
    cu_q = [0]
    for n in q_lens:
        cu_q.append(cu_q[-1] + int(n))
    cu_k = [0]
    for n in k_lens:
        cu_k.append(cu_k[-1] + int(n))
    max_q = max((int(n) for n in q_lens), default=0)
    max_k = max((int(n) for n in k_lens), default=0)
    return cu_q, cu_k, max_q, max_k


# ---------------------------------------------------------------------------
# Paged KV cache held in dicts  ([L] 4.1, [K] paged-cache diagram)
# ---------------------------------------------------------------------------


class PageTable:
    """Per-sequence logical page -> physical page, kept in a dict."""

    def __init__(self, page_size: int):
        self.page_size = int(page_size)
        self.table: dict[tuple[int, int], int] = {}

    def map(self, seq: int, logical_page: int, physical_page: int) -> None:
        self.table[(int(seq), int(logical_page))] = int(physical_page)

    def physical_page(self, seq: int, pos: int) -> int:
        return self.table[(int(seq), int(pos) // self.page_size)]

    def slot(self, seq: int, pos: int) -> int:
        """Physical slot of KV position ``pos`` of sequence ``seq``:
        physical_page * page_size + (pos mod page_size)."""
        return self.physical_page(seq, pos) * self.page_size + int(pos) % self.page_size


def page_table_from_block_tables(block_tables, seqlens_k, page_size) -> PageTable:
    """Dict page table holding, for each sequence, the pages its KV length uses."""
    pt = PageTable(page_size)
    bt = np.asarray(block_tables)
    for s, lk in enumerate(seqlens_k):
        for p in range(-(-int(lk) // int(page_size))):
            pt.map(s, p, int(bt[s, p]))
    return pt


class PagedKVStore:
    """Physical KV storage: dict (physical_page, offset) -> (k, v) bf16 bits.

    k and v are uint16 arrays of shape [num_kv_heads, head_dim].
    """

    def __init__(self, page_size: int, num_kv_heads: int, head_dim: int):
        self.page_size = int(page_size)
        self.num_kv_heads = int(num_kv_heads)
        self.head_dim = int(head_dim)
        self.cells: dict[tuple[int, int], tuple[np.ndarray, np.ndarray]] = {}

    def write_slot(self, slot: int, k_bits, v_bits) -> None:
        key = (int(slot) // self.page_size, int(slot) % self.page_size)
        self.cells[key] = (np.array(k_bits, dtype=np.uint16), np.array(v_bits, dtype=np.uint16))

    def read(self, table: PageTable, seq: int, pos: int):
        slot = table.slot(seq, pos)
        return self.cells[(slot // self.page_size, slot % self.page_size)]

    def gather(self, table: PageTable, seq: int, length: int):
        """K, V of positions 0..length-1 of ``seq`` as float64 [length, H_kv, D]."""
        K = np.empty((length, self.num_kv_heads, self.head_dim), dtype=np.float64)
        V = np.empty_like(K)
        for pos in range(length):
            kb, vb = self.read(table, seq, pos)
            K[pos] = bf16_bits_to_f64(kb)
            V[pos] = bf16_bits_to_f64(vb)
        return K, V

    def materialize(self, num_pages: int, fill_bits: int = 0x7FC0):
        """Dense caches [num_pages, page_size, H_kv, D] of bf16 bits; cells never
        written hold ``fill_bits``."""
        shape = (int(num_pages), self.page_size, self.num_kv_heads, self.head_dim)
        kc = np.full(shape, fill_bits, dtype=np.uint16)
        vc = np.full(shape, fill_bits, dtype=np.uint16)
        for (page, off), (kb, vb) in self.cells.items():
            kc[page, off] = kb
            vc[page, off] = vb
        return kc, vc


def new_token_slots(table: PageTable, cu_seqlens_q, seqlens_k) -> np.ndarray:
    """slot_mapping for this step's tokens ([W] "输入组装").

    The tokens of segment s are its last Lq positions: token t sits at position
    (Lk - Lq) + (t - cu_seqlens_q[s]).
    """
    cu = [int(x) for x in cu_seqlens_q]
    out = np.empty(cu[-1], dtype=np.int64)
    for s in range(len(cu) - 1):
        lq = cu[s + 1] - cu[s]
        hist = int(seqlens_k[s]) - lq
        for t in range(cu[s], cu[s + 1]):
            out[t] = table.slot(s, hist + (t - cu[s]))
    return out


def append(store: PagedKVStore, slot_mapping, k_new_bits, v_new_bits) -> None:
    """Write each new token's K/V into its slot; a negative slot is skipped
    ([W] "输入组装"; [L] 4.2)."""
    for t, slot in enumerate(np.asarray(slot_mapping)):
        if int(slot) >= 0:
            store.write_slot(int(slot), k_new_bits[t], v_new_bits[t])


# ---------------------------------------------------------------------------
# Attention  ([W] "Flash Attention 的 varlen 接口")
# ---------------------------------------------------------------------------


def visible_keys(i: int, q_len: int, k_len: int) -> int:
    """Number of keys query i (0-based within its segment) sees: positions
    0 .. i + (k_len - q_len), i.e. the whole history plus chunk tokens <= i."""
    return int(i) + (int(k_len) - int(q_len)) + 1


def kv_head_of(h: int, num_q_heads: int, num_kv_heads: int) -> int:
    """kv head used by q head h: contiguous groups of H_q / H_kv q heads."""
    return int(h) // (int(num_q_heads) // int(num_kv_heads))


def mixed_attention(q, store: PagedKVStore, table: PageTable, cu_seqlens_q, seqlens_k,
                    num_kv_heads: int, sm_scale: float, tokens=None, row_block: int = 256):
    """Attention of every query token of the step against its own segment's keys.

    q: float [T, H_q, D].  Returns (out [T, H_q, D], lse [T, H_q]) in float64;
    lse is natural-log.  ``tokens`` (optional iterable of stream indices) limits
    the work to those rows; the other rows are NaN.
    """
    q = np.asarray(q, dtype=np.float64)
    T, H_q, D = q.shape
    out = np.full((T, H_q, D), np.nan)
    lse = np.full((T, H_q), np.nan)
    cu = [int(x) for x in cu_seqlens_q]
    want = None if tokens is None else np.zeros(T, dtype=bool)
    if want is not None:
        want[np.asarray(list(tokens), dtype=np.int64)] = True
    for s in range(len(cu) - 1):
        lq = cu[s + 1] - cu[s]
        lk = int(seqlens_k[s])
        if lq == 0:
            continue
        local = np.arange(lq)
        if want is not None:
            local = local[want[cu[s]:cu[s + 1]]]
            if local.size == 0:
                continue
        K, V = store.gather(table, s, lk)
        n_vis = np.array([visible_keys(i, lq, lk) for i in local])
        cols = np.arange(lk)
        for h in range(H_q):
            g = kv_head_of(h, H_q, num_kv_heads)
            Kg, Vg = K[:, g, :], V[:, g, :]
            for b0 in range(0, local.size, row_block):
                li = local[b0:b0 + row_block]
                nv = n_vis[b0:b0 + row_block]
                S = (q[cu[s] + li, h, :] @ Kg.T) * sm_scale
                S[cols[None, :] >= nv[:, None]] = -np.inf
                m = S.max(axis=1)
                E = np.exp(S - m[:, None])
                l = E.sum(axis=1)
                out[cu[s] + li, h, :] = (E @ Vg) / l[:, None]
                lse[cu[s] + li, h] = m + np.log(l)
    return out, lse


def merge_states(o_parts, lse_parts):
    """Combine attention results over disjoint key sets.

    o_parts [n, ..., D] are each normalised by their own softmax sum; lse_parts
    [n, ...] their natural-log sums.  With M = max_k lse_k and w_k = exp(lse_k - M):
    O = sum_k w_k O_k / sum_k w_k and LSE = M + ln sum_k w_k.  A part with
    lse = -inf (no keys) has weight 0.
    """
    o = np.asarray(o_parts, dtype=np.float64)
    lse = np.asarray(lse_parts, dtype=np.float64)
    M = lse.max(axis=0)
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    w = np.where(np.isfinite(lse), np.exp(lse - Ms[None]), 0.0)
    wsum = w.sum(axis=0)
    num = (w[..., None] * np.where(np.isfinite(lse)[..., None], o, 0.0)).sum(axis=0)
    safe = np.where(wsum > 0, wsum, 1.0)
    O = np.where((wsum > 0)[..., None], num / safe[..., None], 0.0)
    L = np.where(wsum > 0, Ms + np.log(safe), -math.inf)
    return O, L
