"""Test-side glue: runs the oracle on a synthetic workload.

Test infrastructure: imports the oracle; the product never imports this file.
"""

from __future__ import annotations

import numpy as np

import oracle
import synth


class OracleStep:
    """The oracle's view of one step of a workload.

    History positions 0..Lk-Lq-1 of every segment are written first, as if an
    earlier step had appended them (segments with Lq = Lk = history length);
    then this step's tokens are appended and attention runs.
    """

    def __init__(self, w: synth.Workload, tensors: dict, fill_bits: int = 0x7FC0):
        self.w = w
        self.bt = w.block_tables()
        self.cu_q, self.cu_k, self.max_q, self.max_k = oracle.segment_layout(w.q_lens, w.k_lens)
        self.table = oracle.page_table_from_block_tables(self.bt, w.k_lens, w.page_size)
        self.store = oracle.PagedKVStore(w.page_size, w.num_kv_heads, w.head_dim)
        hist = w.hist_lens
        cu_h, _, _, _ = oracle.segment_layout(hist, hist)
        self.hist_slots = oracle.new_token_slots(self.table, cu_h, hist)
        if "k_hist" in tensors:
            oracle.append(self.store, self.hist_slots, synth.bf16_bits(tensors["k_hist"]),
                          synth.bf16_bits(tensors["v_hist"]))
        self.fill_bits = fill_bits
        self.slots = oracle.new_token_slots(self.table, self.cu_q, w.k_lens)
        self.q = oracle.bf16_bits_to_f64(synth.bf16_bits(tensors["q"]))
        self.k_new_bits = synth.bf16_bits(tensors["k_new"])
        self.v_new_bits = synth.bf16_bits(tensors["v_new"])
        self.appended = False

    def cache_bits(self):
        return self.store.materialize(self.w.num_pages, self.fill_bits)

    def do_append(self):
        oracle.append(self.store, self.slots, self.k_new_bits, self.v_new_bits)
        self.appended = True

    def attention(self, tokens=None):
        assert self.appended
        return oracle.mixed_attention(self.q, self.store, self.table, self.cu_q, self.w.k_lens,
                                      self.w.num_kv_heads, self.w.sm_scale, tokens=tokens)


def rel_rms(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.sqrt(np.mean(b * b))
    return float(np.sqrt(np.mean((a - b) ** 2)) / max(den, 1e-30))
