"""Binding of the native chunked-prefill scheduler (``mcp_sched_*``).

[W] wangyu.me "大语言模型推理优化（二）：Chunked Prefill", sections "Token 预算：
max_num_batched_tokens", "调度器：running 优先，waiting 填充" and "采样"; [X]
m.xxqk.cn "动态批处理中的抢占与优先级调度" (priority admission, preemption by
recompute or swap).  Each ``schedule()`` returns the step's metadata as numpy
arrays; ``finish_step()`` advances the requests once the step ran.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np

from . import _capi, load


@dataclass
class StepPlan:
    request_ids: np.ndarray     # [S] int64
    cu_seqlens_q: np.ndarray    # [S + 1] int32
    seqlens_k: np.ndarray       # [S] int32
    block_tables: np.ndarray    # [S, max_pages_per_seq] int32
    sample_mask: np.ndarray     # [S] uint8
    logits_indices: np.ndarray  # [num_logits] int32
    swap_out: np.ndarray        # [n, 2] int32: (device page, host page)
    swap_in: np.ndarray         # [n, 2] int32: (host page, device page)
    preempted: np.ndarray       # [n] int64

    @property
    def num_seqs(self) -> int:
        return int(self.request_ids.size)

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q)


def _arr(ptr, n, dtype):
    if n == 0:
        return np.zeros(0, dtype=dtype)
    return np.ctypeslib.as_array(ptr, shape=(n,)).astype(dtype, copy=True)


class Scheduler:
    def __init__(self, max_num_batched_tokens, num_pages, max_pages_per_seq, page_size=16,
                 max_num_seqs=256, long_prefill_token_threshold=0, preempt_swap=False,
                 num_host_pages=0):
        self._lib = load()
        if int(max_num_seqs) > 4096:
            raise ValueError("max_num_seqs above 4096 is not supported by this binding")
        self.max_pages_per_seq = int(max_pages_per_seq)
        cfg = _capi.SchedConfig(int(max_num_batched_tokens), int(long_prefill_token_threshold),
                                int(max_num_seqs), int(num_pages), int(page_size),
                                self.max_pages_per_seq, 1 if preempt_swap else 0,
                                int(num_host_pages), (ctypes.c_int32 * 4)())
        h = ctypes.c_void_p()
        _capi.check(self._lib.mcp_sched_create(ctypes.byref(cfg), ctypes.byref(h)), "sched_create")
        self._h = h

    def add_request(self, request_id, prompt_len, max_new_tokens, priority=0):
        _capi.check(self._lib.mcp_sched_add_request(self._h, int(request_id), int(prompt_len),
                                                    int(max_new_tokens), int(priority)),
                    "sched_add_request")

    def schedule(self) -> StepPlan:
        o = _capi.SchedOutput()
        _capi.check(self._lib.mcp_sched_schedule(self._h, ctypes.byref(o)), "sched_schedule")
        S = o.num_seqs
        mp = self.max_pages_per_seq
        bt = _arr(o.block_tables, S * mp, np.int32).reshape(S, mp)
        so = np.stack([_arr(o.swap_out_device_pages, o.num_swap_out, np.int32),
                       _arr(o.swap_out_host_pages, o.num_swap_out, np.int32)], axis=1)
        si = np.stack([_arr(o.swap_in_host_pages, o.num_swap_in, np.int32),
                       _arr(o.swap_in_device_pages, o.num_swap_in, np.int32)], axis=1)
        return StepPlan(_arr(o.request_ids, S, np.int64),
                        _arr(o.cu_seqlens_q, S + 1, np.int32) if S else np.zeros(1, np.int32),
                        _arr(o.seqlens_k, S, np.int32), bt,
                        _arr(o.sample_mask, S, np.uint8),
                        _arr(o.logits_indices, o.num_logits, np.int32), so, si,
                        _arr(o.preempted_ids, o.num_preempted, np.int64))

    def finish_step(self) -> np.ndarray:
        ids = (ctypes.c_int64 * 4096)()
        n = ctypes.c_int32()
        _capi.check(self._lib.mcp_sched_finish_step(self._h, ctypes.byref(n), ids),
                    "sched_finish_step")
        return np.array(ids[:n.value], dtype=np.int64)

    def stats(self) -> dict:
        w, r, sw, fp = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        f = ctypes.c_int64()
        _capi.check(self._lib.mcp_sched_stats(self._h, ctypes.byref(w), ctypes.byref(r),
                                              ctypes.byref(sw), ctypes.byref(f), ctypes.byref(fp)),
                    "sched_stats")
        return dict(waiting=w.value, running=r.value, swapped=sw.value, finished=f.value,
                    free_pages=fp.value)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.mcp_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
