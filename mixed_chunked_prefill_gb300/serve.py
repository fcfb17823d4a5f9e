"""Multi-step serving loop over the library: the step builder (``Scheduler``)
decides each step, preempted sequences' pages are swapped with
``kv_copy_pages``, and the pipelined ``HostStep`` appends and attends.

[W] wangyu.me "大语言模型推理优化（二）：Chunked Prefill", sections "调度器：running
优先，waiting 填充" and "输入组装": every step the scheduler's batch is assembled
into the varlen metadata, the new K/V are written through the slot mapping and
the paged attention runs; [X] m.xxqk.cn "动态批处理中的抢占与优先级调度": swap-out
to host memory and swap-in when memory is free again.  The caller supplies the
step's per-token q / k_new / v_new (the model's projections); the loop owns the
paged KV pools.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import kv_copy_pages
from .sched import Scheduler, StepPlan
from .step import HostStep


@dataclass
class StepResult:
    plan: StepPlan
    ticket: int
    out: object        # page-locked host bf16 [T, H_q, D]
    lse: object        # page-locked host float32 [T, H_q]
    finished: np.ndarray
    _keep: tuple = ()  # index tensors the step's swap copies read


class ServeLoop:
    def __init__(self, num_q_heads, num_kv_heads, head_dim, num_pages, sm_scale,
                 max_num_batched_tokens, max_pages_per_seq, max_num_seqs=256,
                 long_prefill_token_threshold=0, preempt_swap=False, num_host_pages=0,
                 page_size=16, device="cuda", stream=None):
        import torch

        self.hq, self.hkv, self.D, self.P = num_q_heads, num_kv_heads, head_dim, page_size
        self.device = torch.device(device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.sched = Scheduler(max_num_batched_tokens, num_pages, max_pages_per_seq, page_size,
                               max_num_seqs, long_prefill_token_threshold, preempt_swap,
                               num_host_pages)
        shape = (num_pages, page_size, num_kv_heads, head_dim)
        self.k_cache = torch.zeros(shape, dtype=torch.bfloat16, device=self.device)
        self.v_cache = torch.zeros_like(self.k_cache)
        if preempt_swap and num_host_pages > 0:
            hshape = (num_host_pages, page_size, num_kv_heads, head_dim)
            self.host_k = torch.zeros(hshape, dtype=torch.bfloat16).pin_memory()
            self.host_v = torch.zeros(hshape, dtype=torch.bfloat16).pin_memory()
        self.hs = HostStep(num_q_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale,
                           max_tokens=max_num_batched_tokens, max_seqs=max_num_seqs,
                           max_pages_per_seq=max_pages_per_seq, device=self.device,
                           stream=self.stream)

    def add_request(self, request_id, prompt_len, max_new_tokens, priority=0):
        self.sched.add_request(request_id, prompt_len, max_new_tokens, priority)

    def positions(self, plan: StepPlan) -> tuple:
        """(request id, position) of every token of the step, in stream order."""
        rid = np.repeat(plan.request_ids, plan.q_lens)
        pos = np.concatenate([np.arange(k - q, k) for q, k in zip(plan.q_lens, plan.seqlens_k)]) \
            if plan.num_seqs else np.zeros(0, dtype=np.int64)
        return rid, pos

    def step(self, token_fn):
        """Schedule and enqueue one step; ``token_fn(plan)`` returns page-locked
        (q [T, H_q, D], k_new [T, H_kv, D], v_new [T, H_kv, D]) bf16.  Returns a
        StepResult (outputs valid after ``wait``), or None if nothing is runnable."""
        import torch

        plan = self.sched.schedule()
        keep = []
        with torch.cuda.stream(self.stream):
            if len(plan.swap_out):
                src = torch.from_numpy(plan.swap_out[:, 0].copy()).pin_memory()
                dst = torch.from_numpy(plan.swap_out[:, 1].copy()).pin_memory()
                kv_copy_pages(self.k_cache, self.v_cache, self.host_k, self.host_v, src, dst,
                              stream=self.stream)
                keep += [src, dst]
            if len(plan.swap_in):
                src = torch.from_numpy(plan.swap_in[:, 0].copy()).pin_memory()
                dst = torch.from_numpy(plan.swap_in[:, 1].copy()).pin_memory()
                kv_copy_pages(self.host_k, self.host_v, self.k_cache, self.v_cache, src, dst,
                              stream=self.stream)
                keep += [src, dst]
        if plan.num_seqs == 0:
            self.sched.finish_step()
            return None
        q, k, v = token_fn(plan)
        T = plan.total_q
        out = torch.empty((T, self.hq, self.D), dtype=torch.bfloat16).pin_memory()
        lse = torch.empty((T, self.hq), dtype=torch.float32).pin_memory()
        ticket = self.hs.run(q, k, v, plan.cu_seqlens_q, plan.seqlens_k, plan.block_tables,
                             self.k_cache, self.v_cache, out, lse)
        finished = self.sched.finish_step()
        return StepResult(plan, ticket, out, lse, finished, tuple(keep) + (q, k, v))

    def wait(self, result: StepResult):
        self.hs.wait(result.ticket)

    def close(self):
        self.hs.close()
        self.sched.close()
