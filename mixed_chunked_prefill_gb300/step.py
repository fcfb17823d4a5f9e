"""Step runners over the C ABI: the calls one layer of a chunked-prefill
serving step makes ([W] wangyu.me "大语言模型推理优化（二）：Chunked Prefill",
section "输入组装": write the new K/V through slot_mapping, then run the varlen
paged attention).

``MixedStep`` keeps one step's metadata, plan and workspace on the device and
runs append + attention on device tensors.  ``HostStep`` is the end-to-end
path from host buffers: it copies the step's inputs and metadata to the
device, plans, runs, and copies the output back, all on one stream.
"""

from __future__ import annotations

import numpy as np

from . import (
    PlanOptions,
    build_slot_mapping,
    check_device_errors,
    make_desc,
    mixed_attn_fwd,
    mixed_attn_plan,
    paged_kv_append,
    workspace_error_word,
)


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


class MixedStep:
    """Device-side state of one step: metadata, slot mapping, plan, workspace."""

    def __init__(self, num_q_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale,
                 cu_seqlens_q, seqlens_k, block_tables, device="cuda", options=None,
                 stream=None):
        import torch

        self.cu_h = _i32(cu_seqlens_q)
        self.sk_h = _i32(seqlens_k)
        self.bt_h = _i32(block_tables)
        if self.bt_h.ndim != 2:
            raise ValueError("block_tables must be [num_seqs, max_pages_per_seq]")
        S = len(self.sk_h)
        self.desc = make_desc(S, int(self.cu_h[-1]), num_q_heads, num_kv_heads, head_dim,
                              page_size, self.bt_h.shape[1], num_pages, sm_scale)
        self.options = options
        self.stream = stream
        self.device = device
        self.slots_h = build_slot_mapping(self.bt_h, self.cu_h, self.sk_h, page_size, num_pages)
        self.cu_d = torch.from_numpy(self.cu_h).to(device)
        self.sk_d = torch.from_numpy(self.sk_h).to(device)
        self.bt_d = torch.from_numpy(self.bt_h).to(device)
        self.slots_d = torch.from_numpy(self.slots_h).to(device)
        sizing = mixed_attn_plan(self.desc, self.cu_h, self.sk_h, options)
        self.workspace = torch.empty(max(256, int(sizing.workspace_bytes)), dtype=torch.uint8,
                                     device=device)
        self.plan = mixed_attn_plan(self.desc, self.cu_h, self.sk_h, options, self.workspace,
                                    stream)
        self.error_word = workspace_error_word(self.plan, self.workspace)

    def append(self, k_new, v_new, k_cache, v_cache):
        paged_kv_append(k_new, v_new, self.slots_d, k_cache, v_cache, self.error_word,
                        self.stream)

    def attention(self, q, k_cache, v_cache, out, lse=None):
        mixed_attn_fwd(self.plan, q, k_cache, v_cache, self.bt_d, self.cu_d, self.sk_d, out, lse,
                       self.workspace, self.stream)

    def run(self, q, k_new, v_new, k_cache, v_cache, out, lse=None):
        self.append(k_new, v_new, k_cache, v_cache)
        self.attention(q, k_cache, v_cache, out, lse)

    def check(self):
        """Synchronise and raise if a device-side check or bounded wait failed."""
        check_device_errors(self.error_word, self.stream)


def write_history(block_tables, hist_lens, k_hist, v_hist, k_cache, v_cache, page_size,
                  stream=None):
    """Fill positions 0..hist_lens[s]-1 of every sequence from packed k_hist /
    v_hist [sum(hist_lens), H_kv, D] (device bf16), through the same slot
    mapping and append kernel a step uses."""
    import torch

    hist = _i32(hist_lens)
    cu = np.concatenate([[0], np.cumsum(hist)]).astype(np.int32)
    if int(cu[-1]) == 0:
        return
    slots = build_slot_mapping(block_tables, cu, hist, page_size, int(k_cache.shape[0]))
    paged_kv_append(k_hist, v_hist, torch.from_numpy(slots).to(k_cache.device), k_cache, v_cache,
                    stream=stream)


class HostStep:
    """End-to-end step from host memory.

    Per call: host->device copies of q, k_new, v_new and the metadata (block
    tables, cu_seqlens_q, seqlens_k, slot mapping) from pinned buffers; host
    planning and plan upload; append; attention; device->host copy of the
    output into a pinned buffer.  The KV cache is device-resident state.
    """

    def __init__(self, num_q_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale,
                 max_tokens, max_seqs, max_pages_per_seq, device="cuda", options=None,
                 stream=None, workspace_bytes=1 << 26):
        import torch

        self.hq, self.hkv, self.D, self.P = num_q_heads, num_kv_heads, head_dim, page_size
        self.num_pages, self.scale = num_pages, sm_scale
        self.options = options
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        dev = device
        self.q_d = torch.empty((max_tokens, num_q_heads, head_dim), dtype=torch.bfloat16, device=dev)
        self.k_d = torch.empty((max_tokens, num_kv_heads, head_dim), dtype=torch.bfloat16, device=dev)
        self.v_d = torch.empty_like(self.k_d)
        self.out_d = torch.empty_like(self.q_d)
        self.cu_d = torch.empty(max_seqs + 1, dtype=torch.int32, device=dev)
        self.sk_d = torch.empty(max_seqs, dtype=torch.int32, device=dev)
        self.bt_d = torch.empty((max_seqs, max_pages_per_seq), dtype=torch.int32, device=dev)
        self.slots_d = torch.empty(max_tokens, dtype=torch.int64, device=dev)
        self.meta_h = torch.empty(max_seqs * (max_pages_per_seq + 2) + 1, dtype=torch.int32,
                                  pin_memory=True)
        self.slots_h = torch.empty(max_tokens, dtype=torch.int64, pin_memory=True)
        self.workspace = torch.empty(workspace_bytes, dtype=torch.uint8, device=dev)
        self.h2d_bytes = 0
        self.d2h_bytes = 0

    def __call__(self, q_h, k_new_h, v_new_h, cu_seqlens_q, seqlens_k, block_tables, k_cache,
                 v_cache, out_h):
        """q_h / k_new_h / v_new_h / out_h: pinned host bf16 tensors; metadata:
        host int arrays.  Returns out_h after the device->host copy finished."""
        import torch

        cu = _i32(cu_seqlens_q)
        sk = _i32(seqlens_k)
        bt = _i32(block_tables)
        S, T = len(sk), int(cu[-1])
        mp = bt.shape[1]
        slots = build_slot_mapping(bt, cu, sk, self.P, self.num_pages)
        desc = make_desc(S, T, self.hq, self.hkv, self.D, self.P, mp, self.num_pages, self.scale)
        plan = mixed_attn_plan(desc, cu, sk, self.options)
        if plan.workspace_bytes > self.workspace.numel():
            self.workspace = torch.empty(int(plan.workspace_bytes), dtype=torch.uint8,
                                         device=self.workspace.device)
        # pack metadata into one pinned buffer -> one copy
        n_meta = (S + 1) + S + S * mp
        meta = self.meta_h[:n_meta].numpy()
        meta[:S + 1] = cu
        meta[S + 1:2 * S + 1] = sk
        meta[2 * S + 1:] = bt.reshape(-1)
        self.slots_h[:T].numpy()[:] = slots
        s = self.stream
        with torch.cuda.stream(s):
            meta_d = torch.empty(n_meta, dtype=torch.int32, device=self.cu_d.device)
            meta_d.copy_(self.meta_h[:n_meta], non_blocking=True)
            cu_d = meta_d[:S + 1]
            sk_d = meta_d[S + 1:2 * S + 1]
            bt_d = meta_d[2 * S + 1:].view(S, mp)
            slots_d = self.slots_d[:T]
            slots_d.copy_(self.slots_h[:T], non_blocking=True)
            q_d = self.q_d[:T]
            k_d = self.k_d[:T]
            v_d = self.v_d[:T]
            q_d.copy_(q_h, non_blocking=True)
            k_d.copy_(k_new_h, non_blocking=True)
            v_d.copy_(v_new_h, non_blocking=True)
            plan = mixed_attn_plan(desc, cu, sk, self.options, self.workspace, s)
            paged_kv_append(k_d, v_d, slots_d, k_cache, v_cache, stream=s)
            out_d = self.out_d[:T]
            mixed_attn_fwd(plan, q_d, k_cache, v_cache, bt_d, cu_d, sk_d, out_d, None,
                           self.workspace, s)
            out_h.copy_(out_d, non_blocking=True)
        self.h2d_bytes = (n_meta * 4 + T * 8 + q_h.numel() * 2 + k_new_h.numel() * 2
                          + v_new_h.numel() * 2)
        self.d2h_bytes = out_h.numel() * 2
        return out_h
