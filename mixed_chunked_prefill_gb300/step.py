"""Step runners over the C ABI: the calls one layer of a chunked-prefill
serving step makes ([W] wangyu.me "大语言模型推理优化（二）：Chunked Prefill",
section "输入组装": write the new K/V through slot_mapping, then run the varlen
paged attention).

``MixedStep`` keeps one step's metadata, plan and workspace on the device and
runs append + attention on device tensors.  ``HostStep`` is the end-to-end
path from host buffers over the library's pipelined host step: each call
copies the step's inputs and metadata to the device, plans on the host,
appends, attends and copies the output back, with up to two steps in flight
(the copies of one step overlap the kernels of the other).
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
    mixed_attn_plan_rows,
    paged_kv_append,
    workspace_error_word,
)


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


class MixedStep:
    """Device-side state of one step: metadata, slot mapping, plan, workspace."""

    def __init__(self, num_q_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale,
                 cu_seqlens_q, seqlens_k, block_tables, device="cuda", options=None,
                 stream=None, rows=None):
        """``rows``: None for every query row, else the token indices (e.g.
        logits_indices) whose attention rows this step computes."""
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
        if rows is None:
            def planner(ws=None, st=None):
                return mixed_attn_plan(self.desc, self.cu_h, self.sk_h, options, ws, st)
        else:
            self.rows_h = _i32(rows)

            def planner(ws=None, st=None):
                return mixed_attn_plan_rows(self.desc, self.cu_h, self.sk_h, self.rows_h,
                                            options, ws, st)
        sizing = planner()
        self.workspace = torch.empty(max(256, int(sizing.workspace_bytes)), dtype=torch.uint8,
                                     device=device)
        self.plan = planner(self.workspace, stream)
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
    """End-to-end steps from host memory (``mcp_host_step_*``).

    ``run`` enqueues one step and returns its ticket without waiting: the
    copy-in of q, k_new, v_new (page-locked host tensors, left unchanged until
    the step is waited for), host planning, append, attention and the
    copy-out into ``out_h`` (and ``lse_h``).  ``wait(ticket)`` blocks until
    that step's outputs are in host memory and raises on a device-side error.
    Calling the object runs one step and waits for it.  The device and
    page-locked arenas are torch tensors owned by this object; the KV cache
    is the caller's device state.
    """

    def __init__(self, num_q_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale,
                 max_tokens, max_seqs, max_pages_per_seq, device="cuda", stream=None,
                 workspace_bytes=0, list_bytes=0):
        import ctypes

        import torch

        from . import _capi, load

        self._lib = load()
        self.hq, self.hkv, self.D, self.P = num_q_heads, num_kv_heads, head_dim, page_size
        self.mp = int(max_pages_per_seq)
        self.stream = stream if stream is not None else torch.cuda.current_stream(device)
        shape = make_desc(0, 0, num_q_heads, num_kv_heads, head_dim, page_size, 1, num_pages,
                          sm_scale)
        lim = _capi.HostStepLimits(int(max_tokens), int(max_seqs), self.mp, 0,
                                   int(workspace_bytes), int(list_bytes), (ctypes.c_int32 * 4)())
        dbytes, hbytes = ctypes.c_size_t(), ctypes.c_size_t()
        _capi.check(self._lib.mcp_host_step_arena_bytes(ctypes.byref(shape), ctypes.byref(lim),
                                                        ctypes.byref(dbytes), ctypes.byref(hbytes)),
                    "host_step_arena_bytes")
        # arenas: torch's device and page-locked allocations are 256-byte aligned
        self.device_arena = torch.empty(dbytes.value, dtype=torch.uint8, device=device)
        self.host_arena = torch.empty(hbytes.value, dtype=torch.uint8, pin_memory=True)
        handle = ctypes.c_void_p()
        _capi.check(self._lib.mcp_host_step_create(
            ctypes.byref(shape), ctypes.byref(lim), ctypes.c_void_p(self.device_arena.data_ptr()),
            dbytes.value, ctypes.c_void_p(self.host_arena.data_ptr()), hbytes.value,
            ctypes.c_void_p(self.stream.cuda_stream), ctypes.byref(handle)), "host_step_create")
        self._h = handle
        self._keep = {}  # host arrays a ticket's copies still read / write
        self.h2d_bytes = 0
        self.d2h_bytes = 0

    def run(self, q_h, k_new_h, v_new_h, cu_seqlens_q, seqlens_k, block_tables, k_cache,
            v_cache, out_h, lse_h=None) -> int:
        import ctypes

        import torch

        from . import _capi

        cu = _i32(cu_seqlens_q)
        sk = _i32(seqlens_k)
        bt = _i32(block_tables)
        S = len(sk)
        if bt.ndim != 2 or bt.shape[0] != S or bt.shape[1] > self.mp:
            raise ValueError(f"block_tables must be [S, <= {self.mp}]")
        if bt.shape[1] < self.mp:
            full = np.full((S, self.mp), -1, dtype=np.int32)
            full[:, :bt.shape[1]] = bt
            bt = full
        T = int(cu[-1]) if len(cu) else 0
        for t, name, dt in ((q_h, "q", torch.bfloat16), (k_new_h, "k_new", torch.bfloat16),
                            (v_new_h, "v_new", torch.bfloat16), (out_h, "out", torch.bfloat16)):
            if t.is_cuda or t.dtype != dt or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous host {dt} tensor")
        if lse_h is not None and (lse_h.is_cuda or lse_h.dtype != torch.float32):
            raise ValueError("lse must be a host float32 tensor")
        if q_h.numel() < T * self.hq * self.D or out_h.numel() < T * self.hq * self.D:
            raise ValueError("q / out smaller than [T, H_q, D]")
        if k_new_h.numel() < T * self.hkv * self.D or v_new_h.numel() < T * self.hkv * self.D:
            raise ValueError("k_new / v_new smaller than [T, H_kv, D]")
        ticket = ctypes.c_int64(-1)
        st = self._lib.mcp_host_step_run(
            self._h, S, cu.ctypes.data_as(ctypes.c_void_p), sk.ctypes.data_as(ctypes.c_void_p),
            bt.ctypes.data_as(ctypes.c_void_p), ctypes.c_void_p(q_h.data_ptr()),
            ctypes.c_void_p(k_new_h.data_ptr()), ctypes.c_void_p(v_new_h.data_ptr()),
            ctypes.c_void_p(k_cache.data_ptr()), ctypes.c_void_p(v_cache.data_ptr()),
            ctypes.c_void_p(out_h.data_ptr()),
            ctypes.c_void_p(lse_h.data_ptr()) if lse_h is not None else None, ctypes.byref(ticket))
        _capi.check(st, "host_step_run")
        t = int(ticket.value)
        self._keep[t] = (q_h, k_new_h, v_new_h, out_h, lse_h)
        for old in [k for k in self._keep if k < t - 1]:
            del self._keep[old]  # slot reused: that step has finished
        self.h2d_bytes = (cu.nbytes + sk.nbytes + bt.nbytes + T * 8
                          + 2 * T * (self.hq + 2 * self.hkv) * self.D)
        self.d2h_bytes = 2 * T * self.hq * self.D + (4 * T * self.hq if lse_h is not None else 0)
        return t

    def wait(self, ticket: int):
        from . import _capi

        _capi.check(self._lib.mcp_host_step_wait(self._h, int(ticket)), "host_step_wait")
        self._keep.pop(int(ticket), None)

    def __call__(self, q_h, k_new_h, v_new_h, cu_seqlens_q, seqlens_k, block_tables, k_cache,
                 v_cache, out_h, lse_h=None):
        self.wait(self.run(q_h, k_new_h, v_new_h, cu_seqlens_q, seqlens_k, block_tables,
                           k_cache, v_cache, out_h, lse_h))
        return out_h

    def close(self):
        from . import _capi

        if getattr(self, "_h", None) is not None and self._h.value:
            h, self._h = self._h, None
            _capi.check(self._lib.mcp_host_step_destroy(h), "host_step_destroy")
            self._keep.clear()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
