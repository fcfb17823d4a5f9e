"""Mixed chunked-prefill + decode paged attention for GB300 (sm_103a).

Python binding of the C ABI in ``include/mcp.h``.  The functions here only
check and marshal arguments (torch tensors -> device pointers, the current
CUDA stream); every step of the computation runs in the library's CUDA
kernels.  If the library is not built, every call raises: there is no CPU or
PyTorch fallback.
"""

from __future__ import annotations

import ctypes

import numpy as np

from . import _capi
from ._capi import (  # noqa: F401
    DEVERR_ITEM_KIND,
    DEVERR_PAGE_RANGE,
    DEVERR_ROW_RANGE,
    DEVERR_SLOT_DUP,
    DEVERR_SLOT_RANGE,
    DEVERR_TIMEOUT,
    AttnDesc,
    MCPError,
    Plan,
    PlanOptions,
)

__all__ = [
    "AttnDesc", "Plan", "PlanOptions", "MCPError", "load", "abi_version", "paged_kv_append",
    "build_slot_mapping", "mixed_attn_plan", "mixed_attn_fwd", "check_device_errors",
    "workspace_error_word", "merge_states", "make_desc", "mixed_attn_fwd_noalloc",
    "mixed_attn_plan_rows", "build_logits_indices", "gather_rows", "kv_copy_pages",
    "mixed_attn_varlen",
]


def load():
    return _capi.load()


def abi_version() -> int:
    return int(load().mcp_abi_version())


def _stream(stream):
    import torch

    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if hasattr(stream, "cuda_stream"):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t, dtype, name):
    import torch

    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _host_i32(a, name):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.ctypes.data_as(ctypes.c_void_p)


def make_desc(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, page_size,
              max_pages_per_seq, num_pages, sm_scale) -> AttnDesc:
    return AttnDesc(int(num_seqs), int(total_q), int(num_q_heads), int(num_kv_heads),
                    int(head_dim), int(page_size), int(max_pages_per_seq), int(num_pages),
                    float(sm_scale))


def paged_kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, error_word=None, stream=None):
    """Scatter k_new/v_new [T, H_kv, D] (bf16) into the paged caches
    [num_pages, P, H_kv, D] at slot_mapping [T] (int64; < 0 skips).
    ``error_word``: None, an int32 CUDA tensor, or a device address."""
    import torch

    lib = load()
    T = int(k_new.shape[0]) if k_new.dim() > 0 else 0
    num_pages, P, Hkv, D = (int(x) for x in k_cache.shape)
    if tuple(k_new.shape) != (T, Hkv, D) or tuple(v_new.shape) != (T, Hkv, D):
        raise ValueError("k_new / v_new must be [T, H_kv, D] matching the cache")
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache shapes differ")
    if tuple(slot_mapping.shape) != (T,):
        raise ValueError("slot_mapping must be [T]")
    if error_word is None or isinstance(error_word, torch.Tensor):
        ew = _dev(error_word, torch.int32, "error_word")
    else:  # a device address, e.g. workspace_error_word(plan, workspace)
        ew = ctypes.c_void_p(int(error_word))
    st = lib.mcp_paged_kv_append(
        _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
        _dev(slot_mapping, torch.int64, "slot_mapping"), T, Hkv, D, P, num_pages,
        _dev(k_cache, torch.bfloat16, "k_cache"), _dev(v_cache, torch.bfloat16, "v_cache"),
        ew, _stream(stream))
    _capi.check(st, "paged_kv_append")


def build_slot_mapping(block_tables, cu_seqlens_q, seqlens_k, page_size, num_pages) -> np.ndarray:
    """Host-side slot mapping of the step's new tokens (int64 numpy array)."""
    lib = load()
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    S = bt.shape[0]
    cu, cu_p = _host_i32(cu_seqlens_q, "cu_seqlens_q")
    sk, sk_p = _host_i32(seqlens_k, "seqlens_k")
    out = np.empty(int(cu[-1]), dtype=np.int64)
    st = lib.mcp_build_slot_mapping(bt.ctypes.data_as(ctypes.c_void_p), S,
                                    bt.shape[1] if bt.ndim == 2 else 0, int(page_size),
                                    int(num_pages), cu_p, sk_p,
                                    out.ctypes.data_as(ctypes.c_void_p))
    _capi.check(st, "build_slot_mapping")
    return out


def mixed_attn_plan(desc: AttnDesc, cu_seqlens_q, seqlens_k, options: PlanOptions | None = None,
                    workspace=None, stream=None) -> Plan:
    """Plan a step from HOST metadata; with ``workspace`` (uint8 CUDA tensor)
    also copy the work lists into it."""
    import torch

    lib = load()
    cu, cu_p = _host_i32(cu_seqlens_q, "cu_seqlens_q")
    sk, sk_p = _host_i32(seqlens_k, "seqlens_k")
    plan = Plan()
    ws = _dev(workspace, torch.uint8, "workspace") if workspace is not None else None
    nbytes = int(workspace.numel()) if workspace is not None else 0
    st = lib.mcp_mixed_attn_plan(ctypes.byref(desc), cu_p, sk_p,
                                 ctypes.byref(options) if options is not None else None,
                                 ctypes.byref(plan), ws, nbytes,
                                 _stream(stream) if workspace is not None else None)
    _capi.check(st, "mixed_attn_plan")
    return plan


def mixed_attn_plan_rows(desc: AttnDesc, cu_seqlens_q, seqlens_k, rows,
                         options: PlanOptions | None = None, workspace=None,
                         stream=None) -> Plan:
    """Plan attention for the listed query rows only (HOST token indices,
    strictly increasing); with ``workspace`` also copy the work lists into it."""
    import torch

    lib = load()
    cu, cu_p = _host_i32(cu_seqlens_q, "cu_seqlens_q")
    sk, sk_p = _host_i32(seqlens_k, "seqlens_k")
    rw, rw_p = _host_i32(rows, "rows")
    plan = Plan()
    ws = _dev(workspace, torch.uint8, "workspace") if workspace is not None else None
    nbytes = int(workspace.numel()) if workspace is not None else 0
    st = lib.mcp_mixed_attn_plan_rows(ctypes.byref(desc), cu_p, sk_p, rw_p, int(rw.size),
                                      ctypes.byref(options) if options is not None else None,
                                      ctypes.byref(plan), ws, nbytes,
                                      _stream(stream) if workspace is not None else None)
    _capi.check(st, "mixed_attn_plan_rows")
    return plan


def build_logits_indices(cu_seqlens_q, sample_mask=None) -> np.ndarray:
    """The last token of every segment with a token this step (optionally only
    segments with a non-zero ``sample_mask``): int32 numpy array."""
    lib = load()
    cu, cu_p = _host_i32(cu_seqlens_q, "cu_seqlens_q")
    S = int(cu.size) - 1
    out = np.empty(max(S, 1), dtype=np.int32)
    count = ctypes.c_int32()
    mask_p = None
    if sample_mask is not None:
        m = np.ascontiguousarray(np.asarray(sample_mask, dtype=np.uint8))
        if m.size != S:
            raise ValueError("sample_mask must have one entry per segment")
        mask_p = m.ctypes.data_as(ctypes.c_void_p)
    st = lib.mcp_build_logits_indices(S, cu_p, mask_p, out.ctypes.data_as(ctypes.c_void_p),
                                      ctypes.byref(count))
    _capi.check(st, "build_logits_indices")
    return out[:count.value].copy()


def kv_copy_pages(k_src, v_src, k_dst, v_dst, src_pages, dst_pages, error_word=None,
                  stream=None) -> None:
    """Copy whole KV pages between two pools ([pages, P, H_kv, D] bf16 tensors,
    device or page-locked host): dst[dst_pages[i]] = src[src_pages[i]].
    ``src_pages`` / ``dst_pages``: int32 tensors on the device (or pinned)."""
    import torch

    lib = load()
    n = int(src_pages.numel())
    if int(dst_pages.numel()) != n:
        raise ValueError("src_pages and dst_pages differ in length")
    for t, name in ((k_src, "k_src"), (v_src, "v_src"), (k_dst, "k_dst"), (v_dst, "v_dst")):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 page pool")
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{name} must be device or page-locked host memory")
    if tuple(k_src.shape[1:]) != tuple(k_dst.shape[1:]) or k_src.shape != v_src.shape \
            or k_dst.shape != v_dst.shape:
        raise ValueError("pools must have the same page shape")
    for t, name in ((src_pages, "src_pages"), (dst_pages, "dst_pages")):
        if t.dtype != torch.int32 or not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{name} must be an int32 device (or pinned) tensor")
    page_bytes = int(k_src[0].numel()) * 2
    if error_word is None or isinstance(error_word, torch.Tensor):
        ew = _dev(error_word, torch.int32, "error_word")
    else:
        ew = ctypes.c_void_p(int(error_word))
    st = lib.mcp_kv_copy_pages(ctypes.c_void_p(k_src.data_ptr()), ctypes.c_void_p(v_src.data_ptr()),
                               int(k_src.shape[0]), ctypes.c_void_p(k_dst.data_ptr()),
                               ctypes.c_void_p(v_dst.data_ptr()), int(k_dst.shape[0]), page_bytes,
                               ctypes.c_void_p(src_pages.data_ptr()),
                               ctypes.c_void_p(dst_pages.data_ptr()), n, ew, _stream(stream))
    _capi.check(st, "kv_copy_pages")


def gather_rows(src, rows, dst, error_word=None, stream=None) -> None:
    """dst[i] = src[rows[i]] along the first dimension (device tensors; rows int32)."""
    import torch

    lib = load()
    n = int(rows.numel())
    if dst.shape[0] != n or tuple(dst.shape[1:]) != tuple(src.shape[1:]) or dst.dtype != src.dtype:
        raise ValueError("dst must be [len(rows), *src.shape[1:]] of src's dtype")
    if not (src.is_cuda and dst.is_cuda and src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("src / dst must be contiguous CUDA tensors")
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] else dst[0].numel() * dst.element_size()
    if error_word is None or isinstance(error_word, torch.Tensor):
        ew = _dev(error_word, torch.int32, "error_word")
    else:
        ew = ctypes.c_void_p(int(error_word))
    st = lib.mcp_gather_rows(ctypes.c_void_p(src.data_ptr()), int(src.shape[0]), int(row_bytes),
                             _dev(rows, torch.int32, "rows"), n, ctypes.c_void_p(dst.data_ptr()),
                             ew, _stream(stream))
    _capi.check(st, "gather_rows")


def mixed_attn_fwd(plan: Plan, q, k_cache, v_cache, block_tables, cu_seqlens_q, seqlens_k, out,
                   lse=None, workspace=None, stream=None) -> None:
    """Fused mixed attention forward on device tensors (see include/mcp.h)."""
    import torch

    lib = load()
    st = lib.mcp_mixed_attn_fwd(
        ctypes.byref(plan), _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(block_tables, torch.int32, "block_tables"),
        _dev(cu_seqlens_q, torch.int32, "cu_seqlens_q"), _dev(seqlens_k, torch.int32, "seqlens_k"),
        _dev(out, torch.bfloat16, "out"), _dev(lse, torch.float32, "lse"),
        _dev(workspace, torch.uint8, "workspace"),
        int(workspace.numel()) if workspace is not None else 0, _stream(stream))
    _capi.check(st, "mixed_attn_fwd")


def mixed_attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, sm_scale, out=None, lse=None,
                      options: PlanOptions | None = None, stream=None):
    """Right-aligned causal attention over packed non-paged K/V ([W] "Flash
    Attention 的 varlen 接口"): q [T, H_q, D], k / v [total_k, H_kv, D] bf16
    CUDA tensors; cu_seqlens_q / cu_seqlens_k host int arrays.  Plans, runs
    and checks the device error word; returns ``out`` (and fills ``lse``)."""
    import torch

    lib = load()
    cu_q = np.ascontiguousarray(np.asarray(cu_seqlens_q, dtype=np.int32))
    cu_k = np.ascontiguousarray(np.asarray(cu_seqlens_k, dtype=np.int32))
    S = int(cu_q.size) - 1
    if cu_k.size != S + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k differ in length")
    sk = np.diff(cu_k).astype(np.int32)
    T, Hq, D = (int(x) for x in q.shape)
    total_k, Hkv = int(k.shape[0]), int(k.shape[1])
    if int(cu_k[-1]) != total_k or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k / v must be [cu_seqlens_k[-1], H_kv, D]")
    mp = max(1, int((sk.max() + 15) // 16)) if S else 1
    desc = make_desc(S, T, Hq, Hkv, D, 16, mp, 1, sm_scale)
    sizing = mixed_attn_plan(desc, cu_q, sk, options)
    ws = torch.empty(max(256, int(sizing.workspace_bytes)), dtype=torch.uint8, device=q.device)
    plan = mixed_attn_plan(desc, cu_q, sk, options, ws, stream)
    if out is None:
        out = torch.empty_like(q)
    cu_q_d = torch.from_numpy(cu_q).to(q.device)
    cu_k_d = torch.from_numpy(cu_k).to(q.device)
    st = lib.mcp_mixed_attn_fwd_varlen(
        ctypes.byref(plan), _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"),
        _dev(v, torch.bfloat16, "v"), _dev(cu_q_d, torch.int32, "cu_seqlens_q"),
        _dev(cu_k_d, torch.int32, "cu_seqlens_k"), total_k, _dev(out, torch.bfloat16, "out"),
        _dev(lse, torch.float32, "lse"), _dev(ws, torch.uint8, "workspace"), int(ws.numel()),
        _stream(stream))
    _capi.check(st, "mixed_attn_fwd_varlen")
    check_device_errors(workspace_error_word(plan, ws), stream)
    return out


def workspace_error_word(plan: Plan, workspace) -> int:
    lib = load()
    return int(lib.mcp_workspace_error_word(ctypes.byref(plan), ctypes.c_void_p(workspace.data_ptr())))


def check_device_errors(error_word_ptr: int, stream=None) -> None:
    """Synchronise, read and clear a device error word; raise on a set bit."""
    lib = load()
    st = lib.mcp_check_device_errors(ctypes.c_void_p(int(error_word_ptr)), _stream(stream))
    _capi.check(st, "check_device_errors")


def merge_states(o_parts, lse_parts, out, lse_out=None, stream=None) -> None:
    """Merge split attention states: o_parts [n, R, H, D] fp32, lse_parts [n, R, H]."""
    import torch

    lib = load()
    n, R, H, D = (int(x) for x in o_parts.shape)
    if tuple(lse_parts.shape) != (n, R, H) or tuple(out.shape) != (R, H, D):
        raise ValueError("shape mismatch")
    st = lib.mcp_merge_states(_dev(o_parts, torch.float32, "o_parts"),
                              _dev(lse_parts, torch.float32, "lse_parts"), n, R, H, D,
                              _dev(out, torch.bfloat16, "out"),
                              _dev(lse_out, torch.float32, "lse_out"), _stream(stream))
    _capi.check(st, "merge_states")


def mixed_attn_fwd_noalloc(desc: AttnDesc, h_cu_seqlens_q, h_seqlens_k, q, k_cache, v_cache,
                           block_tables, cu_seqlens_q, seqlens_k, out, lse=None,
                           options: PlanOptions | None = None, stream=None) -> int:
    """Mixed attention forward without a workspace (for callers that cannot
    allocate device memory): plans from the HOST metadata and keeps its scratch
    in the library's fixed 16 MiB device array.  Returns the device address of
    this call's error word (for check_device_errors).  Calls that overlap on
    the GPU race; make the first call on a device before any stream capture."""
    import torch

    lib = load()
    cu, cu_p = _host_i32(h_cu_seqlens_q, "h_cu_seqlens_q")
    sk, sk_p = _host_i32(h_seqlens_k, "h_seqlens_k")
    ew = ctypes.c_void_p()
    st = lib.mcp_mixed_attn_fwd_noalloc(
        ctypes.byref(desc), cu_p, sk_p, ctypes.byref(options) if options is not None else None,
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(block_tables, torch.int32, "block_tables"),
        _dev(cu_seqlens_q, torch.int32, "cu_seqlens_q"), _dev(seqlens_k, torch.int32, "seqlens_k"),
        _dev(out, torch.bfloat16, "out"), _dev(lse, torch.float32, "lse"), ctypes.byref(ew),
        _stream(stream))
    _capi.check(st, "mixed_attn_fwd_noalloc")
    return int(ew.value or 0)
