"""ctypes view of the C ABI declared in include/mcp.h (argument marshalling only)."""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int32, c_int64, c_size_t, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libmcp.so")

MCP_OK = 0
MCP_ERR_INVALID_ARG = 1
MCP_ERR_UNSUPPORTED = 2
MCP_ERR_WORKSPACE_TOO_SMALL = 3
MCP_ERR_CUDA = 4
MCP_ERR_TIMEOUT = 5
MCP_ERR_DEVICE_CHECK = 6

DEVERR_TIMEOUT = 0x1
DEVERR_PAGE_RANGE = 0x2
DEVERR_SLOT_RANGE = 0x4
DEVERR_ROW_RANGE = 0x8
DEVERR_ITEM_KIND = 0x10
DEVERR_SLOT_DUP = 0x20
BUILD_CHECKED = 0x1


class AttnDesc(ctypes.Structure):
    _fields_ = [
        ("num_seqs", c_int32),
        ("total_q", c_int32),
        ("num_q_heads", c_int32),
        ("num_kv_heads", c_int32),
        ("head_dim", c_int32),
        ("page_size", c_int32),
        ("max_pages_per_seq", c_int32),
        ("num_pages", c_int32),
        ("sm_scale", c_float),
    ]


class PlanOptions(ctypes.Structure):
    _fields_ = [
        ("num_sms", c_int32),
        ("decode_split_tokens", c_int32),
        ("prefill_split_tokens", c_int32),
        ("test_stall", c_int32),
        ("reserved", c_int32 * 4),
    ]


class Plan(ctypes.Structure):
    _fields_ = [
        ("magic", c_int32),
        ("num_items", c_int32),
        ("num_decode_items", c_int32),
        ("num_prefill_items", c_int32),
        ("num_combine", c_int32),
        ("decode_split_tokens", c_int32),
        ("prefill_split_tokens", c_int32),
        ("num_sms", c_int32),
        ("partial_rows", c_int64),
        ("off_items", c_int64),
        ("off_combine", c_int64),
        ("off_part_o", c_int64),
        ("off_part_lse", c_int64),
        ("off_error", c_int64),
        ("workspace_bytes", c_int64),
        ("desc", AttnDesc),
        ("combine_rows", c_int32),
        ("test_stall", c_int32),
        ("reserved", c_int32 * 6),
    ]


class SchedConfig(ctypes.Structure):
    _fields_ = [
        ("max_num_batched_tokens", c_int32),
        ("long_prefill_token_threshold", c_int32),
        ("max_num_seqs", c_int32),
        ("num_pages", c_int32),
        ("page_size", c_int32),
        ("max_pages_per_seq", c_int32),
        ("preempt_swap", c_int32),
        ("num_host_pages", c_int32),
        ("reserved", c_int32 * 4),
    ]


class SchedOutput(ctypes.Structure):
    _fields_ = [
        ("num_seqs", c_int32),
        ("total_q", c_int32),
        ("request_ids", POINTER(c_int64)),
        ("cu_seqlens_q", POINTER(c_int32)),
        ("seqlens_k", POINTER(c_int32)),
        ("block_tables", POINTER(c_int32)),
        ("sample_mask", POINTER(ctypes.c_uint8)),
        ("logits_indices", POINTER(c_int32)),
        ("num_logits", c_int32),
        ("num_swap_out", c_int32),
        ("swap_out_device_pages", POINTER(c_int32)),
        ("swap_out_host_pages", POINTER(c_int32)),
        ("num_swap_in", c_int32),
        ("swap_in_host_pages", POINTER(c_int32)),
        ("swap_in_device_pages", POINTER(c_int32)),
        ("num_preempted", c_int32),
        ("preempted_ids", POINTER(c_int64)),
        ("reserved", c_int32 * 4),
    ]


class HostStepLimits(ctypes.Structure):
    _fields_ = [
        ("max_tokens", c_int32),
        ("max_seqs", c_int32),
        ("max_pages_per_seq", c_int32),
        ("reserved0", c_int32),
        ("workspace_bytes", c_int64),
        ("list_bytes", c_int64),
        ("reserved", c_int32 * 4),
    ]


# name -> (restype, argtypes); every symbol include/mcp.h declares
SIGNATURES = {
    "mcp_status_string": (c_char_p, [c_int32]),
    "mcp_last_error": (c_char_p, []),
    "mcp_abi_version": (c_int32, []),
    "mcp_build_flags": (c_int32, []),
    "mcp_paged_kv_append": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                      c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
    "mcp_build_slot_mapping": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p,
                                         c_void_p, c_void_p]),
    "mcp_mixed_attn_plan": (c_int32, [POINTER(AttnDesc), c_void_p, c_void_p, POINTER(PlanOptions),
                                      POINTER(Plan), c_void_p, c_size_t, c_void_p]),
    "mcp_mixed_attn_plan_host": (c_int32, [POINTER(AttnDesc), c_void_p, c_void_p,
                                           POINTER(PlanOptions), POINTER(Plan), c_void_p,
                                           c_size_t]),
    "mcp_mixed_attn_fwd": (c_int32, [POINTER(Plan), c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                     c_void_p]),
    "mcp_mixed_attn_fwd_noalloc": (c_int32, [POINTER(AttnDesc), c_void_p, c_void_p,
                                             POINTER(PlanOptions), c_void_p, c_void_p, c_void_p,
                                             c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                             c_void_p, c_void_p]),
    "mcp_mixed_attn_fwd_varlen": (c_int32, [POINTER(Plan), c_void_p, c_void_p, c_void_p,
                                            c_void_p, c_void_p, c_int64, c_void_p, c_void_p,
                                            c_void_p, c_size_t, c_void_p]),
    "mcp_check_device_errors": (c_int32, [c_void_p, c_void_p]),
    "mcp_workspace_error_word": (c_void_p, [POINTER(Plan), c_void_p]),
    "mcp_merge_states": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32,
                                   c_void_p, c_void_p, c_void_p]),
    "mcp_build_logits_indices": (c_int32, [c_int32, c_void_p, c_void_p, c_void_p,
                                           POINTER(c_int32)]),
    "mcp_mixed_attn_plan_rows": (c_int32, [POINTER(AttnDesc), c_void_p, c_void_p, c_void_p,
                                           c_int32, POINTER(PlanOptions), POINTER(Plan),
                                           c_void_p, c_size_t, c_void_p]),
    "mcp_mixed_attn_plan_rows_host": (c_int32, [POINTER(AttnDesc), c_void_p, c_void_p,
                                                c_void_p, c_int32, POINTER(PlanOptions),
                                                POINTER(Plan), c_void_p, c_size_t]),
    "mcp_kv_copy_pages": (c_int32, [c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int32,
                                    c_int32, c_void_p, c_void_p, c_int32, c_void_p, c_void_p]),
    "mcp_gather_rows": (c_int32, [c_void_p, c_int32, c_int32, c_void_p, c_int32, c_void_p,
                                  c_void_p, c_void_p]),
    "mcp_sched_create": (c_int32, [POINTER(SchedConfig), POINTER(c_void_p)]),
    "mcp_sched_add_request": (c_int32, [c_void_p, c_int64, c_int32, c_int32, c_int32]),
    "mcp_sched_schedule": (c_int32, [c_void_p, POINTER(SchedOutput)]),
    "mcp_sched_finish_step": (c_int32, [c_void_p, POINTER(c_int32), c_void_p]),
    "mcp_sched_stats": (c_int32, [c_void_p, POINTER(c_int32), POINTER(c_int32), POINTER(c_int32),
                                  POINTER(c_int64), POINTER(c_int32)]),
    "mcp_sched_destroy": (c_int32, [c_void_p]),
    "mcp_host_step_arena_bytes": (c_int32, [POINTER(AttnDesc), POINTER(HostStepLimits),
                                            POINTER(c_size_t), POINTER(c_size_t)]),
    "mcp_host_step_create": (c_int32, [POINTER(AttnDesc), POINTER(HostStepLimits), c_void_p,
                                       c_size_t, c_void_p, c_size_t, c_void_p,
                                       POINTER(c_void_p)]),
    "mcp_host_step_run": (c_int32, [c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    POINTER(c_int64)]),
    "mcp_host_step_wait": (c_int32, [c_void_p, c_int64]),
    "mcp_host_step_destroy": (c_int32, [c_void_p]),
}

_lib = None


def open_library(path: str):
    """A ctypes handle on the library at ``path`` with every signature set."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(the CUDA library is required; there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str = LIB_PATH):
    """Load the CUDA library; raise if it was not built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = open_library(path)
    return _lib


class MCPError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        self.status = status
        msg = lib.mcp_last_error().decode(errors="replace")
        name = lib.mcp_status_string(status).decode()
        super().__init__(f"{where}: {name}: {msg}")


def check(status: int, where: str) -> None:
    if status != MCP_OK:
        raise MCPError(status, where)
