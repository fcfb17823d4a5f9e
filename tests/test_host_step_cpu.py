"""Host-side checks of the pipelined host step (``mcp_host_step_*``): arena
sizing and argument validation, all before any CUDA call."""

from __future__ import annotations

import ctypes

import pytest

import mixed_chunked_prefill_gb300 as mcp
from mixed_chunked_prefill_gb300 import _capi


def shape(hq=32, hkv=8, d=128, p=16, pages=1000, scale=0.088):
    return mcp.make_desc(0, 0, hq, hkv, d, p, 1, pages, scale)


def limits(tokens=2048, seqs=64, pages=512, ws=0, lists=0, r0=0, res=(0, 0, 0, 0)):
    return _capi.HostStepLimits(tokens, seqs, pages, r0, ws, lists, (ctypes.c_int32 * 4)(*res))


def sizes(sh, lim):
    lib = mcp.load()
    d, h = ctypes.c_size_t(), ctypes.c_size_t()
    st = lib.mcp_host_step_arena_bytes(ctypes.byref(sh), ctypes.byref(lim), ctypes.byref(d),
                                       ctypes.byref(h))
    return st, d.value, h.value


def test_arena_bytes_cover_two_slots():
    T, S, mp = 2048, 64, 512
    st, dbytes, hbytes = sizes(shape(), limits(T, S, mp))
    assert st == 0
    per_slot_tokens = T * (2 * 32 + 2 * 8) * 128 * 2 + T * 32 * 4 + T * 8  # q, out, k, v, lse, slots
    per_slot_meta = ((S + 1) + S + S * mp) * 4
    assert dbytes >= 2 * (per_slot_tokens + per_slot_meta + (64 << 20))  # default workspace
    assert hbytes >= 2 * (per_slot_meta + T * 8 + (4 << 20))             # default list bytes
    assert dbytes % 256 == 0 and hbytes % 256 == 0
    st, d2, h2 = sizes(shape(), limits(T, S, mp, ws=1 << 20, lists=1 << 16))
    assert st == 0 and d2 < dbytes and h2 < hbytes


@pytest.mark.parametrize("sh,lim,code", [
    (shape(d=80), limits(), 2),
    (shape(p=4), limits(), 2),
    (shape(hq=30, hkv=8), limits(), 1),
    (shape(scale=0.0), limits(), 1),
    (shape(), limits(tokens=0), 1),
    (shape(), limits(seqs=-1), 1),
    (shape(), limits(r0=1), 1),
    (shape(), limits(res=(0, 1, 0, 0)), 1),
    (shape(), limits(ws=-5), 1),
])
def test_arena_bytes_validation(sh, lim, code):
    st, _, _ = sizes(sh, lim)
    assert st == code, mcp.load().mcp_last_error()


def test_create_and_calls_reject_null_before_cuda():
    lib = mcp.load()
    sh, lim = shape(), limits()
    out = ctypes.c_void_p()
    assert lib.mcp_host_step_create(ctypes.byref(sh), ctypes.byref(lim), None, 0, None, 0, None,
                                    ctypes.byref(out)) == 1
    assert out.value is None
    # misaligned arenas are rejected before any device query
    assert lib.mcp_host_step_create(ctypes.byref(sh), ctypes.byref(lim), ctypes.c_void_p(0x1008),
                                    1 << 40, ctypes.c_void_p(0x2008), 1 << 40, None,
                                    ctypes.byref(out)) == 1
    # arenas smaller than the sizing call says
    _, dbytes, hbytes = sizes(sh, lim)
    assert lib.mcp_host_step_create(ctypes.byref(sh), ctypes.byref(lim), ctypes.c_void_p(0x1000),
                                    dbytes - 256, ctypes.c_void_p(0x2000), hbytes, None,
                                    ctypes.byref(out)) == 3
    t = ctypes.c_int64()
    assert lib.mcp_host_step_run(None, 0, None, None, None, None, None, None, None, None, None,
                                 None, ctypes.byref(t)) == 1
    assert lib.mcp_host_step_wait(None, 0) == 1
    assert lib.mcp_host_step_destroy(None) == 0


@pytest.mark.parametrize("d,p", [(64, 16), (96, 16), (256, 16), (128, 1), (128, 8), (256, 64)])
def test_arena_bytes_for_every_built_shape(d, p):
    """Every built head_dim / page size sizes its arenas; the device arena
    grows with head_dim (q, out, k_new, v_new rows of 2 * d bytes)."""
    T = 1024
    st, dbytes, hbytes = sizes(shape(d=d, p=p, scale=1.0 / d ** 0.5), limits(T, 32, 2048))
    assert st == 0 and dbytes % 256 == 0 and hbytes % 256 == 0
    assert dbytes >= 2 * T * (2 * 32 + 2 * 8) * d * 2
    st64, d64, _ = sizes(shape(d=64, p=p), limits(T, 32, 2048))
    assert st64 == 0 and (d == 64 or dbytes > d64)
