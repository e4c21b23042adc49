"""Host-side checks of libh2o.so: it builds for sm_103a, loads, exports every symbol include/h2o.h
declares, and rejects bad arguments before any CUDA call (so these run without a GPU)."""

import ctypes
import os
import re

import pytest

import kv_cache_eviction_step_gb300 as h2o
from kv_cache_eviction_step_gb300 import build as h2o_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    h2o_build.build()
    return h2o.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "h2o.h")).read()
    return re.findall(r"H2O_API\s+[\w\s\*]+?\b(h2o_\w+)\s*\(", text)


def test_header_declares_the_abi():
    names = declared_symbols()
    assert set(names) == set(h2o.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        ctypes.cast(getattr(lib, name), ctypes.c_void_p)


def test_only_the_abi_is_exported(lib):
    out = os.popen(f"nm -D --defined-only {h2o_build.LIB}").read()
    syms = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert {s for s in syms if s.startswith("h2o_")} == set(h2o.EXPORTS)


def test_status_strings(lib):
    assert h2o.status_string(h2o.OK) == "ok"
    assert "invalid" in h2o.status_string(h2o.ERR_INVALID_ARG)
    assert h2o.status_string(99) == "unknown status"


def dims(**kw):
    base = dict(units_b=2, heads=4, head_dim=128, budget=8, k_heavy=4, k_local=4, dtype=h2o.BF16)
    base.update(kw)
    return h2o.Dims(**base)


def test_workspace_bytes(lib):
    d = dims()
    units, P = 8, 100
    per = (units * P * 4 + 255) // 256 * 256
    assert h2o.h2o_prefill_workspace_bytes(d, P) == 3 * per
    assert h2o.h2o_prefill_workspace_bytes(dims(k_heavy=5), P) == 0
    assert h2o.h2o_prefill_workspace_bytes(d, 0) == 0


@pytest.mark.parametrize("bad,status", [
    (dict(k_heavy=5), h2o.ERR_INVALID_ARG),          # k_heavy + k_local != budget
    (dict(budget=0, k_heavy=0, k_local=0), h2o.ERR_INVALID_ARG),
    (dict(k_local=-1, k_heavy=9), h2o.ERR_INVALID_ARG),
    (dict(heads=0), h2o.ERR_INVALID_ARG),
    (dict(dtype=7), h2o.ERR_INVALID_ARG),
    (dict(head_dim=96), h2o.ERR_UNSUPPORTED),
])
def test_decode_rejects_bad_dims(lib, bad, status):
    d = dims(**bad)
    rc = lib.h2o_decode_step(ctypes.byref(d), 10, *([16] * 10), None)
    assert rc == status


def test_decode_rejects_null_misaligned_and_position(lib):
    d = dims()
    ptrs = [4096 * (i + 1) for i in range(10)]
    assert lib.h2o_decode_step(ctypes.byref(d), 0, *ptrs, None) == h2o.ERR_INVALID_ARG
    for i in range(10):
        p = list(ptrs)
        p[i] = None
        assert lib.h2o_decode_step(ctypes.byref(d), 10, *p, None) == h2o.ERR_INVALID_ARG
        # q, k_new, v_new, k_cache, v_cache need 16 bytes; scores, positions, out and the
        # eviction indices need their element's alignment
        p[i] = ptrs[i] + (8 if i < 5 else 1)
        assert lib.h2o_decode_step(ctypes.byref(d), 10, *p, None) == h2o.ERR_INVALID_ARG


def test_prefetch_hint_rejects_null_and_misaligned_members(lib):
    """h2o_decode_step_prefetch checks the next-call hint before any CUDA call: every member
    non-NULL, the K/V caches 16-byte aligned, scores and positions 4-byte aligned. (A good hint with
    position 0 still fails on the position, so nothing is launched.)"""
    d = dims()
    ptrs = [4096 * (i + 1) for i in range(10)]
    good = [1 << 20, 2 << 20, 3 << 20, 4 << 20]
    call = lambda nxt, pos: lib.h2o_decode_step_prefetch(ctypes.byref(d), None, pos, *ptrs,
                                                         ctypes.byref(h2o.NextCache(*nxt)), None)
    assert call(good, 0) == h2o.ERR_INVALID_ARG
    for i in range(4):
        bad = list(good)
        bad[i] = None
        assert call(bad, 10) == h2o.ERR_INVALID_ARG
        bad[i] = good[i] + (8 if i < 2 else 2)
        assert call(bad, 10) == h2o.ERR_INVALID_ARG
    assert lib.h2o_decode_step_prefetch(ctypes.byref(d), None, 0, *ptrs, None, None) == h2o.ERR_INVALID_ARG


def test_prefill_rejects_bad_arguments(lib):
    d = dims()
    ws = h2o.h2o_prefill_workspace_bytes(d, 64)
    args = [4096 * (i + 1) for i in range(7)]
    # prompt length out of range
    assert lib.h2o_prefill_select(ctypes.byref(d), 0, *args, 4096, ws * 10, None) == h2o.ERR_INVALID_ARG
    assert lib.h2o_prefill_select(ctypes.byref(d), 16385, *args, 4096, 1 << 40, None) == h2o.ERR_UNSUPPORTED
    # workspace too small
    assert lib.h2o_prefill_select(ctypes.byref(d), 64, *args, 4096, ws - 1, None) == h2o.ERR_INVALID_ARG
    # misaligned cache pointer
    bad = list(args)
    bad[3] += 4
    assert lib.h2o_prefill_select(ctypes.byref(d), 64, *bad, 4096, ws, None) == h2o.ERR_INVALID_ARG
    assert lib.h2o_prefill_scores(ctypes.byref(d), 64, 4096, 8192, None, 4096, ws, None) == h2o.ERR_INVALID_ARG


def test_zero_units_is_a_noop(lib):
    d = dims(units_b=0)
    assert lib.h2o_decode_step(ctypes.byref(d), 10, *([None] * 10), None) == h2o.OK
    assert lib.h2o_prefill_select(ctypes.byref(d), 64, *([None] * 7), None, 0, None) == h2o.OK


@pytest.mark.parametrize("pol", [
    h2o.Policy(7),                                       # unknown kind
    h2o.Policy(-1),
    h2o.Policy(h2o.POLICY_SINK_WINDOW, n_sink=8),        # n_sink must stay below the budget
    h2o.Policy(h2o.POLICY_SINK_WINDOW, n_sink=-1),
    h2o.Policy(h2o.POLICY_STRIDED, stride=0),
])
def test_policy_entry_points_reject_bad_policies(lib, pol):
    d = dims()
    ptrs = [4096 * (i + 1) for i in range(10)]
    assert lib.h2o_decode_step_policy(ctypes.byref(d), ctypes.byref(pol), 10, *ptrs, None) \
        == h2o.ERR_INVALID_ARG
    ws = h2o.h2o_prefill_workspace_bytes(d, 64)
    assert lib.h2o_prefill_select_policy(ctypes.byref(d), ctypes.byref(pol), 64, *ptrs[:7], 4096, ws,
                                         None) == h2o.ERR_INVALID_ARG
    # rejected even when there is no unit to process
    d0 = dims(units_b=0)
    assert lib.h2o_decode_step_policy(ctypes.byref(d0), ctypes.byref(pol), 10, *([None] * 10), None) \
        == h2o.ERR_INVALID_ARG


@pytest.mark.parametrize("pol", [None, h2o.Policy(), h2o.Policy(h2o.POLICY_LOCAL),
                                 h2o.Policy(h2o.POLICY_SINK_WINDOW, n_sink=7),
                                 h2o.Policy(h2o.POLICY_TOPK), h2o.Policy(h2o.POLICY_STRIDED, stride=3)])
def test_policy_entry_points_accept_valid_policies(lib, pol):
    d0 = dims(units_b=0)
    ref = None if pol is None else ctypes.byref(pol)
    assert lib.h2o_decode_step_policy(ctypes.byref(d0), ref, 10, *([None] * 10), None) == h2o.OK
    assert lib.h2o_prefill_select_policy(ctypes.byref(d0), ref, 64, *([None] * 7), None, 0, None) == h2o.OK
    # the same argument checks as the plain entry points
    d = dims()
    assert lib.h2o_decode_step_policy(ctypes.byref(d), ref, 0, *([4096] * 10), None) == h2o.ERR_INVALID_ARG


def test_prefill_forward_needs_an_aligned_output(lib):
    d = dims()
    ws = h2o.h2o_prefill_workspace_bytes(d, 64)
    args = [4096 * (i + 1) for i in range(3)]
    rest = [4096 * (i + 5) for i in range(4)]
    assert lib.h2o_prefill_forward(ctypes.byref(d), None, 64, *args, None, *rest, 4096, ws, None) \
        == h2o.ERR_INVALID_ARG
    assert lib.h2o_prefill_forward(ctypes.byref(d), None, 64, *args, 4096 + 8, *rest, 4096, ws, None) \
        == h2o.ERR_INVALID_ARG
    bad = h2o.Policy(h2o.POLICY_STRIDED, stride=0)
    assert lib.h2o_prefill_forward(ctypes.byref(d), ctypes.byref(bad), 64, *args, 4096, *rest, 4096, ws,
                                   None) == h2o.ERR_INVALID_ARG
    d0 = dims(units_b=0)
    assert lib.h2o_prefill_forward(ctypes.byref(d0), None, 64, *([None] * 9), 0, None) == h2o.OK


@pytest.mark.parametrize("bad,status", [
    (dict(head_dim=64), h2o.ERR_UNSUPPORTED),
    (dict(dtype=h2o.F32), h2o.ERR_UNSUPPORTED),
    (dict(budget=520, k_heavy=260, k_local=260), h2o.ERR_UNSUPPORTED),
])
def test_e4m3_entry_points_reject_unsupported_shapes(lib, bad, status):
    d = dims(**bad)
    ptrs = [4096 * (i + 1) for i in range(12)]
    assert lib.h2o_decode_step_e4m3(ctypes.byref(d), None, 10, *ptrs, None) == status
    ws = h2o.h2o_prefill_workspace_bytes(d, 64)
    assert lib.h2o_prefill_select_e4m3(ctypes.byref(d), None, 64, *ptrs[:9], 4096, ws, None) == status


def test_e4m3_entry_points_need_aligned_scales(lib):
    d = dims()
    ptrs = [4096 * (i + 1) for i in range(12)]
    for i in (5, 6):  # k_scale, v_scale (after q, k_new, v_new, k_cache, v_cache)
        p = list(ptrs)
        p[i] = None
        assert lib.h2o_decode_step_e4m3(ctypes.byref(d), None, 10, *p, None) == h2o.ERR_INVALID_ARG
        p[i] = ptrs[i] + 2
        assert lib.h2o_decode_step_e4m3(ctypes.byref(d), None, 10, *p, None) == h2o.ERR_INVALID_ARG
