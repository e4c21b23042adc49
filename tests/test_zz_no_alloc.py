"""h2o_prefill_select_static -- the prefill entry point for callers that cannot allocate device
memory (a serving engine whose pool owns all device memory, a plugin inside a framework that owns
the allocator); its scratch is a fixed array inside the library -- against h2o_prefill_select with a
caller-allocated workspace. Collected last, so that a run stopping at the first failure has already
run every other test."""

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _state(w):
    import torch
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    return (torch.full((w.units, w.budget, w.head_dim), 7, dtype=dt, device="cuda"),
            torch.full((w.units, w.budget, w.head_dim), 7, dtype=dt, device="cuda"),
            torch.full((w.units, w.budget), -3.0, dtype=torch.float32, device="cuda"),
            torch.full((w.units, w.budget), -9, dtype=torch.int32, device="cuda"))


def _dev(a):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a))
    return (t.view(torch.bfloat16) if a.dtype == np.uint16 else t).cuda()


def _dims(h2o, w):
    return h2o.Dims(units_b=w.units_b, heads=w.heads, head_dim=w.head_dim, budget=w.budget,
                    k_heavy=w.k_heavy, k_local=w.k_local,
                    dtype=h2o.F32 if w.dtype == "f32" else h2o.BF16)


def test_static_scratch_prefill_matches_workspace_entry_point():
    """Several calls in a row with different shapes: each later call finds the previous call's
    leftovers in the shared scratch array and must still match the workspace entry point exactly
    (same kernels, so the tolerance is zero)."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    assert torch.cuda.is_available()
    for w in (synth.WORKLOADS["opt-6.7b"].with_(layers=1, batch=2, heads=8),
              synth.WORKLOADS["llama-7b"].with_(batch=1, heads=5),
              synth.WORKLOADS["tiny"]):
        dims = _dims(h2o, w)
        inp = synth.generate(w, steps=0)
        q, k, v = _dev(inp.q_prompt), _dev(inp.k_prompt), _dev(inp.v_prompt)
        ref = _state(w)
        ws = torch.empty(h2o.h2o_prefill_workspace_bytes(dims, w.prompt_len), dtype=torch.uint8,
                         device="cuda")
        h2o.h2o_prefill_select(dims, w.prompt_len, q, k, v, *ref, ws)
        got = _state(w)
        h2o.h2o_prefill_select_static(dims, w.prompt_len, q, k, v, *got)
        torch.cuda.synchronize()
        # The first call on the device looks the array up (and so loads the module that holds it):
        # it must leave no CUDA error behind.
        assert h2o.last_cuda_error() == "cudaSuccess"
        for a, b in zip(ref, got):
            assert torch.equal(a, b), w.name
        assert h2o.h2o_get_device_error() == 0


def test_static_scratch_call_allocates_no_device_memory():
    """Once every shape below has run once (its kernels are loaded), further calls of all of them
    leave the device's free memory exactly where it was: the entry point allocates nothing."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    calls = []
    for w in (synth.WORKLOADS["opt-6.7b"].with_(layers=1, batch=2, heads=8),
              synth.WORKLOADS["llama-7b"].with_(batch=1, heads=5),
              synth.WORKLOADS["opt-30b"].with_(batch=1, heads=7, prompt_len=333),
              synth.WORKLOADS["tiny"]):
        inp = synth.generate(w, steps=0)
        calls.append((_dims(h2o, w), w.prompt_len, _dev(inp.q_prompt), _dev(inp.k_prompt),
                      _dev(inp.v_prompt), _state(w)))
    for dims, P, q, k, v, st in calls:  # warm-up: every kernel these shapes use is loaded
        h2o.h2o_prefill_select_static(dims, P, q, k, v, *st)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        for dims, P, q, k, v, st in calls:
            h2o.h2o_prefill_select_static(dims, P, q, k, v, *st)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert h2o.h2o_get_device_error() == 0


def test_static_scratch_rejects_oversized_calls():
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    w = synth.WORKLOADS["opt-6.7b"]  # 8192 units x 512 tokens needs 48 MiB of scratch
    dims = _dims(h2o, w)
    assert h2o.h2o_prefill_workspace_bytes(dims, w.prompt_len) > h2o.STATIC_SCRATCH_BYTES
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(h2o.H2OError) as e:
        h2o.h2o_prefill_select_static(dims, w.prompt_len, x, x, x, x, x, x, x)
    assert e.value.status == h2o.ERR_UNSUPPORTED
    assert torch.count_nonzero(x) == 0
