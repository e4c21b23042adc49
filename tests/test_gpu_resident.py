"""The one-CTA-per-unit decode kernel with the whole unit resident in shared memory (bf16, D = 128,
budget <= 208, at least one and fewer than four units per SM: one layer's batch x heads per launch)
against the oracle through the C ABI, and the next-call L2 prefetch hint of h2o_decode_step_prefetch
(needs a GB300)."""

import numpy as np
import pytest

import oracle
import parity
import synth

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
UNITS = 160  # >= one per SM (152) and < four per SM: the resident kernel's window


def _assert(rep: parity.Report):
    parity.check(rep)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    h2o.load()
    torch.cuda.init()
    yield
    assert h2o.h2o_get_device_error() == 0


def _shape(budget: int, P: int, k_local: int, steps: int, units: int = UNITS) -> synth.Workload:
    return W["opt-6.7b"].with_(layers=1, batch=units, heads=1, prompt_len=P, decode_steps=steps,
                               budget=budget, k_heavy=budget - k_local, k_local=k_local)


@pytest.mark.parametrize("budget,P,k_local", [
    (1, 40, 0),        # one slot, no protected window
    (2, 1, 1),         # cache fills during decode
    (31, 50, 15),      # one partial 32-slot block
    (32, 20, 16),      # one full block, filled during decode
    (33, 80, 1),       # a block of one slot
    (64, 64, 32),      # prompt exactly the budget
    (100, 60, 50),     # appends then evictions across block edges
    (204, 512, 102),   # the OPT-6.7B layer shape
    (208, 150, 104),   # the largest budget the kernel takes, filled during decode
    (208, 300, 0),     # ... with no protected window
])
def test_resident_kernel_budgets(budget, P, k_local):
    """Budgets from 1 to 208 slots (one to seven 32-slot warp blocks, full and partial), prompts
    shorter than, equal to and longer than the budget (slots appended, then evicted), k_local from 0
    to k/2; the oracle follows 12 sampled units through every step, state compared every 8 steps."""
    steps = max(24, budget - P + 24)
    w = _shape(budget, P, k_local, steps)
    units = np.linspace(0, w.units - 1, 12).astype(int)
    _assert(parity.run(w, check_units=units, state_every=8))


POLICIES = {
    "local": (oracle.POLICY_LOCAL, 0, 1),
    "sink4": (oracle.POLICY_SINK_WINDOW, 4, 1),
    "topk": (oracle.POLICY_TOPK, 0, 1),
    "strided3": (oracle.POLICY_STRIDED, 0, 3),
}


@pytest.mark.parametrize("pol", list(POLICIES))
def test_resident_kernel_policies(pol):
    """The baseline eviction policies on the resident kernel (OPT-6.7B budget, 160 units)."""
    w = _shape(204, 512, 102, 48)
    units = np.linspace(0, w.units - 1, 10).astype(int)
    _assert(parity.run(w, check_units=units, state_every=16, policy=POLICIES[pol]))


@pytest.mark.parametrize("units", [152, 256, 607])
def test_resident_kernel_unit_counts(units):
    """The ends of the resident kernel's unit window and the per-layer OPT-6.7B count."""
    w = _shape(204, 512, 102, 24, units=units)
    check = [0, units // 3, units // 2, units - 1]
    _assert(parity.run(w, check_units=check, state_every=8))


def _two_layer_run(hint: str, steps: int = 24):
    """Two 256-unit caches (two layers) stepped alternately on one stream, as a model launches the
    step once per layer; ``hint``: "none", "next" (each call names the other layer's cache, the next
    call's) or "self" (each call names its own cache). Returns every output and the final state."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    w = W["opt-6.7b"].with_(layers=1, decode_steps=steps)
    dims = parity.dims_of(w)
    keys = ("q_prompt", "k_prompt", "v_prompt", "q_dec", "k_dec", "v_dec")
    dev = []
    for i in range(2):
        inp = synth.generate(w, seed=synth.DEFAULT_SEED + 7 * i)
        dev.append({k: parity.to_device(getattr(inp, k), w.dtype) for k in keys})
    caches = [h2o.H2OCache(dims, w.prompt_len) for _ in range(2)]
    for c, d in zip(caches, dev):
        c.prefill(d["q_prompt"], d["k_prompt"], d["v_prompt"])
    S, U, D = w.decode_steps, w.units, w.head_dim
    outs = [torch.empty((S, U, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    evs = [torch.empty((S, U), dtype=torch.int32, device="cuda") for _ in range(2)]
    evp = [torch.empty((S, U), dtype=torch.int32, device="cuda") for _ in range(2)]
    for s in range(S):
        for l in range(2):
            d = dev[l]
            nxt = {"none": None, "next": caches[1 - l], "self": caches[l]}[hint]
            caches[l].step(d["q_dec"][s], d["k_dec"][s], d["v_dec"][s], out=outs[l][s], evicted_slot=evs[l][s],
                           evicted_pos=evp[l][s], prefetch=nxt)
    torch.cuda.synchronize()
    assert h2o.h2o_get_device_error() == 0
    got = outs + evs + evp
    for c in caches:
        got += [c.k_cache, c.v_cache, c.scores, c.slot_pos]
    return got


def test_prefetch_hint_leaves_results_unchanged():
    """The hint is a prefetch only: outputs, evictions and both caches' state are bit-identical with
    no hint, with the next call's cache named, and with the call's own cache named."""
    import torch
    base = _two_layer_run("none")
    for hint in ("next", "self"):
        got = _two_layer_run(hint)
        assert len(got) == len(base)
        for i, (x, y) in enumerate(zip(got, base)):
            assert torch.equal(x, y), (hint, i)


def test_prefetch_hint_on_other_kernels_is_ignored():
    """Shapes run by the other kernels (six units: the cluster-split kernel; 640 units: the persistent
    kernel) take the hint and give the plain call's results, bit for bit."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    for batch, heads in ((2, 3), (20, 32)):
        w = W["opt-6.7b"].with_(layers=1, batch=batch, heads=heads, decode_steps=6)
        dims = parity.dims_of(w)
        inp = synth.generate(w)
        dv = {k: parity.to_device(getattr(inp, k), w.dtype) for k in ("q_prompt", "k_prompt", "v_prompt",
                                                                       "q_dec", "k_dec", "v_dec")}
        runs = []
        for hinted in (False, True):
            a, b = h2o.H2OCache(dims, w.prompt_len), h2o.H2OCache(dims, w.prompt_len)
            for c in (a, b):
                c.prefill(dv["q_prompt"], dv["k_prompt"], dv["v_prompt"])
            outs = []
            for s in range(w.decode_steps):
                o, es, ep = a.step(dv["q_dec"][s], dv["k_dec"][s], dv["v_dec"][s], prefetch=b if hinted else None)
                outs += [o.clone(), es.clone(), ep.clone()]
            torch.cuda.synchronize()
            runs.append(outs + [a.k_cache, a.v_cache, a.scores, a.slot_pos])
        for i, (x, y) in enumerate(zip(*runs)):
            assert torch.equal(x, y), (batch, heads, i)
