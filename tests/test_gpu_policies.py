"""The eviction-policy variants (Local, sink + window, Top-K, strided, and H2O through the policy entry
points) on the GPU against the oracle under the same policy, through the C ABI (needs a GB300).

Each policy runs on all three decode kernels: the CUDA-core kernel (fp32 or D = 64), the cluster-split
tensor-core kernel (few bf16 units of D = 128) and the persistent tensor-core kernel (at least four
bf16 units of D = 128 per SM)."""

import numpy as np
import pytest

import oracle
import parity
import synth

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS

POLICIES = {
    "h2o": (oracle.POLICY_H2O, 0, 1),
    "local": (oracle.POLICY_LOCAL, 0, 1),
    "sink4": (oracle.POLICY_SINK_WINDOW, 4, 1),
    "topk": (oracle.POLICY_TOPK, 0, 1),
    "strided3": (oracle.POLICY_STRIDED, 0, 3),
}


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


@pytest.mark.parametrize("pol", list(POLICIES))
def test_policy_cuda_core_kernel_every_unit(pol):
    """fp32, D = 64, budget 32 (16 + 16): every unit, every step, state compared every 8 steps."""
    _assert(parity.run(W["tiny"], state_every=8, policy=POLICIES[pol]))


@pytest.mark.parametrize("pol", list(POLICIES))
def test_policy_split_tensor_core_kernel(pol):
    """Six bf16 units of D = 128 with the OPT-6.7B budget (102 + 102 of a 512-token prompt): each unit
    split over a CTA cluster."""
    w = W["opt-6.7b"].with_(layers=1, batch=2, heads=3, decode_steps=160)
    _assert(parity.run(w, state_every=32, policy=POLICIES[pol]))


@pytest.mark.parametrize("pol", list(POLICIES))
def test_policy_persistent_tensor_core_kernel(pol):
    """640 bf16 units of D = 128 (the persistent tcgen05 kernel); the oracle follows 8 sampled units."""
    w = W["opt-6.7b"].with_(layers=1, batch=20, heads=32, decode_steps=64)
    assert w.units >= 608
    units = np.linspace(0, w.units - 1, 8).astype(int)
    _assert(parity.run(w, check_units=units, state_every=16, policy=POLICIES[pol]))


def _policy_sweep():
    rng = np.random.default_rng(11)
    cases = []
    kinds = list(POLICIES)
    for i in range(15):
        D = int(rng.choice([64, 128]))
        dtype = "f32" if i % 3 == 0 else "bf16"
        budget = int(rng.choice([1, 2, 5, 17, 33, 100, 129, 256]))
        P = int(rng.integers(1, 3 * budget + 2))
        kl = int(rng.choice([0, 1, budget // 2, budget]))
        name = kinds[i % len(kinds)]
        kind, n_sink, stride = POLICIES[name]
        if kind == oracle.POLICY_SINK_WINDOW:
            n_sink = int(rng.integers(0, budget))
        if kind == oracle.POLICY_STRIDED:
            stride = int(rng.choice([1, 2, 5, 8]))
        w = synth.Workload(
            f"{name}{i}", layers=1, batch=int(rng.choice([1, 3, 40])), heads=int(rng.choice([1, 2, 5])),
            head_dim=D, dtype=dtype, prompt_len=P, decode_steps=int(rng.integers(1, 60)), budget=budget,
            k_heavy=budget - kl, k_local=kl, hh_kind="pareto", hh_count=max(1, (P + 60) // 20),
            q_boost=1.0)
        cases.append((w, (kind, n_sink, stride)))
    return cases


@pytest.mark.parametrize("w,pol", _policy_sweep(),
                         ids=lambda x: (f"{x.name}-D{x.head_dim}-{x.dtype}-k{x.budget}-kl{x.k_local}"
                                        f"-P{x.prompt_len}-u{x.units}") if isinstance(x, synth.Workload)
                         else f"n_sink{x[1]}-stride{x[2]}")
def test_policy_sweep(w, pol):
    """Odd budgets (1 to 256), prompts shorter and longer than the budget, k_local in {0, 1, k/2, k},
    sink counts from 0 to budget - 1, strides 1 to 8, fp32 and bf16, D in {64, 128}."""
    check = None if w.units <= 64 else np.linspace(0, w.units - 1, 24).astype(int)
    _assert(parity.run(w, check_units=check, state_every=16, policy=pol))


def test_policy_decisions_differ():
    """Sanity: on the same inputs the policies evict different positions (so a policy field that
    never reached the kernel would show)."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    w = W["opt-6.7b"].with_(layers=1, batch=1, heads=2, decode_steps=8)
    inp = synth.generate(w)
    dims = parity.dims_of(w)
    seen = {}
    for name, pol in POLICIES.items():
        cache = h2o.H2OCache(dims, w.prompt_len, policy=h2o.Policy(*pol))
        cache.prefill(*(parity.to_device(a, w.dtype) for a in (inp.q_prompt, inp.k_prompt, inp.v_prompt)))
        evicted = []
        for s in range(w.decode_steps):
            _, _, ep = cache.step(*(parity.to_device(a[s], w.dtype) for a in (inp.q_dec, inp.k_dec, inp.v_dec)))
            evicted.append(ep.cpu().numpy().copy())
        torch.cuda.synchronize()
        seen[name] = np.stack(evicted)
    # Local keeps the last `budget` prompt positions and evicts the oldest of them first; sink + window
    # keeps positions 0-3 and the last budget - 4, evicting the oldest of the window
    P, k = w.prompt_len, w.budget
    assert np.array_equal(seen["local"][:, 0], P - k + np.arange(8))
    assert np.array_equal(seen["sink4"][:, 0], P - (k - 4) + np.arange(8))
    keys = [seen[n].tobytes() for n in ("h2o", "local", "sink4", "strided3")]
    assert len(set(keys)) == len(keys)
