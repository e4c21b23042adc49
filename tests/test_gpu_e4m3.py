"""The quantised cache (FP8 E4M3 codes with one float32 scale per row) on the GPU against the
oracle's quantised cache, through the C ABI (needs a GB300): eviction decisions and slot maps
exact (near ties as for bf16), codes and scales bit for bit, outputs within the bf16 tolerance."""

import numpy as np
import pytest

import oracle
import parity
import synth

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


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


@pytest.mark.parametrize("name,kw", [
    ("opt-6.7b", dict(layers=1, batch=2, heads=3, decode_steps=160)),            # k = 204, 2 tiles
    ("llama-7b", dict(batch=1, heads=3, decode_steps=48)),                       # k = 460, 4 tiles
    ("opt-30b", dict(batch=1, heads=3, prompt_len=333, decode_steps=64)),        # k = 307
    ("opt-6.7b", dict(layers=1, batch=1, heads=4, prompt_len=100, decode_steps=150)),  # cache fills up
    ("opt-6.7b", dict(layers=1, batch=1, heads=2, prompt_len=600, budget=512, k_heavy=511, k_local=1,
                      decode_steps=40)),
])
def test_e4m3_every_unit(name, kw):
    w = W[name].with_(**kw)
    _assert(parity.run(w, state_every=16, e4m3=True))


def test_e4m3_many_units_sampled():
    """640 units (the persistent kernel on every SM, several units per CTA); 8 sampled."""
    w = W["opt-6.7b"].with_(layers=1, batch=20, heads=32, decode_steps=64)
    units = np.linspace(0, w.units - 1, 8).astype(int)
    _assert(parity.run(w, check_units=units, state_every=16, e4m3=True))


def test_e4m3_per_layer_launch_shape():
    """One OPT-6.7B layer per launch (256 units: one or two per CTA); 16 sampled."""
    w = W["opt-6.7b"].with_(layers=1, decode_steps=96)
    units = np.linspace(0, w.units - 1, 16).astype(int)
    _assert(parity.run(w, check_units=units, state_every=32, e4m3=True))


@pytest.mark.slow
@pytest.mark.parametrize("name,check", [("opt-6.7b", 8), ("llama-7b", 4), ("opt-30b", 6)])
def test_e4m3_full_size_workload_sampled_units(name, check):
    """The full workload over the E4M3 cache in the launch shape the benchmark times (both kernel
    instantiations: two tiles for OPT-6.7B, four for LLaMA-7B and OPT-30B); sampled units."""
    w = W[name]
    units = np.linspace(0, w.units - 1, check).astype(int)
    _assert(parity.run(w, check_units=units, state_every=64, e4m3=True))


@pytest.mark.parametrize("policy", [(oracle.POLICY_LOCAL, 0, 1), (oracle.POLICY_SINK_WINDOW, 4, 1),
                                    (oracle.POLICY_TOPK, 0, 1), (oracle.POLICY_STRIDED, 0, 3)])
def test_e4m3_policies(policy):
    w = W["opt-6.7b"].with_(layers=1, batch=2, heads=2, decode_steps=64)
    _assert(parity.run(w, state_every=16, policy=policy, e4m3=True))


def _sweep():
    rng = np.random.default_rng(21)
    out = []
    for i in range(10):
        budget = int(rng.choice([1, 2, 5, 33, 128, 129, 255, 512]))
        P = int(rng.integers(1, 2 * budget + 3))
        kl = int(rng.choice([0, 1, budget // 2, budget]))
        out.append(synth.Workload(
            f"e4m3sweep{i}", layers=1, batch=int(rng.choice([1, 3, 7])), heads=int(rng.choice([1, 2])),
            head_dim=128, dtype="bf16", prompt_len=P, decode_steps=int(rng.integers(1, 50)),
            budget=budget, k_heavy=budget - kl, k_local=kl, hh_kind="pareto",
            hh_count=max(1, (P + 50) // 20), q_boost=1.0))
    return out


@pytest.mark.parametrize("w", _sweep(), ids=lambda w: f"{w.name}-k{w.budget}-kl{w.k_local}-P{w.prompt_len}-u{w.units}")
def test_e4m3_sweep(w):
    """Budgets 1 to 512 (partial and whole tiles), prompts shorter and longer than the budget."""
    _assert(parity.run(w, state_every=8, e4m3=True))


def test_e4m3_rejects_unsupported_shapes():
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    for kw, status in [(dict(head_dim=64), h2o.ERR_UNSUPPORTED), (dict(dtype=h2o.F32), h2o.ERR_UNSUPPORTED),
                       (dict(budget=600, k_heavy=300, k_local=300), h2o.ERR_UNSUPPORTED)]:
        base = dict(units_b=1, heads=1, head_dim=128, budget=8, k_heavy=4, k_local=4, dtype=h2o.BF16)
        base.update(kw)
        d = h2o.Dims(**base)
        z = torch.zeros(16, dtype=torch.float32, device="cuda")
        with pytest.raises(h2o.H2OError) as e:
            h2o.h2o_decode_step_e4m3(d, None, 10, z, z, z, z, z, z, z, z, z, z, z, z)
        assert e.value.status == status
