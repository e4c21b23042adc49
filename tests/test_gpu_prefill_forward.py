"""h2o_prefill_forward on the GPU: the prompt's causal attention output against the oracle's float64
one (within 2e-2 absolute for bf16, 1e-5 for fp32), with the cache it builds checked like
h2o_prefill_select's and then decoded (needs a GB300)."""

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
    ("tiny", {}),                                                       # fp32, D = 64: CUDA cores
    ("opt-6.7b", dict(layers=1, batch=2, heads=3, decode_steps=32)),   # bf16 D = 128, 4 tiles
    ("llama-7b", dict(batch=1, heads=2, decode_steps=16)),             # 16 tiles of 128 rows
    ("opt-30b", dict(batch=1, heads=3, prompt_len=333, decode_steps=16)),  # ragged last tile
    ("opt-6.7b", dict(layers=1, batch=2, heads=2, head_dim=64, prompt_len=300, decode_steps=16)),
    ("opt-6.7b", dict(layers=1, batch=1, heads=2, prompt_len=1, decode_steps=8)),
    ("opt-6.7b", dict(layers=1, batch=1, heads=2, prompt_len=128, decode_steps=8)),
    ("opt-6.7b", dict(layers=1, batch=1, heads=2, prompt_len=129, decode_steps=8)),
    ("opt-6.7b", dict(layers=1, batch=1, heads=2, dtype="f32", prompt_len=200, decode_steps=8)),
])
def test_prefill_forward_output_and_cache(name, kw):
    w = W[name].with_(**kw)
    _assert(parity.run(w, state_every=8, prefill_out=True))


def test_prefill_forward_many_units_sampled():
    """640 units (the launch shape of a real layer batch); the oracle checks 8 of them."""
    w = W["opt-6.7b"].with_(layers=1, batch=20, heads=32, decode_steps=8)
    units = np.linspace(0, w.units - 1, 8).astype(int)
    _assert(parity.run(w, check_units=units, prefill_out=True))


@pytest.mark.parametrize("policy", [(oracle.POLICY_TOPK, 0, 1), (oracle.POLICY_SINK_WINDOW, 4, 1)])
def test_prefill_forward_under_policies(policy):
    w = W["opt-6.7b"].with_(layers=1, batch=2, heads=2, decode_steps=24)
    _assert(parity.run(w, state_every=8, prefill_out=True, policy=policy))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_growing_logits_force_rescaling(dtype):
    """Keys aligned with the queries and growing along the prompt: every 128-key tile's maximum is
    ~11 above the previous one, so the bf16 kernel rescales its running output at every tile."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    P, D, units = 512, 128, 3
    rng = np.random.default_rng(5)
    u = rng.standard_normal(D)
    u /= np.linalg.norm(u)
    q = np.tile(16.0 * u, (units, P, 1)) + 0.1 * rng.standard_normal((units, P, D))
    k = (np.arange(P)[None, :, None] / 16.0) * u[None, None, :] + 0.1 * rng.standard_normal((units, P, D))
    v = rng.standard_normal((units, P, D))
    conv = (lambda a: a.astype(np.float32)) if dtype == "f32" else \
        (lambda a: synth.to_bf16_bits(a.astype(np.float32)))
    q, k, v = conv(q), conv(k), conv(v)
    dims = h2o.Dims(units_b=units, heads=1, head_dim=D, budget=64, k_heavy=32, k_local=32,
                    dtype=h2o.F32 if dtype == "f32" else h2o.BF16)
    dq, dk, dv = (parity.to_device(a, dtype) for a in (q, k, v))
    out = torch.empty_like(dq)
    cache = h2o.H2OCache(dims, P)
    cache.prefill(dq, dk, dv, out=out)
    torch.cuda.synchronize()
    got = parity.widen(parity.to_host(out, dtype))
    ref = oracle.prefill_attention(q, k, v)
    err = float(np.max(np.abs(got - ref)))
    assert err <= parity.OUT_TOL[dtype], err
    # the column sums the cache was built from (the workspace's third array)
    arr = (units * P * 4 + 255) // 256 * 256
    colsum = cache.workspace[2 * arr: 2 * arr + units * P * 4].view(torch.float32).view(units, P)
    orc = oracle.Oracle(64, 32, 32)
    st = orc.new_state(units, D, q.dtype)
    c, _ = orc.prefill_select(q, k, v, st, want_colsum=True)
    rel = np.abs(colsum.cpu().numpy() - c) / np.maximum(c, 1e-3)
    assert rel.max() < 2e-5, rel.max()
