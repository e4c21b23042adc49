"""The one-pass prefill column sums (bf16 prompts of at most four 128-token tiles, at least one unit
per SM): every column sum of sampled units against the oracle's float64 sums around the dispatch
boundaries (units per SM, prompt tiles), the kept slot maps and decode steps that follow, and bit-for-
bit repeatability (needs a GB300)."""

import numpy as np
import pytest

import oracle
import parity
import synth

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    h2o.load()
    torch.cuda.init()
    yield
    assert h2o.h2o_get_device_error() == 0


def _sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


def _colsums(w):
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    inp = synth.generate(w, steps=0)
    dims = parity.dims_of(w)
    q, k = parity.to_device(inp.q_prompt, w.dtype), parity.to_device(inp.k_prompt, w.dtype)
    colsum = torch.empty((w.units, w.prompt_len), dtype=torch.float32, device="cuda")
    ws = torch.empty(h2o.h2o_prefill_workspace_bytes(dims, w.prompt_len), dtype=torch.uint8, device="cuda")
    h2o.h2o_prefill_scores(dims, w.prompt_len, q, k, colsum, ws)
    first = colsum.clone()
    h2o.h2o_prefill_scores(dims, w.prompt_len, q, k, colsum, ws)
    torch.cuda.synchronize()
    return inp, first, colsum


@pytest.mark.parametrize("P", [1, 77, 128, 129, 256, 385, 512, 513])
@pytest.mark.parametrize("per_sm", [0, 1])
def test_column_sums_around_the_dispatch(P, per_sm):
    """Units = SMs - 1 (two passes, work spread over the CTAs) and = SMs (one pass, one unit per CTA);
    prompts of one token, of ragged and full tiles up to 512 tokens (four tiles, the one-pass limit)
    and of 513 (five tiles: two passes). Every column sum of 12 sampled units within 2e-5 relative of
    the oracle's float64 sums; each row of the causal attention sums to 1, so the column sums of a unit
    add up to P; a second call gives the same bits."""
    units = _sms() - 1 + per_sm
    w = W["opt-6.7b"].with_(layers=1, batch=units, heads=1, prompt_len=P, decode_steps=0)
    inp, first, colsum = _colsums(w)
    import torch
    assert torch.equal(first, colsum)
    got = colsum.cpu().numpy().astype(np.float64)
    sample = np.linspace(0, w.units - 1, 12).astype(int)
    orc = oracle.Oracle(w.budget, w.k_heavy, w.k_local)
    st = orc.new_state(len(sample), w.head_dim, synth.storage_dtype(w))
    ref, _ = orc.prefill_select(inp.q_prompt[sample], inp.k_prompt[sample], inp.v_prompt[sample], st,
                                want_colsum=True)
    rel = np.abs(got[sample] - ref) / np.maximum(ref, 1e-3)
    assert rel.max() < 2e-5, rel.max()
    assert np.allclose(got.sum(axis=1), P, rtol=1e-5)


@pytest.mark.parametrize("P,budget,k_local", [(200, 64, 32), (512, 204, 102), (390, 400, 200)])
def test_one_pass_prefill_then_decode(P, budget, k_local):
    """The kept sets the one-pass column sums lead to (heavy hitters plus the local window, a budget
    above the prompt keeping every token) and 16 decode steps after them, 16 sampled units of 304
    (two per SM), decisions exact under the near-tie rule."""
    w = W["opt-6.7b"].with_(layers=1, batch=2 * _sms(), heads=1, prompt_len=P, decode_steps=16,
                            budget=budget, k_heavy=budget - k_local, k_local=k_local)
    units = np.linspace(0, w.units - 1, 16).astype(int)
    parity.check(parity.run(w, check_units=units, state_every=8))


@pytest.mark.parametrize("P", [1, 100, 300, 512])
def test_one_pass_head_dim_64(P):
    """The one-pass kernel's D = 64 shape (one 64-column TMA box per 32-row block, an 8-deep streamed
    ring, four K steps per tile product) at one unit per SM: every column sum of 12 sampled units
    against the oracle, a repeated call bit-identical, then the kept slot maps and 8 decode steps."""
    import torch
    units = _sms()
    w = W["opt-6.7b"].with_(layers=1, batch=units, heads=1, head_dim=64, prompt_len=P, decode_steps=8,
                            budget=64, k_heavy=32, k_local=32)
    inp, first, colsum = _colsums(w)
    assert torch.equal(first, colsum)
    got = colsum.cpu().numpy().astype(np.float64)
    sample = np.linspace(0, w.units - 1, 12).astype(int)
    orc = oracle.Oracle(w.budget, w.k_heavy, w.k_local)
    st = orc.new_state(len(sample), w.head_dim, synth.storage_dtype(w))
    ref, _ = orc.prefill_select(inp.q_prompt[sample], inp.k_prompt[sample], inp.v_prompt[sample], st,
                                want_colsum=True)
    rel = np.abs(got[sample] - ref) / np.maximum(ref, 1e-3)
    assert rel.max() < 2e-5, rel.max()
    parity.check(parity.run(w, check_units=sample, state_every=4))
