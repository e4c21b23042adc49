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


@pytest.mark.parametrize("gain,P", [(8.0, 512), (40.0, 512), (40.0, 300)])
@pytest.mark.parametrize("per_sm", [0, 1])
def test_column_sums_with_wide_logit_ranges(gain, P, per_sm):
    """Queries scaled by 8 and by 40 (then rounded to bf16; the oracle takes the same bits): logits
    spread over tens to hundreds of natural-log units, so rows are close to one-hot, a row's running
    maximum jumps between key tiles (the rescale path) and most exponentials underflow. One pass (152
    units) and two passes (151 units): every column sum of 12 sampled units against the oracle's
    float64 sums, the sums of each unit adding up to P, and a repeated call giving the same bits.
    Tolerance: the logits are fp32 sums of 128 exact bf16 products, whose rounding grows with the
    logit's size L (log2 units) and enters every weight's exponent, so relative 2e-5 + 2^-21 L (L the
    unit's largest |q.k| log2(e) / sqrt(D)); 2e-5 at the unscaled inputs."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    units = _sms() - 1 + per_sm
    w = W["opt-6.7b"].with_(layers=1, batch=units, heads=1, prompt_len=P, decode_steps=0)
    inp = synth.generate(w, steps=0)
    qs = synth.to_bf16_bits(synth.bf16_bits_to_f32(inp.q_prompt) * np.float32(gain))
    dims = parity.dims_of(w)
    q, k = parity.to_device(qs, w.dtype), parity.to_device(inp.k_prompt, w.dtype)
    colsum = torch.empty((w.units, P), dtype=torch.float32, device="cuda")
    ws = torch.empty(h2o.h2o_prefill_workspace_bytes(dims, P), dtype=torch.uint8, device="cuda")
    h2o.h2o_prefill_scores(dims, P, q, k, colsum, ws)
    first = colsum.clone()
    h2o.h2o_prefill_scores(dims, P, q, k, colsum, ws)
    torch.cuda.synchronize()
    assert torch.equal(first, colsum)
    got = colsum.cpu().numpy().astype(np.float64)
    sample = np.linspace(0, w.units - 1, 12).astype(int)
    orc = oracle.Oracle(w.budget, w.k_heavy, w.k_local)
    st = orc.new_state(len(sample), w.head_dim, synth.storage_dtype(w))
    ref, _ = orc.prefill_select(qs[sample], inp.k_prompt[sample], inp.v_prompt[sample], st, want_colsum=True)
    q64, k64 = synth.bf16_bits_to_f32(qs[sample]).astype(np.float64), synth.bf16_bits_to_f32(inp.k_prompt[sample]).astype(np.float64)
    lmax = np.abs(np.einsum("uid,ujd->uij", q64, k64)).max(axis=(1, 2)) / np.sqrt(w.head_dim) / np.log(2.0)
    tol = 2e-5 + 2.0 ** -21 * lmax[:, None]
    rel = np.abs(got[sample] - ref) / np.maximum(ref, 1e-3)
    print(f"gain {gain}, P {P}, units {units}: largest logit {lmax.max():.0f} (log2 units), "
          f"column sums max rel err {rel.max():.2e}, worst err / tol {(rel / tol).max():.2f}")
    assert (rel < tol).all(), (rel / tol).max()
    assert np.allclose(got.sum(axis=1), P, rtol=1e-5)
