"""CUDA path vs the CPU oracle, through the C ABI, on the same seeded inputs (needs a GB300)."""

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


def test_tiny_workload_every_unit_every_step():
    """batch 1, 2 heads, d=64 fp32, 64+64, k=32 (16+16): the whole workload against the oracle."""
    _assert(parity.run(W["tiny"], state_every=8))


@pytest.mark.parametrize("name,kw", [
    ("opt-6.7b", dict(layers=1, batch=2, heads=3)),
    ("llama-7b", dict(batch=1, heads=3)),
    ("opt-30b", dict(batch=1, heads=3)),
    ("streaming", dict(heads=2, decode_steps=4800)),
])
def test_workload_shapes_on_few_units(name, kw):
    """Each workload's prompt length, budget split, head dim and dtype on a few units, so the oracle
    runs every unit; few units also make the decode step split each unit over a CTA cluster."""
    w = W[name].with_(**kw)
    _assert(parity.run(w, state_every=128))


def _sweep_cases():
    rng = np.random.default_rng(7)
    cases = []
    for i in range(14):
        D = int(rng.choice([64, 128]))
        dtype = "f32" if i % 3 == 0 else "bf16"
        budget = int(rng.choice([1, 2, 5, 17, 33, 63, 100, 129]))
        regime = i % 4
        P = {0: max(1, budget // 2), 1: budget, 2: budget + 1 + int(rng.integers(0, 60)),
             3: int(rng.integers(1, 3 * budget + 2))}[regime]
        kl = int(rng.choice([0, 1, budget, budget // 2]))
        units_b = int(rng.choice([1, 3, 40, 200]))
        heads = int(rng.choice([1, 2, 5]))
        cases.append(synth.Workload(
            f"sweep{i}", layers=1, batch=units_b, heads=heads, head_dim=D, dtype=dtype,
            prompt_len=P, decode_steps=int(rng.integers(1, 70)), budget=budget,
            k_heavy=budget - kl, k_local=kl, hh_kind="pareto",
            hh_count=max(1, (P + 70) // 20), q_boost=1.0))
    return cases


@pytest.mark.parametrize("w", _sweep_cases(), ids=lambda w: f"{w.name}-D{w.head_dim}-{w.dtype}-k{w.budget}"
                         f"-kl{w.k_local}-P{w.prompt_len}-u{w.units}")
def test_sweep(w):
    """Odd budgets, prompts shorter / equal / longer than the budget, k_local in {0, 1, k/2, k},
    D in {64, 128}, fp32 and bf16, 1 to 1000 units (1 to 16 CTAs per unit)."""
    check = None if w.units <= 64 else np.linspace(0, w.units - 1, 24).astype(int)
    _assert(parity.run(w, check_units=check, state_every=16))


@pytest.mark.parametrize("name,kw", [
    ("opt-6.7b", dict(layers=1, batch=20, heads=32, decode_steps=96)),
    ("llama-7b", dict(batch=20, heads=32, decode_steps=48)),
    ("opt-30b", dict(batch=12, heads=56, decode_steps=64, prompt_len=100, budget=300, k_heavy=150,
                     k_local=150)),
    ("opt-6.7b", dict(layers=1, batch=20, heads=32, decode_steps=40, prompt_len=600, budget=512,
                      k_heavy=511, k_local=1)),
])
def test_tensor_core_decode_path(name, kw):
    """At least 4 units per SM with bf16, D = 128 and budgets up to 512 take the tcgen05 decode
    kernel: 2 and 4 tiles of 128 slots, a cache that grows from 100 to 300 slots before evicting,
    and the largest budget with k_local = 1. The oracle follows sampled units through every step."""
    w = W[name].with_(**kw)
    assert w.units >= 608 and w.head_dim == 128 and w.dtype == "bf16" and w.budget <= 512
    units = np.linspace(0, w.units - 1, 10).astype(int)
    _assert(parity.run(w, check_units=units, state_every=16))


def test_prefill_column_sums_elementwise():
    """P1-P2 alone: h2o_prefill_scores against the oracle's float64 column sums, every element."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    for name, kw in [("opt-6.7b", dict(layers=1, batch=1, heads=4)), ("tiny", {}),
                     ("llama-7b", dict(batch=1, heads=2)), ("opt-30b", dict(batch=1, heads=2, prompt_len=333))]:
        w = W[name].with_(**kw)
        inp = synth.generate(w, steps=0)
        dims = parity.dims_of(w)
        q, k = parity.to_device(inp.q_prompt, w.dtype), parity.to_device(inp.k_prompt, w.dtype)
        colsum = torch.empty((w.units, w.prompt_len), dtype=torch.float32, device="cuda")
        ws = torch.empty(h2o.h2o_prefill_workspace_bytes(dims, w.prompt_len), dtype=torch.uint8, device="cuda")
        h2o.h2o_prefill_scores(dims, w.prompt_len, q, k, colsum, ws)
        got = colsum.cpu().numpy().astype(np.float64)
        orc = oracle.Oracle(w.budget, w.k_heavy, w.k_local)
        st = orc.new_state(w.units, w.head_dim, synth.storage_dtype(w))
        ref, _ = orc.prefill_select(inp.q_prompt, inp.k_prompt, inp.v_prompt, st, want_colsum=True)
        rel = np.abs(got - ref) / np.maximum(ref, 1e-3)
        assert rel.max() < 2e-5, (name, rel.max())
        assert np.allclose(got.sum(axis=1), w.prompt_len, rtol=1e-5)


def test_exact_ties_evict_lowest_position():
    """Hand-built full caches whose updated scores tie exactly (all-zero keys and queries give
    equal weights): the GPU must evict the lowest position, like the oracle."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    budget, D = 8, 64
    for t, kl, pos, sc, want in [
        (14, 1, [7, 3, 9, 5, 12, 4, 11, 10], [0.5] * 8, 1),                     # lowest position 3
        (15, 3, [12, 3, 14, 5, 2, 9, 13, 10], [0.25] * 8, 4),                   # 2 (13, 14 protected)
        (15, 2, [5, 8, 2, 9, 10, 11, 12, 13], [0.25, 0.5, 0.25, 0.75, 1, 1, 1, 1], 2),  # 5 vs 2 -> 2
        (14, 8, [7, 6, 9, 8, 10, 11, 12, 13], [0.0, 9.0, 0, 0, 0, 0, 0, 0], 1),  # window: only 6
    ]:
        d = h2o.Dims(units_b=1, heads=1, head_dim=D, budget=budget, k_heavy=budget - kl, k_local=kl,
                     dtype=h2o.BF16)
        z = torch.zeros((1, D), dtype=torch.bfloat16, device="cuda")
        kc = torch.zeros((1, budget, D), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        scores = torch.tensor([sc], dtype=torch.float32, device="cuda")
        sp = torch.tensor([pos], dtype=torch.int32, device="cuda")
        out = torch.empty_like(z)
        es = torch.empty(1, dtype=torch.int32, device="cuda")
        ep = torch.empty_like(es)
        h2o.h2o_decode_step(d, t, z, z, z + 1, kc, vc, scores, sp, out, es, ep)
        torch.cuda.synchronize()
        assert es.item() == want and ep.item() == pos[want], (kl, es.item(), ep.item())
        assert sp[0, want].item() == t
        assert torch.all(vc[0, want] == 1)
        # oracle on the same state agrees
        orc = oracle.Oracle(budget, budget - kl, kl)
        st = orc.new_state(1, D, np.uint16)
        st.slot_pos[0], st.scores[0] = pos, sc
        zz = np.zeros((1, D), dtype=np.uint16)
        _, oes, _, _, _ = orc.decode_step(t, zz, zz, zz, st)
        assert oes[0] == want
        assert np.array_equal(scores.cpu().numpy(), st.scores)


def test_device_error_word_reports_a_timed_out_wait():
    """The bounded wait gives up on a barrier nothing completes, sets the error word and returns;
    the context stays usable."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    assert h2o.h2o_get_device_error() == 0
    h2o.h2o_selftest_wait_timeout()
    assert h2o.h2o_get_device_error() == h2o.DEVERR_WAIT_TIMEOUT
    assert h2o.h2o_get_device_error() == 0  # cleared
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


def test_rejected_calls_leave_state_untouched():
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    d = h2o.Dims(units_b=1, heads=2, head_dim=64, budget=4, k_heavy=2, k_local=2, dtype=h2o.F32)
    kc = torch.full((2, 4, 64), 3.0, device="cuda")
    with pytest.raises(h2o.H2OError):
        bad = h2o.Dims(units_b=1, heads=2, head_dim=64, budget=4, k_heavy=3, k_local=2, dtype=h2o.F32)
        z = torch.zeros((2, 64), device="cuda")
        s = torch.zeros((2, 4), device="cuda")
        p = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
        e = torch.zeros(2, dtype=torch.int32, device="cuda")
        h2o.h2o_decode_step(bad, 5, z, z, z, kc, kc, s, p, z, e, e)
    assert torch.all(kc == 3.0)


@pytest.mark.slow
@pytest.mark.parametrize("name,check", [("opt-6.7b", 8), ("llama-7b", 4), ("opt-30b", 6)])
def test_full_size_workload_sampled_units(name, check):
    """The full workload in the launch shape the benchmark times; the oracle follows sampled units
    (spread over layers, sequences and heads) through every step."""
    w = W[name]
    units = np.linspace(0, w.units - 1, check).astype(int)
    _assert(parity.run(w, check_units=units, state_every=64))


def test_per_layer_launch_shape():
    """One OPT-6.7B layer per launch (batch 8 x 32 heads = 256 units, k = 204), the shape of the
    benchmark's per-layer decode timing: between one and four units per SM with a budget of at most
    208, so the resident one-CTA-per-unit kernel runs; the oracle follows 16 sampled units through
    every step."""
    w = W["opt-6.7b"].with_(layers=1, decode_steps=96)
    assert w.units == 256
    units = np.linspace(0, w.units - 1, 16).astype(int)
    _assert(parity.run(w, check_units=units, state_every=32))


def test_streaming_segments_small():
    """The segmented long-run check of the streaming workload on a short run (2 units, 4800 steps,
    segments of 1024 steps: growth to the budget inside the first segment, then evicting steps),
    so that the machinery the full-length test relies on is itself checked quickly."""
    w = W["streaming"].with_(heads=2, decode_steps=4800, budget=2048, k_heavy=1024, k_local=1024)
    _assert(parity.run_segments(w, check_units=[0, 1], seg_len=1024))


@pytest.mark.slow
def test_streaming_full_length_every_step_against_the_oracle():
    """512 + 262144 steps at budget 4096 (2048 heavy + 2048 local), all 32 units on the GPU. Every
    step of units 0, 17 and 31 is checked against the oracle (evictions exact, outputs within 2e-2), in 16
    segments of 16384 steps run on all host cores; each segment starts from the GPU state, which
    must equal where the oracle's previous segment ended (slot map and K/V rows exactly, scores within
    the float32 tolerance). Every 4096 steps, invariants that hold at any length are checked on every
    unit: slot map valid, recent window resident, K/V rows equal to the generated rows of their
    positions, scores finite and bounded by the number of queries."""
    import torch

    w = W["streaming"]
    U, k, kl, P = w.units, w.budget, w.k_local, w.prompt_len
    sample_units = [0, 13, 31]

    def props(cache, t):
        sp = parity.to_host(cache.slot_pos, "i32")
        sc = parity.to_host(cache.scores, "f32")
        n = min(t + 1, k)
        for u in range(U):
            pos = sp[u][sp[u] >= 0]
            assert len(pos) == n and len(np.unique(pos)) == n, (t, u)
            recent = np.arange(max(0, t - kl + 1), t + 1)
            assert np.isin(recent, pos).all(), (t, u)
        assert np.isfinite(sc).all() and (sc >= 0).all()
        assert (sc.sum(axis=1, dtype=np.float64) <= t + 1 + 1e-2).all()
        kc = parity.to_host(cache.k_cache, w.dtype)
        vc = parity.to_host(cache.v_cache, w.dtype)
        lo = max(0, t + 1 - 4096)  # regenerate the most recent 4096 positions only
        for u in sample_units:
            rows = sp[u]
            gen = synth.unit_sequence(w, synth.DEFAULT_SEED, u, lo, t + 1)
            sel = rows >= lo
            assert np.array_equal(kc[u][sel], gen[1][rows[sel] - lo]), (t, u)
            assert np.array_equal(vc[u][sel], gen[2][rows[sel] - lo]), (t, u)

    rep = parity.run_segments(w, check_units=[0, 17, 31], seg_len=16384, property_checks=props)
    assert rep.decisions >= 3 * (w.decode_steps - (k - P)), rep.decisions
    _assert(rep)
    torch.cuda.synchronize()


@pytest.mark.parametrize("e4m3", [False, True])
def test_layer_interleaved_steps_match_one_cache_at_a_time(e4m3):
    """Per-layer decoding: two caches (two layers of 256 units, k = 204) stepped alternately on one
    stream, so that every launch may load its cache before the previous launch (the other layer's)
    has finished, give outputs, evictions and cache state bit-identical to stepping one cache at a
    time (where consecutive launches share a cache and each waits for the last)."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    w = W["opt-6.7b"].with_(layers=1, decode_steps=40)
    dims = parity.dims_of(w)
    keys = ("q_prompt", "k_prompt", "v_prompt", "q_dec", "k_dec", "v_dec")
    dev = []
    for i in range(2):
        inp = synth.generate(w, seed=synth.DEFAULT_SEED + 101 * i)
        dev.append({k: parity.to_device(getattr(inp, k), w.dtype) for k in keys})
    S, U, D = w.decode_steps, w.units, w.head_dim

    def run(interleaved):
        caches = [h2o.H2OCache(dims, w.prompt_len, e4m3=e4m3) for _ in range(2)]
        outs = [torch.empty((S, U, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        evs = [torch.empty((S, U), dtype=torch.int32, device="cuda") for _ in range(2)]
        evp = [torch.empty((S, U), dtype=torch.int32, device="cuda") for _ in range(2)]
        for c, d in zip(caches, dev):
            c.prefill(d["q_prompt"], d["k_prompt"], d["v_prompt"])
        order = ([(s, l) for s in range(S) for l in range(2)] if interleaved else
                 [(s, l) for l in range(2) for s in range(S)])
        for s, l in order:
            d = dev[l]
            caches[l].step(d["q_dec"][s], d["k_dec"][s], d["v_dec"][s], out=outs[l][s],
                           evicted_slot=evs[l][s], evicted_pos=evp[l][s])
        torch.cuda.synchronize()
        got = outs + evs + evp
        for c in caches:
            got += [c.k_cache, c.v_cache, c.scores, c.slot_pos]
            if e4m3:
                got += [c.k_scale, c.v_scale]
        return got

    a, b = run(True), run(False)
    assert len(a) == len(b)
    for i, (x, y) in enumerate(zip(a, b)):
        assert torch.equal(x, y), i
    assert h2o.h2o_get_device_error() == 0


@pytest.mark.parametrize("units,e4m3", [(151, False), (152, False), (153, False), (607, False), (608, False),
                                         (609, False), (151, True), (152, True), (153, True)])
def test_unit_counts_around_the_dispatch_and_grid_boundaries(units, e4m3):
    """Unit counts on both sides of one unit per SM (152: the persistent kernels' grid) and of four
    per SM (608: where the bf16 step moves from the cluster-split to the persistent kernel), with the
    OPT-6.7B budget; the first, last and middle units checked through every step."""
    w = W["opt-6.7b"].with_(layers=1, batch=units, heads=1, decode_steps=24)
    assert w.units == units
    check = [0, units // 2, units - 1]
    _assert(parity.run(w, check_units=check, state_every=8, e4m3=e4m3))


@pytest.mark.slow
@pytest.mark.parametrize("budget,P,steps", [
    (6000, 6100, 12),     # n > 4096: the tensor-core step split over 16-CTA clusters
    (9000, 9100, 12),     # n > 8192: the CUDA-core step
    (16384, 16384, 4),    # the largest prompt and budget the library takes (cache full from t = P)
])
def test_long_caches_and_largest_sizes(budget, P, steps):
    """One unit (bf16, D = 128) with caches beyond 4096 and 8192 slots and at the size limits: the
    prefill's selection over long prompts and evicting decode steps, every step checked."""
    kh = budget // 2
    w = W["streaming"].with_(heads=1, prompt_len=P, decode_steps=steps, budget=budget, k_heavy=kh,
                             k_local=budget - kh)
    assert w.units == 1
    _assert(parity.run(w, state_every=4))


def test_long_prompt_column_sums_and_selection():
    """A 4096-token prompt (32 tiles of 128 rows per unit) on the tensor-core passes: every column sum
    against the oracle, the kept slot map, and a few decode steps."""
    w = W["llama-7b"].with_(batch=1, heads=2, prompt_len=4096, decode_steps=4, budget=1024,
                            k_heavy=512, k_local=512)
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    inp = synth.generate(w, steps=0)
    dims = parity.dims_of(w)
    q, k = parity.to_device(inp.q_prompt, w.dtype), parity.to_device(inp.k_prompt, w.dtype)
    colsum = torch.empty((w.units, w.prompt_len), dtype=torch.float32, device="cuda")
    ws = torch.empty(h2o.h2o_prefill_workspace_bytes(dims, w.prompt_len), dtype=torch.uint8, device="cuda")
    h2o.h2o_prefill_scores(dims, w.prompt_len, q, k, colsum, ws)
    got = colsum.cpu().numpy().astype(np.float64)
    orc = oracle.Oracle(w.budget, w.k_heavy, w.k_local)
    st = orc.new_state(w.units, w.head_dim, synth.storage_dtype(w))
    ref, _ = orc.prefill_select(inp.q_prompt, inp.k_prompt, inp.v_prompt, st, want_colsum=True)
    rel = np.abs(got - ref) / np.maximum(ref, 1e-3)
    assert rel.max() < 2e-5, rel.max()
    _assert(parity.run(w, state_every=2))


@pytest.mark.parametrize("middle", ["select", "forward", "select_e4m3"])
def test_prefill_between_decodes_of_different_caches(middle):
    """decode(A) -> prefill(B) -> decode(B) on one stream, six rounds, B prefilled again each round,
    in the per-layer launch shape (256 units, k = 204), where a decode launch may read its cache
    before waiting for the launch before it: the prefill in between writes B's cache, so decode(B)
    must see all of it. Outputs, evictions and both caches' state must be bit-identical to the same
    calls with the stream synchronised after each one."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    e4m3 = middle == "select_e4m3"
    w = W["opt-6.7b"].with_(layers=1, decode_steps=12)
    dims = parity.dims_of(w)
    keys = ("q_prompt", "k_prompt", "v_prompt", "q_dec", "k_dec", "v_dec")
    dev = []
    for i in range(2):
        inp = synth.generate(w, seed=synth.DEFAULT_SEED + 37 * i)
        dev.append({k: parity.to_device(getattr(inp, k), w.dtype) for k in keys})
    U, D, P = w.units, w.head_dim, w.prompt_len
    rounds = 6

    def run(sync):
        a = h2o.H2OCache(dims, P, e4m3=e4m3)
        b = h2o.H2OCache(dims, P, e4m3=e4m3)
        a.prefill(dev[0]["q_prompt"], dev[0]["k_prompt"], dev[0]["v_prompt"])
        torch.cuda.synchronize()
        pout = torch.empty((U, P, D), dtype=torch.bfloat16, device="cuda")
        got = []
        for r in range(rounds):
            o = torch.empty((2, U, D), dtype=torch.bfloat16, device="cuda")
            es = torch.empty((2, U), dtype=torch.int32, device="cuda")
            ep = torch.empty((2, U), dtype=torch.int32, device="cuda")
            a.step(dev[0]["q_dec"][r], dev[0]["k_dec"][r], dev[0]["v_dec"][r], out=o[0],
                   evicted_slot=es[0], evicted_pos=ep[0])
            if sync:
                torch.cuda.synchronize()
            b.prefill(dev[1]["q_prompt"], dev[1]["k_prompt"], dev[1]["v_prompt"],
                      out=pout if middle == "forward" else None)
            if sync:
                torch.cuda.synchronize()
            b.step(dev[1]["q_dec"][r], dev[1]["k_dec"][r], dev[1]["v_dec"][r], out=o[1],
                   evicted_slot=es[1], evicted_pos=ep[1])
            if sync:
                torch.cuda.synchronize()
            got += [o, es, ep]
        torch.cuda.synchronize()
        for c in (a, b):
            got += [c.k_cache, c.v_cache, c.scores, c.slot_pos]
            if e4m3:
                got += [c.k_scale, c.v_scale]
        return got

    x, y = run(False), run(True)
    assert len(x) == len(y)
    for i, (p, q) in enumerate(zip(x, y)):
        assert torch.equal(p, q), i
    assert h2o.h2o_get_device_error() == 0


@pytest.mark.parametrize("P", [100, 256, 300, 512])
def test_prefill_with_many_units(P):
    """At least 8 units per SM, prompts of 1 to 4 tiles: the one-pass column sums (CTAs take whole
    units). 1280 OPT-6.7B-shaped units: every column sum of 40 sampled units against the oracle's
    float64 sums, then the kept slot maps and 8 decode steps."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o
    w = W["opt-6.7b"].with_(layers=1, batch=40, heads=32, decode_steps=8, prompt_len=P)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert w.units >= 8 * sms
    units = np.linspace(0, w.units - 1, 40).astype(int)
    inp = synth.generate(w, steps=0)
    dims = parity.dims_of(w)
    q, k = parity.to_device(inp.q_prompt, w.dtype), parity.to_device(inp.k_prompt, w.dtype)
    colsum = torch.empty((w.units, w.prompt_len), dtype=torch.float32, device="cuda")
    ws = torch.empty(h2o.h2o_prefill_workspace_bytes(dims, w.prompt_len), dtype=torch.uint8, device="cuda")
    h2o.h2o_prefill_scores(dims, w.prompt_len, q, k, colsum, ws)
    got = colsum.cpu().numpy().astype(np.float64)
    orc = oracle.Oracle(w.budget, w.k_heavy, w.k_local)
    st = orc.new_state(len(units), w.head_dim, synth.storage_dtype(w))
    ref, _ = orc.prefill_select(inp.q_prompt[units], inp.k_prompt[units], inp.v_prompt[units], st,
                                want_colsum=True)
    rel = np.abs(got[units] - ref) / np.maximum(ref, 1e-3)
    print(f"P={P}: column sums max rel err {rel.max():.2e}")
    assert rel.max() < 2e-5, rel.max()
    assert np.allclose(got.sum(axis=1), w.prompt_len, rtol=1e-5)
    _assert(parity.run(w, check_units=units, state_every=8))
