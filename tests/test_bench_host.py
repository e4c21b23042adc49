"""bench.py's host-side pieces on CPU: the algorithmic bytes per unit behind every roofline figure,
the kernel each workload's decode step dispatches to, and the oracle baseline's record."""

import argparse
import os

import bench
import synth


def test_decode_bytes_per_unit():
    # n (2 D eb + 12) + 6 D eb + 16: K and V rows, score read + write and position read per slot;
    # q / k_new / v_new in, the victim's K/V row and the output row out; score, position, indices
    assert bench.decode_bytes_per_unit(204, 128, 2) == 204 * 524 + 1552 == 108_448
    assert 8192 * bench.decode_bytes_per_unit(204, 128, 2) == 888_406_016  # one OPT-6.7B launch
    assert bench.decode_bytes_per_unit(32, 64, 4) == 32 * 524 + 1552   # tiny: fp32, D = 64
    # E4M3: codes (2 n D), row scales (8 n), scores and positions (12 n); bf16 q/k/v/out (8 D),
    # the victim's codes (2 D) and scales (8); score, position, indices (16)
    assert bench.decode_bytes_per_unit_e4m3(204, 128) == 204 * 276 + 1304
    assert bench.decode_bytes_per_unit(0, 128, 2) == 6 * 128 * 2 + 16  # empty cache: the token only


def test_decode_kernel_dispatch():
    W = synth.WORKLOADS
    k = lambda name, **kw: bench.decode_kernel(W[name].with_(**kw), 152)[0]
    assert k("opt-6.7b") == "h2o_decode_tc_kernel"             # 8192 units, k = 204
    assert k("llama-7b") == "h2o_decode_tc_kernel"             # 2048 units, k = 460
    assert k("opt-30b") == "h2o_decode_tc_kernel"              # 1792 units, k = 307
    assert k("opt-6.7b", layers=1) == "h2o_decode_resident_kernel"  # 256 units: one layer
    assert k("opt-6.7b", layers=1, budget=209, k_heavy=105) == "h2o_decode_tc_split_kernel"
    assert k("opt-6.7b", layers=1, batch=4) == "h2o_decode_tc_split_kernel"  # 128 units < one per SM
    assert k("streaming") == "h2o_decode_tc_split_kernel"      # 32 units, k = 4096
    assert k("tiny") == "h2o_decode_step_kernel"               # fp32, D = 64
    assert bench.decode_kernel(W["opt-6.7b"], 152, e4m3=True)[0] == "h2o_decode_e4m3_kernel"


def test_prefill_launch_count():
    """One score launch (the one-pass column sums) for bf16 prompts of <= 4 tiles with >= one unit per
    SM, two otherwise; plus the selection."""
    W = synth.WORKLOADS
    n = lambda name, **kw: bench.prefill_launches(W[name].with_(**kw), 152)
    assert n("opt-6.7b") == 2                           # 8192 units x 512 tokens
    assert n("opt-30b") == 2                            # 1792 units x 512
    assert n("opt-6.7b", prompt_len=513) == 3           # five tiles
    assert n("opt-6.7b", layers=1, batch=4) == 3        # 128 units < one per SM
    assert n("opt-6.7b", layers=1, batch=19, heads=8) == 2  # 152 units
    assert n("llama-7b") == 3                           # 2048-token prompts
    assert n("streaming") == 3                          # 32 units
    assert n("tiny") == 3                               # fp32
    k = lambda name, **kw: bench.prefill_score_kernels(W[name].with_(**kw), 152)
    assert k("opt-30b") == "prefill_tc_kernel<D, one pass>"
    assert k("llama-7b").startswith("prefill_tc_kernel<D, row stats>")
    assert "CUDA cores" in k("tiny")


def test_oracle_baseline_record():
    b = bench.cpu_oracle_baseline(synth.WORKLOADS["tiny"], synth.DEFAULT_SEED, target_s=0.2)
    assert b["kind"] == "oracle" and b["unit"] == "tokens/s" and b["cores"] >= 1
    assert b["value"] > 0 and "units" in b["sample"]


def test_config_names_the_workload():
    w = synth.WORKLOADS["opt-6.7b"]
    args = argparse.Namespace(gpus=1, kv_cache="bf16")
    c = bench.config_of(w, args)
    assert c["workload"].startswith("opt-6.7b") and c["units"] == 8192 and c["budget"] == 204
    assert (c["k_heavy"], c["k_local"], c["prompt_len"], c["decode_steps"]) == (102, 102, 512, 512)
    assert "model" not in c


def test_recorded_traffic_is_keyed_by_launch_size():
    """A DRAM-traffic record applies only to launches of the size it was captured on: the E4M3 kernel's
    all-layers record (8192 units per launch) must not be reported for its per-layer launches."""
    import json
    with open(bench.TRAFFIC_FILE) as f:
        recs = json.load(f)["records"]
    assert recs and all(isinstance(r.get("units_per_launch"), int) for r in recs)
    for r in recs:
        src = os.path.join(bench.CSRC, {"h2o_decode_tc_kernel": "h2o_decode_tc.cu",
                                        "h2o_decode_e4m3_kernel": "h2o_decode_e4m3.cu",
                                        "h2o_decode_resident_kernel": "h2o_decode_resident.cu"}[r["kernel"]])
        other = r["units_per_launch"] * 2
        assert bench.recorded_traffic(r["workload"], r["kernel"], src, other) is None


def test_per_layer_calls_and_prefetch_hints():
    """The benchmark's decode step: one call per layer on that layer's slice of every array, each
    naming the next layer's cache arrays as the prefetch hint (layer 0's after the last layer), the
    last launch of a job naming none; E4M3 caches: one plain E4M3 call per layer."""
    import types

    import torch

    import kv_cache_eviction_step_gb300 as h2o
    L, B, H, D, K = 3, 2, 4, 8, 5
    dims = h2o.Dims(units_b=L * B, heads=H, head_dim=D, budget=K, k_heavy=3, k_local=2, dtype=h2o.BF16)
    U = dims.units
    log = []

    def rec(name):
        return lambda *a: log.append((name, a))

    fake = types.SimpleNamespace(
        next_cache=lambda k, v, s, p: ("next", k.data_ptr(), v.data_ptr(), s.data_ptr(), p.data_ptr()),
        h2o_decode_step_prefetch=rec("prefetch"), h2o_decode_step=rec("plain"),
        h2o_decode_step_e4m3=rec("e4m3"))
    cache = types.SimpleNamespace(k_cache=torch.zeros(U, K, D), v_cache=torch.zeros(U, K, D),
                                  scores=torch.zeros(U, K), slot_pos=torch.zeros(U, K, dtype=torch.int32),
                                  k_scale=torch.zeros(U, K), v_scale=torch.zeros(U, K))
    io = [torch.zeros(U, D) for _ in range(4)] + [torch.zeros(U, dtype=torch.int32)] * 2
    q, kn, vn, out, evs, evp = io
    calls = bench.Calls(fake, dims, cache, e4m3=False, layers=L)
    ul = U // L
    for last in (False, True):
        log.clear()
        calls.decode(7, q, kn, vn, out, evs, evp, 0, last=last)
        assert [n for n, _ in log] == ["prefetch"] * L
        for l, (_, a) in enumerate(log):
            d, pol, t = a[0], a[1], a[2]
            assert d.units == ul and pol is None and t == 7
            assert a[3].data_ptr() == q[l * ul:].data_ptr() and a[6].data_ptr() == cache.k_cache[l * ul:].data_ptr()
            nl = (l + 1) % L
            want = ("next", cache.k_cache[nl * ul:].data_ptr(), cache.v_cache[nl * ul:].data_ptr(),
                    cache.scores[nl * ul:].data_ptr(), cache.slot_pos[nl * ul:].data_ptr())
            assert a[-2] == (None if last and l == L - 1 else want), (last, l)
    log.clear()
    calls.decode(7, q, kn, vn, out, evs, evp, 0, hint=False)
    assert [n for n, _ in log] == ["plain"] * L
    log.clear()
    bench.Calls(fake, dims, cache, e4m3=True, layers=L).decode(7, q, kn, vn, out, evs, evp, 0)
    assert [n for n, _ in log] == ["e4m3"] * L
