"""Seeded synthetic inputs for the H2O decode-step and prefill workloads.

This module only draws numbers. It holds none of the H2O arithmetic (no attention, no scores,
no eviction), so both the CUDA path and the CPU oracle can take their inputs from it without
sharing any of the method's code.

Workloads are shaped like the attention layers the H2O summary post (ttsmallhot.github.io,
§3.1.2 测试的模型) lists -- OPT-6.7B, LLaMA-7B, OPT-30B -- and like its padded fixed-length
prompt+generation runs (§3.2.2 效率实验: 512+512, 512+1024). No dataset is used; the
heavy-hitter structure that makes eviction non-trivial is planted on purpose: a fixed unit
direction ``u`` is added to some keys, and every query leans towards ``u``, so those keys soak
up attention (the power-law "Heavy-Hitter" observation of the same post, §2.1.2). Boosted
positions are shared by all layers and heads of one sequence (heavy-hitter sets overlap across
heads: "H2O Heavy-Hitter Oracle 分析", §3.1) and differ between sequences.

Recipe (all draws from numpy's PCG64 through ``SeedSequence`` so any subset of units and
positions can be regenerated independently and identically):

* ``u``: a standard normal vector in R^D from stream ``[seed, 0x5EED_0001]``, normalised.
* Boosted positions of sequence ``b``: stream ``[seed, 0x5EED_0002, b]``.  ``"fixed"`` workloads
  pick ``hh_count`` distinct prompt positions and add ``k_boost * u``; ``"pareto"`` workloads pick
  ``hh_count`` distinct positions over prompt+generation and add ``beta * u`` with
  ``beta = min(cap, (1 - U) ** (-1 / alpha))`` (classical Pareto, x_m = 1).
* Q/K/V of unit ``g`` (g = (layer * batch + b) * heads + h), positions ``[1024 j, 1024 j + 1024)``:
  float32 standard normals of shape (3, 1024, D) from stream ``[seed, 0x5EED_0003, g, j]``.
* Every query gets ``+ q_boost * u``.  Sums are taken in float64, rounded to float32, and for bf16
  workloads rounded once more to bf16 with round-to-nearest-even (stored as uint16 bit patterns).

Layouts: prompt tensors ``[units, P, D]``; per-step decode tensors ``[S, units, D]`` so one step's
inputs are contiguous.
"""

from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

BLOCK = 1024  # positions per independent normal stream block

_TAG_U = 0x5EED_0001
_TAG_HH = 0x5EED_0002
_TAG_QKV = 0x5EED_0003


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and heavy-hitter recipe of one synthetic workload."""

    name: str
    layers: int
    batch: int
    heads: int
    head_dim: int
    dtype: str  # "f32" or "bf16"
    prompt_len: int
    decode_steps: int
    budget: int
    k_heavy: int
    k_local: int
    hh_kind: str  # "fixed" or "pareto"
    hh_count: int  # boosted positions per sequence
    k_boost: float = 3.0  # "fixed": key += k_boost * u
    pareto_alpha: float = 1.5
    pareto_cap: float = 8.0
    q_boost: float = 1.0
    note: str = ""

    @property
    def units_b(self) -> int:
        """Independent (layer, sequence) rows; each has ``heads`` units."""
        return self.layers * self.batch

    @property
    def units(self) -> int:
        return self.layers * self.batch * self.heads

    @property
    def total_len(self) -> int:
        return self.prompt_len + self.decode_steps

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    "tiny": Workload(
        "tiny", layers=1, batch=1, heads=2, head_dim=64, dtype="f32",
        prompt_len=64, decode_steps=64, budget=32, k_heavy=16, k_local=16,
        hh_kind="fixed", hh_count=4, k_boost=3.0, q_boost=1.5,
        note="batch 1, 1 layer, 2 heads, d=64 fp32; 64+64; k=32 (16+16); 4 prompt keys += 3u, q += 1.5u"),
    "opt-6.7b": Workload(
        "opt-6.7b", layers=32, batch=8, heads=32, head_dim=128, dtype="bf16",
        prompt_len=512, decode_steps=512, budget=204, k_heavy=102, k_local=102,
        hh_kind="pareto", hh_count=51, q_boost=1.0,
        note="OPT-6.7B-shaped: 32 layers x batch 8 x 32 heads, d=128 bf16; 512+512; k=204 (102+102); "
             "5% of positions key += beta u, beta ~ Pareto(1.5) capped at 8; q += 1.0u"),
    "llama-7b": Workload(
        "llama-7b", layers=1, batch=64, heads=32, head_dim=128, dtype="bf16",
        prompt_len=2048, decode_steps=256, budget=460, k_heavy=230, k_local=230,
        hh_kind="fixed", hh_count=4, k_boost=3.0, q_boost=1.5,
        note="LLaMA-7B-shaped: batch 64 x 32 heads, d=128 bf16, one layer (of 32); 2048+256; "
             "k=460 (230+230); 4 prompt keys += 3u, q += 1.5u"),
    "streaming": Workload(
        "streaming", layers=1, batch=1, heads=32, head_dim=128, dtype="bf16",
        prompt_len=512, decode_steps=262144, budget=4096, k_heavy=2048, k_local=2048,
        hh_kind="pareto", hh_count=(512 + 262144) // 100, q_boost=1.0,
        note="streaming: batch 1 x 32 heads, d=128 bf16; 512 + 262144 decode; k=4096 (2048+2048); "
             "1% of positions key += beta u, beta ~ Pareto(1.5) capped at 8; q += 1.0u"),
    "opt-30b": Workload(
        "opt-30b", layers=1, batch=32, heads=56, head_dim=128, dtype="bf16",
        prompt_len=512, decode_steps=1024, budget=307, k_heavy=154, k_local=153,
        hh_kind="pareto", hh_count=(512 + 1024) * 5 // 100, q_boost=1.0,
        note="OPT-30B-shaped: batch 32 x 56 heads, d=128 bf16, one layer; 512+1024; k=307 (154+153); "
             "5% Pareto(1.5) heavy hitters capped at 8; q += 1.0u"),
}

DEFAULT_SEED = 0x48324F00


def _rng(*words: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(w) for w in words])))


def heavy_hitter_direction(seed: int, head_dim: int) -> np.ndarray:
    """The fixed unit vector ``u`` (float64) shared by every head, layer and sequence."""
    z = _rng(seed, _TAG_U).standard_normal(head_dim)
    return z / np.linalg.norm(z)


def boosted_positions(w: Workload, seed: int, b: int) -> tuple[np.ndarray, np.ndarray]:
    """Boosted positions of sequence ``b`` (ascending int64) and their boost factors (float64)."""
    rng = _rng(seed, _TAG_HH, b)
    if w.hh_kind == "fixed":
        pool = w.prompt_len
        count = min(w.hh_count, pool)
        pos = np.sort(rng.choice(pool, size=count, replace=False))
        beta = np.full(count, w.k_boost, dtype=np.float64)
    elif w.hh_kind == "pareto":
        pool = w.total_len
        count = min(w.hh_count, pool)
        pos = np.sort(rng.choice(pool, size=count, replace=False))
        uu = rng.random(count)
        beta = np.minimum(w.pareto_cap, (1.0 - uu) ** (-1.0 / w.pareto_alpha))
    elif w.hh_kind == "none":
        pos = np.zeros(0, dtype=np.int64)
        beta = np.zeros(0, dtype=np.float64)
    else:
        raise ValueError(f"unknown heavy-hitter kind {w.hh_kind!r}")
    return pos.astype(np.int64), beta


def to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); uint16 bit patterns."""
    bits = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    rounded = (bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def storage_dtype(w: Workload):
    return np.float32 if w.dtype == "f32" else np.uint16


def _store(x64: np.ndarray, dtype: str) -> np.ndarray:
    x32 = x64.astype(np.float32)
    return x32 if dtype == "f32" else to_bf16_bits(x32)


def unit_sequence(w: Workload, seed: int, g: int, pos0: int, pos1: int,
                  u: np.ndarray | None = None,
                  hh: tuple[np.ndarray, np.ndarray] | None = None) -> np.ndarray:
    """Q, K, V of unit ``g`` for positions ``[pos0, pos1)``: array (3, pos1-pos0, D) in storage dtype."""
    D = w.head_dim
    if u is None:
        u = heavy_hitter_direction(seed, D)
    if hh is None:
        b = (g // w.heads) % w.batch
        hh = boosted_positions(w, seed, b)
    n = pos1 - pos0
    out = np.empty((3, n, D), dtype=np.float64)
    j0, j1 = pos0 // BLOCK, (pos1 - 1) // BLOCK if n > 0 else pos0 // BLOCK - 1
    for j in range(j0, j1 + 1):
        z = _rng(seed, _TAG_QKV, g, j).standard_normal((3, BLOCK, D), dtype=np.float32)
        a0, a1 = max(pos0, j * BLOCK), min(pos1, (j + 1) * BLOCK)
        out[:, a0 - pos0:a1 - pos0] = z[:, a0 - j * BLOCK:a1 - j * BLOCK]
    out[0] += w.q_boost * u
    hpos, beta = hh
    sel = (hpos >= pos0) & (hpos < pos1)
    for p, bt in zip(hpos[sel], beta[sel]):
        out[1, p - pos0] += bt * u
    return _store(out, w.dtype)


@dataclasses.dataclass
class Inputs:
    """Host arrays of one workload (or a subset of its units / steps)."""

    workload: Workload
    units: np.ndarray  # global unit ids present, ascending
    q_prompt: np.ndarray  # [n_units, P, D]
    k_prompt: np.ndarray
    v_prompt: np.ndarray
    step0: int  # first decode step held (step s is position P + s)
    q_dec: np.ndarray  # [n_steps, n_units, D]
    k_dec: np.ndarray
    v_dec: np.ndarray


def generate(w: Workload, seed: int = DEFAULT_SEED, units=None, step0: int = 0,
             steps: int | None = None, prompt: bool = True, threads: int | None = None) -> Inputs:
    """Generate the prompt and decode-step inputs for ``units`` (default: all) and decode steps
    ``[step0, step0 + steps)`` (default: all)."""
    if units is None:
        units = np.arange(w.units)
    units = np.asarray(units, dtype=np.int64)
    if steps is None:
        steps = w.decode_steps - step0
    D, P = w.head_dim, w.prompt_len
    sd = storage_dtype(w)
    nu = len(units)
    qp = np.empty((nu, P if prompt else 0, D), dtype=sd)
    kp = np.empty_like(qp)
    vp = np.empty_like(qp)
    qd = np.empty((steps, nu, D), dtype=sd)
    kd = np.empty_like(qd)
    vd = np.empty_like(qd)
    u = heavy_hitter_direction(seed, D)
    hh_cache = {}

    def hh_of(b):
        if b not in hh_cache:
            hh_cache[b] = boosted_positions(w, seed, b)
        return hh_cache[b]

    for b in sorted({int((g // w.heads) % w.batch) for g in units}):
        hh_of(b)

    def work(i):
        g = int(units[i])
        hh = hh_cache[int((g // w.heads) % w.batch)]
        if prompt:
            s = unit_sequence(w, seed, g, 0, P, u, hh)
            qp[i], kp[i], vp[i] = s[0], s[1], s[2]
        if steps > 0:
            s = unit_sequence(w, seed, g, P + step0, P + step0 + steps, u, hh)
            qd[:, i], kd[:, i], vd[:, i] = s[0], s[1], s[2]

    nthreads = threads or min(32, os.cpu_count() or 1)
    if nu * (P + steps) * D < (1 << 20) or nthreads == 1:
        for i in range(nu):
            work(i)
    else:
        with _cf.ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(work, range(nu)))
    return Inputs(w, units, qp, kp, vp, step0, qd, kd, vd)

