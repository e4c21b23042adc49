"""Python handle on the CPU oracle of the H2O budgeted KV-cache eviction step.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package. The product path
(``kv_cache_eviction_step_gb300``) never imports it, and this package never imports the product.

The arithmetic lives in ``h2o_oracle.c`` (plain C, float64); this module only compiles it with gcc
and marshals numpy arrays. See that file's header for the pages it restates and the readings taken.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "h2o_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libh2o_oracle.so")

F32, BF16 = 0, 1
NO_EVICTION, RULE, NEAR_TIE, ERROR_BOUND, REJECTED = range(5)
KIND_NAMES = ["no_eviction", "rule", "near_tie", "error_bound", "rejected"]

# The near-tie threshold of the parity rule: two candidate scores closer than this (relative) are a tie.
TIE_REL = 1e-6


POLICY_H2O, POLICY_LOCAL, POLICY_SINK_WINDOW, POLICY_TOPK, POLICY_STRIDED = range(5)


class Policy(ctypes.Structure):
    """Eviction policy: H2O (default) or one of the baselines; see h2o_oracle.c."""
    _fields_ = [("kind", ctypes.c_int32), ("n_sink", ctypes.c_int32), ("stride", ctypes.c_int32)]


class StepInfo(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("rule_victim", ctypes.c_int32),
                ("victim", ctypes.c_int32), ("evicted_pos", ctypes.c_int32),
                ("written_slot", ctypes.c_int32), ("n_candidates", ctypes.c_int32),
                ("gap_rel", ctypes.c_double)]


class PrefillInfo(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("kept", ctypes.c_int32), ("gap_rel", ctypes.c_double)]


_lock = threading.Lock()
_libs: dict[str, ctypes.CDLL] = {}


def build(src: str = SRC, out: str = LIB, extra_flags=()) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, no vectorisation flags that reorder sums)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
           *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i32, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_double
    lib.h2o_oracle_prefill_select.argtypes = [i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                              vp, vp, vp, vp, f64, f64, vp]
    lib.h2o_oracle_prefill_select.restype = ctypes.c_int
    lib.h2o_oracle_decode_step.argtypes = [i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                           vp, vp, vp, vp, vp, vp, f64, f64, vp]
    lib.h2o_oracle_decode_step.restype = ctypes.c_int
    lib.h2o_oracle_prefill_select_policy.argtypes = [i32, i32, i32, i32, i32, i32, i32, vp, vp, vp,
                                                     vp, vp, vp, vp, vp, vp, vp, f64, f64, vp]
    lib.h2o_oracle_prefill_select_policy.restype = ctypes.c_int
    lib.h2o_oracle_decode_step_policy.argtypes = [i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                                  vp, vp, vp, vp, vp, vp, vp, vp, vp, f64, f64, vp]
    lib.h2o_oracle_decode_step_policy.restype = ctypes.c_int
    lib.h2o_oracle_run_unit.argtypes = [i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                        ctypes.c_int64, vp, vp, vp, vp, vp]
    lib.h2o_oracle_run_unit.restype = ctypes.c_int
    lib.h2o_oracle_prefill_attention.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp]
    lib.h2o_oracle_prefill_attention.restype = ctypes.c_int
    lib.h2o_oracle_prefill_select_e4m3.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                                   vp, vp, vp, vp, vp, vp, vp, f64, f64, vp]
    lib.h2o_oracle_prefill_select_e4m3.restype = ctypes.c_int
    lib.h2o_oracle_decode_step_e4m3.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                                vp, vp, vp, vp, vp, vp, vp, vp, vp, f64, f64, vp]
    lib.h2o_oracle_decode_step_e4m3.restype = ctypes.c_int
    lib.h2o_oracle_e4m3_code.argtypes = [ctypes.c_float]
    lib.h2o_oracle_e4m3_code.restype = ctypes.c_uint8
    lib.h2o_oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.h2o_oracle_e4m3_value.restype = ctypes.c_double
    return lib


def load(path: str = LIB) -> ctypes.CDLL:
    """Load (building first if needed) an oracle shared library."""
    with _lock:
        if path in _libs:
            return _libs[path]
        if path == LIB and (not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC)):
            build()
        lib = _declare(ctypes.CDLL(path))
        _libs[path] = lib
        return lib


def prefill_attention(q, k, v, lib_path: str = LIB) -> np.ndarray:
    """Causal attention output of every prompt row, float64 [units, P, D]; q/k/v: [units, P, D]
    float32 or bf16 bits (uint16)."""
    q, k, v = (np.ascontiguousarray(a) for a in (q, k, v))
    units, P, D = q.shape
    out = np.empty((units, P, D), dtype=np.float64)
    rc = load(lib_path).h2o_oracle_prefill_attention(units, D, _dtype_code(q), P, _ptr(q), _ptr(k),
                                                     _ptr(v), _ptr(out))
    if rc != 0:
        raise ValueError(f"h2o_oracle_prefill_attention failed (code {rc})")
    return out


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle inputs must be float32 or uint16 (bf16 bits), got {arr.dtype}")


def e4m3_code(f: float, lib_path: str = LIB) -> int:
    """E4M3 code of a float32 (to nearest, ties to even, saturating at +-448)."""
    return int(load(lib_path).h2o_oracle_e4m3_code(f))


def e4m3_value(code: int, lib_path: str = LIB) -> float:
    return float(load(lib_path).h2o_oracle_e4m3_value(code))


class State:
    """One H2O cache state on the host: K/V slots, fp32 score table and slot-to-position map. With
    ``e4m3`` the K/V slots hold E4M3 codes (uint8) and ``k_scale``/``v_scale`` one scale per slot."""

    def __init__(self, units: int, budget: int, head_dim: int, dtype, e4m3: bool = False):
        cdt = np.uint8 if e4m3 else dtype
        self.k_cache = np.zeros((units, budget, head_dim), dtype=cdt)
        self.v_cache = np.zeros((units, budget, head_dim), dtype=cdt)
        self.k_scale = np.zeros((units, budget), dtype=np.float32) if e4m3 else None
        self.v_scale = np.zeros((units, budget), dtype=np.float32) if e4m3 else None
        self.scores = np.zeros((units, budget), dtype=np.float32)
        self.slot_pos = np.full((units, budget), -1, dtype=np.int32)

    @property
    def e4m3(self) -> bool:
        return self.k_scale is not None

    def copy(self) -> "State":
        c = State.__new__(State)
        c.k_cache, c.v_cache = self.k_cache.copy(), self.v_cache.copy()
        c.k_scale = None if self.k_scale is None else self.k_scale.copy()
        c.v_scale = None if self.v_scale is None else self.v_scale.copy()
        c.scores, c.slot_pos = self.scores.copy(), self.slot_pos.copy()
        return c


class Oracle:
    """The oracle's two operations on numpy arrays (host memory)."""

    def __init__(self, budget: int, k_heavy: int, k_local: int, lib_path: str = LIB,
                 policy: Policy | None = None):
        self.lib = load(lib_path)
        self.budget, self.k_heavy, self.k_local = budget, k_heavy, k_local
        self.policy = policy

    def _pol(self):
        return None if self.policy is None else ctypes.cast(ctypes.pointer(self.policy), ctypes.c_void_p)

    def new_state(self, units: int, head_dim: int, dtype, e4m3: bool = False) -> State:
        return State(units, self.budget, head_dim, dtype, e4m3)

    def prefill_select(self, q, k, v, state: State, prefer_pos=None, tie_rel=TIE_REL,
                       err_rel=TIE_REL, want_colsum=False):
        """Prefill score pass + selection. q/k/v: [units, P, D]. Returns (colsum or None, infos)."""
        q, k, v = (np.ascontiguousarray(a) for a in (q, k, v))
        units, P, D = q.shape
        colsum = np.empty((units, P), dtype=np.float64) if want_colsum else None
        infos = (PrefillInfo * max(units, 1))()
        pref = None if prefer_pos is None else np.ascontiguousarray(prefer_pos, dtype=np.int32)
        if state.e4m3:
            if _dtype_code(q) != BF16:
                raise TypeError("the E4M3 cache takes bf16 inputs")
            rc = self.lib.h2o_oracle_prefill_select_e4m3(
                units, D, self.budget, self.k_heavy, self.k_local, P, _ptr(q), _ptr(k), _ptr(v),
                _ptr(state.k_cache), _ptr(state.v_cache), _ptr(state.k_scale), _ptr(state.v_scale),
                _ptr(state.scores), _ptr(state.slot_pos), _ptr(colsum), self._pol(), _ptr(pref),
                tie_rel, err_rel, ctypes.cast(infos, ctypes.c_void_p))
        else:
            rc = self.lib.h2o_oracle_prefill_select_policy(
                units, D, self.budget, self.k_heavy, self.k_local, _dtype_code(q), P,
                _ptr(q), _ptr(k), _ptr(v), _ptr(state.k_cache), _ptr(state.v_cache),
                _ptr(state.scores), _ptr(state.slot_pos), _ptr(colsum), self._pol(), _ptr(pref),
                tie_rel, err_rel, ctypes.cast(infos, ctypes.c_void_p))
        if rc != 0:
            raise ValueError(f"h2o_oracle_prefill_select rejected its arguments (code {rc})")
        return colsum, infos[:units]

    def decode_step(self, t: int, q, k_new, v_new, state: State, prefer_victim=None,
                    tie_rel=TIE_REL, err_rel=TIE_REL, want_probs=False):
        """One decode step at position t. q/k_new/v_new: [units, D].
        Returns (out float64 [units, D], evicted_slot, evicted_pos, probs or None, infos)."""
        q, k_new, v_new = (np.ascontiguousarray(a) for a in (q, k_new, v_new))
        units, D = q.shape
        out = np.empty((units, D), dtype=np.float64)
        ev_slot = np.empty(units, dtype=np.int32)
        ev_pos = np.empty(units, dtype=np.int32)
        probs = np.full((units, self.budget + 1), np.nan) if want_probs else None
        infos = (StepInfo * max(units, 1))()
        pref = None if prefer_victim is None else np.ascontiguousarray(prefer_victim, dtype=np.int32)
        if state.e4m3:
            if _dtype_code(q) != BF16:
                raise TypeError("the E4M3 cache takes bf16 inputs")
            rc = self.lib.h2o_oracle_decode_step_e4m3(
                units, D, self.budget, self.k_heavy, self.k_local, t, _ptr(q), _ptr(k_new),
                _ptr(v_new), _ptr(state.k_cache), _ptr(state.v_cache), _ptr(state.k_scale),
                _ptr(state.v_scale), _ptr(state.scores), _ptr(state.slot_pos), _ptr(out),
                _ptr(probs), _ptr(ev_slot), _ptr(ev_pos), self._pol(), _ptr(pref), tie_rel,
                err_rel, ctypes.cast(infos, ctypes.c_void_p))
        else:
            rc = self.lib.h2o_oracle_decode_step_policy(
                units, D, self.budget, self.k_heavy, self.k_local, _dtype_code(q), t,
                _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(state.k_cache), _ptr(state.v_cache),
                _ptr(state.scores), _ptr(state.slot_pos), _ptr(out), _ptr(probs), _ptr(ev_slot),
                _ptr(ev_pos), self._pol(), _ptr(pref), tie_rel, err_rel,
                ctypes.cast(infos, ctypes.c_void_p))
        if rc != 0:
            raise ValueError(f"h2o_oracle_decode_step rejected its arguments (code {rc})")
        return out, ev_slot, ev_pos, probs, infos[:units]

    def run_unit(self, q, k, v, q_dec, k_dec, v_dec, state: State, unit: int = 0):
        """One unit's prefill + decode steps in one call (for timing). q/k/v: [P, D] of the unit;
        q_dec/k_dec/v_dec: [S, units, D] arrays, the unit's rows taken at index ``unit``."""
        q, k, v = (np.ascontiguousarray(a) for a in (q, k, v))
        P, D = q.shape
        S, nu, _ = q_dec.shape
        for a in (q_dec, k_dec, v_dec):
            assert a.flags.c_contiguous
        off = unit * D * q_dec.itemsize
        base = lambda a: ctypes.c_void_p(a.ctypes.data + off)
        rc = self.lib.h2o_oracle_run_unit(
            D, self.budget, self.k_heavy, self.k_local, _dtype_code(q), P, S, _ptr(q), _ptr(k),
            _ptr(v), base(q_dec), base(k_dec), base(v_dec), nu * D, _ptr(state.k_cache),
            _ptr(state.v_cache), _ptr(state.scores), _ptr(state.slot_pos), None)
        if rc != 0:
            raise ValueError(f"h2o_oracle_run_unit failed (code {rc})")
