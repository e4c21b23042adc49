"""H2O (Heavy-Hitter Oracle) budgeted KV-cache eviction on GB300: Python binding of libh2o.so.

Every step of the path runs in the library's CUDA kernels; this module only marshals arguments
(device pointers taken from torch tensors, the current torch stream) into the C ABI declared in
``include/h2o.h`` and turns a non-zero status into an exception. There is no CPU fallback: if the
library cannot be loaded, every call raises.

    dims = Dims(units_b=layers * batch, heads=H, head_dim=128, budget=204, k_heavy=102,
                k_local=102, dtype=BF16)
    cache = H2OCache(dims, prompt_len=512, device="cuda")
    cache.prefill(q, k, v)                 # [units, P, D] each
    out, ev_slot, ev_pos = cache.step(q_t, k_t, v_t)   # [units, D] each, position advances
"""

from __future__ import annotations

import ctypes
import os

from . import build as _build

F32, BF16 = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE = range(5)
DEVERR_NONE, DEVERR_WAIT_TIMEOUT, DEVERR_NO_CANDIDATE = range(3)
POLICY_H2O, POLICY_LOCAL, POLICY_SINK_WINDOW, POLICY_TOPK, POLICY_STRIDED = range(5)

STATIC_SCRATCH_BYTES = 16 << 20  # H2O_STATIC_SCRATCH_BYTES

EXPORTS = ("h2o_prefill_workspace_bytes", "h2o_prefill_scores", "h2o_prefill_select",
           "h2o_prefill_select_static", "h2o_prefill_select_policy", "h2o_prefill_forward",
           "h2o_decode_step", "h2o_decode_step_policy", "h2o_decode_step_prefetch",
           "h2o_prefill_select_e4m3",
           "h2o_decode_step_e4m3", "h2o_get_device_error",
           "h2o_selftest_wait_timeout", "h2o_last_cuda_error", "h2o_status_string")


class Dims(ctypes.Structure):
    """``h2o_dims``: units_b = layers * batch rows of ``heads`` units each."""

    _fields_ = [("units_b", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("budget", ctypes.c_int32),
                ("k_heavy", ctypes.c_int32), ("k_local", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]

    @property
    def units(self) -> int:
        return self.units_b * self.heads

    def __repr__(self):
        return ("Dims(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")")


class NextCache(ctypes.Structure):
    """``h2o_next_cache``: the cache arrays of the next decode call on the stream (an L2 prefetch
    hint for h2o_decode_step_prefetch)."""

    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("scores", ctypes.c_void_p), ("slot_pos", ctypes.c_void_p)]


class Policy(ctypes.Structure):
    """``h2o_policy``: which slot a decode step evicts (and which prompt positions prefill keeps)."""

    _fields_ = [("kind", ctypes.c_int32), ("n_sink", ctypes.c_int32), ("stride", ctypes.c_int32)]

    def __init__(self, kind: int = POLICY_H2O, n_sink: int = 0, stride: int = 1):
        super().__init__(kind, n_sink, stride)

    def __repr__(self):
        return f"Policy(kind={self.kind}, n_sink={self.n_sink}, stride={self.stride})"


class H2OError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        detail = f", {last_cuda_error()}" if status == ERR_CUDA else ""
        super().__init__(f"{fn} failed: {status_string(status)} (status {status}{detail})")


_lib: ctypes.CDLL | None = None


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libh2o.so from this package's ``_build`` directory (building it first if it is missing
    and nvcc is available). Raises if the library cannot be loaded."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libh2o.so not built ({path}); run kv_cache_eviction_step_gb300.build")
        _build.build()
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    dp = ctypes.POINTER(Dims)
    lib.h2o_prefill_workspace_bytes.argtypes = [dp, i32]
    lib.h2o_prefill_workspace_bytes.restype = sz
    lib.h2o_prefill_scores.argtypes = [dp, i32, vp, vp, vp, vp, sz, vp]
    lib.h2o_prefill_scores.restype = ctypes.c_int
    lib.h2o_prefill_select.argtypes = [dp, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.h2o_prefill_select.restype = ctypes.c_int
    lib.h2o_prefill_select_static.argtypes = [dp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.h2o_prefill_select_static.restype = ctypes.c_int
    lib.h2o_decode_step.argtypes = [dp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.h2o_decode_step.restype = ctypes.c_int
    pp = ctypes.POINTER(Policy)
    lib.h2o_prefill_select_policy.argtypes = [dp, pp, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.h2o_prefill_select_policy.restype = ctypes.c_int
    lib.h2o_decode_step_policy.argtypes = [dp, pp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.h2o_decode_step_policy.restype = ctypes.c_int
    lib.h2o_decode_step_prefetch.argtypes = [dp, pp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                             ctypes.POINTER(NextCache), vp]
    lib.h2o_decode_step_prefetch.restype = ctypes.c_int
    lib.h2o_prefill_forward.argtypes = [dp, pp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.h2o_prefill_forward.restype = ctypes.c_int
    lib.h2o_prefill_select_e4m3.argtypes = [dp, pp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.h2o_prefill_select_e4m3.restype = ctypes.c_int
    lib.h2o_decode_step_e4m3.argtypes = [dp, pp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.h2o_decode_step_e4m3.restype = ctypes.c_int
    lib.h2o_get_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    lib.h2o_get_device_error.restype = ctypes.c_int
    lib.h2o_selftest_wait_timeout.argtypes = [vp]
    lib.h2o_selftest_wait_timeout.restype = ctypes.c_int
    lib.h2o_last_cuda_error.argtypes = []
    lib.h2o_last_cuda_error.restype = ctypes.c_char_p
    lib.h2o_status_string.argtypes = [ctypes.c_int]
    lib.h2o_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().h2o_status_string(status).decode()


def last_cuda_error() -> str:
    """Name of the CUDA error behind the last ERR_CUDA on this thread."""
    return load().h2o_last_cuda_error().decode()


def _ptr(x) -> int | None:
    """Device address of a tensor (or an int address / None)."""
    if x is None or isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(x) -> int:
    return x.numel() * x.element_size()


def _check(fn: str, status: int):
    if status != OK:
        raise H2OError(fn, status)


def h2o_prefill_workspace_bytes(dims: Dims, prompt_len: int) -> int:
    return int(load().h2o_prefill_workspace_bytes(ctypes.byref(dims), prompt_len))


def h2o_prefill_scores(dims: Dims, prompt_len: int, q, k, colsum, workspace, stream=None,
                       workspace_bytes: int | None = None):
    """Causal column sums of Softmax(QK^T/sqrt(D)) per unit into ``colsum`` [units, P] float32."""
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    _check("h2o_prefill_scores", load().h2o_prefill_scores(
        ctypes.byref(dims), prompt_len, _ptr(q), _ptr(k), _ptr(colsum), _ptr(workspace), wb,
        _stream(stream)))


def h2o_prefill_select(dims: Dims, prompt_len: int, q, k, v, k_cache, v_cache, scores, slot_pos,
                       workspace, stream=None, workspace_bytes: int | None = None):
    """Prefill score pass, heavy-hitter + recent selection and gather into the budgeted caches."""
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    _check("h2o_prefill_select", load().h2o_prefill_select(
        ctypes.byref(dims), prompt_len, _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
        _ptr(scores), _ptr(slot_pos), _ptr(workspace), wb, _stream(stream)))


def h2o_prefill_select_static(dims: Dims, prompt_len: int, q, k, v, k_cache, v_cache, scores,
                              slot_pos, stream=None):
    """h2o_prefill_select with its scratch in the library's fixed 16 MiB device array, for callers
    that cannot allocate device memory (a memory pool that owns the whole device, a plugin inside a
    framework that owns the allocator). Calls on one device share that array: order them on one
    stream. units * prompt_len must not exceed 1,398,080."""
    _check("h2o_prefill_select_static", load().h2o_prefill_select_static(
        ctypes.byref(dims), prompt_len, _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
        _ptr(scores), _ptr(slot_pos), _stream(stream)))


def h2o_decode_step(dims: Dims, position: int, q, k_new, v_new, k_cache, v_cache, scores,
                    slot_pos, out, evicted_slot, evicted_pos, stream=None):
    """One fused budgeted decode step at absolute ``position`` for every unit."""
    _check("h2o_decode_step", load().h2o_decode_step(
        ctypes.byref(dims), position, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
        _ptr(v_cache), _ptr(scores), _ptr(slot_pos), _ptr(out), _ptr(evicted_slot),
        _ptr(evicted_pos), _stream(stream)))


def _policy_ref(policy: Policy | None):
    return None if policy is None else ctypes.byref(policy)


def h2o_prefill_select_policy(dims: Dims, policy: Policy | None, prompt_len: int, q, k, v, k_cache,
                              v_cache, scores, slot_pos, workspace, stream=None,
                              workspace_bytes: int | None = None):
    """h2o_prefill_select under ``policy`` (None = H2O)."""
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    _check("h2o_prefill_select_policy", load().h2o_prefill_select_policy(
        ctypes.byref(dims), _policy_ref(policy), prompt_len, _ptr(q), _ptr(k), _ptr(v),
        _ptr(k_cache), _ptr(v_cache), _ptr(scores), _ptr(slot_pos), _ptr(workspace), wb,
        _stream(stream)))


def h2o_prefill_forward(dims: Dims, policy: Policy | None, prompt_len: int, q, k, v, out, k_cache,
                        v_cache, scores, slot_pos, workspace, stream=None,
                        workspace_bytes: int | None = None):
    """h2o_prefill_select_policy that also writes the prompt's causal attention output ``out``
    [units, P, D]."""
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    _check("h2o_prefill_forward", load().h2o_prefill_forward(
        ctypes.byref(dims), _policy_ref(policy), prompt_len, _ptr(q), _ptr(k), _ptr(v), _ptr(out),
        _ptr(k_cache), _ptr(v_cache), _ptr(scores), _ptr(slot_pos), _ptr(workspace), wb,
        _stream(stream)))


def h2o_decode_step_policy(dims: Dims, policy: Policy | None, position: int, q, k_new, v_new,
                           k_cache, v_cache, scores, slot_pos, out, evicted_slot, evicted_pos,
                           stream=None):
    """h2o_decode_step under ``policy`` (None = H2O)."""
    _check("h2o_decode_step_policy", load().h2o_decode_step_policy(
        ctypes.byref(dims), _policy_ref(policy), position, _ptr(q), _ptr(k_new), _ptr(v_new),
        _ptr(k_cache), _ptr(v_cache), _ptr(scores), _ptr(slot_pos), _ptr(out), _ptr(evicted_slot),
        _ptr(evicted_pos), _stream(stream)))


def next_cache(k_cache, v_cache, scores, slot_pos) -> NextCache:
    """The ``h2o_next_cache`` of a cache's arrays (tensors or raw pointers)."""
    return NextCache(_ptr(k_cache), _ptr(v_cache), _ptr(scores), _ptr(slot_pos))


def h2o_decode_step_prefetch(dims: Dims, policy: Policy | None, position: int, q, k_new, v_new,
                             k_cache, v_cache, scores, slot_pos, out, evicted_slot, evicted_pos,
                             next: NextCache | None, stream=None):
    """h2o_decode_step_policy, asking L2 for ``next``'s rows while it runs (None: no hint)."""
    _check("h2o_decode_step_prefetch", load().h2o_decode_step_prefetch(
        ctypes.byref(dims), _policy_ref(policy), position, _ptr(q), _ptr(k_new), _ptr(v_new),
        _ptr(k_cache), _ptr(v_cache), _ptr(scores), _ptr(slot_pos), _ptr(out), _ptr(evicted_slot),
        _ptr(evicted_pos), None if next is None else ctypes.byref(next), _stream(stream)))


def h2o_prefill_select_e4m3(dims: Dims, policy: Policy | None, prompt_len: int, q, k, v, k_cache,
                            v_cache, k_scale, v_scale, scores, slot_pos, workspace, stream=None,
                            workspace_bytes: int | None = None):
    """Prefill selection into an E4M3 cache (uint8 codes + float32 per-row scales)."""
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    _check("h2o_prefill_select_e4m3", load().h2o_prefill_select_e4m3(
        ctypes.byref(dims), _policy_ref(policy), prompt_len, _ptr(q), _ptr(k), _ptr(v),
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(scores), _ptr(slot_pos),
        _ptr(workspace), wb, _stream(stream)))


def h2o_decode_step_e4m3(dims: Dims, policy: Policy | None, position: int, q, k_new, v_new, k_cache,
                         v_cache, k_scale, v_scale, scores, slot_pos, out, evicted_slot, evicted_pos,
                         stream=None):
    """One decode step over an E4M3 cache."""
    _check("h2o_decode_step_e4m3", load().h2o_decode_step_e4m3(
        ctypes.byref(dims), _policy_ref(policy), position, _ptr(q), _ptr(k_new), _ptr(v_new),
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(scores), _ptr(slot_pos),
        _ptr(out), _ptr(evicted_slot), _ptr(evicted_pos), _stream(stream)))


def h2o_get_device_error(stream=None) -> int:
    """Synchronise ``stream``, return and clear the device error word (0 = none)."""
    code = ctypes.c_int32(0)
    st = load().h2o_get_device_error(_stream(stream), ctypes.byref(code))
    if st not in (OK, ERR_DEVICE):
        raise H2OError("h2o_get_device_error", st)
    return int(code.value)


def h2o_selftest_wait_timeout(stream=None):
    """Launch the bounded-wait self-test (sets the device error word to DEVERR_WAIT_TIMEOUT)."""
    _check("h2o_selftest_wait_timeout", load().h2o_selftest_wait_timeout(_stream(stream)))


class H2OCache:
    """Device buffers of one budgeted cache (caller-owned memory, allocated here with torch) and the
    running position. A convenience wrapper over the ABI calls; it computes nothing itself."""

    def __init__(self, dims: Dims, prompt_len: int, device="cuda", policy: Policy | None = None,
                 e4m3: bool = False):
        """``e4m3``: the K/V caches hold E4M3 codes with per-row scales (bf16, head_dim 128)."""
        import torch
        self.dims = dims
        self.policy = policy
        self.e4m3 = e4m3
        self.prompt_len = prompt_len
        self.position = prompt_len
        dt = torch.float32 if dims.dtype == F32 else torch.bfloat16
        u, k, d = dims.units, dims.budget, dims.head_dim
        self.dtype = dt
        cdt = torch.uint8 if e4m3 else dt
        self.k_cache = torch.empty((u, k, d), dtype=cdt, device=device)
        self.v_cache = torch.empty((u, k, d), dtype=cdt, device=device)
        self.k_scale = torch.empty((u, k), dtype=torch.float32, device=device) if e4m3 else None
        self.v_scale = torch.empty((u, k), dtype=torch.float32, device=device) if e4m3 else None
        self.scores = torch.empty((u, k), dtype=torch.float32, device=device)
        self.slot_pos = torch.empty((u, k), dtype=torch.int32, device=device)
        self.workspace = torch.empty(h2o_prefill_workspace_bytes(dims, prompt_len), dtype=torch.uint8,
                                     device=device)
        self.out = torch.empty((u, d), dtype=dt, device=device)
        self.evicted_slot = torch.empty(u, dtype=torch.int32, device=device)
        self.evicted_pos = torch.empty(u, dtype=torch.int32, device=device)

    def prefill(self, q, k, v, out=None, stream=None):
        """Build the cache from the prompt; with ``out`` ([units, P, D]) also write the prompt's
        attention output."""
        if self.e4m3:
            if out is not None:
                raise ValueError("the prompt output is not produced with an E4M3 cache")
            h2o_prefill_select_e4m3(self.dims, self.policy, self.prompt_len, q, k, v, self.k_cache,
                                    self.v_cache, self.k_scale, self.v_scale, self.scores,
                                    self.slot_pos, self.workspace, stream)
        elif out is None:
            h2o_prefill_select_policy(self.dims, self.policy, self.prompt_len, q, k, v, self.k_cache,
                                      self.v_cache, self.scores, self.slot_pos, self.workspace, stream)
        else:
            h2o_prefill_forward(self.dims, self.policy, self.prompt_len, q, k, v, out, self.k_cache,
                                self.v_cache, self.scores, self.slot_pos, self.workspace, stream)
        self.position = self.prompt_len

    def step(self, q, k_new, v_new, out=None, evicted_slot=None, evicted_pos=None, stream=None,
             prefetch: "H2OCache | None" = None):
        """One decode step. ``prefetch``: the cache the next step on this stream will decode (same
        dims), asked of L2 while this step runs (h2o_decode_step_prefetch; bf16 caches only)."""
        out = self.out if out is None else out
        es = self.evicted_slot if evicted_slot is None else evicted_slot
        ep = self.evicted_pos if evicted_pos is None else evicted_pos
        if prefetch is not None:
            if self.e4m3 or prefetch.e4m3:
                raise ValueError("the next-call prefetch hint is for bf16 / fp32 caches")
            h2o_decode_step_prefetch(self.dims, self.policy, self.position, q, k_new, v_new,
                                     self.k_cache, self.v_cache, self.scores, self.slot_pos, out, es,
                                     ep, next_cache(prefetch.k_cache, prefetch.v_cache,
                                                    prefetch.scores, prefetch.slot_pos), stream)
        elif self.e4m3:
            h2o_decode_step_e4m3(self.dims, self.policy, self.position, q, k_new, v_new, self.k_cache,
                                 self.v_cache, self.k_scale, self.v_scale, self.scores, self.slot_pos,
                                 out, es, ep, stream)
        else:
            h2o_decode_step_policy(self.dims, self.policy, self.position, q, k_new, v_new,
                                   self.k_cache, self.v_cache, self.scores, self.slot_pos, out, es,
                                   ep, stream)
        self.position += 1
        return out, es, ep
