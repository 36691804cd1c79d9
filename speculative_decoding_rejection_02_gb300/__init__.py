"""GB300 speculative-sampling verifier: Python binding of the C ABI.

Thin ``ctypes`` marshalling over ``libspecverify.so`` (declared in
``include/spec_verify.h``). Every step of the verification runs in the
library's CUDA kernels; PyTorch only supplies device memory and streams.
There is no CPU fallback: if the library is missing or fails to load, every
entry point raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

from . import _build

SPEC_OK = 0
SPEC_ERR = {
    -1: "SPEC_ERR_INVALID_ARG", -2: "SPEC_ERR_UNSUPPORTED", -3: "SPEC_ERR_CUDA",
    -4: "SPEC_ERR_NOT_INIT", -5: "SPEC_ERR_CAPACITY", -6: "SPEC_ERR_DEVICE_STATUS",
}
SPEC_F32, SPEC_BF16 = 0, 1

STATUS_NONFINITE = 0x1
STATUS_NO_FINITE = 0x2
STATUS_BAD_TOKEN = 0x4
STATUS_EMPTY_RESIDUAL = 0x8
STATUS_BAD_OFFSETS = 0x10
STATUS_TIMEOUT = 0x20
STATUS_UNSETTLED = 0x40

SHARD_HIST_INTS = 6148  # ints per row of the sharded window histogram

FLAG_NAIVE = 0x1
FLAG_SAMPLER_MATCH = 0x2
FLAG_EARLY_EXIT = 0x4

CONFIG_TEST_WAIT_TIMEOUT = 0x1  # test only: early-exit queue waits run out
CONFIG_EARLY_QUEUE = 0x2        # test only: early exit always takes the work queue
CONFIG_EARLY_FULL_PASS = 0x4    # test only: early exit always reads every row
CONFIG_EARLY_RESIDENT = 0x8     # early exit keeps each judged row in a cluster's shared memory

# The entry points declared in include/spec_verify.h.
ENTRY_POINTS = (
    "spec_verify_init", "spec_verify_run", "spec_verify_greedy", "spec_verify_status",
    "spec_verify_check_batch", "spec_verify_set_phase_events", "spec_verify_run_noalloc",
    "spec_verify_destroy", "spec_verify_strerror",
    "spec_verify_shard_rows", "spec_verify_shard_rescale", "spec_verify_shard_judge",
    "spec_verify_shard_race_p", "spec_verify_shard_emit",
)

_SHARD_CALLS = ENTRY_POINTS[-5:]


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {SPEC_ERR.get(code, code)} ({code})")
        self.code = code


class Config(C.Structure):
    _fields_ = [("device", C.c_int), ("max_batch", C.c_int), ("max_rows", C.c_longlong),
                ("max_vocab", C.c_int), ("flags", C.c_uint)]


class Batch(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("V", C.c_int), ("N", C.c_int),
        ("cu_num_draft", C.c_void_p), ("draft_token_ids", C.c_void_p),
        ("target_logits", C.c_void_p), ("logits_dtype", C.c_int),
        ("draft_probs", C.c_void_p), ("temperature", C.c_void_p),
        ("top_k", C.c_void_p), ("top_p", C.c_void_p),
        ("seed", C.c_ulonglong), ("request_base", C.c_longlong), ("flags", C.c_uint),
        ("out_tokens", C.c_void_p), ("num_accepted", C.c_void_p), ("p_at_draft", C.c_void_p),
    ]


class Shard(C.Structure):
    _fields_ = [
        ("v0", C.c_longlong), ("V_global", C.c_int),
        ("m", C.c_void_p), ("z", C.c_void_p), ("argmax", C.c_void_p), ("lx", C.c_void_p),
        ("qx", C.c_void_p), ("hist", C.c_void_p), ("hist_w", C.c_void_p),
        ("best", C.c_void_p), ("best_p", C.c_void_p),
    ]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """Load libspecverify.so (building it first if the sources are newer)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise ImportError(f"the CUDA verifier library is not built ({path}); "
                                  "run __graft_entry__.build()")
            L = C.CDLL(path)
            L.spec_verify_init.argtypes = [C.POINTER(C.c_void_p), C.POINTER(Config)]
            L.spec_verify_run.argtypes = [C.c_void_p, C.POINTER(Batch), C.c_void_p]
            L.spec_verify_greedy.argtypes = [C.c_void_p, C.POINTER(Batch), C.c_void_p]
            L.spec_verify_status.argtypes = [C.c_void_p, C.POINTER(C.c_uint)]
            L.spec_verify_check_batch.argtypes = [C.POINTER(Config), C.POINTER(Batch)]
            L.spec_verify_set_phase_events.argtypes = [C.c_void_p, C.c_void_p, C.c_int]
            L.spec_verify_run_noalloc.argtypes = [C.POINTER(Batch), C.c_void_p, C.c_void_p]
            L.spec_verify_destroy.argtypes = [C.c_void_p]
            L.spec_verify_destroy.restype = None
            L.spec_verify_strerror.argtypes = [C.c_int]
            L.spec_verify_strerror.restype = C.c_char_p
            for name in _SHARD_CALLS:
                getattr(L, name).argtypes = [C.c_void_p, C.POINTER(Batch), C.POINTER(Shard),
                                             C.c_void_p]
            for name in ENTRY_POINTS:
                getattr(L, name)  # raises if the library lacks a declared symbol
            _lib = L
    return _lib


def _check(rc: int, what: str):
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, what)


def _ptr(t):
    return None if t is None else t.data_ptr()


class DeviceBatch:
    """Device tensors of one verification call (inputs and outputs).

    ``target_logits`` is a [(N+B), V] torch tensor of dtype bfloat16 or
    float32; the others follow include/spec_verify.h.
    """

    def __init__(self, *, cu_num_draft, draft_token_ids, target_logits, draft_probs,
                 temperature, top_k=None, top_p=None, seed=0, request_base=0, flags=0,
                 out_tokens=None, num_accepted=None, p_at_draft=None, N=None, V=None):
        import torch
        self.cu_num_draft = cu_num_draft
        self.draft_token_ids = draft_token_ids
        self.target_logits = target_logits
        self.draft_probs = draft_probs
        self.temperature = temperature
        self.top_k = top_k
        self.top_p = top_p
        self.seed = int(seed)
        self.request_base = int(request_base)
        self.flags = int(flags)
        self.B = int(cu_num_draft.numel()) - 1
        self.V = int(V if V is not None else target_logits.shape[-1])
        self.N = int(N if N is not None else draft_token_ids.numel())
        dev = target_logits.device
        self.out_tokens = out_tokens if out_tokens is not None else torch.empty(
            self.N + self.B, dtype=torch.int32, device=dev)
        self.num_accepted = num_accepted if num_accepted is not None else torch.empty(
            self.B, dtype=torch.int32, device=dev)
        self.p_at_draft = p_at_draft

    def struct(self) -> Batch:
        import torch
        dt = self.target_logits.dtype
        if dt == torch.bfloat16:
            code = SPEC_BF16
        elif dt == torch.float32:
            code = SPEC_F32
        else:
            raise TypeError(f"target_logits must be bfloat16 or float32, not {dt}")
        return Batch(B=self.B, V=self.V, N=self.N, cu_num_draft=_ptr(self.cu_num_draft),
                     draft_token_ids=_ptr(self.draft_token_ids),
                     target_logits=_ptr(self.target_logits), logits_dtype=code,
                     draft_probs=_ptr(self.draft_probs), temperature=_ptr(self.temperature),
                     top_k=_ptr(self.top_k), top_p=_ptr(self.top_p), seed=self.seed,
                     request_base=self.request_base, flags=self.flags,
                     out_tokens=_ptr(self.out_tokens), num_accepted=_ptr(self.num_accepted),
                     p_at_draft=_ptr(self.p_at_draft))


def upload(batch: dict, device="cuda", with_p=True, pin=False) -> DeviceBatch:
    """Copy a host batch (numpy arrays, see ``synth``) to device tensors."""
    import numpy as np
    import torch

    def t(a, dtype=None):
        if a is None:
            return None
        x = torch.from_numpy(np.ascontiguousarray(a))
        if dtype is not None:
            x = x.view(dtype)
        return x.to(device, non_blocking=False)

    if batch["logits_dtype"] == "bf16":
        logits = t(np.ascontiguousarray(batch["target_logits"]).view(np.int16), torch.bfloat16)
    else:
        logits = t(batch["target_logits"])
    N = int(batch["cu_num_draft"][-1])
    db = DeviceBatch(cu_num_draft=t(batch["cu_num_draft"]),
                     draft_token_ids=t(batch["draft_token_ids"]), target_logits=logits,
                     draft_probs=t(batch["draft_probs"]), temperature=t(batch["temperature"]),
                     top_k=t(batch.get("top_k")), top_p=t(batch.get("top_p")),
                     seed=batch["seed"], request_base=batch.get("request_base", 0),
                     flags=batch.get("flags", 0), N=N, V=batch["V"])
    if with_p:
        db.p_at_draft = torch.empty(N, dtype=torch.float32, device=logits.device)
    return db


class Verifier:
    """One library handle (one workspace) on one CUDA device."""

    def __init__(self, max_batch: int, max_rows: int, max_vocab: int, device: int = 0,
                 config_flags: int = 0):
        self._lib = lib()
        self.cfg = Config(device=device, max_batch=max_batch, max_rows=max_rows,
                          max_vocab=max_vocab, flags=config_flags)
        h = C.c_void_p()
        _check(self._lib.spec_verify_init(C.byref(h), C.byref(self.cfg)), "spec_verify_init")
        self._h = h

    def _stream(self, stream):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream(self.cfg.device)
        return C.c_void_p(stream.cuda_stream)

    def run(self, b: DeviceBatch, stream=None):
        s = b.struct()
        _check(self._lib.spec_verify_run(self._h, C.byref(s), self._stream(stream)),
               "spec_verify_run")
        return b

    def greedy(self, b: DeviceBatch, stream=None):
        s = b.struct()
        _check(self._lib.spec_verify_greedy(self._h, C.byref(s), self._stream(stream)),
               "spec_verify_greedy")
        return b

    def shard(self, step: str, b: DeviceBatch, sh: "ShardBuffers", stream=None):
        """One step of a vocab-sharded call: "rows", "rescale", "judge",
        "race_p" or "emit" (the caller all-reduces in between; see tp.py)."""
        name = f"spec_verify_shard_{step}"
        s, shs = b.struct(), sh.struct()
        _check(getattr(self._lib, name)(self._h, C.byref(s), C.byref(shs), self._stream(stream)),
               name)

    def status(self) -> int:
        bits = C.c_uint(0)
        rc = self._lib.spec_verify_status(self._h, C.byref(bits))
        if rc not in (SPEC_OK, -6):
            raise SpecVerifyError(rc, "spec_verify_status")
        return int(bits.value)

    def set_phase_events(self, events):
        """Record ``events`` (4 torch.cuda.Event) around the phases of later calls:
        [start, after the row pass, after the accept scan, after the race]."""
        if not events:
            _check(self._lib.spec_verify_set_phase_events(self._h, None, 0), "set_phase_events")
            self._events = None
            return
        for e in events:
            e.record()  # materialise the underlying cudaEvent_t
        arr = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
        _check(self._lib.spec_verify_set_phase_events(self._h, arr, len(events)),
               "set_phase_events")
        self._events = list(events)

    def close(self):
        if getattr(self, "_h", None):
            self._lib.spec_verify_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class ShardBuffers:
    """Device arrays exchanged between the ranks of a vocab-sharded call."""

    def __init__(self, b: DeviceBatch, v0: int, V_global: int, filters: bool):
        import torch
        dev = b.target_logits.device
        R, N, B = b.N + b.B, b.N, b.B
        self.v0, self.V_global = int(v0), int(V_global)
        self.m = torch.empty(R, dtype=torch.float32, device=dev)
        self.z = torch.empty(R, dtype=torch.float32, device=dev)
        self.argmax = torch.empty(R, dtype=torch.int32, device=dev)
        self.lx = torch.empty(R, dtype=torch.float32, device=dev)
        self.qx = (torch.empty(max(N, 1), dtype=torch.float32, device=dev)
                   if b.draft_probs is not None else None)
        self.hist = (torch.empty((R, SHARD_HIST_INTS), dtype=torch.int32, device=dev)
                     if filters else None)
        self.hist_w = torch.empty((R, 2), dtype=torch.float32, device=dev) if filters else None
        # (score bits << 32) | ~index: non-negative as int64, so MAX combines them
        self.best = torch.empty(max(B, 1), dtype=torch.int64, device=dev)
        self.best_p = torch.empty(max(B, 1), dtype=torch.int64, device=dev)

    def struct(self) -> Shard:
        return Shard(v0=self.v0, V_global=self.V_global, m=_ptr(self.m), z=_ptr(self.z),
                     argmax=_ptr(self.argmax), lx=_ptr(self.lx), qx=_ptr(self.qx),
                     hist=_ptr(self.hist), hist_w=_ptr(self.hist_w), best=_ptr(self.best),
                     best_p=_ptr(self.best_p))


def check_batch(cfg: Config, b: Batch) -> int:
    """Host-side argument checks only (no device needed)."""
    return lib().spec_verify_check_batch(C.byref(cfg), C.byref(b))


def strerror(code: int) -> str:
    return lib().spec_verify_strerror(code).decode()
