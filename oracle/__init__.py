"""CPU oracle of the speculative-sampling verifier (TEST INFRASTRUCTURE).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its Python binding) never imports, links or executes anything here, and this
package imports nothing from the product: the two share only the seeded
input generators in ``synth``.

The arithmetic lives in ``spec_oracle.cpp`` (plain single-threaded C++,
fp64); this module compiles it with gcc (``build()``) and marshals numpy
arrays through ctypes.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libspecoracle.so")

_lock = threading.Lock()
_lib = None

# Per-request status bits written by the oracle.
ST_NONFINITE = 1
ST_NO_FINITE = 2
ST_BAD_TOKEN = 4
ST_EMPTY_RESIDUAL = 8

FLAG_NAIVE = 1
FLAG_SAMPLER_MATCH = 2
FLAG_EARLY_EXIT = 4


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libspecoracle.so`` (gcc, -O2)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC",
           "-Wno-free-nonheap-object", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Batch(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("V", C.c_int),
        ("cu_num_draft", C.c_void_p), ("draft_token_ids", C.c_void_p),
        ("target_logits", C.c_void_p), ("logits_dtype", C.c_int),
        ("draft_probs", C.c_void_p), ("temperature", C.c_void_p),
        ("top_k", C.c_void_p), ("top_p", C.c_void_p),
        ("seed", C.c_uint64), ("request_base", C.c_int64),
        ("flags", C.c_uint),
    ]


class _Outputs(C.Structure):
    _fields_ = [
        ("out_tokens", C.c_void_p), ("num_accepted", C.c_void_p),
        ("p_at_draft", C.c_void_p), ("accept_margin", C.c_void_p),
        ("topp_margin", C.c_void_p), ("race_margin", C.c_void_p),
        ("req_status", C.c_void_p), ("row_race_margin", C.c_void_p),
    ]


class _RowInfo(C.Structure):
    _fields_ = [
        ("m", C.c_double), ("argmax", C.c_int), ("n_kept", C.c_int),
        ("theta", C.c_double), ("z_kept", C.c_double),
        ("topp_margin", C.c_double), ("status", C.c_int),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = C.CDLL(path)
            L.or_philox4x32_10.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p]
            L.or_accept_uniform.argtypes = [C.c_uint64, C.c_int64, C.c_int32]
            L.or_accept_uniform.restype = C.c_double
            L.or_race_uniform.argtypes = [C.c_uint64, C.c_int64, C.c_int32, C.c_int64]
            L.or_race_uniform.restype = C.c_float
            L.or_bf16_to_double.argtypes = [C.c_uint16]
            L.or_bf16_to_double.restype = C.c_double
            L.or_argmax.argtypes = [C.c_void_p, C.c_int]
            L.or_argmax.restype = C.c_int
            L.or_target_probs.argtypes = [C.c_void_p, C.c_int, C.c_double, C.c_int,
                                          C.c_double, C.c_void_p, C.POINTER(_RowInfo)]
            L.or_target_probs.restype = C.c_int
            L.or_accept.argtypes = [C.c_double, C.c_double, C.c_double]
            L.or_accept.restype = C.c_int
            L.or_residual_weights.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                              C.c_int, C.c_void_p]
            L.or_race.argtypes = [C.c_void_p, C.c_int, C.c_uint64, C.c_int64, C.c_int32,
                                  C.POINTER(C.c_double)]
            L.or_race.restype = C.c_int
            L.or_verify.argtypes = [C.POINTER(_Batch), C.POINTER(_Outputs)]
            L.or_verify.restype = C.c_int
            L.or_verify_requests.argtypes = [C.POINTER(_Batch), C.c_void_p, C.c_int,
                                             C.POINTER(_Outputs)]
            L.or_verify_requests.restype = C.c_int
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


# ---------------------------------------------------------------------------
# Building blocks (each mirrors one function of spec_oracle.cpp)
# ---------------------------------------------------------------------------

def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().or_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def accept_uniform(seed: int, request: int, position: int) -> float:
    return lib().or_accept_uniform(seed, request, position)


def race_uniform(seed: int, request: int, position: int, j: int) -> float:
    return lib().or_race_uniform(seed, request, position, j)


def bf16_to_double(bits: int) -> float:
    return lib().or_bf16_to_double(bits)


def argmax(logits) -> int:
    l = np.ascontiguousarray(logits, dtype=np.float64)
    return lib().or_argmax(_ptr(l), l.size)


def target_probs(logits, T: float, top_k: int = 0, top_p: float = 1.0):
    """p after temperature / top-k / top-p, plus the row summary."""
    l = np.ascontiguousarray(logits, dtype=np.float64)
    p = np.zeros_like(l)
    info = _RowInfo()
    st = lib().or_target_probs(_ptr(l), l.size, float(T), int(top_k), float(top_p),
                               _ptr(p), C.byref(info))
    return p, {"m": info.m, "argmax": info.argmax, "n_kept": info.n_kept,
               "theta": info.theta, "z_kept": info.z_kept,
               "topp_margin": info.topp_margin, "status": st}


def accept(p_x: float, q_x: float, u: float) -> bool:
    return bool(lib().or_accept(p_x, q_x, u))


def residual_weights(p, q, x: int, mode: int):
    p = np.ascontiguousarray(p, dtype=np.float64)
    qq = np.ascontiguousarray(q if q is not None else np.zeros_like(p), dtype=np.float64)
    w = np.zeros_like(p)
    lib().or_residual_weights(_ptr(p), _ptr(qq), int(x), int(mode), p.size, _ptr(w))
    return w


def race(w, seed: int, request: int, position: int):
    w = np.ascontiguousarray(w, dtype=np.float64)
    margin = C.c_double()
    idx = lib().or_race(_ptr(w), w.size, seed, request, position, C.byref(margin))
    return idx, margin.value


# ---------------------------------------------------------------------------
# Whole-batch verification
# ---------------------------------------------------------------------------

def _batch_struct(batch, keep):
    """Build the ctypes batch; `keep` collects arrays that must stay alive."""
    def arr(name, dtype):
        a = batch.get(name)
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=dtype)
        keep.append(a)
        return a

    cu = arr("cu_num_draft", np.int32)
    ids = arr("draft_token_ids", np.int32)
    dt = batch["logits_dtype"]
    logits = arr("target_logits", np.uint16 if dt == "bf16" else np.float32)
    q = arr("draft_probs", np.float32)
    temp = arr("temperature", np.float32)
    tk = arr("top_k", np.int32)
    tp = arr("top_p", np.float32)
    B = int(cu.size - 1)
    b = _Batch(B=B, V=int(batch["V"]), cu_num_draft=_ptr(cu), draft_token_ids=_ptr(ids),
               target_logits=_ptr(logits), logits_dtype=1 if dt == "bf16" else 0,
               draft_probs=_ptr(q), temperature=_ptr(temp), top_k=_ptr(tk),
               top_p=_ptr(tp), seed=int(batch["seed"]) & 0xFFFFFFFFFFFFFFFF,
               request_base=int(batch.get("request_base", 0)),
               flags=int(batch.get("flags", 0)))
    return b, B, int(cu[-1])


def verify(batch, requests=None, threads: int = 1):
    """Run the oracle over a batch dict (see ``synth``) and return a dict of
    outputs and decision margins. ``requests`` restricts the work to a list of
    request indices (the other requests' slots keep their fill values:
    tokens -2, counts -1, NaN margins).

    ``threads`` > 1 splits the requests into that many disjoint sets (every
    t-th request) and runs the unchanged single-threaded oracle on each set in
    its own thread, all writing into the same output arrays: a request's
    verification reads only the batch and writes only that request's slots,
    so the result is the same as one thread's."""
    keep = []
    b, B, N = _batch_struct(batch, keep)
    R = N + B
    out = {
        "out_tokens": np.full(R, -2, np.int32),
        "num_accepted": np.full(B, -1, np.int32),
        "p_at_draft": np.full(N, np.nan),
        "accept_margin": np.full(N, np.nan),
        "topp_margin": np.full(R, np.nan),
        "race_margin": np.full(B, np.nan),
        "req_status": np.zeros(B, np.uint32),
        "row_race_margin": np.full(R, np.nan),
    }
    o = _Outputs(**{k: _ptr(v) for k, v in out.items()})
    if requests is None and threads <= 1:
        rc = lib().or_verify(C.byref(b), C.byref(o))
    else:
        reqs = np.ascontiguousarray(np.arange(B) if requests is None else requests,
                                    dtype=np.int32)
        L = lib()
        if threads <= 1 or reqs.size < 2:
            rc = L.or_verify_requests(C.byref(b), _ptr(reqs), reqs.size, C.byref(o))
        else:
            from concurrent.futures import ThreadPoolExecutor
            parts = [np.ascontiguousarray(reqs[t::threads]) for t in range(threads)]
            parts = [p for p in parts if p.size]
            with ThreadPoolExecutor(len(parts)) as ex:
                rcs = list(ex.map(lambda p: L.or_verify_requests(C.byref(b), _ptr(p), p.size,
                                                                 C.byref(o)), parts))
            rc = next((r for r in rcs if r != 0), 0)
    if rc != 0:
        raise ValueError(f"oracle verify failed ({rc})")
    return out


def host_threads() -> int:
    """Host cores this process may run on (for ``verify(threads=...)``)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1
