"""The C-ABI library loads on any machine and exports every declared entry
point; the host-side argument checks work without a device."""
import ctypes as C
import os
import re

import pytest

import speculative_decoding_rejection_02_gb300 as sv
from speculative_decoding_rejection_02_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(spec_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return sv.lib()


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 7
    for n in names:
        assert hasattr(L, n), n
    assert set(sv.ENTRY_POINTS) <= set(names)


def _cfg():
    return sv.Config(device=0, max_batch=8, max_rows=64, max_vocab=1000, flags=0)


def _batch(**kw):
    fake = 0x1000  # host-side checks never dereference
    base = dict(B=4, V=100, N=10, cu_num_draft=fake, draft_token_ids=fake, target_logits=fake,
                logits_dtype=sv.SPEC_BF16, draft_probs=None, temperature=fake, top_k=None,
                top_p=None, seed=1, request_base=0, flags=0, out_tokens=fake,
                num_accepted=fake, p_at_draft=None)
    base.update(kw)
    return sv.Batch(**base)


def test_check_batch(L):
    cfg = _cfg()
    assert sv.check_batch(cfg, _batch()) == 0
    assert sv.check_batch(cfg, _batch(B=0, cu_num_draft=None)) == 0
    assert sv.check_batch(cfg, _batch(cu_num_draft=None)) == -1
    assert sv.check_batch(cfg, _batch(target_logits=None)) == -1
    assert sv.check_batch(cfg, _batch(out_tokens=None)) == -1
    assert sv.check_batch(cfg, _batch(temperature=None)) == -1
    assert sv.check_batch(cfg, _batch(logits_dtype=7)) == -1
    assert sv.check_batch(cfg, _batch(V=0)) == -1
    assert sv.check_batch(cfg, _batch(N=-1)) == -1
    assert sv.check_batch(cfg, _batch(B=9)) == -5
    assert sv.check_batch(cfg, _batch(V=1001)) == -5
    assert sv.check_batch(cfg, _batch(N=61)) == -5
    assert sv.check_batch(cfg, _batch(N=0, draft_token_ids=None)) == 0


def test_check_batch_flags(L):
    cfg = _cfg()
    assert sv.check_batch(cfg, _batch(flags=sv.FLAG_NAIVE)) == 0
    assert sv.check_batch(cfg, _batch(flags=sv.FLAG_SAMPLER_MATCH)) == 0
    # the two rules exclude each other; unknown bits are refused
    assert sv.check_batch(cfg, _batch(flags=sv.FLAG_NAIVE | sv.FLAG_SAMPLER_MATCH)) == -1
    assert sv.check_batch(cfg, _batch(flags=0x8)) == -1
    assert sv.check_batch(cfg, _batch(flags=0x80000000)) == -1


def test_check_batch_early_exit(L):
    cfg = _cfg()
    early = sv.FLAG_EARLY_EXIT
    # bf16 rows of 96 values are 192 bytes: aligned; filters allowed on bf16
    assert sv.check_batch(cfg, _batch(V=96, flags=early)) == 0
    assert sv.check_batch(cfg, _batch(V=96, flags=early | sv.FLAG_NAIVE, top_p=0x1000)) == 0
    # any row layout and dtype (rows the queue cannot take get the full pass)
    assert sv.check_batch(cfg, _batch(V=100, flags=early)) == 0
    assert sv.check_batch(cfg, _batch(V=96, flags=early, target_logits=0x1008)) == 0
    assert sv.check_batch(cfg, _batch(V=96, logits_dtype=sv.SPEC_F32, flags=early)) == 0
    assert sv.check_batch(cfg, _batch(V=96, logits_dtype=sv.SPEC_F32, flags=early,
                                      top_k=0x1000)) == 0
    # not with sampler-match
    assert sv.check_batch(cfg, _batch(V=96, flags=early | sv.FLAG_SAMPLER_MATCH)) == -1


def test_strerror(L):
    for code in (0, -1, -2, -3, -4, -5, -6, 99):
        assert isinstance(sv.strerror(code), str) and sv.strerror(code)


def test_null_handle_and_bad_config(L):
    assert L.spec_verify_run(None, C.byref(_batch()), None) == -4
    assert L.spec_verify_greedy(None, C.byref(_batch()), None) == -4
    L.spec_verify_destroy(None)
    h = C.c_void_p()
    bad = sv.Config(device=0, max_batch=0, max_rows=1, max_vocab=1, flags=0)
    assert L.spec_verify_init(C.byref(h), C.byref(bad)) == -1


def test_config_flags_checked_before_the_device(L):
    """Unknown handle flags, and the cluster schedule combined with a forced
    early-exit schedule, are rejected before any device is touched."""
    h = C.c_void_p()
    for flags in (0x100, sv.CONFIG_EARLY_RESIDENT | sv.CONFIG_EARLY_QUEUE,
                  sv.CONFIG_EARLY_RESIDENT | sv.CONFIG_EARLY_FULL_PASS):
        cfg = sv.Config(device=0, max_batch=4, max_rows=16, max_vocab=64, flags=flags)
        assert L.spec_verify_init(C.byref(h), C.byref(cfg)) == -1
        assert not h.value


def test_init_without_gpu_fails_cleanly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = C.c_void_p()
    assert L.spec_verify_init(C.byref(h), C.byref(_cfg())) == -3
    assert not h.value


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(sv, "_lib", None)
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(ImportError):
        sv.lib()
