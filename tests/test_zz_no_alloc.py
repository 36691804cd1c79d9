"""spec_verify_run_noalloc: the verification entry point for callers that
cannot allocate device memory (code inside an allocator or memory-pool
callback, processes whose device memory belongs to another framework's
caching allocator, loops that must not pay for a cudaMalloc). Its scratch is
a fixed device array inside the library, so this test checks, through the C
ABI, that it returns exactly what spec_verify_run returns on the same batch,
on two calls in a row (the second call finds the array holding the first
call's contents), on every part of the array: plain rows, misaligned rows,
aligned bf16 rows with top-k / top-p (the window histogram and its list of
unsettled rows) and early exit through the work queue; that it agrees with
the oracle; and that it refuses batches beyond its stated limits.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decoding_rejection_02_gb300 as sv
from parity import assert_parity, check_structure, compare

pytestmark = pytest.mark.gpu


def _run_handle(batch):
    R = batch["target_logits"].shape[0]
    ver = sv.Verifier(max_batch=batch["B"], max_rows=R, max_vocab=batch["V"])
    db = sv.upload(batch, "cuda:0")
    ver.run(db)
    torch.cuda.synchronize()
    out = (db.out_tokens.cpu().numpy(), db.num_accepted.cpu().numpy(), db.p_at_draft.cpu().numpy())
    assert ver.status() == 0
    ver.close()
    return out


def _run_noalloc(batch):
    L = sv.lib()
    db = sv.upload(batch, "cuda:0")
    db.out_tokens.fill_(-7)
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    s = db.struct()
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.spec_verify_run_noalloc(C.byref(s), C.c_void_p(stream), C.c_void_p(status.data_ptr()))
    assert rc == 0, sv.strerror(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return db.out_tokens.cpu().numpy(), db.num_accepted.cpu().numpy(), db.p_at_draft.cpu().numpy()


@pytest.mark.parametrize("name,B,V,early", [
    ("c5", 40, 65536, False),   # bf16 rows through the bulk-copy row pass
    ("c3", 27, 30011, False),   # misaligned rows: slice partials, exact filter kernel
    ("c3", 27, 30008, False),   # aligned bf16 rows with top-k / top-p: window histogram
    ("c2", 8, 32000, False),    # fp32 rows
    ("c5", 700, 4096, True),    # early exit through the work queue (B >= 2 x row-pass CTAs)
    ("c3", 640, 4000, True),    # early exit with filtered rows through the work queue
])
def test_noalloc_matches_handle_entry_point(name, B, V, early):
    batch = synth.make(name, B=B, V=V)
    if early:
        batch["flags"] = sv.FLAG_EARLY_EXIT
    ref_tok, ref_acc, ref_p = _run_handle(batch)
    for _ in range(2):  # two calls in a row share the array
        tok, acc, p = _run_noalloc(batch)
        assert np.array_equal(tok, ref_tok)
        assert np.array_equal(acc, ref_acc)
        np.testing.assert_allclose(p, ref_p, rtol=1e-6, atol=0)
    gpu = dict(out_tokens=tok, num_accepted=acc, p_at_draft=p, status=0)
    check_structure(batch, gpu)
    assert_parity(compare(batch, gpu, oracle.verify(batch, threads=oracle.host_threads())))


def test_noalloc_rejects_batches_beyond_its_limits():
    L = sv.lib()
    fake = 0x1000  # never dereferenced: the size check comes first
    base = dict(V=100, cu_num_draft=fake, draft_token_ids=fake, target_logits=fake,
                logits_dtype=sv.SPEC_BF16, draft_probs=None, temperature=fake, top_k=None,
                top_p=None, seed=1, request_base=0, flags=0, out_tokens=fake, num_accepted=fake,
                p_at_draft=None)
    too_many = sv.Batch(B=2049, N=2049, **base)
    assert L.spec_verify_run_noalloc(C.byref(too_many), None, None) == -5
    too_long = sv.Batch(B=10, N=8190, **base)
    assert L.spec_verify_run_noalloc(C.byref(too_long), None, None) == -5
    wide = sv.Batch(B=1, N=1, **dict(base, V=262145))
    assert L.spec_verify_run_noalloc(C.byref(wide), None, None) == -5
