"""Vocab-sharded verification on the GPU: n ranks (processes on cuda:0,
gloo collectives through host memory, no kernel waits on another rank)
each hold a slice of the vocabulary and run the library's sharded steps
with speculative_decoding_rejection_02_gb300.tp; every rank's outputs must
equal the oracle's for the whole vocabulary (parity rules of parity.py)."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth
from parity import assert_parity, check_structure, compare

pytestmark = pytest.mark.gpu


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _columns(batch, v0, v1):
    part = dict(batch)
    part["target_logits"] = np.ascontiguousarray(batch["target_logits"][:, v0:v1])
    if batch["draft_probs"] is not None:
        part["draft_probs"] = np.ascontiguousarray(batch["draft_probs"][:, v0:v1])
    part["V"] = v1 - v0
    return part


def _cuts(V, world, align):
    cuts = [k * V // world // align * align for k in range(world)] + [V]
    return cuts


def _worker(rank, world, port, name, B, V, align, out_dir):
    import torch

    import speculative_decoding_rejection_02_gb300 as sv
    from speculative_decoding_rejection_02_gb300 import tp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    batch = synth.make(name, B=B, V=V)
    cuts = _cuts(batch["V"], world, align)
    v0, v1 = cuts[rank], cuts[rank + 1]
    part = _columns(batch, v0, v1)
    R = part["target_logits"].shape[0]
    ver = sv.Verifier(max_batch=part["B"], max_rows=R, max_vocab=part["V"])
    db = sv.upload(part, "cuda:0")
    filters = part.get("top_k") is not None or part.get("top_p") is not None
    sh = sv.ShardBuffers(db, v0, batch["V"], filters)
    tp.verify_sharded(ver, db, sh)
    torch.cuda.synchronize()
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), out_tokens=db.out_tokens.cpu().numpy(),
             num_accepted=db.num_accepted.cpu().numpy(), p_at_draft=db.p_at_draft.cpu().numpy(),
             status=np.array([ver.status()]))
    ver.close()
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("name,B,V,world", [
    ("c2", None, None, 2),    # fp32 logits and probabilistic draft: q(x) and the residual race
    ("c3", 27, 40008, 3),     # every temperature / filter combination over three slices
    ("c4", 24, 50000, 2),     # one-hot drafts, top-p
    ("c5", 40, 70000, 2),     # argmax and probabilistic requests, ragged rounds
])
def test_sharded_equals_the_whole_vocabulary(tmp_path, name, B, V, world):
    batch = synth.make(name, B=B, V=V)
    align = 8 if batch["logits_dtype"] == "bf16" else 4  # 16-byte rows, v0 a multiple of 4
    mp.spawn(_worker, args=(world, _free_port(), name, B, V, align, str(tmp_path)),
             nprocs=world, join=True)
    ref = oracle.verify(batch)
    outs = [np.load(tmp_path / f"rank{k}.npz") for k in range(world)]
    for o in outs[1:]:  # every rank holds the same outputs
        assert np.array_equal(o["out_tokens"], outs[0]["out_tokens"])
        assert np.array_equal(o["num_accepted"], outs[0]["num_accepted"])
    gpu = {k: outs[0][k] for k in ("out_tokens", "num_accepted", "p_at_draft")}
    assert int(outs[0]["status"][0]) == 0
    check_structure(batch, gpu)
    rep = compare(batch, gpu, ref)
    assert_parity(rep)
    assert rep["requests"] > 0
