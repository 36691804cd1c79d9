"""The multi-GPU path on CPU ranks (gloo, world size 2).

The verifier partitions by request: a rank verifies its own requests with
request_base = the global index of its first one, so every rank's results
equal the slice of the unpartitioned call, with no exchange on the data
path. Checked here with the CPU oracle standing in for each rank's GPU (the
host logic of the sharding is what is under test), plus bench.py's rank
helpers (request numbering and the max-over-ranks timing reduction).
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth

WORLD = 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def shard(batch, lo, hi):
    """Requests [lo, hi) of a batch as a batch of their own."""
    cu = batch["cu_num_draft"]
    n0, n1 = int(cu[lo]), int(cu[hi])
    part = dict(batch)
    part.update(B=hi - lo, cu_num_draft=(cu[lo:hi + 1] - n0).astype(np.int32),
                draft_token_ids=batch["draft_token_ids"][n0:n1],
                target_logits=batch["target_logits"][n0 + lo:n1 + hi],
                draft_probs=None if batch["draft_probs"] is None else batch["draft_probs"][n0:n1],
                temperature=batch["temperature"][lo:hi],
                top_k=None if batch.get("top_k") is None else batch["top_k"][lo:hi],
                top_p=None if batch.get("top_p") is None else batch["top_p"][lo:hi],
                request_base=batch.get("request_base", 0) + lo)
    return part


def _worker(rank, port, out_dir):
    import torch

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    batch = synth.make("c3", B=20, V=3001)
    B = batch["B"]
    lo, hi = rank * B // WORLD, (rank + 1) * B // WORLD
    o = oracle.verify(shard(batch, lo, hi))
    toks = [None] * WORLD
    accs = [None] * WORLD
    dist.all_gather_object(toks, o["out_tokens"].tolist())
    dist.all_gather_object(accs, o["num_accepted"].tolist())
    t = bench.max_over_ranks(0.5 + rank, torch.device("cpu"))
    base = bench.rank_request_base(rank, B)
    if rank == 0:
        np.save(os.path.join(out_dir, "tok.npy"), np.concatenate([np.array(x) for x in toks]))
        np.save(os.path.join(out_dir, "acc.npy"), np.concatenate([np.array(x) for x in accs]))
        np.save(os.path.join(out_dir, "t.npy"), np.array([t, base]))
    dist.barrier()
    dist.destroy_process_group()


def test_request_sharded_ranks_equal_the_whole_batch(tmp_path):
    mp.spawn(_worker, args=(_free_port(), str(tmp_path)), nprocs=WORLD, join=True)
    batch = synth.make("c3", B=20, V=3001)
    whole = oracle.verify(batch)
    assert np.array_equal(np.load(tmp_path / "tok.npy"), whole["out_tokens"])
    assert np.array_equal(np.load(tmp_path / "acc.npy"), whole["num_accepted"])
    t, base = np.load(tmp_path / "t.npy")
    assert t == 1.5  # max over ranks of 0.5 + rank
    assert base == 0


def test_rank_request_base_is_disjoint():
    import bench
    B = 1024
    bases = [bench.rank_request_base(r, B) for r in range(8)]
    assert bases == [r * B for r in range(8)]
