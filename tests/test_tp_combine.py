"""The collectives of the vocab-sharded path on CPU ranks (gloo, world
sizes 2 and 3).

Each rank holds a slice of the vocabulary; speculative_decoding_rejection_02_gb300.tp
combines the ranks' per-row statistics between the library's sharded steps.
Here each rank's local statistics are computed in fp64 numpy (standing in
for its GPU), put through tp's combine functions, and must equal the
statistics of the whole rows: the max, the lowest argmax, the sum of
exp((l - m) / T) rescaled to the global max, the draft token's logit, q at
the draft token, the value histogram, and the race winner packed as
(score bits << 32) | ~index.
"""
import os
import socket
import types

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


R, V, N = 12, 64, 9


def _data():
    rng = np.random.default_rng(5)
    l = np.round(rng.normal(0, 2, size=(R, V)) * 4) / 4  # ties across slices
    l[3, :] = -np.inf
    l[3, 40] = 1.0      # the only finite value of row 3 sits in the last slice
    T = rng.uniform(0.5, 2, size=R)
    x = rng.integers(0, V, size=R)
    q = rng.random((N, V))
    qx_ids = rng.integers(0, V, size=N)
    score = rng.random((R, V))
    return l, T, x, q, qx_ids, score


def _pack(score, j):
    bits = np.float32(score).view(np.uint32).astype(np.int64)
    return int((bits << 32) | (0xFFFFFFFF - int(j)))


def _worker(rank, world, port, out_dir):
    from speculative_decoding_rejection_02_gb300 import tp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    l, T, x, q, qx_ids, score = _data()
    cuts = [k * V // world // 4 * 4 for k in range(world)] + [V]
    v0, v1 = cuts[rank], cuts[rank + 1]
    loc = l[:, v0:v1]
    with np.errstate(invalid="ignore"):
        m_loc = loc.max(1)
    arg_loc = np.array([v0 + int(np.argmax(loc[i])) if np.isfinite(m_loc[i]) else 2**31 - 1
                        for i in range(R)])
    z_loc = np.array([np.exp((loc[i] - m_loc[i]) / T[i]).sum() if np.isfinite(m_loc[i]) else 0.0
                      for i in range(R)])
    sh = types.SimpleNamespace(
        m=torch.tensor(m_loc), z=torch.zeros(R, dtype=torch.float64),
        argmax=torch.tensor(arg_loc, dtype=torch.int32),
        lx=torch.tensor([l[i, x[i]] if v0 <= x[i] < v1 else -np.inf for i in range(R)]),
        qx=torch.tensor([q[n, qx_ids[n]] if v0 <= qx_ids[n] < v1 else 0.0 for n in range(N)]),
        hist=torch.tensor(np.stack([np.histogram(loc[i][np.isfinite(loc[i])], bins=32,
                                                 range=(-10, 10))[0] for i in range(R)]),
                          dtype=torch.int32),
        hist_w=torch.tensor(np.ones((R, 2)) * (rank + 1)),
        best=torch.zeros(R, dtype=torch.int64))
    tp.combine_max(sh)
    mg = sh.m.numpy()
    # the rescale step (on the GPU the library's kernel)
    for i in range(R):
        sh.z[i] = z_loc[i] * np.exp((m_loc[i] - mg[i]) / T[i]) if np.isfinite(m_loc[i]) else 0.0
        if m_loc[i] != mg[i]:
            sh.argmax[i] = 2**31 - 1
    tp.combine_rescaled(sh)
    sc = score[:, v0:v1]
    sh.best = torch.tensor([_pack(sc[i].max(), v0 + int(np.argmax(sc[i]))) for i in range(R)],
                           dtype=torch.int64)
    tp.combine_best(sh.best)
    if rank == 0:
        np.savez(os.path.join(out_dir, "out.npz"), m=sh.m.numpy(), z=sh.z.numpy(),
                 argmax=sh.argmax.numpy(), lx=sh.lx.numpy(), qx=sh.qx.numpy(),
                 hist=sh.hist.numpy(), hist_w=sh.hist_w.numpy(), best=sh.best.numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_combined_statistics_equal_the_whole_rows(tmp_path, world):
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    o = np.load(tmp_path / "out.npz")
    l, T, x, q, qx_ids, score = _data()
    m = l.max(1)
    assert np.array_equal(o["m"], m)
    assert np.array_equal(o["argmax"], np.argmax(l, 1))  # lowest index of the max
    z = np.array([np.exp((l[i] - m[i]) / T[i]).sum() for i in range(R)])
    np.testing.assert_allclose(o["z"], z, rtol=1e-12)
    assert np.array_equal(o["lx"], l[np.arange(R), x])
    np.testing.assert_allclose(o["qx"], q[np.arange(N), qx_ids], rtol=0)
    whole = np.stack([np.histogram(l[i][np.isfinite(l[i])], bins=32, range=(-10, 10))[0]
                      for i in range(R)])
    assert np.array_equal(o["hist"], whole)
    np.testing.assert_allclose(o["hist_w"], np.full((R, 2), world * (world + 1) / 2))
    want = [_pack(score[i].max(), int(np.argmax(score[i]))) for i in range(R)]
    assert np.array_equal(o["best"], np.array(want))
