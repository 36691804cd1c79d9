"""Vocab-sharded (tensor-parallel) verification across ranks.

Each rank holds the target logits (and draft probabilities) of a contiguous
slice of the vocabulary. The library's five sharded steps run on every
rank; between them the ranks all-reduce small per-row arrays (the order and
the reduce operations are fixed by include/spec_verify.h):

    rows     -> MAX m
    rescale  -> SUM z, qx, hist, hist_w;  MIN argmax;  MAX lx
    judge    -> MAX best
    race_p   -> MAX best_p
    emit

so every rank ends with the out_tokens / num_accepted a single device
verifying the whole vocabulary gives. Only collectives and library calls
happen here; the arithmetic is in the kernels.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import DeviceBatch, ShardBuffers, Verifier


def all_reduce(t: torch.Tensor, op, group=None) -> None:
    """In-place all-reduce; through host memory when the group's backend
    cannot reduce device tensors (gloo)."""
    if t is None:
        return
    if t.is_cuda and dist.get_backend(group) == "gloo":
        h = t.cpu()
        dist.all_reduce(h, op=op, group=group)
        t.copy_(h)
    else:
        dist.all_reduce(t, op=op, group=group)


def combine_max(sh: ShardBuffers, group=None) -> None:
    """After the rows step: every rank's m becomes the global row max."""
    all_reduce(sh.m, dist.ReduceOp.MAX, group)


def combine_rescaled(sh: ShardBuffers, group=None) -> None:
    """After the rescale step: sums over the ranks' columns, the global
    argmax (lowest index among the ranks holding the max), the draft token's
    logit from the rank that holds it."""
    all_reduce(sh.z, dist.ReduceOp.SUM, group)
    all_reduce(sh.qx, dist.ReduceOp.SUM, group)
    all_reduce(sh.hist, dist.ReduceOp.SUM, group)
    all_reduce(sh.hist_w, dist.ReduceOp.SUM, group)
    all_reduce(sh.argmax, dist.ReduceOp.MIN, group)
    all_reduce(sh.lx, dist.ReduceOp.MAX, group)


def combine_best(t: torch.Tensor, group=None) -> None:
    """After a race step: the winner over all columns."""
    all_reduce(t, dist.ReduceOp.MAX, group)


def verify_sharded(ver: Verifier, b: DeviceBatch, sh: ShardBuffers, group=None,
                   stream=None) -> DeviceBatch:
    """Verify one batch whose logits are vocab-sharded over the group."""
    ver.shard("rows", b, sh, stream)
    combine_max(sh, group)
    ver.shard("rescale", b, sh, stream)
    combine_rescaled(sh, group)
    ver.shard("judge", b, sh, stream)
    combine_best(sh.best, group)
    ver.shard("race_p", b, sh, stream)
    combine_best(sh.best_p, group)
    ver.shard("emit", b, sh, stream)
    return b
