"""A tensor sharded across ranks by whole 65,536-element chunks, and the one
exchange that a single stream of the whole tensor needs.

Each rank encodes its shard on its own GPU into a self-contained stream.  The
stream of the whole tensor (what ``sz_concat`` builds from the shard streams)
places shard k's escape records after those of every shard before it and
shifts its chunk-header offsets by their number: an exclusive scan of the
shard escape counts.  A shard's escape count follows from its element count
and stream size by the closed-form size, so one all-gather of two integers
per rank gives every rank the whole layout.  Host arithmetic only; the data
path is the library's.
"""
from __future__ import annotations

import torch

from . import splitzip as S

CHUNK = S.SZ_CHUNK_ELEMS


def shard(n: int, world: int, rank: int) -> tuple[int, int]:
    """[start, end) of rank's shard: whole chunks, the last shard taking the
    partial chunk; empty (start == end) for ranks beyond the chunk count."""
    chunks = -(-n // CHUNK)
    per = -(-chunks // max(1, world))
    a0 = min(n, rank * per * CHUNK)
    return a0, min(n, a0 + per * CHUNK)


def escapes(dt: int, n: int, nbytes: int) -> int:
    """Escape count of a stream of nbytes bytes encoding n elements."""
    fixed = S.sz_encoded_size(dt, n, 0)
    if nbytes < fixed or (nbytes - fixed) % 3:
        raise ValueError("not a stream size for this element count")
    return (nbytes - fixed) // 3


def exchange_sizes(dist, n_local: int, bytes_local: int, device="cpu", group=None) -> tuple[list[int], list[int]]:
    """All ranks' element counts and stream sizes, in rank order (one
    all-gather; `device` is where the backend wants its tensors)."""
    mine = torch.tensor([n_local, bytes_local], dtype=torch.int64, device=device)
    got = [torch.empty_like(mine) for _ in range(dist.get_world_size(group))]
    dist.all_gather(got, mine, group=group)
    pairs = [t.cpu().tolist() for t in got]
    return [p[0] for p in pairs], [p[1] for p in pairs]


def escapes_before(dt: int, ns, sizes) -> list[int]:
    """Exclusive scan of the shard escape counts: the offset to add to shard
    k's chunk headers (and its record index) in the whole tensor's stream."""
    out, acc = [], 0
    for n, b in zip(ns, sizes):
        out.append(acc)
        acc += escapes(dt, n, b)
    return out


def joined_size(dt: int, ns, sizes) -> int:
    """Size of the whole tensor's stream built from these shard streams."""
    return S.sz_encoded_size(dt, sum(ns), sum(escapes(dt, n, b) for n, b in zip(ns, sizes)))
