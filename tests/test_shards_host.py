"""Sharding by whole chunks and the size exchange that a single stream of the
whole tensor needs (CPU): ranges, escape counts from stream sizes, the
exclusive scan, and the all-gather run as two gloo ranks on 127.0.0.1."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import oracle as O

C = 65536


def _shards():
    from lossless_kv_cache_bf16_gb300 import shards

    return shards


@pytest.mark.parametrize("n", [0, 1, C - 1, C, 3 * C + 7, 10 * C])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shards_cover_the_tensor_in_whole_chunks(n, world):
    sh = _shards()
    ranges = [sh.shard(n, world, r) for r in range(world)]
    at = 0
    for a0, a1 in ranges:
        assert a0 == at and a1 >= a0
        at = a1
    assert at == n
    nonempty = [r for r in ranges if r[1] > r[0]]
    for a0, a1 in nonempty[:-1]:
        assert a0 % C == 0 and a1 % C == 0


@pytest.mark.parametrize("n", [1, C, 3 * C + 7, 10 * C, 17 * C + 1])
@pytest.mark.parametrize("parts", [1, 2, 3, 8])
def test_shards_are_the_transfer_segments(n, parts):
    # The offload pipeline's segments and the ranks' shards cut alike, so a
    # rank's offloaded segments join exactly like its shards.
    from lossless_kv_cache_bf16_gb300 import transfer as T

    sh = _shards()
    ranges = [sh.shard(n, parts, r) for r in range(parts)]
    assert [r for r in ranges if r[1] > r[0]] == T.segments(n, parts)


def _bf16_bytes(n, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(n) * 30).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16).view(np.uint8)  # truncated to bf16 bit patterns


def test_escape_scan_and_joined_size_match_the_oracle(orc):
    from lossless_kv_cache_bf16_gb300 import splitzip as S

    sh = _shards()
    cb = np.arange(120, 136, dtype=np.uint8)
    n, world = 5 * C + 321, 3
    xb = _bf16_bytes(n, 1)
    ns, sizes, counts = [], [], []
    for r in range(world):
        a0, a1 = sh.shard(n, world, r)
        s = orc.encode(O.BF16, cb, xb[2 * a0:2 * a1])
        ns.append(a1 - a0)
        sizes.append(s.size)
        counts.append(orc.count_escapes(O.BF16, cb, xb[2 * a0:2 * a1]))
    assert [sh.escapes(S.SZ_BF16, m, b) for m, b in zip(ns, sizes)] == counts
    assert sh.escapes_before(S.SZ_BF16, ns, sizes) == [0, counts[0], counts[0] + counts[1]]
    assert sh.joined_size(S.SZ_BF16, ns, sizes) == orc.encode(O.BF16, cb, xb).size
    with pytest.raises(ValueError):
        sh.escapes(S.SZ_BF16, 10, S.sz_encoded_size(S.SZ_BF16, 10, 0) + 1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from lossless_kv_cache_bf16_gb300 import shards as sh
    from lossless_kv_cache_bf16_gb300 import splitzip as S

    orc = O.default()
    cb = np.arange(120, 136, dtype=np.uint8)
    n = 3 * C + 99
    xb = _bf16_bytes(n, 2)  # every rank draws the same tensor and encodes its shard
    a0, a1 = sh.shard(n, world, rank)
    s = orc.encode(O.BF16, cb, xb[2 * a0:2 * a1])
    ns, sizes = sh.exchange_sizes(dist, a1 - a0, s.size)
    q.put((rank, ns, sizes, sh.escapes_before(S.SZ_BF16, ns, sizes), sh.joined_size(S.SZ_BF16, ns, sizes)))
    dist.destroy_process_group()


def test_two_ranks_exchange_their_shard_sizes(orc):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    cb = np.arange(120, 136, dtype=np.uint8)
    n = 3 * C + 99
    xb = _bf16_bytes(n, 2)
    from lossless_kv_cache_bf16_gb300 import shards as sh

    want_ns, want_sizes = [], []
    for r in range(2):
        a0, a1 = sh.shard(n, 2, r)
        want_ns.append(a1 - a0)
        want_sizes.append(orc.encode(O.BF16, cb, xb[2 * a0:2 * a1]).size)
    whole = orc.encode(O.BF16, cb, xb).size
    for rank, ns, sizes, before, joined in out:
        assert ns == want_ns and sizes == want_sizes
        assert before[0] == 0 and joined == whole
