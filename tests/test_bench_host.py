"""bench.py host logic (CPU): throughput aggregation, the link model, the
profile-traffic lookup, and the N>1 path's max-over-ranks timing run as two
gloo ranks on 127.0.0.1."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_aggregate_uses_slowest_rank():
    value, t = bench.aggregate(10 ** 9, [0.5, 0.25])
    assert t == 0.5 and value == pytest.approx(2 * 10 ** 9 / 0.5 / 1e9)


def test_link_model():
    m = bench.link_model(10 ** 9, 750_000_000, 0.001, 0.0005)
    raw = 10 ** 9 / 50e9
    coded = 0.001 + 750_000_000 / 50e9 + 0.0005
    assert m["50GBps"]["speedup"] == pytest.approx(raw / coded)
    assert m["100GBps"]["raw_ms"] == pytest.approx(10.0)


def test_traffic_is_null_without_matching_profile(tmp_path, monkeypatch):
    assert bench.profiled_traffic("encode_bf16", "no_such_workload") is None
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "profiles")
    csrc = tmp_path / "lossless_kv_cache_bf16_gb300" / "csrc"
    os.makedirs(csrc)
    for name in bench.KERNEL_SOURCES["encode_bf16"]:
        (csrc / name).write_text('#include "sz_hdr.cuh"\nv1')
    (csrc / "sz_hdr.cuh").write_text("h1")
    assert "sz_hdr.cuh" in bench.source_closure(bench.KERNEL_SOURCES["encode_bf16"])

    def record():
        h = bench.kernel_source_hash("encode_bf16")
        (tmp_path / "profiles" / "encode_bf16_w.txt").write_text(
            f"kernel_source_sha256_16: {h}\ndram_bytes_per_launch: 1234\n")

    record()
    assert bench.profiled_traffic("encode_bf16", "w") == 1234
    (csrc / "sz_hdr.cuh").write_text("h2")   # an included header changed since the capture
    assert bench.profiled_traffic("encode_bf16", "w") is None
    record()
    (csrc / "sz_bf16.cu").write_text('#include "sz_hdr.cuh"\nv2')   # the kernel itself changed
    assert bench.profiled_traffic("encode_bf16", "w") is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [0.75, 0.5][rank]
    per_rank = bench.gather_elapsed(dist, elapsed, torch.device("cpu"))
    value, t = bench.aggregate(3 * 10 ** 9, per_rank)
    q.put((rank, per_rank, value, t))
    dist.destroy_process_group()


def test_two_rank_max_over_ranks():
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
    for rank, per_rank, value, t in out:
        assert per_rank == [0.75, 0.5]
        assert t == 0.75
        assert value == pytest.approx(2 * 3 * 10 ** 9 / 0.75 / 1e9)


def test_bench_legs_are_defined():
    # Every leg main() calls exists at module level (a missing one would only
    # show where a GPU runs the bench).
    import ast

    tree = ast.parse(open(bench.__file__).read())
    defined = {n.name for n in tree.body if isinstance(n, (ast.FunctionDef, ast.ClassDef))}
    main = next(n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name == "main")
    called = {c.func.id for c in ast.walk(main) if isinstance(c, ast.Call) and isinstance(c.func, ast.Name)}
    local = {n.name for n in ast.walk(main) if isinstance(n, ast.FunctionDef)}
    local |= {n.id for n in ast.walk(main) if isinstance(n, ast.Name) and isinstance(n.ctx, ast.Store)}
    import builtins

    missing = {name for name in called - local - defined if not hasattr(builtins, name)}
    assert not missing, missing


def test_rates_and_codec_roofline():
    # 1 GB in, 0.75 GB stream: the codec moves 1.75 GB per call; at 1 ms per
    # encode and 0.5 ms per decode against a 7,000 GB/s copy peak.
    r = bench.rates(10 ** 9, 750_000_000, 0.001, 0.0005, 7000.0)
    assert r["encode_gbs"] == pytest.approx(1000.0) and r["decode_gbs"] == pytest.approx(2000.0)
    assert r["encode_frac_of_codec_roofline"] == pytest.approx(1750.0 / 7000.0)
    assert r["decode_frac_of_codec_roofline"] == pytest.approx(3500.0 / 7000.0)
    assert r["codec_roofline_gbs"] == pytest.approx(7000.0 / 1.75)


def test_default_run_headlines_the_largest_graded_workload():
    from lossless_kv_cache_bf16_gb300 import workloads as W

    largest = max(bench.GRADED, key=lambda name: W.CONFIGS[name].numel * (2 if W.CONFIGS[name].dtype == "bf16" else 1))
    assert largest == "long_ctx_gqa"
    import inspect

    assert '"--config", default="long_ctx_gqa"' in inspect.getsource(bench.main)
