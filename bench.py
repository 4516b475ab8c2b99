#!/usr/bin/env python3
"""SplitZip codec bench: encode + decode throughput on GB300.

One step = one pass of the whole hot path over one batch: sz_encode of the
workload tensor (split, code, pack, ordered escape compaction), then
sz_decode of the stream (dense LUT pass + escape overwrite).  The default
workload is the Llama-3-8B-shaped BF16 prefill KV cache [32, 2, 8192, 8, 128]
(1.07 GB).  Throughput is uncompressed bytes / time.  Inputs (1.07 GB) are
larger than L2 (129 MB), so no L2 flush is needed between steps.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on
the host instead.  For N > 1 (torchrun), every rank runs its own copy of the
workload on its own GPU (independent shards, no data-path collective: weak
scaling); a barrier and a max-over-ranks of the elapsed time bracket the
timed region.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "encode / decode GB/s (uncompressed) on 1 GB300, % of codec HBM roofline, ratio"
UNIT = "GB/s"
LINKS_GBS = (50.0, 100.0)   # inter-node links of the pages' transfer setting
PAPER_ENCODE_GBS = 613.3    # pages' encode throughput (hardware not named): context only
PAPER_DECODE_GBS = 2181.8
PAPER_E5M2_RATIO = 1.14     # pages' E5M2 compression ratio (about 8/7)
SPEC_HBM_GBS = 8000.0       # GB300 HBM3e, nominal

# Each timed operation, the kernels it launches and the translation units they
# are built from (their included headers count too, see kernel_source_hash).
# sz_encode is two launches (the streaming encode kernel, then finish_kernel);
# sz_decode is one.
OPS = {
    "encode_bf16": (["encode_bf16_kernel", "finish_kernel"], ["sz_bf16.cu", "sz_finish.cu"]),
    "decode_bf16": (["decode_bf16_kernel"], ["sz_bf16.cu"]),
    "encode_e5m2": (["encode_e5m2_kernel", "finish_kernel"], ["sz_e5m2.cu", "sz_finish.cu"]),
    "decode_e5m2": (["decode_e5m2_kernel"], ["sz_e5m2.cu"]),
}
KERNEL_SOURCES = {op: srcs for op, (_, srcs) in OPS.items()}


def _csrc() -> str:
    return os.path.join(ROOT, "lossless_kv_cache_bf16_gb300", "csrc")


def source_closure(names) -> list[str]:
    """The given csrc files and every csrc header they include, transitively,
    sorted."""
    import re

    seen, todo = set(), list(names)
    while todo:
        name = todo.pop()
        if name in seen or not os.path.exists(os.path.join(_csrc(), name)):
            continue
        seen.add(name)
        with open(os.path.join(_csrc(), name)) as f:
            todo += re.findall(r'^#include "([A-Za-z0-9_.]+)"', f.read(), re.M)
    return sorted(seen)


def kernel_source_hash(op: str) -> str:
    h = hashlib.sha256()
    for name in source_closure(KERNEL_SOURCES[op]):
        with open(os.path.join(_csrc(), name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(op: str, workload: str):
    """DRAM bytes per call of `op` (summed over its kernels) from a committed
    ncu summary, or None if there is none or a source changed since it was
    taken."""
    path = os.path.join(ROOT, "profiles", f"{op}_{workload}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            k, sep, v = line.partition(":")
            if sep:
                fields[k.strip()] = v.strip()
    if fields.get("kernel_source_sha256_16") != kernel_source_hash(op):
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def link_model(n_bytes: int, stream_bytes: int, t_enc_s: float, t_dec_s: float):
    """Modelled transfer over a link of L GB/s: raw = bytes / L; with the codec
    = encode + stream / L + decode."""
    out = {}
    for L in LINKS_GBS:
        raw = n_bytes / (L * 1e9)
        coded = t_enc_s + stream_bytes / (L * 1e9) + t_dec_s
        out[f"{int(L)}GBps"] = {"raw_ms": raw * 1e3, "splitzip_ms": coded * 1e3, "speedup": raw / coded}
    return out


def gather_elapsed(dist, elapsed_s: float, device) -> list[float]:
    """Every rank's elapsed time (for the max-over-ranks); [elapsed] alone
    without a process group."""
    if dist is None:
        return [elapsed_s]
    import torch

    parts = [torch.zeros(1, dtype=torch.float64, device=device) for _ in range(dist.get_world_size())]
    dist.all_gather(parts, torch.tensor([elapsed_s], dtype=torch.float64, device=device))
    return [float(t.item()) for t in parts]


def aggregate(bytes_per_rank: int, elapsed_per_rank_s: list[float]):
    """Whole-job throughput: all ranks' bytes over the slowest rank's time."""
    t = max(elapsed_per_rank_s)
    return len(elapsed_per_rank_s) * bytes_per_rank / t / 1e9, t


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.started = False
        self.gpu = gpu_index

    def start(self):
        self.started = True
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            why = "nvidia-smi unavailable" if self.started else "not sampled (--profile)"
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [why], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [[c.strip() for c in line.split(",")] for line in out.splitlines() if line.count(",") >= 7]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                smax.append(float(r[1]))
            except ValueError:
                continue
            for name, v in zip(names, r[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        loaded = [s for s in sm if s > 0]
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons), "samples": len(sm)}


SWEEP_POINTS = (("p=0", 0.0), ("p=0.001", 0.001), ("p=0.01", 0.01), ("p=0.05", 0.05), ("adversarial", None),
                ("all_escape", None))
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2


def escape_sweep_leg(S, W, dt, cb, x, out, ob, est, ws, dst, dev, stream, peak, iters=20):
    """Encode and decode throughput as the escape share grows: the sweep's
    planted-escape tensors (same size and codebook as the p = 0 tensor x),
    uniformly random non-NaN patterns, and a tensor with every exponent
    outside the codebook.  Each point is checked bit-exact before it is
    timed; the roofline fraction uses the point's own stream size.  The
    tensors are only twice the L2, so repeated calls on the same buffers would
    find part of their input still in L2: every timed call is preceded by a
    write of a buffer twice the L2 and timed on its own."""
    import torch

    n = x.numel()
    n_bytes = 2 * n
    y = torch.empty_like(x)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    e = [torch.cuda.Event(enable_timing=True) for _ in range(4 * iters)]
    res = {}
    for name, p in SWEEP_POINTS:
        if p is not None:
            t = W.escape_sweep(p, cb, dev, n=n)
        elif name == "adversarial":
            t = W.adversarial(dev, n=n)
        else:
            t = W.all_escape(cb, dev, n=n)
        S.sz_encode(dt, cb, t, out, ob, est, ws)
        torch.cuda.synchronize()
        size = int(ob.item())
        S.sz_decode(dt, out, size, n, y, dst)
        torch.cuda.synchronize()
        assert int(est.item()) == 0 and int(dst.item()) == 0, name
        assert torch.equal(y.view(torch.uint8), t.view(torch.uint8)), f"{name}: round trip is not bit-exact"
        for _ in range(3):
            S.sz_encode(dt, cb, t, out, ob, est, ws)
            S.sz_decode(dt, out, size, n, y, dst)
        for i in range(iters):
            flush.fill_(i & 0xFF)
            e[4 * i].record(stream)
            S.sz_encode(dt, cb, t, out, ob, est, ws)
            e[4 * i + 1].record(stream)
            flush.fill_((i + 1) & 0xFF)
            e[4 * i + 2].record(stream)
            S.sz_decode(dt, out, size, n, y, dst)
            e[4 * i + 3].record(stream)
        torch.cuda.synchronize()
        te = sum(e[4 * i].elapsed_time(e[4 * i + 1]) for i in range(iters)) / iters / 1e3
        td = sum(e[4 * i + 2].elapsed_time(e[4 * i + 3]) for i in range(iters)) / iters / 1e3
        res[name] = {"escape_rate": (size - S.sz_encoded_size(dt, n, 0)) / 3 / n, "ratio": n_bytes / size,
                     "encode_gbs": n_bytes / te / 1e9, "decode_gbs": n_bytes / td / 1e9,
                     "encode_frac_of_codec_roofline": (n_bytes + size) / te / 1e9 / peak,
                     "decode_frac_of_codec_roofline": (n_bytes + size) / td / 1e9 / peak}
        del t
    return res


def offload_leg(S, T, dt, cb, x, y, dev, parts, reps=5):
    """The tensor to pinned host memory and back over this machine's host
    link: raw copies against the pipelined codec (transfer.Pipeline), each
    the median of `reps` host-timed runs; GB/s counts uncompressed bytes."""
    import torch

    n_bytes = x.numel() * x.element_size()
    xb = x.view(torch.uint8).reshape(-1)
    yb = y.view(torch.uint8).reshape(-1)
    raw = torch.empty(n_bytes, dtype=torch.uint8, pin_memory=True)
    pipe = T.Pipeline(dt, cb, n_bytes // S.ELEMENT_BYTES[dt], dev, parts=parts)

    def timed(fn):
        ts = []
        for _ in range(reps + 1):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            ts.append(time.perf_counter() - t0)
        return statistics.median(ts[1:])

    t_raw_d2h = timed(lambda: raw.copy_(xb))
    t_raw_h2d = timed(lambda: yb.copy_(raw))
    held = {}
    t_off = timed(lambda: held.__setitem__("hs", pipe.offload(x)))
    y.fill_(0)
    t_rel = timed(lambda: pipe.reload(held["hs"], y))
    pipe.reload_status()
    assert torch.equal(y.view(torch.uint8), x.view(torch.uint8)), "reloaded tensor is not bit-exact"
    hs = held["hs"]
    return {"segments": len(hs.segs), "raw_bytes": n_bytes, "host_bytes": hs.nbytes,
            "raw_d2h_gbs": n_bytes / t_raw_d2h / 1e9, "raw_h2d_gbs": n_bytes / t_raw_h2d / 1e9,
            "offload_gbs": n_bytes / t_off / 1e9, "reload_gbs": n_bytes / t_rel / 1e9,
            "offload_speedup": t_raw_d2h / t_off, "reload_speedup": t_raw_h2d / t_rel,
            "note": "offload = encode + D2H of the streams, reload = H2D + decode, pipelined over segments; "
                    "raw = one pinned copy of the tensor"}


# ---- the reference arm: the CPU oracle ------------------------------------------

def time_oracle(orc, dt_oracle, cb, xb, n):
    t0 = time.perf_counter()
    s = orc.encode(dt_oracle, cb, xb)
    t1 = time.perf_counter()
    st, y = orc.decode(dt_oracle, s, n)
    t2 = time.perf_counter()
    assert st == 0
    return t1 - t0, t2 - t1, s.size


# ---- main ------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["splitzip", "reference"], default="splitzip")
    ap.add_argument("--config", default="llama8b_prefill",
                    choices=["llama8b_prefill", "long_ctx_gqa", "fp8_e5m2", "escape_sweep", "tiny"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-segments", type=int, default=8,
                    help="whole-chunk segments the end-to-end leg pipelines across three streams")
    ap.add_argument("--layers", type=int, default=None,
                    help="use only the first L layers of a layered workload (smaller captures for ncu)")
    ap.add_argument("--profile", action="store_true",
                    help="only the timed encode/decode steps: no clock warm-up, e2e, memcpy or CPU baseline")
    args = ap.parse_args()
    if args.profile:
        args.no_cpu_baseline = True
        args.e2e_steps = 0
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    import numpy as np
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist = dist_mod
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)

    from lossless_kv_cache_bf16_gb300 import workloads as W

    cfg = W.CONFIGS[args.config]
    is_bf16 = cfg.dtype == "bf16"
    elem_bytes = 2 if is_bf16 else 1

    if args.impl == "reference":
        if rank != 0:
            return 0
        from oracle import oracle as O

        dev = "cuda" if torch.cuda.is_available() else "cpu"
        x = W.workload(args.config, dev)
        sample = W.calibration_sample(args.config, dev, full=x)
        odt = O.BF16 if is_bf16 else O.E5M2
        orc = O.default()
        cb = orc.calibrate(odt, sample.contiguous().view(torch.uint8).reshape(-1).cpu().numpy())
        # Bounded per-step sample: about 30 s for the whole run at ~0.3 GB/s.
        budget = int(30 * 0.3e9 / (args.steps + args.warmup))
        n_s = max(65536, min(cfg.numel, budget // elem_bytes))
        n_s -= n_s % 65536 if n_s > 65536 else 0
        xb = x.reshape(-1)[:n_s].contiguous().view(torch.uint8).cpu().numpy()
        del x
        for _ in range(args.warmup):
            time_oracle(orc, odt, cb, xb, n_s)
        t = 0.0
        for _ in range(args.steps):
            te, td, _ = time_oracle(orc, odt, cb, xb, n_s)
            t += te + td
        value = args.steps * n_s * elem_bytes / t / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16" if is_bf16 else "u8",
                "data": "synthetic", "config": {"workload": args.config, "elements_per_step": n_s},
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                                 "sample": f"first {n_s} elements of {args.config} per step (encode + decode)"},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    from lossless_kv_cache_bf16_gb300 import build as B

    B.build()
    from lossless_kv_cache_bf16_gb300 import splitzip as S
    from lossless_kv_cache_bf16_gb300 import transfer as T

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dt = S.SZ_BF16 if is_bf16 else S.SZ_FP8_E5M2
    stream = torch.cuda.current_stream()

    x = W.workload(args.config, dev)
    sample = W.calibration_sample(args.config, dev, full=x)
    if args.layers is not None:
        assert x.dim() == 5 and 0 < args.layers <= x.shape[0], "--layers needs a layered workload"
        x = x[: args.layers].contiguous()
    hist = torch.empty(S.sz_histogram_bins(dt), dtype=torch.int64, device=dev)
    cb = S.sz_calibrate(dt, sample, hist)
    del sample
    n = x.numel()
    n_bytes = n * elem_bytes
    cap = S.sz_encoded_size(dt, n, n)
    out = torch.empty(cap, dtype=torch.uint8, device=dev)
    ws = torch.empty(S.sz_workspace_size(dt, n), dtype=torch.uint8, device=dev)
    ob = torch.zeros(1, dtype=torch.int64, device=dev)
    est = torch.zeros(1, dtype=torch.int32, device=dev)
    dst = torch.zeros(1, dtype=torch.int32, device=dev)
    y = torch.empty_like(x)

    def encode():
        S.sz_encode(dt, cb, x, out, ob, est, ws)

    def decode(size):
        S.sz_decode(dt, out, size, n, y, dst)

    # Size of the stream (fixed for a given input), then check the round trip.
    encode()
    torch.cuda.synchronize()
    size = int(ob.item())
    decode(size)
    torch.cuda.synchronize()
    assert int(est.item()) == 0 and int(dst.item()) == 0, "codec reported an error"
    assert torch.equal(y.view(torch.uint8), x.view(torch.uint8)), "round trip is not bit-exact"
    n_esc = (size - S.sz_encoded_size(dt, n, 0)) // 3

    for _ in range(args.warmup):
        encode()
        decode(size)
    # Keep the GPU busy for a moment so the clock sampler sees it under load.
    sampler = ClockSampler(local_rank)
    if not args.profile:
        sampler.start()
        t_end = time.time() + 0.6
        while time.time() < t_end:
            encode()
            decode(size)
            torch.cuda.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for e0, e1, e2 in ev:
        e0.record(stream)
        encode()
        e1.record(stream)
        decode(size)
        e2.record(stream)
    t_stop.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    elapsed = t_start.elapsed_time(t_stop) / 1e3
    t_enc = [a.elapsed_time(b) / 1e3 for a, b, _ in ev]
    t_dec = [b.elapsed_time(c) / 1e3 for _, b, c in ev]
    assert int(est.item()) == 0 and int(dst.item()) == 0

    value, t_max = aggregate(K * n_bytes, gather_elapsed(dist, elapsed, dev))

    online = None
    if not args.profile:
        # Online (per-tensor) calibration on the device, the alternative to the
        # offline codebook that the pages' calibration ablation weighs: the
        # histogram of one 128-byte line in every run of s lines plus the top-16, then an
        # encode that reads that codebook from device memory.
        dcb = torch.empty(16, dtype=torch.uint8, device=dev)
        dhist = torch.empty(S.sz_histogram_bins(dt), dtype=torch.int64, device=dev)
        online = {}
        for stride in (1, 16):
            for _ in range(3):
                S.sz_calibrate_device(dt, x, dhist, dcb, sample_stride=stride)
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            for _ in range(20):
                S.sz_calibrate_device(dt, x, dhist, dcb, sample_stride=stride)
            c1.record(stream)
            torch.cuda.synchronize()
            online[f"calibrate_us_stride{stride}"] = c0.elapsed_time(c1) / 20 * 1e3
        for _ in range(3):
            S.sz_encode_dcb(dt, dcb, x, out, ob, est, ws)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(20):
            S.sz_encode_dcb(dt, dcb, x, out, ob, est, ws)
        c1.record(stream)
        torch.cuda.synchronize()
        assert int(est.item()) == 0
        online_size = int(ob.item())
        online.update({"sample": "one 128-byte line in every run of 16 lines (hashed position) of the tensor itself",
                       "encode_dcb_gbs": n_bytes / (c0.elapsed_time(c1) / 20 / 1e3) / 1e9,
                       "codebook": dcb.cpu().tolist(), "offline_codebook": [int(v) for v in cb],
                       "ratio": n_bytes / online_size, "ratio_offline": n_bytes / size})

    paged = None
    if not args.profile:
        # Paged KV: the tensor seen as a pool of pages of 16 tokens (x heads x
        # head_dim elements), a shuffled block table over all of them, encoded
        # straight from the pages and decoded straight into a second pool.
        page_elems = 16 * x.shape[-1] * x.shape[-2] if x.dim() == 5 else 16384
        if n % page_elems == 0:
            pages = n // page_elems
            gperm = torch.Generator(device="cpu")
            gperm.manual_seed(7)
            ids = torch.randperm(pages, generator=gperm).to(torch.int32).to(dev)
            pout = torch.empty(S.sz_encoded_size(dt, n, n), dtype=torch.uint8, device=dev)
            for _ in range(3):
                S.sz_encode_paged(dt, cb, x, page_elems, ids, n, pout, ob, est, ws)
            torch.cuda.synchronize()
            psize = int(ob.item())
            for _ in range(3):
                S.sz_decode_paged(dt, pout, psize, n, y, page_elems, ids, dst)
            ev3 = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev3[0].record(stream)
            for _ in range(20):
                S.sz_encode_paged(dt, cb, x, page_elems, ids, n, pout, ob, est, ws)
            ev3[1].record(stream)
            for _ in range(20):
                S.sz_decode_paged(dt, pout, psize, n, y, page_elems, ids, dst)
            ev3[2].record(stream)
            torch.cuda.synchronize()
            assert int(est.item()) == 0 and int(dst.item()) == 0
            assert torch.equal(y.view(torch.uint8), x.view(torch.uint8)), "paged round trip is not bit-exact"
            paged = {"page_elems": page_elems, "pages": pages, "block_table": "random permutation of all pages",
                     "encode_gbs": n_bytes / (ev3[0].elapsed_time(ev3[1]) / 20 / 1e3) / 1e9,
                     "decode_gbs": n_bytes / (ev3[1].elapsed_time(ev3[2]) / 20 / 1e3) / 1e9,
                     "stream_bytes": psize}
            # Restore y as the plain decode of the contiguous stream for what follows.
            S.sz_decode(dt, out, size, n, y, dst)

    ablation = None
    if not args.profile:
        # Codebook ablation on this tensor: exact stream sizes under Top-16
        # (this format), Top-8 and Top-15 + sentinel, from the device
        # histogram of the whole tensor.
        fh = torch.empty(S.sz_histogram_bins(dt), dtype=torch.int64, device=dev)
        S.sz_histogram(dt, x, fh)
        counts = fh.cpu().tolist()
        s16, s8, s15 = S.sz_ablation_sizes(dt, counts, n)
        top = sorted(counts, reverse=True)
        ablation = {"ratio_top16": n_bytes / s16, "ratio_top8": n_bytes / s8, "ratio_top15_sentinel": n_bytes / s15,
                    "coverage_top16": sum(top[:16]) / n, "coverage_top8": sum(top[:8]) / n,
                    "coverage_top15": sum(top[:15]) / n,
                    "note": "sizes from the whole-tensor exponent histogram; the Top-8 and sentinel layouts are "
                            "readings (codes + the same headers; Top-8 keeps position records, the sentinel "
                            "stores only exponent bytes)"}
        if is_bf16:
            # Decode speed of the alternative designs on this tensor (their
            # encoders are plain and not timed).
            speeds = {"top16": n_bytes / statistics.mean(t_dec) / 1e9}
            for variant, name in ((S.SZ_ABL_TOP8, "top8"), (S.SZ_ABL_SENTINEL, "top15_sentinel")):
                acb = S.sz_ablation_codebook(variant, counts)
                aout = torch.empty(S.sz_ablation_encoded_size(variant, n, n), dtype=torch.uint8, device=dev)
                aws = torch.empty(S.sz_ablation_workspace_size(n), dtype=torch.uint8, device=dev)
                S.sz_ablation_encode(variant, acb, x, aout, ob, aws)
                torch.cuda.synchronize()
                asize = int(ob.item())
                for _ in range(3):
                    S.sz_ablation_decode(variant, aout, asize, n, y, dst)
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                for _ in range(20):
                    S.sz_ablation_decode(variant, aout, asize, n, y, dst)
                a1.record(stream)
                torch.cuda.synchronize()
                assert int(dst.item()) == 0 and torch.equal(y.view(torch.uint8), x.view(torch.uint8)), name
                speeds[name] = n_bytes / (a0.elapsed_time(a1) / 20 / 1e3) / 1e9
                del aout, aws
            ablation["decode_gbs"] = speeds
            ablation["decode_slowdown_vs_top16"] = {k: speeds["top16"] / v for k, v in speeds.items()}
            S.sz_decode(dt, out, size, n, y, dst)

    sweep = None
    if not args.profile and args.config == "escape_sweep":
        sweep = escape_sweep_leg(S, W, dt, cb, x, out, ob, est, ws, dst, dev, stream, peak=measured_peaks()[0])
        S.sz_encode(dt, cb, x, out, ob, est, ws)
        S.sz_decode(dt, out, size, n, y, dst)

    e2e = None
    memcpy_gbs = None
    if not args.profile and args.e2e_steps > 0:
        # End to end through the C ABI with host buffers, every step: pinned H2D
        # of the input, encode, decode, D2H of the decoded tensor.  The tensor
        # is cut into segments of whole 65,536-element chunks, each encoded as
        # its own self-contained stream (the layout of an independent shard),
        # so that the H2D copy of one segment, the codec on the previous one
        # and the D2H copy of the one before overlap on three streams.
        xh = torch.empty(n_bytes, dtype=torch.uint8, pin_memory=True)
        xh.copy_(x.view(torch.uint8).reshape(-1))
        yh = torch.empty(n_bytes, dtype=torch.uint8, pin_memory=True)
        segs = T.segments(n, args.e2e_segments)
        xf, yf = x.reshape(-1), y.reshape(-1)
        seg_cap = [S.sz_encoded_size(dt, a1 - a0, a1 - a0) for a0, a1 in segs]
        seg_at = [sum((c + 255) // 256 * 256 for c in seg_cap[:i]) for i in range(len(segs))]
        seg_buf = torch.empty(seg_at[-1] + seg_cap[-1], dtype=torch.uint8, device=dev)
        seg_out = [seg_buf[o:o + c] for o, c in zip(seg_at, seg_cap)]
        seg_size = []  # per-segment stream sizes (fixed for this input)
        for (a0, a1), o in zip(segs, seg_out):
            S.sz_encode(dt, cb, xf[a0:a1], o, ob, est, ws)
            torch.cuda.synchronize()
            seg_size.append(int(ob.item()))
        s_in, s_cod, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        in_done = [ev() for _ in segs]     # H2D of segment i landed
        enc_done = [ev() for _ in segs]    # encode of segment i has read its input
        dec_done = [ev() for _ in segs]    # decode of segment i wrote its output
        out_done = [ev() for _ in segs]    # D2H of segment i has read its output
        started = [False]

        def e2e_step():
            for i, ((a0, a1), o, sz) in enumerate(zip(segs, seg_out, seg_size)):
                b0, b1 = a0 * elem_bytes, a1 * elem_bytes
                with torch.cuda.stream(s_in):
                    if started[0]:
                        s_in.wait_event(enc_done[i])  # the previous step's encode has read it
                    x.view(torch.uint8).reshape(-1)[b0:b1].copy_(xh[b0:b1], non_blocking=True)
                    in_done[i].record(s_in)
                with torch.cuda.stream(s_cod):
                    s_cod.wait_event(in_done[i])
                    if started[0]:
                        s_cod.wait_event(out_done[i])  # the previous step's D2H has read it
                    S.sz_encode(dt, cb, xf[a0:a1], o, ob, est, ws)
                    enc_done[i].record(s_cod)
                    S.sz_decode(dt, o, sz, a1 - a0, yf[a0:a1], dst)
                    dec_done[i].record(s_cod)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(dec_done[i])
                    yh[b0:b1].copy_(y.view(torch.uint8).reshape(-1)[b0:b1], non_blocking=True)
                    out_done[i].record(s_out)
            started[0] = True

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_a.record(stream)
        for s_ in (s_in, s_cod, s_out):
            s_.wait_event(e_a)
        for _ in range(args.e2e_steps):
            e2e_step()
        for s_ in (s_in, s_cod, s_out):
            stream.wait_stream(s_)
        e_b.record(stream)
        torch.cuda.synchronize()
        e2e_t = e_a.elapsed_time(e_b) / 1e3
        e2e_value, _ = aggregate(args.e2e_steps * n_bytes, gather_elapsed(dist, e2e_t, dev))
        assert int(est.item()) == 0 and int(dst.item()) == 0, "codec reported an error"
        assert torch.equal(yh, xh), "end-to-end round trip is not bit-exact"

        # Device-to-device copy bandwidth in the same run (bytes = read + write).
        a = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
        b = torch.empty_like(a)
        for _ in range(3):
            b.copy_(a)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(10):
            b.copy_(a)
        c1.record(stream)
        torch.cuda.synchronize()
        memcpy_gbs = 2 * a.numel() * 10 / (c0.elapsed_time(c1) / 1e3) / 1e9
        del a, b

        e2e = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": n_bytes, "d2h_bytes_per_step": n_bytes,
               "steps": args.e2e_steps, "segments": len(segs), "streams": 3,
               "stream_bytes_per_step": sum(seg_size)}
    offload = None
    if not args.profile and args.e2e_steps > 0 and world == 1:
        offload = offload_leg(S, T, dt, cb, x, y, dev, parts=args.e2e_segments)

    te, td = statistics.mean(t_enc), statistics.mean(t_dec)
    enc_gbs, dec_gbs = n_bytes / te / 1e9, n_bytes / td / 1e9
    peak, peak_src = measured_peaks()
    moved = n_bytes + size
    suffix = "bf16" if is_bf16 else "e5m2"
    ops = {f"encode_{suffix}": te, f"decode_{suffix}": td}
    dominant = max(ops, key=ops.get)
    achieved = moved / ops[dominant] / 1e9
    traffic = profiled_traffic(dominant, args.config)
    roofline = {"bound": "hbm", "kernel": " + ".join(OPS[dominant][0]), "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "peak_source": f"{peak_src} hbm_gbs (copy)",
                "algorithmic_bytes_per_launch": moved}

    def dram_view(op, t):
        """Achieved HBM GB/s of one call: its ncu DRAM bytes over this run's time."""
        tr = profiled_traffic(op, args.config)
        if tr is None:
            return None
        g = tr / t / 1e9
        return {"dram_bytes_per_call": tr, "dram_gbs": g, "frac_of_spec": g / SPEC_HBM_GBS,
                "frac_of_memcpy": g / memcpy_gbs if memcpy_gbs else None, "frac_of_measured_copy": g / peak}

    hbm = {"encode": dram_view(f"encode_{suffix}", te), "decode": dram_view(f"decode_{suffix}", td),
           "source": "ncu dram__bytes_read.sum + dram__bytes_write.sum per call (profiles/), over this run's "
                     "CUDA-event time; null without a capture of the current kernels for this workload"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import oracle as O

        orc = O.default()
        odt = O.BF16 if is_bf16 else O.E5M2
        xb = x.view(torch.uint8).reshape(-1).cpu().numpy()
        tenc, tdec, osize = time_oracle(orc, odt, np.array(cb, dtype=np.uint8), xb, n)
        assert osize == size
        cpu = {"value": n_bytes / (tenc + tdec) / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"the whole {args.config} tensor ({n_bytes} bytes), one encode + one decode",
               "encode_gbs": n_bytes / tenc / 1e9, "decode_gbs": n_bytes / tdec / 1e9}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": t_max / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8" if not is_bf16 else "u16", "data": "synthetic",
        "config": {"workload": args.config + (f"[:{args.layers} layers]" if args.layers else ""), "elements": n, "input_bytes": n_bytes,
                   "step": "one sz_encode + one sz_decode of the whole tensor",
                   "l2": "inputs larger than L2 (129 MB); no flush", "parallelism": f"{world} independent shards"},
        "encode_gbs": enc_gbs, "decode_gbs": dec_gbs,
        "encode_frac_of_codec_roofline": (n_bytes + size) / te / 1e9 / peak,
        "decode_frac_of_codec_roofline": (n_bytes + size) / td / 1e9 / peak,
        "codec_roofline_gbs": peak * n_bytes / (n_bytes + size),
        "ratio": n_bytes / size, "escape_rate": n_esc / n, "stream_bytes": size,
        "memcpy_d2d_gbs": memcpy_gbs, "spec_hbm_gbs": SPEC_HBM_GBS, "hbm_achieved": hbm,
        "link_model": link_model(n_bytes, size, te, td),
        "paper_context": {"encode_gbs": PAPER_ENCODE_GBS, "decode_gbs": PAPER_DECODE_GBS,
                          "e5m2_ratio": PAPER_E5M2_RATIO, "hardware": "not named on the pages"},
        "roofline": roofline, "cpu_baseline": cpu, "online_calibration": online, "ablation": ablation, "paged": paged,
        "escape_sweep": sweep,
        "escape_sweep_timing": sweep and "each call timed on its own after a 256 MiB write that flushes L2",
        "offload": offload, "e2e": e2e,
        "gpu_launches": sum(len(OPS[op][0]) for op in ops) * K, "clocks": clocks,
    }
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
