"""Pipelined KV offload to host memory and reload, through the codec.

The pages' setting moves KV caches over a link between machines, and the
codec pays for itself when it shrinks the bytes on the link by more than it
costs (SplitZip abstract, arXiv 2605.01708v2; technical summary,
gist.science/es, "Resultados" > "Transferencia").  On one GB300 the link at
hand is the one to the host, so this module offloads a tensor to pinned host
memory as SplitZip streams and reloads it, with the codec overlapped with the
copies:

* the tensor is cut into segments of whole 65,536-element chunks, and each
  segment is encoded as its own self-contained stream (the layout of an
  independent shard);
* offload: the encode of segment i+1 on the codec stream overlaps the
  device-to-host copy of segment i's stream on the copy stream (two device
  staging buffers);
* reload: the host-to-device copy of segment i+1's stream overlaps the decode
  of segment i.

Every step runs in the library's kernels and CUDA copies; this module only
orders them.  Offload waits, on the host, for each segment's encode to learn
how many bytes to copy (the kernel writes the size into pinned host memory);
the GPU keeps working meanwhile.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import splitzip as S

CHUNK = S.SZ_CHUNK_ELEMS


def segments(n: int, parts: int) -> list[tuple[int, int]]:
    """[start, end) element ranges of at most `parts` segments of whole
    65,536-element chunks (the last one may be partial) covering n elements;
    [(0, 0)] when n is 0."""
    chunks = max(1, -(-n // CHUNK))
    per = -(-chunks // max(1, parts))
    out = []
    for c0 in range(0, chunks, per):
        a0, a1 = c0 * CHUNK, min(n, (c0 + per) * CHUNK)
        if a1 > a0:
            out.append((a0, a1))
    return out or [(0, 0)]


@dataclass
class HostStreams:
    """An offloaded tensor: segment i's stream is host[offsets[i]:offsets[i] +
    sizes[i]].  `host` is the pipeline's pinned buffer, rewritten by its next
    offload."""
    dt: int
    n: int
    segs: list
    offsets: list
    sizes: list
    host: torch.Tensor

    @property
    def nbytes(self) -> int:
        return sum(self.sizes)


class Pipeline:
    """Offload/reload of tensors of n elements of type dt with codebook cb,
    on `device`, cut into `parts` segments.  Buffers are allocated once:
    two device staging buffers and a workspace for the largest segment, and a
    pinned host buffer of host_bytes (default: the worst case of all
    segments, every element an escape).  The streams are packed one after
    the other in the host buffer; an offload whose streams do not fit raises
    SplitZipError with SZ_ERR_CAPACITY."""

    def __init__(self, dt: int, cb, n: int, device, parts: int = 8, host_bytes: int | None = None):
        self.dt, self.cb, self.n = dt, [int(v) for v in cb], n
        self.device = torch.device(device)
        self.segs = segments(n, parts)
        self.caps = [S.sz_encoded_size(dt, a1 - a0, a1 - a0) for a0, a1 in self.segs]
        big = max(a1 - a0 for a0, a1 in self.segs)
        self.dev = [torch.empty(max(self.caps), dtype=torch.uint8, device=self.device) for _ in range(2)]
        self.ws = torch.empty(S.sz_workspace_size(dt, big), dtype=torch.uint8, device=self.device)
        self.host = torch.empty(sum(self.caps) if host_bytes is None else host_bytes, dtype=torch.uint8,
                                pin_memory=True)
        k = len(self.segs)
        self.sizes_h = torch.zeros(k, dtype=torch.int64, pin_memory=True)
        self.status = torch.zeros(k, dtype=torch.int32, device=self.device)
        self.codec = torch.cuda.Stream(self.device)
        self.copy = torch.cuda.Stream(self.device)

    def _flat(self, t: torch.Tensor) -> torch.Tensor:
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return t.view(torch.uint8).reshape(-1)

    def _check_status(self, what: str):
        bad = [int(v) for v in self.status.cpu().tolist() if int(v) != S.SZ_OK]
        if bad:
            raise S.SplitZipError(what, bad[0])

    def offload(self, x: torch.Tensor) -> HostStreams:
        """Streams of x in pinned host memory (synchronises with the copies)."""
        dt, esize = self.dt, S.ELEMENT_BYTES[self.dt]
        if x.numel() * x.element_size() != self.n * esize:
            raise ValueError("tensor size differs from the pipeline's")
        xb = self._flat(x)
        k = len(self.segs)
        enc = [torch.cuda.Event() for _ in range(k)]
        freed = [torch.cuda.Event() for _ in range(2)]  # staging buffer b no longer read by a copy
        self.status.zero_()
        self.codec.wait_stream(torch.cuda.current_stream(self.device))

        def encode(i):
            a0, a1 = self.segs[i]
            b = i % 2
            with torch.cuda.stream(self.codec):
                if i >= 2:
                    self.codec.wait_event(freed[b])
                # The size lands in pinned host memory straight from the
                # kernel: a copy would queue behind the stream copies.
                S.sz_encode(dt, self.cb, xb[a0 * esize:a1 * esize], self.dev[b], self.sizes_h[i:i + 1],
                            self.status[i:i + 1], self.ws, n=a1 - a0)
                enc[i].record(self.codec)

        sizes, offsets, o = [], [], 0
        encode(0)
        for i in range(k):
            if i + 1 < k:
                encode(i + 1)
            enc[i].synchronize()  # host learns segment i's size; the GPU runs on
            size = int(self.sizes_h[i])
            if o + size > self.host.numel():
                self.codec.synchronize()
                self.copy.synchronize()
                raise S.SplitZipError("offload", S.SZ_ERR_CAPACITY)
            sizes.append(size)
            offsets.append(o)
            with torch.cuda.stream(self.copy):
                self.copy.wait_event(enc[i])
                self.host[o:o + size].copy_(self.dev[i % 2][:size], non_blocking=True)
                freed[i % 2].record(self.copy)
            o += size
        self.copy.synchronize()
        self._check_status("offload")
        return HostStreams(dt, self.n, list(self.segs), offsets, sizes, self.host)

    def reload(self, hs: HostStreams, y: torch.Tensor) -> None:
        """Decodes hs into y on the device; y is ready on the current stream
        when this returns (asynchronous otherwise)."""
        dt, esize = self.dt, S.ELEMENT_BYTES[self.dt]
        if y.numel() * y.element_size() != self.n * esize or hs.n != self.n:
            raise ValueError("tensor size differs from the pipeline's")
        yb = self._flat(y)
        k = len(hs.segs)
        landed = [torch.cuda.Event() for _ in range(k)]
        freed = [torch.cuda.Event() for _ in range(2)]  # staging buffer b decoded
        self.status.zero_()
        cur = torch.cuda.current_stream(self.device)
        self.copy.wait_stream(cur)
        self.codec.wait_stream(cur)
        for i, ((a0, a1), o, size) in enumerate(zip(hs.segs, hs.offsets, hs.sizes)):
            b = i % 2
            with torch.cuda.stream(self.copy):
                if i >= 2:
                    self.copy.wait_event(freed[b])
                self.dev[b][:size].copy_(hs.host[o:o + size], non_blocking=True)
                landed[i].record(self.copy)
            with torch.cuda.stream(self.codec):
                self.codec.wait_event(landed[i])
                S.sz_decode(dt, self.dev[b], size, a1 - a0, yb[a0 * esize:a1 * esize], self.status[i:i + 1])
                freed[b].record(self.codec)
        cur.wait_stream(self.codec)

    def reload_status(self) -> None:
        """Raises if a reload's decode reported an error (synchronises)."""
        self._check_status("reload")
