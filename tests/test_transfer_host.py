"""Host logic of the pipelined offload/reload (no GPU): how a tensor is cut
into segments of whole 65,536-element chunks."""
import pytest

from lossless_kv_cache_bf16_gb300 import transfer as T


@pytest.mark.parametrize("n,parts", [(536870912, 8), (939524096, 8), (65537, 8), (100, 3), (0, 8),
                                     (131072 * 3, 2), (65536 * 5, 8), (1, 1)])
def test_segments_cover_whole_chunks(n, parts):
    segs = T.segments(n, parts)
    assert 1 <= len(segs) <= max(1, parts)
    assert segs[0][0] == 0 and segs[-1][1] == n
    for (a0, a1), (b0, _) in zip(segs, segs[1:]):
        assert a1 == b0 and a0 % 65536 == 0 and a1 % 65536 == 0 and a1 > a0


def test_segments_balance():
    # 8 parts of a 32-chunk tensor: 4 chunks each.
    assert T.segments(32 * 65536, 8) == [(4 * 65536 * i, 4 * 65536 * (i + 1)) for i in range(8)]
    # More parts than chunks: one chunk each.
    assert T.segments(3 * 65536, 8) == [(0, 65536), (65536, 131072), (131072, 196608)]
