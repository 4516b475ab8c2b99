"""The codec captured into a CUDA graph on its very first use in a process:
the launchers' one-time per-kernel setup (shared memory limit, occupancy
query) must be legal inside a stream capture.  Runs in a child process so
that nothing has touched the library before the capture."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
from lossless_kv_cache_bf16_gb300 import splitzip as S
from tests.oracle_pins import CB_E5_MID, CB_MID
for dt, cb in ((S.SZ_BF16, CB_MID), (S.SZ_FP8_E5M2, CB_E5_MID)):
    n = 3 * 65536 + 17
    g = torch.Generator(device="cuda"); g.manual_seed(5)
    if dt == S.SZ_BF16:
        x = (torch.randn(n, generator=g, device="cuda") * 30).to(torch.bfloat16)
    else:
        x = torch.randint(0, 256, (n,), generator=g, device="cuda", dtype=torch.uint8)
    out = torch.empty(S.sz_encoded_size(dt, n, n), dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(dt, n), dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.empty_like(x)
    cap = S.sz_encoded_size(dt, n, n)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            S.sz_encode(dt, cb, x, out, size, st, ws)
    torch.cuda.current_stream().wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    s = int(size.item())
    S.sz_decode(dt, out, s, n, y, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.equal(y.view(torch.uint8), x.view(torch.uint8))
print("ok")
"""


def test_first_use_inside_a_graph_capture():
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
