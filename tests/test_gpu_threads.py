"""First calls from several host threads at once.

Every kernel configuration sets its shared-memory attribute on its first
launch on a device (once, under a lock).  In a fresh process, six threads
launch six different configurations at the same moment, each on its own
stream; the results must be the same bits as the same calls made one after
the other afterwards, and no error may be reported.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
import torch
import mx_gemm_gb300 as fg
from tests.gpu_util import Case
import inputs

shapes = [("fp8_tensor", 1, 2048, 7168), ("fp8_block128", 16, 2048, 2048), ("mxfp4", 1, 4096, 2048),
          ("bf16", 300, 512, 1024), ("mxfp8", 64, 512, 1024), ("fp8_block128", 300, 512, 1024)]
cases = [Case(m, *inputs.operands(m, M, N, K, 7 + i, 17 + i, 27 + i)) for i, (m, M, N, K) in enumerate(shapes)]
torch.cuda.synchronize()
outs = [None] * len(cases)
streams = [torch.cuda.Stream() for _ in cases]
start = threading.Barrier(len(cases))
errors = []

def run(i):
    try:
        start.wait()
        with torch.cuda.stream(streams[i]):
            c = cases[i]
            ws = torch.empty(max(4, fg.gemm_workspace_size(c.mode, c.M, c.N, c.K)) // 4, dtype=torch.float32,
                             device="cuda")
            outs[i] = fg.gemm(c.dA, c.pb, c.da_s, workspace=ws, stream=streams[i])
    except Exception as e:  # reported by the parent
        errors.append(repr(e))

threads = [threading.Thread(target=run, args=(i,)) for i in range(len(cases))]
for t in threads:
    t.start()
for t in threads:
    t.join()
torch.cuda.synchronize()
assert not errors, errors
assert fg.get_error() == fg.FG_OK
for i, c in enumerate(cases):
    ws = torch.empty(max(4, fg.gemm_workspace_size(c.mode, c.M, c.N, c.K)) // 4, dtype=torch.float32, device="cuda")
    again = fg.gemm(c.dA, c.pb, c.da_s, workspace=ws)
    assert torch.equal(outs[i].view(torch.int16), again.view(torch.int16)), shapes[i]
print("ok", len(cases))
"""


def test_first_calls_from_several_threads():
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "ok 6" in r.stdout
