"""A library call captured into a CUDA graph as the process's very first call:
the one-time device set-up (function attributes, the co-resident cluster
query, the tensor-map encoder lookup) then runs while the stream is being
captured.  The capture must succeed, and the replayed graph must produce the
GEMM.  It runs in a fresh Python process so that no earlier test has done the
set-up already; the parent compares the result with the oracle."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from multistage_smem_pipeline_gb300 import synthetic
from tolerance import compare

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np
import torch
from multistage_smem_pipeline_gb300 import binding, synthetic
M, N, K, out_path = int(sys.argv[1]), int(sys.argv[2]), int(sys.argv[3]), sys.argv[4]
dev = torch.device("cuda", 0)
a = torch.from_numpy(synthetic.uniform_pm1(501, (M, K)).view(np.float16)).to(dev)
b = torch.from_numpy(synthetic.uniform_pm1(502, (N, K)).view(np.float16)).to(dev)
d = torch.zeros((M, N), dtype=torch.float16, device=dev)
side = torch.cuda.Stream(dev)
side.wait_stream(torch.cuda.current_stream(dev))
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=side):
    binding.gemm_tn_f16(a, b, out=d, stream=torch.cuda.current_stream(dev))
for _ in range(2):
    g.replay()
torch.cuda.synchronize()
status, raw = binding.get_device_error()
assert status == 0, hex(raw)
np.save(out_path, d.cpu().numpy().view(np.uint16))
"""


@pytest.mark.parametrize("M,N,K", [(512, 768, 1024), (1024, 1536, 2048)])
def test_first_call_inside_a_graph_capture(gpu, tmp_path, M, N, K):
    out = str(tmp_path / "d.npy")
    r = subprocess.run([sys.executable, "-c", CHILD, str(M), str(N), str(K), out], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    got = np.load(out)
    a = synthetic.uniform_pm1(501, (M, K))
    b = synthetic.uniform_pm1(502, (N, K))
    st = compare(got, oracle.gemm_tn(a, b), K, a, b)
    assert st["bad"] == 0, st
