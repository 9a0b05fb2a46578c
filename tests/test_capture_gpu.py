"""A launch shape's first call on a device, captured into a CUDA graph.

The first call of a launch shape makes one-time device queries (the kernel's
shared-memory limit, its occupancy, the tensor-map encoder's entry point).
CUDA refuses such calls while the thread captures a stream in the default
(global) mode; the library makes them in relaxed mode, so the capture succeeds.
The call runs in a fresh process (nothing cached yet), its graph is replayed,
and the outputs are compared with the oracle here.
"""

import os
import subprocess
import sys

import pytest
import torch

from grouped_gemm_epilogues_gb300 import workloads as wl

from test_gemm_gpu import _check_plain

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
from grouped_gemm_epilogues_gb300 import binding, workloads as wl
cg, out_path = int(sys.argv[2]), sys.argv[3]
w = wl.small("gemm_act_4096_bf16_gelu", 300, 520, 200, 2)
t = {k: v.cuda() for k, v in wl.make(w).items() if isinstance(v, torch.Tensor)}
D = torch.full((2, 300, 520), float("nan"), dtype=torch.bfloat16, device="cuda")
P = torch.full_like(D, float("nan"))
binding.workspace(torch.device("cuda", 0), 64 << 20)   # made (and zeroed) before the capture
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g):
    binding.gge_gemm_act(t["A"], t["B"], P, w.act, D=D, C=t["C"], alpha=w.alpha, beta=w.beta,
                         config=binding.make_config(cta_group=cg, tile_n=256))
assert torch.isnan(D.float()).all(), "the captured call ran during the capture"
g.replay()
torch.cuda.synchronize()
assert binding.gge_read_device_status()[0] == "GGE_OK"
torch.save({"D": D.cpu(), "P": P.cpu()}, out_path)
"""


@pytest.mark.parametrize("cta_group", [1, 2])
def test_first_call_inside_graph_capture(tmp_path, cta_group):
    out_path = str(tmp_path / "out.pt")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, str(cta_group), out_path],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    got = torch.load(out_path)
    w = wl.small("gemm_act_4096_bf16_gelu", 300, 520, 200, 2)
    _check_plain(w, wl.make(w), got)
