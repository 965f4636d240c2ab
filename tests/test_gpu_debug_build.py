"""The MOE_DEBUG build (device-side checks of the tile decompositions' invariants: every
weight-streaming tile inside its K range, slice, part and rows; every grouped-GEMM tile
inside its A tensor) reports nothing on the decode, weight-streaming and grouped-GEMM
paths, and gives the normal build's output bit for bit. It runs in a child process that
loads the debug library (MOE_GB300_LIB)."""
import os
import subprocess
import sys
import tempfile

import pytest
import torch

from mixture_experts_layer_gemv_gb300 import binding as B
from mixture_experts_layer_gemv_gb300.synth import WORKLOADS, make_tokens, make_weights

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CASES = [("tiny_t8", 1), ("tiny_t8", 8), ("tiny_t8", 37), ("tiny_t8", 300), ("dsv2_decode_t1", 1),
         ("dsv2_decode_t1", 64)]

CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
from mixture_experts_layer_gemv_gb300 import binding as B
from mixture_experts_layer_gemv_gb300.synth import WORKLOADS, make_tokens, make_weights
outs = {}
for name, T in eval(sys.argv[2]):
    cfg = WORKLOADS[name].cfg
    W = make_weights(cfg, 31, "cuda")
    x = make_tokens(cfg, T, 32 + T, "cuda")
    ws = B.alloc_workspace(cfg, T)
    out = torch.empty_like(x)
    B.moe_forward(cfg, x, W, out, ws=ws)
    torch.cuda.synchronize()
    outs[(name, T)] = (out.cpu(), B.moe_read_device_status(ws))
torch.save(outs, sys.argv[3])
"""


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_layer_gemv_gb300 import build
    build.build()
    build.build(debug=True)
    B.lib()


def test_debug_build_reports_nothing_and_matches():
    from mixture_experts_layer_gemv_gb300 import build
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "outs.pt")
        env = dict(os.environ, MOE_GB300_LIB=build.DEBUG_LIB)
        r = subprocess.run([sys.executable, "-c", CHILD, ROOT, repr(CASES), path], env=env, capture_output=True,
                           text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-3000:]
        debug = torch.load(path)
    for name, T in CASES:
        cfg = WORKLOADS[name].cfg
        W = make_weights(cfg, 31, "cuda")
        x = make_tokens(cfg, T, 32 + T, "cuda")
        ws = B.alloc_workspace(cfg, T)
        out = torch.empty_like(x)
        B.moe_forward(cfg, x, W, out, ws=ws)
        torch.cuda.synchronize()
        d_out, d_status = debug[(name, T)]
        assert d_status == 0, (name, T, d_status)
        assert torch.equal(out.cpu(), d_out), (name, T)
