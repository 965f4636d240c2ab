"""moe_forward_trace: the layer's output is moe_forward's, bit for bit, and the per-CTA
global-timer stamps of the decode kernels are present and ordered (start <= wait done <=
done within a CTA; each kernel starts no earlier than the one before it starts), to within
the timer's agreement across SMs."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_gemv_gb300 import binding as B
from mixture_experts_layer_gemv_gb300.synth import WORKLOADS, make_tokens, make_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_layer_gemv_gb300 import build
    build.build()
    B.lib()


@pytest.mark.parametrize("name,T", [("tiny_t8", 8), ("dsv2_decode_t1", 1), ("dsv2_decode_t1", 37)])
def test_trace_matches_forward_and_stamps_are_ordered(name, T):
    wl = WORKLOADS[name]
    cfg = wl.cfg
    W = make_weights(cfg, wl.seed, "cuda")
    x = make_tokens(cfg, T, wl.seed, "cuda")
    ws = B.alloc_workspace(cfg, T)
    ref = torch.empty_like(x)
    B.moe_forward(cfg, x, W, ref, ws=ws)
    out = torch.empty_like(x)
    tr = torch.zeros(B.TRACE_WORDS, dtype=torch.int64, device="cuda")
    B.moe_forward_trace(cfg, x, W, out, tr, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert B.moe_read_device_status(ws) == 0
    t = tr.view(len(B.TRACE_KERNELS), B.TRACE_CTAS, len(B.TRACE_EVENTS)).cpu().numpy()
    # the router has one CTA per routed expert, every one of which stamps start, wait and done
    route = t[0, :cfg.n_routed]
    assert (route[:, [0, 1, 3]] > 0).all()
    starts = []
    for k in range(len(B.TRACE_KERNELS)):
        rows = t[k][(t[k, :, 0] > 0) & (t[k, :, 3] > 0)]  # CTAs without work leave before "done"
        assert len(rows) > 0, B.TRACE_KERNELS[k]
        # the global timer is read on each SM; reads may disagree by tens of ns, so order
        # is checked with 1 us of slack
        assert (rows[:, 0] <= rows[:, 1] + 1000).all() and (rows[:, 1] <= rows[:, 3] + 1000).all()
        starts.append(rows[:, 0].min())
    assert all(np.diff(starts) >= -1000), starts
