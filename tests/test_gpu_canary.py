"""Out-of-bounds writes, checked without a sanitizer: every output buffer and the workspace
sit between guard regions of a fixed byte pattern, and after each call (fused forward,
MXFP8 forward, stage API) at the decode, weight-streaming and grouped-GEMM token counts
every guard byte must be unchanged. The workspace is passed with its exact size, so a
write past its end lands in the guard."""
import pytest
import torch

from mixture_experts_layer_gemv_gb300 import binding as B
from mixture_experts_layer_gemv_gb300.synth import MoEConfig, WORKLOADS, make_tokens, make_weights, make_weights_mx

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_layer_gemv_gb300 import build
    build.build()
    B.lib()


class Guarded:
    """A device buffer of n bytes between two guard regions."""

    def __init__(self, n: int):
        self.n = n
        self.raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")

    def view(self, dtype, shape):
        return self.raw[GUARD:GUARD + self.n].view(dtype).view(shape)

    def bytes(self):
        return self.raw[GUARD:GUARD + self.n]

    def intact(self) -> bool:
        return bool((self.raw[:GUARD] == PATTERN).all()) and bool((self.raw[GUARD + self.n:] == PATTERN).all())


def _forward_guarded(cfg, T, W, x, mx=False, residual=None):
    H, k = cfg.hidden, cfg.top_k
    n_ws = (B.moe_workspace_size_mx if mx else B.moe_workspace_size)(cfg, T)
    ws = Guarded(n_ws)
    B.moe_workspace_init(ws.bytes())
    out = Guarded(T * H * 2)
    ids = Guarded(T * k * 4)
    fwd = B.moe_forward_mx if mx else B.moe_forward
    for _ in range(2):  # the second call runs on the counters the first left behind
        fwd(cfg, x, W, out.view(torch.bfloat16, (T, H)), residual, ids.view(torch.int32, (T, k)), ws.bytes())
    torch.cuda.synchronize()
    assert B.moe_read_device_status(ws.bytes()) == 0
    return ws, out, ids


TINY = WORKLOADS["tiny_t8"].cfg
CASES = [
    ("tiny", TINY, 1), ("tiny", TINY, 8), ("tiny", TINY, 37), ("tiny", TINY, 64), ("tiny", TINY, 300),
    ("dsv2", WORKLOADS["dsv2_decode_t1"].cfg, 1), ("dsv2", WORKLOADS["dsv2_decode_t1"].cfg, 64),
]


@pytest.mark.parametrize("name,cfg,T", CASES, ids=[f"{c[0]}-T{c[2]}" for c in CASES])
def test_forward_writes_stay_inside_outputs_and_workspace(name, cfg, T):
    W = make_weights(cfg, 21, "cuda")
    x = make_tokens(cfg, T, 22 + T, "cuda")
    res = make_tokens(cfg, T, 23, "cuda", name="residual")
    ws, out, ids = _forward_guarded(cfg, T, W, x, residual=res)
    assert ws.intact() and out.intact() and ids.intact()
    assert bool(((ids.view(torch.int32, (T, cfg.top_k)) >= 0) &
                 (ids.view(torch.int32, (T, cfg.top_k)) < cfg.n_routed)).all())


MX_CFG = MoEConfig(512, 512, 16, 4, 2, 4, 1.0, 1)


@pytest.mark.parametrize("T", [1, 8, 300])
def test_forward_mx_writes_stay_inside_outputs_and_workspace(T):
    W = make_weights_mx(MX_CFG, 24, "cuda")
    x = make_tokens(MX_CFG, T, 25 + T, "cuda")
    ws, out, ids = _forward_guarded(MX_CFG, T, W, x, mx=True)
    assert ws.intact() and out.intact() and ids.intact()


@pytest.mark.parametrize("T", [5, 300])
def test_stage_api_writes_stay_inside_outputs(T):
    cfg = TINY
    H, k, Is = cfg.hidden, cfg.top_k, cfg.shared_inter
    W = make_weights(cfg, 26, "cuda")
    x = make_tokens(cfg, T, 27 + T, "cuda")
    ws = Guarded(B.moe_workspace_size(cfg, T))
    B.moe_workspace_init(ws.bytes())
    ids = Guarded(T * k * 4)
    w = Guarded(T * k * 4)
    B.moe_route(cfg, x, W["w_router"], W["router_bias"], ids.view(torch.int32, (T, k)),
                w.view(torch.float32, (T, k)), ws.bytes())
    offs = Guarded((cfg.n_routed + 1) * 4)
    perm = Guarded(T * k * 4)
    inv = Guarded(T * k * 4)
    B.moe_permute(cfg, ids.view(torch.int32, (T, k)), offs.view(torch.int32, (cfg.n_routed + 1,)),
                  perm.view(torch.int32, (T * k,)), inv.view(torch.int32, (T * k,)), ws.bytes())
    y_perm = Guarded(T * k * H * 2)
    y_sh = Guarded(T * H * 2)
    B.moe_expert_ffn(cfg, x, W, offs.view(torch.int32, (cfg.n_routed + 1,)), perm.view(torch.int32, (T * k,)),
                     w.view(torch.float32, (T, k)), y_perm.view(torch.bfloat16, (T * k, H)),
                     y_sh.view(torch.bfloat16, (T, H)) if Is > 0 else None, ws.bytes())
    out = Guarded(T * H * 2)
    B.moe_combine(cfg, y_perm.view(torch.bfloat16, (T * k, H)), inv.view(torch.int32, (T * k,)),
                  y_sh.view(torch.bfloat16, (T, H)) if Is > 0 else None, None, out.view(torch.bfloat16, (T, H)))
    torch.cuda.synchronize()
    assert B.moe_read_device_status(ws.bytes()) == 0
    for g in (ws, ids, w, offs, perm, inv, y_perm, y_sh, out):
        assert g.intact()
