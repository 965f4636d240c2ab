"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, stage by stage
and for the whole layer, on the five workloads and the edge cases.

Bars: activation codes, expert ids (unflagged tokens), the permutation and row
offsets bit-exact; outputs within max|err| <= 2e-2 * max|ref| + 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_gemv_gb300 import binding as B
from mixture_experts_layer_gemv_gb300.synth import (MoEConfig, WORKLOADS, make_router, make_tokens,
                                                    make_weights)

from _helpers import assert_out_close, effective_routing, host_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_layer_gemv_gb300 import build
    build.build()
    oracle.build()
    B.lib()


# ------------------------------------------------------------ quantisation
@pytest.mark.parametrize("T,H", [(1, 5120), (8, 512), (37, 7168), (300, 1024)])
def test_quant_act_codes_bit_exact(T, H):
    g = torch.Generator(device="cuda").manual_seed(T * 7 + H)
    x = (torch.randn((T, H), generator=g, device="cuda") *
         torch.exp(torch.randn((T, 1), generator=g, device="cuda") * 3)).to(torch.bfloat16)
    x[0, :128] = 0  # an all-zero block
    if H >= 384:
        x[0, 256:384] = 448.0  # a block sitting exactly on the scale boundary
    xq = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    xs = torch.empty((T, H // 128), dtype=torch.float32, device="cuda")
    B.moe_quant_act(x, xq, xs)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_rows(x.float().cpu().numpy().astype(np.float64))
    assert np.array_equal(xs.cpu().numpy().astype(np.float64), s_ref)
    assert np.array_equal(xq.cpu().numpy(), q_ref)


# ----------------------------------------------------------------- routing
ROUTE_CASES = ["tiny_t8", "dsv2_decode_t1", "dsv2_decode_t64", "prefill_t4096", "dsv2_zipf_t2048"]


@pytest.mark.parametrize("name", ROUTE_CASES)
def test_route_ids_bit_exact(name):
    wl = WORKLOADS[name]
    cfg = wl.cfg
    wr, bias = make_router(cfg, wl.seed, "cuda", zipf=wl.zipf_bias)
    x = make_tokens(cfg, wl.T, wl.seed, "cuda")
    ids = torch.empty((wl.T, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, cfg.top_k), dtype=torch.float32, device="cuda")
    ws = B.alloc_workspace(cfg, wl.T)
    B.moe_route(cfg, x, wr, bias, ids, w, ws)
    torch.cuda.synchronize()
    ids_o, w_o, p_o, margin = oracle.route(cfg, x.cpu(), wr.cpu(), None if bias is None else bias.cpu())
    ids_eff, w_eff, nflag = effective_routing(cfg, ids.cpu().numpy(), ids_o, p_o, margin)
    np.testing.assert_allclose(w.cpu().numpy(), w_eff, rtol=2e-5, atol=1e-7)
    assert B.moe_read_device_status(ws) == 0


# The large-T router on tcgen05 at expert counts that are not multiples of 16 (zero rows
# up to the MMA's N) or of 4 (the partial logits stored one float at a time), the largest
# count (256: 16 column chunks per epilogue thread), ragged token tiles and several K splits.
@pytest.mark.parametrize("E,G,Gk,k,T,H", [(18, 3, 2, 4, 65, 512), (36, 4, 2, 6, 600, 512),
                                          (20, 4, 4, 3, 300, 1024), (256, 8, 4, 8, 130, 512)])
def test_large_t_router_ids_bit_exact(E, G, Gk, k, T, H):
    cfg = MoEConfig(H, 256, E, G, Gk, k, 2.5, 1)
    wr, _ = make_router(cfg, 50 + E, "cuda")
    bias = (torch.arange(E, device="cuda", dtype=torch.float32) % 5) * 1e-3
    x = make_tokens(cfg, T, 51 + T, "cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = B.alloc_workspace(cfg, T)
    B.moe_route(cfg, x, wr, bias, ids, w, ws)
    torch.cuda.synchronize()
    ids_o, w_o, p_o, margin = oracle.route(cfg, x.cpu(), wr.cpu(), bias.cpu())
    ids_eff, w_eff, _ = effective_routing(cfg, ids.cpu().numpy(), ids_o, p_o, margin)
    np.testing.assert_allclose(w.cpu().numpy(), w_eff, rtol=2e-5, atol=1e-7)
    assert B.moe_read_device_status(ws) == 0


# ------------------------------------------------------------- permutation
@pytest.mark.parametrize("T,E,k", [(1, 160, 6), (37, 16, 4), (64, 160, 6), (4096, 64, 8), (2048, 160, 6),
                                   (5000, 256, 16)])
def test_permute_bit_exact(T, E, k):
    cfg = MoEConfig(128, 128, E, 1, 1, k, 1.0, 0)
    g = torch.Generator(device="cpu").manual_seed(T + E + k)
    # skewed ids: a few hot experts, each token's ids distinct
    scores = torch.rand((T, E), generator=g) * torch.linspace(1.0, 4.0, E)[torch.randperm(E, generator=g)]
    ids = scores.topk(k, dim=1).indices.to(torch.int32)
    ids_d = ids.cuda()
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    ps = torch.empty(T * k, dtype=torch.int32, device="cuda")
    ip = torch.empty(T * k, dtype=torch.int32, device="cuda")
    ws = B.alloc_workspace(cfg, T)
    B.moe_permute(cfg, ids_d, off, ps, ip, ws)
    torch.cuda.synchronize()
    o_ref, ps_ref, ip_ref = oracle.permute(cfg, ids.numpy())
    assert np.array_equal(off.cpu().numpy(), o_ref)
    assert np.array_equal(ps.cpu().numpy(), ps_ref)
    assert np.array_equal(ip.cpu().numpy(), ip_ref)


# --------------------------------------------------------- whole-layer parity
# Sampled tokens for the workloads the oracle cannot finish in seconds at full size:
# every parity case spans several weight tiles and a ragged token tail.
SAMPLES = {"tiny_t8": None, "dsv2_decode_t1": None, "dsv2_decode_t64": 24, "prefill_t4096": 12,
           "dsv2_zipf_t2048": 16}

_layers = {}


def _layer(name):
    if name not in _layers:
        _layers.clear()
        torch.cuda.empty_cache()
        wl = WORKLOADS[name]
        W = make_weights(wl.cfg, wl.seed, "cuda", zipf=wl.zipf_bias)
        x = make_tokens(wl.cfg, wl.T, wl.seed, "cuda")
        _layers[name] = (wl, W, x, host_weights(W))
    return _layers[name]


def _sample(T, n, seed):
    if n is None or n >= T:
        return np.arange(T, dtype=np.int32)
    rng = np.random.default_rng(seed)
    s = rng.choice(T, n, replace=False)
    s[:2] = [0, T - 1]
    return np.sort(s).astype(np.int32)


@pytest.mark.parametrize("name", list(SAMPLES))
def test_forward_matches_oracle(name):
    wl, W, x, Wc = _layer(name)
    cfg = wl.cfg
    out, ids = B.forward(cfg, x, W, return_ids=True)
    torch.cuda.synchronize()
    ids_o, w_o, p_o, margin = oracle.route(cfg, x.cpu(), Wc["w_router"], Wc["router_bias"])
    ids_eff, w_eff, _ = effective_routing(cfg, ids.cpu().numpy(), ids_o, p_o, margin)
    tokens = _sample(wl.T, SAMPLES[name], wl.seed)
    ref = oracle.forward_tokens(cfg, oracle.Weights(Wc), x.cpu(), ids_eff, w_eff, tokens)
    assert_out_close(out[torch.from_numpy(tokens).long().cuda()], ref, name)


@pytest.mark.parametrize("name", ["tiny_t8", "dsv2_decode_t64", "prefill_t4096"])
def test_stage_pipeline_with_oracle_routing(name):
    """moe_permute -> moe_expert_ffn -> moe_combine fed the oracle's routing, so an FFN
    error cannot hide behind a routing difference."""
    wl, W, x, Wc = _layer(name)
    cfg, T, k = wl.cfg, wl.T, wl.cfg.top_k
    ids_o, w_o, _, _ = oracle.route(cfg, x.cpu(), Wc["w_router"], Wc["router_bias"])
    ids = torch.from_numpy(ids_o).cuda()
    w = torch.from_numpy(w_o.astype(np.float32)).cuda()
    ws = B.alloc_workspace(cfg, T)
    off = torch.empty(cfg.n_routed + 1, dtype=torch.int32, device="cuda")
    ps = torch.empty(T * k, dtype=torch.int32, device="cuda")
    ip = torch.empty(T * k, dtype=torch.int32, device="cuda")
    B.moe_permute(cfg, ids, off, ps, ip, ws)
    y_perm = torch.empty((T * k, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    y_sh = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    B.moe_expert_ffn(cfg, x, W, off, ps, w, y_perm, y_sh, ws)
    res = make_tokens(cfg, T, wl.seed + 100, "cuda", name="residual")
    out = torch.empty_like(x)
    B.moe_combine(cfg, y_perm, ip, y_sh, res, out)
    torch.cuda.synchronize()
    tokens = _sample(T, SAMPLES[name], wl.seed + 1)
    OW = oracle.Weights(Wc)
    # per-row expert outputs
    inv = ip.cpu().numpy()
    for t in tokens[:4]:
        for j in range(k):
            y_ref, _ = oracle.expert_row(cfg, OW, x[t].cpu(), int(ids_o[t, j]), float(w_o[t, j]))
            assert_out_close(y_perm[inv[t * k + j]], y_ref, f"{name} row ({t},{j})")
        assert_out_close(y_sh[t], oracle.shared_row(cfg, OW, x[t].cpu()), f"{name} shared {t}")
    ref = oracle.forward_tokens(cfg, OW, x.cpu(), ids_o, w_o, tokens, residual_bf16=res.cpu())
    assert_out_close(out[torch.from_numpy(tokens).long().cuda()], ref, name)


def test_combine_sums_in_fp32_and_rounds_once():
    cfg = MoEConfig(256, 128, 8, 1, 1, 3, 1.0, 1)
    T, k, H = 5, 3, 256
    g = torch.Generator(device="cuda").manual_seed(3)
    y_perm = torch.randn((T * k, H), generator=g, device="cuda").to(torch.bfloat16)
    y_sh = torch.randn((T, H), generator=g, device="cuda").to(torch.bfloat16)
    inv = torch.randperm(T * k, device="cuda").to(torch.int32)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    B.moe_combine(cfg, y_perm, inv, y_sh, None, out)
    torch.cuda.synchronize()
    yp = y_perm.double().cpu().numpy()
    ref = yp[inv.cpu().numpy().astype(np.int64)].reshape(T, k, H).sum(1) + y_sh.double().cpu().numpy()
    ref_bf16 = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    got = out.double().cpu().numpy()
    # fp32 accumulation of 4 bf16 terms: within one bf16 rounding of the exact sum
    assert np.all(np.abs(got - ref) <= np.abs(ref_bf16 - ref) + 2.0 ** -8 * np.abs(ref) + 1e-30)


# --------------------------------------------------------------- edge cases
def _run_and_check(cfg, W, x, residual=None, tokens=None):
    out, ids = B.forward(cfg, x, W, residual=residual, return_ids=True)
    torch.cuda.synchronize()
    Wc = host_weights(W)
    ids_o, w_o, p_o, margin = oracle.route(cfg, x.cpu(), Wc["w_router"], Wc["router_bias"])
    ids_eff, w_eff, _ = effective_routing(cfg, ids.cpu().numpy(), ids_o, p_o, margin)
    T = x.shape[0]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else tokens
    ref = oracle.forward_tokens(cfg, oracle.Weights(Wc), x.cpu(), ids_eff, w_eff, tokens,
                                residual_bf16=None if residual is None else residual.cpu())
    assert_out_close(out[torch.from_numpy(tokens).long().cuda()], ref, str(cfg))
    return out, ids


def test_T_zero_is_a_noop():
    cfg = WORKLOADS["tiny_t8"].cfg
    W = make_weights(cfg, 0, "cuda")
    x = torch.empty((0, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((0, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    ws = B.alloc_workspace(cfg, 1)
    B.moe_forward(cfg, x, W, out, ws=ws)
    torch.cuda.synchronize()


@pytest.mark.parametrize("T", [1, 9, 63, 64, 65, 130])
def test_ragged_token_counts_across_the_small_large_boundary(T):
    cfg = MoEConfig(384, 256, 12, 3, 2, 3, 1.5, 1)
    W = make_weights(cfg, 21, "cuda")
    x = make_tokens(cfg, T, 21 + T, "cuda")
    _run_and_check(cfg, W, x)


@pytest.mark.parametrize("G,Gk,k", [(1, 1, 1), (4, 4, 2), (1, 1, 8), (8, 1, 1)])
def test_group_and_topk_degenerate_cases(G, Gk, k):
    cfg = MoEConfig(256, 128, 16, G, Gk, k, 2.0, 0)
    W = make_weights(cfg, 30 + G * 10 + k, "cuda")
    x = make_tokens(cfg, 70, 31, "cuda")
    _run_and_check(cfg, W, x)


@pytest.mark.parametrize("T", [5, 200, 300])
def test_one_expert_receives_every_token(T):
    cfg = MoEConfig(256, 256, 8, 2, 1, 2, 1.0, 1)
    W = make_weights(cfg, 40, "cuda")
    bias = torch.zeros(8, device="cuda")
    bias[5] = 30.0  # expert 5 dominates every token; more than 8 rows per expert
    W["router_bias"] = bias
    x = make_tokens(cfg, T, 41, "cuda")
    out, ids = _run_and_check(cfg, W, x)
    assert (ids[:, 0] == 5).all()


def test_zero_routing_weight_leaves_only_shared_and_residual():
    cfg = MoEConfig(256, 128, 8, 2, 1, 2, 0.0, 1)
    W = make_weights(cfg, 50, "cuda")
    x = make_tokens(cfg, 6, 51, "cuda")
    res = make_tokens(cfg, 6, 52, "cuda", name="residual")
    out, _ = _run_and_check(cfg, W, x, residual=res)
    cfg0 = MoEConfig(256, 128, 8, 2, 1, 2, 0.0, 1)
    Wc = host_weights(W)
    OW = oracle.Weights(Wc)
    for t in range(6):
        ref = oracle.shared_row(cfg0, OW, x[t].cpu()) + res[t].double().cpu().numpy()
        assert_out_close(out[t], ref, "shared + residual")


def test_no_shared_experts():
    cfg = MoEConfig(512, 256, 16, 4, 2, 4, 1.0, 0)
    W = make_weights(cfg, 60, "cuda")
    x = make_tokens(cfg, 20, 61, "cuda")
    _run_and_check(cfg, W, x)


def test_repeated_calls_are_deterministic_and_status_clean():
    wl, W, x, _ = _layer("tiny_t8")
    ws = B.alloc_workspace(wl.cfg, wl.T)
    outs = []
    for _ in range(3):
        out = torch.empty_like(x)
        B.moe_forward(wl.cfg, x, W, out, ws=ws)
        outs.append(out)
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    assert B.moe_read_device_status(ws) == 0


@pytest.mark.parametrize("name", ["dsv2_decode_t1", "dsv2_decode_t64"])
def test_repeated_forwards_bit_identical_over_dirty_workspaces(name):
    # every call gets a fresh workspace laid over memory just filled with random bytes:
    # a partial-sum buffer read before the kernels wrote it, or a race between the
    # streaming kernels, shows up as a difference between two calls on the same input
    wl, W, x, _ = _layer(name)
    n = B.moe_workspace_size(wl.cfg, wl.T)
    gen = torch.Generator(device="cuda").manual_seed(7)
    ref = None
    for i in range(12):
        junk = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=gen)
        del junk
        ws = B.alloc_workspace(wl.cfg, wl.T)
        out = torch.empty_like(x)
        B.moe_forward(wl.cfg, x, W, out, ws=ws)
        torch.cuda.synchronize()
        assert B.moe_read_device_status(ws) == 0
        if ref is None:
            ref = out.clone()
        else:
            assert torch.equal(ref, out), f"call {i} differs from call 0"


def test_invalid_expert_id_is_reported_not_faulted():
    cfg = MoEConfig(128, 128, 8, 1, 1, 2, 1.0, 0)
    ids = torch.tensor([[0, 1], [9, 2]], dtype=torch.int32, device="cuda")  # 9 >= E
    off = torch.empty(9, dtype=torch.int32, device="cuda")
    ps = torch.empty(4, dtype=torch.int32, device="cuda")
    ip = torch.empty(4, dtype=torch.int32, device="cuda")
    ws = B.alloc_workspace(cfg, 2)
    B.moe_permute(cfg, ids, off, ps, ip, ws)
    assert B.moe_read_device_status(ws) == -1  # MOE_ERR_INVALID_ARG
    assert B.moe_read_device_status(ws) == 0   # cleared by the read


@pytest.mark.parametrize("T", [9, 16, 24])
def test_second_shared_row_group_on_the_dsv2_layer(T):
    # several 8-token groups of the shared experts: every CTA, wherever its range
    # starts, must build the operand of the group it begins in
    wl, W, x64, Wc = _layer("dsv2_decode_t64")
    x = x64[:T].contiguous()
    out, ids = B.forward(wl.cfg, x, W, return_ids=True)
    torch.cuda.synchronize()
    ids_o, w_o, p_o, margin = oracle.route(wl.cfg, x.cpu(), Wc["w_router"], Wc["router_bias"])
    ids_eff, w_eff, _ = effective_routing(wl.cfg, ids.cpu().numpy(), ids_o, p_o, margin)
    tokens = np.array([0, 7, 8, T - 1], dtype=np.int32)
    ref = oracle.forward_tokens(wl.cfg, oracle.Weights(Wc), x.cpu(), ids_eff, w_eff, tokens)
    assert_out_close(out[torch.from_numpy(tokens).long().cuda()], ref, f"T={T}")
    assert torch.isfinite(out.float()).all()


# ------------------------------------- grouped tensor-core GEMM path (T > 64 tokens)
GEMM_CFG = MoEConfig(512, 256, 16, 4, 2, 4, 1.0, 2)


@pytest.mark.parametrize("T", [65, 129, 257, 600])
def test_grouped_gemm_path_every_token(T):
    # 128-row token tiles: several per expert, ragged last tiles, and a shared-expert
    # tile with a single row at T = 129 and T = 257
    W = make_weights(GEMM_CFG, 70, "cuda")
    x = make_tokens(GEMM_CFG, T, 71 + T, "cuda")
    res = make_tokens(GEMM_CFG, T, 72, "cuda", name="residual")
    _run_and_check(GEMM_CFG, W, x, residual=res)


def test_grouped_gemm_expert_segments_on_tile_boundaries():
    """moe_permute -> moe_expert_ffn with hand-made ids: expert segments of exactly 128,
    256, 1 and 0 rows, so tiles start and end on every kind of boundary; every
    permuted row is checked against the oracle's expert row."""
    cfg = MoEConfig(512, 256, 16, 4, 2, 4, 1.0, 1)
    T, k = 160, 4
    t = np.arange(T)
    ids = np.stack([np.where(t < 128, 0, 3),                 # expert 0: 128 rows
                    np.full(T, 1),                           # expert 1: 160 + 96 = 256 rows
                    np.where(t < 64, 2, 1),                  # expert 2: 64 rows
                    np.where(t == 5, 4, 5 + t % 11)], 1)     # expert 4: 1 row; experts 5..15
    assert (np.bincount(ids.ravel(), minlength=16)[[0, 1, 4]] == [128, 256, 1]).all()
    rng = np.random.default_rng(80)
    w = rng.uniform(0.1, 2.0, (T, k))
    W = make_weights(cfg, 81, "cuda")
    x = make_tokens(cfg, T, 82, "cuda")
    ws = B.alloc_workspace(cfg, T)
    ids_d = torch.from_numpy(ids.astype(np.int32)).cuda()
    w_d = torch.from_numpy(w.astype(np.float32)).cuda()
    off = torch.empty(cfg.n_routed + 1, dtype=torch.int32, device="cuda")
    ps = torch.empty(T * k, dtype=torch.int32, device="cuda")
    ip = torch.empty(T * k, dtype=torch.int32, device="cuda")
    B.moe_permute(cfg, ids_d, off, ps, ip, ws)
    y_perm = torch.empty((T * k, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    y_sh = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    B.moe_expert_ffn(cfg, x, W, off, ps, w_d.float(), y_perm, y_sh, ws)
    torch.cuda.synchronize()
    assert B.moe_read_device_status(ws) == 0
    OW = oracle.Weights(host_weights(W))
    xc = x.cpu()
    inv = ip.cpu().numpy()
    for tok in range(T):
        for j in range(k):
            y_ref, _ = oracle.expert_row(cfg, OW, xc[tok], int(ids[tok, j]), float(w[tok, j]))
            assert_out_close(y_perm[inv[tok * k + j]], y_ref, f"row ({tok},{j}) expert {ids[tok, j]}")
        assert_out_close(y_sh[tok], oracle.shared_row(cfg, OW, xc[tok]), f"shared {tok}")


@pytest.mark.parametrize("name", ["dsv2_decode_t1", "dsv2_decode_t64", "tiny_t8"])
def test_back_to_back_forwards_on_one_workspace(name):
    # 60 forwards enqueued back to back on one workspace, no synchronisation between them,
    # alternating two inputs whose routings differ, so that a kernel reading the previous
    # call's routing data (a stale work list, permutation or weight) would change its
    # output: every call must equal the same input's result computed alone
    wl, W, x, _ = _layer(name)
    xb = make_tokens(wl.cfg, wl.T, wl.seed + 77, "cuda", name="x_other")
    ws = B.alloc_workspace(wl.cfg, wl.T)
    refs = []
    for xi in (x, xb):
        o = torch.empty_like(xi)
        B.moe_forward(wl.cfg, xi, W, o, ws=ws)
        torch.cuda.synchronize()
        refs.append(o)
    assert not torch.equal(refs[0], refs[1])
    outs = [torch.empty_like(x) for _ in range(60)]
    for i, o in enumerate(outs):
        B.moe_forward(wl.cfg, x if i % 2 == 0 else xb, W, o, ws=ws)
    torch.cuda.synchronize()
    assert B.moe_read_device_status(ws) == 0
    bad = [i for i, o in enumerate(outs) if not torch.equal(o, refs[i % 2])]
    assert not bad, f"calls {bad[:10]} differ from their input's result"
