"""Pins of the oracle's router, group-limited top-k and permutation.

Stage N (router GEMV) and stage O (softmax, group-limited greedy top-k,
w = score x routed_scaling_factor) of the MoE subgraph on "DSV2-236B-MegaKernel"
(README, stage flowchart; per-stage table rows "M+N" and "O"). Pinned by
brute-force enumeration on tiny inputs, reductions to library routines
(numpy/scipy fp64) and the invariants the pages state (top-3 of 8 groups,
exactly top_k distinct ids, w = p x 16.0).
"""
import itertools

import numpy as np
import pytest
import scipy.special
import torch

from mixture_experts_layer_gemv_gb300.synth import MoEConfig, WORKLOADS, make_weights, make_tokens


def _bf16_bits(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_vals(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


# ------------------------------------------------------------------- router
def test_router_unit_vector_selects_a_column(orc):
    cfg = MoEConfig(256, 128, 16, 4, 2, 4, 1.0, 0)
    rng = np.random.default_rng(0)
    wr = rng.normal(0, 0.02, (16, 256)).astype(np.float32)
    x = np.zeros((3, 256), np.float32)
    for t, i in enumerate([0, 17, 255]):
        x[t, i] = 1.0
    lg = orc.router_logits(cfg, _bf16_bits(x), wr)
    for t, i in enumerate([0, 17, 255]):
        assert np.array_equal(lg[t], wr[:, i].astype(np.float64))


def test_router_matches_fp64_matmul_with_bias(orc):
    cfg = MoEConfig(512, 128, 32, 4, 2, 3, 1.0, 0)
    rng = np.random.default_rng(1)
    wr = rng.normal(0, 0.02, (32, 512)).astype(np.float32)
    b = rng.normal(0, 1, 32).astype(np.float32)
    xb = _bf16_bits(rng.normal(0, 1, (5, 512)))
    lg = orc.router_logits(cfg, xb, wr, b)
    ref = _bf16_vals(xb) @ wr.astype(np.float64).T + b.astype(np.float64)
    np.testing.assert_allclose(lg, ref, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------- top-k
def _brute_force(p, G, Gk, k):
    """Max-sum group subset, then max-sum expert subset (distinct values => unique)."""
    E = len(p)
    per = E // G
    gs = np.array([p[g * per:(g + 1) * per].max() for g in range(G)])
    best_groups = max(itertools.combinations(range(G), Gk), key=lambda S: sum(gs[list(S)]))
    cand = [e for g in best_groups for e in range(g * per, (g + 1) * per)]
    best = max(itertools.combinations(cand, k), key=lambda S: sum(p[list(S)]))
    return set(best), set(best_groups)


@pytest.mark.parametrize("E,G,Gk,k", [(16, 4, 2, 4), (8, 4, 2, 2), (12, 3, 1, 3), (16, 8, 3, 5),
                                       (16, 4, 4, 6), (9, 1, 1, 4), (16, 4, 1, 1), (10, 5, 3, 6)])
def test_topk_equals_brute_force(orc, E, G, Gk, k):
    cfg = MoEConfig(128, 128, E, G, Gk, k, 2.5, 0)
    rng = np.random.default_rng(E * 100 + G * 10 + k)
    logits = rng.normal(0, 1.5, (40, E))
    ids, w, p, margin = orc.topk(cfg, logits)
    p_ref = scipy.special.softmax(logits, axis=1)
    np.testing.assert_allclose(p, p_ref, rtol=1e-13, atol=0)
    for t in range(40):
        sel, groups = _brute_force(p_ref[t], G, Gk, k)
        assert set(ids[t].tolist()) == sel
        assert len(set(ids[t].tolist())) == k
        assert all((e // (E // G)) in groups for e in ids[t])
        # listed by score descending
        assert np.all(np.diff(p_ref[t, ids[t]]) <= 0)
        np.testing.assert_allclose(w[t], p_ref[t, ids[t]] * 2.5, rtol=1e-13)
        assert margin[t] > 0


def test_topk_plain_when_one_group_or_all_groups_kept(orc):
    rng = np.random.default_rng(5)
    logits = rng.normal(0, 2, (64, 24))
    p_ref = scipy.special.softmax(logits, axis=1)
    plain = np.argsort(-p_ref, axis=1, kind="stable")[:, :5]
    for G, Gk in [(1, 1), (6, 6), (4, 4)]:
        cfg = MoEConfig(128, 128, 24, G, Gk, 5, 1.0, 0)
        ids, w, _, _ = orc.topk(cfg, logits)
        assert np.array_equal(ids, plain)
        t = torch.topk(torch.from_numpy(p_ref), 5, dim=1)
        np.testing.assert_allclose(w, t.values.numpy(), rtol=1e-13)


def test_topk_ties_go_to_lower_index(orc):
    cfg = MoEConfig(128, 128, 8, 4, 2, 3, 1.0, 0)
    logits = np.zeros((1, 8))  # every expert and group ties
    ids, w, _, margin = orc.topk(cfg, logits)
    assert ids[0].tolist() == [0, 1, 2]   # groups 0 and 1 kept, lowest experts first
    assert margin[0] == 0.0
    # groups {0,1} {2,3} {4,5} tie at the top: the two lower groups are kept, then
    # experts 1 and 2 lead and the tie among 0 and 3 goes to 0
    logits = np.array([[0.0, 1.0, 1.0, 0.0, 1.0, 0.0, 0.0, 0.0]])
    ids, _, _, _ = orc.topk(cfg, logits)
    assert ids[0].tolist() == [1, 2, 0]


def test_dsv2_selected_experts_lie_in_top3_of_8_groups(orc):
    wl = WORKLOADS["dsv2_decode_t64"]
    cfg = wl.cfg
    W = make_weights(MoEConfig(cfg.hidden, 128, cfg.n_routed, cfg.n_group, cfg.topk_group, cfg.top_k,
                               cfg.routed_scaling_factor, 0), wl.seed)  # router only matters here
    x = make_tokens(cfg, 64, wl.seed)
    ids, w, p, margin = orc.route(cfg, x, W["w_router"])
    per = cfg.n_routed // cfg.n_group
    for t in range(64):
        gs = p[t].reshape(cfg.n_group, per).max(1)
        top3 = set(np.argsort(-gs, kind="stable")[:3].tolist())
        assert {e // per for e in ids[t]} <= top3
        assert len(set(ids[t].tolist())) == 6
        np.testing.assert_allclose(w[t], p[t, ids[t]] * 16.0, rtol=1e-14)
    # near-uniform routing: most experts are touched once or a few times
    assert len(np.unique(ids)) > 120


# -------------------------------------------------------------- permutation
@pytest.mark.parametrize("T,E,k", [(1, 16, 4), (8, 16, 4), (37, 20, 6), (300, 64, 8), (0, 8, 2)])
def test_permute_is_stable_sort_by_expert(orc, T, E, k):
    cfg = MoEConfig(128, 128, E, 1, 1, k, 1.0, 0)
    rng = np.random.default_rng(T + E)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32) if T else \
        np.zeros((0, k), np.int32)
    off, perm_src, inv_pos = orc.permute(cfg, ids)
    flat = ids.reshape(-1)
    assert np.array_equal(perm_src, np.argsort(flat, kind="stable"))
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    assert off[-1] == T * k
    assert np.array_equal(inv_pos[perm_src], np.arange(T * k))
    for e in range(E):
        assert np.all(flat[perm_src[off[e]:off[e + 1]]] == e)


def test_zipf_workload_top16_share_is_about_sixty_percent(orc):
    # load-imbalance workload: the top 16 of 160 experts take ~60% of assignments
    from mixture_experts_layer_gemv_gb300.synth import make_router
    wl = WORKLOADS["dsv2_zipf_t2048"]
    wr, bias = make_router(wl.cfg, wl.seed, zipf=True)
    x = make_tokens(wl.cfg, wl.T, wl.seed)
    ids, _, _, _ = orc.route(wl.cfg, x, wr, bias)
    counts = np.bincount(ids.ravel(), minlength=wl.cfg.n_routed)
    share = np.sort(counts)[::-1][:16].sum() / counts.sum()
    assert 0.57 <= share <= 0.63, share
