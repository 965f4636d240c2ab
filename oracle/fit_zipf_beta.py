"""Fit the Zipf strength of the load-imbalanced workload with the oracle's routing.

The DeepSeek-V2-shaped layer at T=2048 gets a per-expert router bias
-beta * 1.1 * ln(rank_e) (rank_e a seeded permutation of 1..160), so that expert
popularity follows Zipf(1.1) with the top 16 experts taking about 60% of the
assignments. Routing through the group limit distorts the shares, so beta is fitted
by bisection on a separate calibration batch (seeded, name "x_calib"), using only
the oracle's router and top-k. The printed value is the ZIPF_BETA constant of the
synthetic-input module.

    python oracle/fit_zipf_beta.py
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
from mixture_experts_layer_gemv_gb300.synth import WORKLOADS, make_router, make_tokens, zipf_bias  # noqa: E402

TARGET = 0.60


def top16_share(cfg, logits, beta, seed):
    b = zipf_bias(cfg, seed, "cpu", beta).numpy().astype(np.float64)
    ids, _, _, _ = oracle.topk(cfg, logits + b[None, :])
    counts = np.bincount(ids.ravel(), minlength=cfg.n_routed)
    return np.sort(counts)[::-1][:16].sum() / counts.sum()


def fit(T=2048):
    wl = WORKLOADS["dsv2_zipf_t2048"]
    cfg = wl.cfg
    wr, _ = make_router(cfg, wl.seed, "cpu", zipf=False)
    x = make_tokens(cfg, T, wl.seed, "cpu", name="x_calib")
    logits = oracle.router_logits(cfg, x, wr)
    lo, hi = 0.0, 4.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        if top16_share(cfg, logits, mid, wl.seed) < TARGET:
            lo = mid
        else:
            hi = mid
    beta = round(0.5 * (lo + hi), 4)
    return beta, top16_share(cfg, logits, beta, wl.seed)


if __name__ == "__main__":
    beta, share = fit()
    print(f"ZIPF_BETA = {beta}  (top-16 share {share:.4f})")
