"""Shared parity helpers for the GPU tests (the CUDA path against the oracle)."""
import numpy as np
import torch

# Near-tie threshold in softmax-probability units: tokens whose oracle routing margin
# is below it are flagged, and a different (equally valid) selection is accepted.
FLAG_MARGIN = 1e-5


def out_tolerance(ref: np.ndarray) -> float:
    """Output bar: max |out - ref| <= 2e-2 * max |ref| + 1e-3 (bf16 output)."""
    return 2e-2 * float(np.abs(ref).max()) + 1e-3


def assert_out_close(out, ref, what=""):
    o = out.float().cpu().numpy() if hasattr(out, "cpu") else np.asarray(out, np.float64)
    err = float(np.abs(o - ref).max())
    tol = out_tolerance(ref)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    assert err <= tol, f"{what}: max|err| {err:.4e} > tol {tol:.4e} (max|ref| {np.abs(ref).max():.4e})"
    return err, tol


def effective_routing(cfg, ids_gpu, ids_ref, probs_ref, margin):
    """Check the GPU routing against the oracle and return the (ids, w) to score outputs with.

    Unflagged tokens must match bit-exactly (ids and order). A flagged token may differ
    only among near-tied candidates: the oracle's probabilities of the GPU's choices must
    equal its own choices' to within FLAG_MARGIN, position by position.
    """
    ids_gpu = np.asarray(ids_gpu)
    same = (ids_gpu == ids_ref).all(axis=1)
    flagged = margin < FLAG_MARGIN
    bad = ~same & ~flagged
    assert not bad.any(), f"routing mismatch on unflagged tokens {np.where(bad)[0][:10].tolist()}"
    ids_eff = ids_ref.copy()
    for t in np.where(~same)[0]:
        pg = probs_ref[t, ids_gpu[t]]
        po = probs_ref[t, ids_ref[t]]
        assert np.all(np.abs(pg - po) < FLAG_MARGIN), f"token {t}: GPU choice not a near-tie"
        assert len(set(ids_gpu[t].tolist())) == cfg.top_k
        ids_eff[t] = ids_gpu[t]
    w_eff = np.take_along_axis(probs_ref, ids_eff.astype(np.int64), axis=1) * cfg.routed_scaling_factor
    return ids_eff, w_eff, int(flagged.sum())


def host_weights(W):
    return {k: (None if v is None else v.detach().cpu()) for k, v in W.items()}


def bf16_np(x: torch.Tensor) -> np.ndarray:
    return x.detach().float().cpu().numpy().astype(np.float64)
