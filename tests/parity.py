"""Comparison rules between the CUDA path and the fp64 oracle (test helpers).

Floating outputs: max |gpu - oracle| <= 2e-2 and mean |gpu - oracle| <= 2e-3
(bf16 operands, fp32 accumulation).  Top-k sets: identical, except that a
boundary near-tie may swap: with s_k the oracle's k-th score and
tau = 1e-6 * max(|s_k|, s_top1 if s_k == 0), every index the GPU chose that
the oracle did not must score >= s_k - tau, and every index the oracle chose
that the GPU did not must score <= s_k + tau (scores are the oracle's fp64
values).  Index lists are compared as sets; padding (-1) must match and
trail, and the real entries must be in ascending index order (the order the
library documents for its index lists).  A row whose set differs from the
oracle's by an accepted near-tie is still checked in full: its float outputs
are compared with the oracle's attention over the GPU's own index set
(``decoupled``), so every row's attention is verified.
"""
import numpy as np
import torch

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """Host uint16 bit patterns of a bf16 tensor."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t):
    """numpy view of an input tensor for the oracle (bf16 -> uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return bits(t)
    return t.detach().cpu().numpy()


def assert_close(gpu, ref, what="", max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    d = np.abs(g - r)
    assert np.all(np.isfinite(d)), f"{what}: non-finite difference"
    assert d.max() <= max_abs, f"{what}: max abs diff {d.max():.3e} > {max_abs}"
    assert d.mean() <= mean_abs, f"{what}: mean abs diff {d.mean():.3e} > {mean_abs}"
    return float(d.max()), float(d.mean())


def assert_lse_close(gpu, ref, what="", tol=1e-3):
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    ninf_g, ninf_r = np.isneginf(g), np.isneginf(r)
    assert np.array_equal(ninf_g, ninf_r), f"{what}: empty-branch pattern differs"
    if (~ninf_r).any():
        d = np.abs(g[~ninf_r] - r[~ninf_r])
        assert d.max() <= tol, f"{what}: lse max diff {d.max():.3e}"


def topk_set_ok(gpu_idx, oracle_idx, scores, kth, k):
    """Check one row's index set against the oracle under the near-tie rule.

    Returns (ok, exact) where exact says the sets are identical.
    """
    g = np.asarray(gpu_idx)
    o = np.asarray(oracle_idx)
    gs, os_ = set(g[g >= 0].tolist()), set(o[o >= 0].tolist())
    if len(gs) != (g >= 0).sum():
        return False, False                      # duplicates
    if (g >= 0).sum() != (o >= 0).sum():
        return False, False
    # padding must trail the real entries, which come in ascending index order
    if np.any(g[(g >= 0).sum():] != -1):
        return False, False
    if np.any(np.diff(g[: (g >= 0).sum()]) <= 0):
        return False, False
    if gs == os_:
        return True, True
    if not np.isfinite(kth):
        return False, False                      # fewer than k visible: all must be taken
    top1 = float(np.max(scores)) if len(scores) else 0.0
    tau = 1e-6 * max(abs(kth), top1 if kth == 0 else 0.0)
    for j in gs - os_:
        if not (j < len(scores) and scores[j] >= kth - tau):
            return False, False
    for j in os_ - gs:
        if not scores[j] <= kth + tau:
            return False, False
    return True, False


def check_topk_rows(gpu_idx_rows, oracle_rows, k, what=""):
    """oracle_rows: list of dicts with idx, scores, kth.  Returns number of near-tie rows."""
    near = 0
    for r, (g, o) in enumerate(zip(gpu_idx_rows, oracle_rows)):
        ok, exact = topk_set_ok(g, o["idx"], o["scores"], o["kth"], k)
        assert ok, f"{what}: row {r} top-k set differs: gpu-only {sorted(set(g) - set(o['idx']))[:8]} " \
                   f"oracle-only {sorted(set(o['idx']) - set(g))[:8]}"
        near += not exact
    return near


def selected(gpu_idx):
    """The GPU's selected entries of one row (padding dropped)."""
    g = np.asarray(gpu_idx)
    return g[g >= 0]


def decoupled(q_t, Kc_sel, Vc_sel, swa=None, scale=1.0):
    """Oracle attention over the entries the GPU selected (fp64), merged with a
    window branch dict (O, lse) when given.  Returns (O, lse) of the branch and,
    with a window, (O, lse) of the layer."""
    import oracle
    O, L = oracle.attend(q_t, Kc_sel, Vc_sel, scale)
    if swa is None:
        return O, L
    return (O, L), oracle.merge([O, swa["O"]], [L, swa["lse"]])
