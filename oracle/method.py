"""Steps of the hybrid compressed-attention path, in float64 (test infrastructure).

Each function is the plain definition of one step; none is blocked, fused or
reordered.  Citation keys are defined in oracle/__init__.py.
"""
import numpy as np

from .formats import nvfp4_decode, nvfp4_quantize, round_bf16


# ---------------------------------------------------------------------------
# compression (CSA m=4, HCA m=128)
# ---------------------------------------------------------------------------
def pool_weights(g) -> np.ndarray:
    """Softmax of the m gate logits of one block.

    [HYBRID]: CSA merges 4 consecutive tokens into one KV entry by
    softmax-weighted pooling; [VIDEO] "Explained simply": the contribution of
    each token is learned, not a plain mean; HCA merges 128 tokens the same
    way.  Reading R1: one logit per token.
    """
    g = np.asarray(g, dtype=np.float64)
    e = np.exp(g - g.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def pool_exact(K, V, gate, m):
    """Unrounded pooled entries: Kc_j = sum_i a_i K_i, Vc_j = sum_i a_i V_i.

    K, V: [T, D] float64; gate: [T].  Block j covers tokens j*m .. j*m+m-1;
    a trailing T mod m tokens form no entry (they stay raw for the window).
    """
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    T, D = K.shape
    n = T // m
    a = pool_weights(np.asarray(gate, np.float64)[: n * m].reshape(n, m))
    Kc = np.einsum("jm,jmd->jd", a, K[: n * m].reshape(n, m, D))
    Vc = np.einsum("jm,jmd->jd", a, V[: n * m].reshape(n, m, D))
    return Kc, Vc


def pool(K, V, gate, m):
    """Pooled entries as stored: pool_exact rounded to bf16 (reading R1)."""
    Kc, Vc = pool_exact(K, V, gate, m)
    return round_bf16(Kc), round_bf16(Vc)


# ---------------------------------------------------------------------------
# visibility
# ---------------------------------------------------------------------------
def visible_count(t, m, n_valid=None) -> int:
    """Number of compressed entries the query at absolute position t may see.

    Reading R2: entry j is visible iff j*m + m - 1 <= t (its block is
    complete at t), i.e. j < floor((t+1)/m); capped by the entries present.
    """
    v = (int(t) + 1) // int(m)
    return v if n_valid is None else min(v, int(n_valid))


# ---------------------------------------------------------------------------
# lightning indexer + top-k (CSA only)
# ---------------------------------------------------------------------------
def index_scores(qI, w, kI) -> np.ndarray:
    """Indexer score of every given entry for one query.

    [HYBRID]: a light "lightning indexer" scores the compressed entries
    against the query and keeps the top-k; [THREAD] "Top comments": the
    indexer picks the candidates that matter before full attention runs.
    Reading R3: s_j = sum_h w_h * max(0, q_I[h] . k_I[j]).
    qI: [HI, DI], w: [HI], kI: [n, DI] -> s: [n].
    """
    dots = np.asarray(kI, np.float64) @ np.asarray(qI, np.float64).T   # [n, HI]
    return np.maximum(dots, 0.0) @ np.asarray(w, np.float64)


def index_scores_fp4(qI, w, kI_packed, kI_scale) -> np.ndarray:
    """Indexer score with the indexer in FP4.

    [HYBRID]: the lightning indexer computes in FP4; [V41]: the keys it reads are
    kept in FP4.  Reading R16: the query is quantised to NVFP4 (per (head)
    row, groups of 16, nvfp4_quantize) and the keys are NVFP4 (R7); the score
    is R3's on the decoded values.
    qI: [HI, DI] (bf16 values), w: [HI], kI_packed: [n, DI/2], kI_scale: [n, DI/16].
    """
    q = nvfp4_decode(*nvfp4_quantize(qI))
    return index_scores(q, w, nvfp4_decode(kI_packed, kI_scale))


def topk_select(s, k):
    """Indices of the k best scores, as an ascending set padded with -1.

    [HYBRID]: keeps the top-k (typically about 128) entries.  Reading R4:
    order by (score desc, index asc); min(k, n) are kept.
    Returns (idx int64 [k], kth score or -inf when fewer than k exist).
    """
    s = np.asarray(s, np.float64)
    n = s.shape[0]
    order = np.lexsort((np.arange(n), -s))      # primary -s, then index
    keep = order[: min(k, n)]
    out = np.full(k, -1, dtype=np.int64)
    out[: keep.size] = np.sort(keep)
    kth = s[keep[-1]] if keep.size == k else -np.inf
    return out, kth


# ---------------------------------------------------------------------------
# attention over a key set (MQA: all heads share K and V)
# ---------------------------------------------------------------------------
def attend(q, K, V, scale=1.0):
    """Softmax attention of H query heads over n shared key/value rows.

    [HYBRID]: both mechanisms use multi-query attention with shared KV
    projections.  z = scale * q K^T; lse = log sum exp z; O = softmax(z) V.
    Reading R6: with no keys, lse = -inf and O = 0.
    q: [H, D]; K, V: [n, D] -> (O [H, D], lse [H]).
    """
    q = np.asarray(q, np.float64)
    H, D = q.shape
    if len(K) == 0:
        return np.zeros((H, np.asarray(V).shape[-1] if np.ndim(V) == 2 else D)), np.full(H, -np.inf)
    z = scale * (q @ np.asarray(K, np.float64).T)          # [H, n]
    zmax = z.max(axis=1, keepdims=True)
    e = np.exp(z - zmax)
    ssum = e.sum(axis=1, keepdims=True)
    O = (e @ np.asarray(V, np.float64)) / ssum
    lse = (zmax + np.log(ssum))[:, 0]
    return O, lse


def window_positions(t, W, raw_pos0=0, raw_len=None) -> np.ndarray:
    """Absolute positions of the sliding-window keys of the query at t.

    [HYBRID]: a sliding-window branch over recent tokens runs in parallel;
    [VIDEO] "Explained simply": it covers the most recent 128 tokens.
    Reading R5: positions max(0, t-W+1) .. t that the raw buffer holds.
    """
    lo = max(0, int(t) - int(W) + 1, int(raw_pos0))
    hi = int(t)
    if raw_len is not None:
        hi = min(hi, int(raw_pos0) + int(raw_len) - 1)
    return np.arange(lo, hi + 1, dtype=np.int64) if hi >= lo else np.zeros(0, np.int64)


def merge(Os, lses):
    """Combine branch outputs by log-sum-exp (reading R6).

    L = log sum_b exp(lse_b); O = sum_b exp(lse_b - L) O_b.  Equal to one
    softmax over the concatenated key lists of the branches ([HYBRID]: the
    window branch runs in parallel; "three views" at a layer).
    Os: list of [H, D]; lses: list of [H] -> (O [H, D], L [H]).
    """
    L = np.stack([np.asarray(l, np.float64) for l in lses])          # [nb, H]
    Lmax = L.max(axis=0)
    finite = np.isfinite(Lmax)
    safe = np.where(finite, Lmax, 0.0)
    wts = np.where(np.isfinite(L), np.exp(L - safe[None, :]), 0.0)   # [nb, H]
    tot = wts.sum(axis=0)
    Lout = np.where(finite, safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    O = sum(wts[b][:, None] * np.asarray(Os[b], np.float64) for b in range(len(Os)))
    O = np.where(finite[:, None], O / np.where(tot > 0, tot, 1.0)[:, None], 0.0)
    return O, Lout


# ---------------------------------------------------------------------------
# query / KV prologue: RMS normalisation and partial rotary embedding
# ---------------------------------------------------------------------------
def rms_norm(x, gamma, eps):
    """RMS normalisation of each row: x / sqrt(mean(x^2) + eps) * gamma.

    [HYBRID]: both mechanisms apply query and KV normalisation.  Reading R11:
    RMSNorm over the head dimension of every query head and of the shared K
    and V rows, each tensor with its own per-channel gain.
    x: [..., D]; gamma: [D].
    """
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + float(eps)) * np.asarray(gamma, np.float64)


def rope_partial(x, pos, d_rope, base=10000.0):
    """Rotary position embedding on the last d_rope channels of each row.

    [HYBRID]: both mechanisms use partial RoPE.  Reading R11: channels
    D-d_rope .. D-1 form d_rope/2 pairs (c, c + d_rope/2) (the "rotate half"
    pairing); pair i is rotated by the angle pos * base^(-2i/d_rope); the
    first D-d_rope channels are left as they are.
    x: [..., D] (rows of one position pos).
    """
    x = np.array(x, np.float64)
    D = x.shape[-1]
    h = d_rope // 2
    i = np.arange(h, dtype=np.float64)
    ang = float(pos) * np.power(float(base), -2.0 * i / d_rope)
    c, s = np.cos(ang), np.sin(ang)
    x1 = x[..., D - d_rope:D - h].copy()
    x2 = x[..., D - h:].copy()
    x[..., D - d_rope:D - h] = x1 * c - x2 * s
    x[..., D - h:] = x2 * c + x1 * s
    return x


def qkv_prologue(q, k, v, pos, gq, gk, gv, eps, d_rope, base=10000.0):
    """The prologue of the path for one position: q heads and k normalised then
    rotated, v normalised only (RoPE encodes positions in scores, not values).
    q: [H, D], k, v: [D] -> (q, k, v) in float64 (unrounded)."""
    qn = rope_partial(rms_norm(q, gq, eps), pos, d_rope, base)
    kn = rope_partial(rms_norm(k, gk, eps), pos, d_rope, base)
    vn = rms_norm(v, gv, eps)
    return qn, kn, vn
