"""Layer-level compositions of the oracle steps, per query (test infrastructure).

Inputs are numpy arrays: bf16 tensors as uint16 bit patterns, fp32 as float32,
NVFP4 as uint8.  Layouts follow the workload recipes: raw K/V [R, D] (row r is
position raw_pos0 + r), compressed K/V [N, D], queries [H, D] per position.

Layers ([VIDEO] "Key insights": CSA and HCA layers alternate 1:1; [HYBRID]:
the window branch runs beside each):
  CSA layer = merge(CSA sparse branch, window branch)
  HCA layer = merge(HCA dense branch, window branch)
"""
import numpy as np

from .formats import bf16_to_f64, nvfp4_decode, round_bf16
from .method import (attend, index_scores, merge, pool, topk_select, visible_count,
                     window_positions)


def f64(x):
    """uint16 -> bf16 value; float arrays -> float64."""
    x = np.asarray(x)
    return bf16_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64)


def csa_branch(q_t, t, qI_t, w_t, kI, Kc, Vc, m, k, n_valid=None, scale=1.0):
    """Indexer over the visible entries, top-k, then attention over those k."""
    nv = visible_count(t, m, len(kI) if n_valid is None else n_valid)
    s = index_scores(qI_t, w_t, kI[:nv])
    idx, kth = topk_select(s, k)
    sel = idx[idx >= 0]
    O, lse = attend(q_t, Kc[sel], Vc[sel], scale)
    return dict(idx=idx, scores=s, kth=kth, O=O, lse=lse, n_visible=nv)


def hca_branch(q_t, t, Kc, Vc, m, n_valid=None, scale=1.0):
    """Dense attention over every visible compressed entry ([HYBRID], HCA)."""
    nv = visible_count(t, m, len(Kc) if n_valid is None else n_valid)
    O, lse = attend(q_t, Kc[:nv], Vc[:nv], scale)
    return dict(O=O, lse=lse, n_visible=nv)


def swa_branch(q_t, t, Kr, Vr, raw_pos0, W, scale=1.0):
    """Attention over the window positions present in the raw buffer."""
    rows = window_positions(t, W, raw_pos0, len(Kr)) - raw_pos0
    O, lse = attend(q_t, Kr[rows], Vr[rows], scale)
    return dict(O=O, lse=lse, n_keys=len(rows))


def _layer(a, b):
    O, L = merge([a["O"], b["O"]], [a["lse"], b["lse"]])
    return O, L


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def tiny_prefill(inp, cfg, rows=None):
    """All (or the given) queries of the 2048-token CSA+HCA prefill."""
    K, V = f64(inp["K"][0]), f64(inp["V"][0])
    gate = f64(inp["gate"][0])
    Kc4, Vc4 = pool(K, V, gate, cfg.m_csa)
    Kc128, Vc128 = pool(K, V, gate, cfg.m_hca)
    q, qI, w, kI = f64(inp["q"][0]), f64(inp["qI"][0]), f64(inp["w"][0]), f64(inp["kI"][0])
    rows = range(cfg.T) if rows is None else rows
    out = []
    for t in rows:
        c = csa_branch(q[t], t, qI[t], w[t], kI, Kc4, Vc4, cfg.m_csa, cfg.k)
        h = hca_branch(q[t], t, Kc128, Vc128, cfg.m_hca)
        sw = swa_branch(q[t], t, K, V, 0, cfg.W)
        csa_O, csa_L = _layer(c, sw)
        hca_O, hca_L = _layer(h, sw)
        three_O, three_L = merge([c["O"], h["O"], sw["O"]], [c["lse"], h["lse"], sw["lse"]])
        out.append(dict(t=t, csa=c, hca=h, swa=sw, csa_layer=(csa_O, csa_L),
                        hca_layer=(hca_O, hca_L), three=(three_O, three_L)))
    return dict(Kc4=Kc4, Vc4=Vc4, Kc128=Kc128, Vc128=Vc128, rows=out)


def csa_decode(inp, cfg, batches=None):
    """One decode query per sequence against precompressed entries + window."""
    res = []
    for b in (range(cfg.B) if batches is None else batches):
        t = cfg.q_pos
        q, qI, w = f64(inp["q"][b, 0]), f64(inp["qI"][b, 0]), f64(inp["w"][b, 0])
        c = csa_branch(q, t, qI, w, f64(inp["kI"][b]), f64(inp["Kc"][b]), f64(inp["Vc"][b]),
                       cfg.m, cfg.k)
        sw = swa_branch(q, t, f64(inp["Kr"][b]), f64(inp["Vr"][b]), cfg.raw_pos0, cfg.W)
        res.append(dict(b=b, csa=c, swa=sw, layer=_layer(c, sw)))
    return res


def csa_prefill(inp, cfg, t_rows, q_rows):
    """Sampled queries of the 131072-token CSA prefill.

    inp: K, V, gate, kI (full), qI/w rows for t_rows ([n, HI, DI], [n, HI]);
    q_rows: [n, H, D] queries of t_rows.
    """
    K, V = f64(inp["K"][0]), f64(inp["V"][0])
    Kc, Vc = pool(K, V, f64(inp["gate"][0]), cfg.m)
    kI = f64(inp["kI"][0])
    res = []
    for i, t in enumerate(t_rows):
        q = f64(q_rows[i])
        c = csa_branch(q, t, f64(inp["qI_rows"][i]), f64(inp["w_rows"][i]), kI, Kc, Vc,
                       cfg.m, cfg.k)
        sw = swa_branch(q, t, K, V, 0, cfg.W)
        res.append(dict(t=t, csa=c, swa=sw, layer=_layer(c, sw)))
    return dict(Kc=Kc, Vc=Vc, rows=res)


def hca_decode(inp, cfg, batches=None):
    res = []
    for b in (range(cfg.B) if batches is None else batches):
        t = cfg.q_pos
        q = f64(inp["q"][b, 0])
        h = hca_branch(q, t, f64(inp["Kc"][b]), f64(inp["Vc"][b]), cfg.m)
        sw = swa_branch(q, t, f64(inp["Kr"][b]), f64(inp["Vr"][b]), cfg.raw_pos0, cfg.W)
        res.append(dict(b=b, hca=h, swa=sw, layer=_layer(h, sw)))
    return res


def hca_prefill(inp, cfg, i_rows, q_rows):
    """Sampled queries of the 32768-token chunk appended to the 1M context.

    Reading R9: the raw buffer holds the W-1 tokens before the chunk, then
    the chunk; the chunk's blocks are pooled from raw row W-1 onward into
    entries N0, N0+1, ... first ([HYBRID]: HCA pools 128 consecutive tokens
    per entry); query i sits at position ctx + i and sees every complete
    block plus its window ([VIDEO] "Explained simply": the last 128 tokens).
    """
    Kr, Vr, gate = f64(inp["Kr"][0]), f64(inp["Vr"][0]), f64(inp["gate"][0])
    r0 = cfg.W - 1
    Kn, Vn = pool(Kr[r0:], Vr[r0:], gate[r0:], cfg.m)
    Kc = np.concatenate([f64(inp["Kc"][0, :cfg.N0]), Kn])
    Vc = np.concatenate([f64(inp["Vc"][0, :cfg.N0]), Vn])
    res = []
    for n, i in enumerate(i_rows):
        t = cfg.q_pos0 + int(i)
        q = f64(q_rows[n])
        h = hca_branch(q, t, Kc, Vc, cfg.m)
        sw = swa_branch(q, t, Kr, Vr, cfg.raw_pos0, cfg.W)
        res.append(dict(i=int(i), hca=h, swa=sw, layer=_layer(h, sw)))
    return dict(Kc_new=Kn, Vc_new=Vn, rows=res)


def pair_decode(inp, cfg, steps=None, batches=None, kI=None, kc_rows=None):
    """The interleaved CSA/HCA layer pair, decoded step by step (reading R9).

    Step s: the new token (raw row W+s of each layer, position ctx+s) joins
    both raw buffers; when it completes a block of a layer (position+1
    divisible by that layer's m) the block -- raw rows W+s+1-m .. W+s -- is
    pooled into entry (ctx+s+1)/m - 1 before attention ([HYBRID]: entries
    are pools of m consecutive tokens; reading R2: an entry is visible once
    its block is complete); then the shared query attends through the CSA
    layer and through the HCA layer.  At a 1M-token context no HCA block
    completes within 64 steps, but the schedule is the same for both layers.
    kI: optional decoded indexer keys [B, Ncap, DI] (fp64) to avoid repeated
    NVFP4 decoding; kc_rows(b, rows) -> (Kc rows, Vc rows) fp64 may replace
    inp["Kc"] / inp["Vc"] for precompressed entries.  inp["gate_h"] (HCA
    gate logits per raw row) is needed only when an HCA block completes.
    """
    steps = range(cfg.steps) if steps is None else steps
    batches = range(cfg.B) if batches is None else batches
    out = {}
    for b in batches:
        kIb = kI[b] if kI is not None else nvfp4_decode(inp["kI_packed"][b], inp["kI_scale"][b])
        Kr, Vr = f64(inp["Kr"][b]), f64(inp["Vr"][b])
        gate = f64(inp["gate"][b])
        Kr_h, Vr_h = f64(inp["Kr_h"][b]), f64(inp["Vr_h"][b])
        Kc_h, Vc_h = f64(inp["Kc_h"][b]), f64(inp["Vc_h"][b])
        # entries pooled during the run (reading R1: stored in bf16)
        new_K, new_V, new_Kh, new_Vh = {}, {}, {}, {}
        last = max(steps) if len(steps) else -1
        for s in range(last + 1):
            pos = cfg.ctx + s
            r1 = cfg.W + s + 1                       # one past the new token's raw row
            if (pos + 1) % cfg.m_csa == 0:
                j = (pos + 1) // cfg.m_csa - 1
                kc, vc = pool(Kr[r1 - cfg.m_csa:r1], Vr[r1 - cfg.m_csa:r1],
                              gate[r1 - cfg.m_csa:r1], cfg.m_csa)
                new_K[j], new_V[j] = kc[0], vc[0]
            if (pos + 1) % cfg.m_hca == 0:
                j = (pos + 1) // cfg.m_hca - 1
                gh = f64(inp["gate_h"][b])
                kc, vc = pool(Kr_h[r1 - cfg.m_hca:r1], Vr_h[r1 - cfg.m_hca:r1],
                              gh[r1 - cfg.m_hca:r1], cfg.m_hca)
                new_Kh[j], new_Vh[j] = kc[0], vc[0]
            if s not in steps:
                continue
            q, qI, w = f64(inp["q"][s, b]), f64(inp["qI"][s, b]), f64(inp["w"][s, b])
            nv = visible_count(pos, cfg.m_csa, cfg.N_csa + len(new_K))
            sc = index_scores(qI, w, kIb[:nv])
            idx, kth = topk_select(sc, cfg.k)
            sel = idx[idx >= 0]
            old = sel[sel < cfg.N_csa]
            if kc_rows is not None:
                Ko, Vo = kc_rows(b, old)
            else:
                Ko, Vo = f64(inp["Kc"][b][old]), f64(inp["Vc"][b][old])
            Kn = np.array([new_K[j] for j in sel if j >= cfg.N_csa]).reshape(-1, cfg.D)
            Vn = np.array([new_V[j] for j in sel if j >= cfg.N_csa]).reshape(-1, cfg.D)
            cO, cL = attend(q, np.concatenate([Ko, Kn]), np.concatenate([Vo, Vn]))
            rows = window_positions(pos, cfg.W, cfg.raw_pos0, cfg.W + s + 1) - cfg.raw_pos0
            sO, sL = attend(q, Kr[rows], Vr[rows])
            nvh = visible_count(pos, cfg.m_hca, cfg.N_hca + len(new_Kh))
            Kh = np.concatenate([Kc_h[:min(nvh, cfg.N_hca)],
                                 np.array([new_Kh[j] for j in range(cfg.N_hca, nvh)]).reshape(-1, cfg.D)])
            Vh = np.concatenate([Vc_h[:min(nvh, cfg.N_hca)],
                                 np.array([new_Vh[j] for j in range(cfg.N_hca, nvh)]).reshape(-1, cfg.D)])
            hO, hL = attend(q, Kh, Vh)
            shO, shL = attend(q, Kr_h[rows], Vr_h[rows])
            out[(s, b)] = dict(idx=idx, scores=sc, kth=kth,
                               csa=merge([cO, sO], [cL, sL]), hca=merge([hO, shO], [hL, shL]),
                               new_entries={j: (new_K[j], new_V[j]) for j in new_K},
                               new_entries_h={j: (new_Kh[j], new_Vh[j]) for j in new_Kh})
    return out


def swa_replay(inp, cfg, R, batches=None):
    """SWA bounded replay of a CSA/HCA layer pair ([V41], the SWA Bounded
    Replay passage): after the local 128-token window state of a paused
    session has been dropped, the compressed (global) caches are kept and
    only the last R input tokens -- positions ctx-R .. ctx-1 -- are replayed
    to rebuild the current state, instead of recomputing the whole prompt.

    Reading: the replay is an R-token prefill chunk of each layer against its
    kept caches; the rebuilt raw buffer holds only the replayed tokens
    (raw_pos0 = ctx - R), so replayed query i sees a window of min(i+1, W)
    tokens, and the last replayed query (position ctx-1) sees its full window
    when R >= W.  Entries are visible by reading R2 against the kept caches.

    inp: the layer-pair decode inputs (PairDecode recipe layout); the replayed
    tokens' raw K/V are raw rows W-R .. W-1 of each layer's buffer and the
    replayed queries are rq/rqI/rw [R, B, ...].  Returns {(i, b): dict(csa=
    (O, lse), hca=(O, lse), idx, scores, kth)}.
    """
    batches = range(cfg.B) if batches is None else batches
    out = {}
    r0 = cfg.W - R                        # first replayed row of the raw buffers
    pos0 = cfg.ctx - R
    for b in batches:
        kIb = nvfp4_decode(inp["kI_packed"][b], inp["kI_scale"][b])
        Kr, Vr = f64(inp["Kr"][b])[r0:cfg.W], f64(inp["Vr"][b])[r0:cfg.W]
        Kr_h, Vr_h = f64(inp["Kr_h"][b])[r0:cfg.W], f64(inp["Vr_h"][b])[r0:cfg.W]
        Kc, Vc = f64(inp["Kc"][b]), f64(inp["Vc"][b])
        Kc_h, Vc_h = f64(inp["Kc_h"][b]), f64(inp["Vc_h"][b])
        for i in range(R):
            t = pos0 + i
            q, qI, w = f64(inp["rq"][i, b]), f64(inp["rqI"][i, b]), f64(inp["rw"][i, b])
            c = csa_branch(q, t, qI, w, kIb, Kc, Vc, cfg.m_csa, cfg.k, n_valid=cfg.N_csa)
            sw = swa_branch(q, t, Kr, Vr, pos0, cfg.W)
            h = hca_branch(q, t, Kc_h, Vc_h, cfg.m_hca, n_valid=cfg.N_hca)
            swh = swa_branch(q, t, Kr_h, Vr_h, pos0, cfg.W)
            out[(i, b)] = dict(idx=c["idx"], scores=c["scores"], kth=c["kth"], window=sw["n_keys"],
                               csa=merge([c["O"], sw["O"]], [c["lse"], sw["lse"]]),
                               hca=merge([h["O"], swh["O"]], [h["lse"], swh["lse"]]))
    return out


def csa2_group(q_t, t, layers, kI, m, k, n_notes, n_valid=None):
    """CSA2 index sharing across a group of CSA layers for one query ([V41], the
    CSA2 passage: the first layer works in full mode -- reads the context,
    highlights what matters and keeps the notes; a re-index layer takes those
    notes as they are and adds its own marks for its own task; a reuse layer
    copies the previous layer's result as it is).

    Reading R12: a full layer scores every visible entry with its own indexer
    query and weights against the indexer keys kI (the notes' keys), keeps the
    n_notes best as the group's notes and attends to its own top-k (the k best
    of the same scores); a re-index layer scores only the notes with its own
    indexer query and weights against the same keys and attends to its top-k
    among them; a reuse layer attends to the entries the layer before it
    selected.  Each layer attends to its own compressed cache (entry j covers
    the same tokens in every layer).  Ties go to the lower index everywhere.

    layers: list of dicts with mode ("full" | "reindex" | "reuse"), q [H, D],
    and, for full / reindex, qI [HI, DI], w [HI]; and Kc, Vc [N, D] (fp64).
    q_t is unused (each layer brings its own q); kept for a uniform signature.
    Returns per layer dict(idx, scores (of the entries it scored), kth, O, lse).
    """
    nv = visible_count(t, m, len(kI) if n_valid is None else n_valid)
    notes = None
    prev = None
    out = []
    for L in layers:
        if L["mode"] == "full":
            s = index_scores(L["qI"], L["w"], kI[:nv])
            notes, _ = topk_select(s, n_notes)
            idx, kth = topk_select(s, k)
            scored = s
        elif L["mode"] == "reindex":
            cand = notes[notes >= 0]
            s_c = index_scores(L["qI"], L["w"], kI[cand])
            pick, kth = topk_select(s_c, k)           # positions within the candidate list
            sel = np.sort(cand[pick[pick >= 0]])
            idx = np.full(k, -1, dtype=np.int64)
            idx[:sel.size] = sel
            scored = dict(zip(cand.tolist(), s_c.tolist()))
        elif L["mode"] == "reuse":
            idx, kth, scored = prev["idx"], prev["kth"], prev["scores"]
        else:
            raise ValueError(L["mode"])
        sel = idx[idx >= 0]
        O, lse = attend(L["q"], L["Kc"][sel], L["Vc"][sel])
        prev = dict(idx=idx, scores=scored, kth=kth, O=O, lse=lse, notes=notes)
        out.append(prev)
    return out
