"""Layer-level composition of the C ABI calls (argument marshalling only).

A CSA layer is the sparse compressed branch merged with the sliding-window
branch; an HCA layer is the dense compressed branch merged with the same
window ("딥시크 V4 분석: ...", section "주요 인사이트": CSA and HCA layers alternate
1:1; "DeepSeek-V4가 이차적 어텐션 비용 없이 ...", section "두 가지 압축 전략: CSA
및 HCA": the window branch runs in parallel).

A plan preallocates every intermediate (index lists, workspace, output and,
for the branch-by-branch form, the branch partials) for fixed sizes, so
repeated calls allocate nothing and a step can be captured in a CUDA graph.
Every step runs in liblcc's kernels.  ``fused=True`` (default) computes the
layer as one softmax over the union of the compressed and window keys
(lcc_csa_layer / lcc_hca_layer_attn); ``fused=False`` runs the two
branches separately and merges them by log-sum-exp (the same result, with
the branch partials O_c/L_c, O_h/L_h and O_w/L_w kept for inspection).
"""
from __future__ import annotations

import torch

from . import (attn_merge, csa_layer, csa_layer_attn, csa_layer_workspace, csa_sparse_attn, decode_append,
               dense_attn_workspace, hca_dense_attn, hca_layer_attn, index_topk_workspace, layer_attn_workspace,
               lightning_index_topk, lightning_reindex_topk, swa_attn)


class CsaLayerPlan:
    """Buffers for CSA layers of fixed size: indexer -> top-k -> sparse MQA, plus window."""

    def __init__(self, B, Tq, H, D, Ncap, k, W, device="cuda", m=4, scale=1.0, fused=True):
        self.B, self.Tq, self.H, self.D, self.Ncap, self.k, self.W, self.m, self.scale = B, Tq, H, D, Ncap, k, W, m, scale
        self.fused = fused
        f32 = dict(dtype=torch.float32, device=device)
        self.idx = torch.empty((B, Tq, k), dtype=torch.int32, device=device)
        if not fused:
            self.O_c = torch.empty((B, Tq, H, D), **f32)
            self.L_c = torch.empty((B, Tq, H), **f32)
            self.O_w = torch.empty((B, Tq, H, D), **f32)
            self.L_w = torch.empty((B, Tq, H), **f32)
        self.out = torch.empty((B, Tq, H, D), dtype=torch.bfloat16, device=device)
        n = csa_layer_workspace(B, Tq, H, D, Ncap, k, W) if fused else index_topk_workspace(B, Tq, Ncap, k)
        self.ws = torch.empty(max(16, n), dtype=torch.uint8, device=device)

    def __call__(self, q, qI, w, q_pos0, kI, n_valid, Kc, Vc, Kr, Vr, raw_pos0, kI_scale=None, stream=None):
        if self.fused:
            return csa_layer(q, qI, w, q_pos0, kI, n_valid, self.m, self.k, Kc, Vc, Kr, Vr, raw_pos0, self.W,
                             kI_scale=kI_scale, scale=self.scale, idx=self.idx, out=self.out, workspace=self.ws,
                             stream=stream)
        lightning_index_topk(qI, w, q_pos0, kI, n_valid, self.m, self.k, kI_scale=kI_scale, idx=self.idx,
                             workspace=self.ws, stream=stream)
        csa_sparse_attn(q, Kc, Vc, self.idx, self.scale, O=self.O_c, lse=self.L_c, stream=stream)
        swa_attn(q, Kr, Vr, q_pos0, raw_pos0, self.W, self.scale, O=self.O_w, lse=self.L_w, stream=stream)
        return attn_merge([(self.O_c, self.L_c), (self.O_w, self.L_w)], out=self.out, stream=stream)


class HcaLayerPlan:
    """Buffers for HCA layers of fixed size: dense MQA over visible entries, plus window."""

    def __init__(self, B, Tq, H, D, Ncap, W, device="cuda", m=128, scale=1.0, fused=True):
        self.B, self.Tq, self.H, self.D, self.Ncap, self.W, self.m, self.scale = B, Tq, H, D, Ncap, W, m, scale
        self.fused = fused
        f32 = dict(dtype=torch.float32, device=device)
        if not fused:
            self.O_h = torch.empty((B, Tq, H, D), **f32)
            self.L_h = torch.empty((B, Tq, H), **f32)
            self.O_w = torch.empty((B, Tq, H, D), **f32)
            self.L_w = torch.empty((B, Tq, H), **f32)
        self.out = torch.empty((B, Tq, H, D), dtype=torch.bfloat16, device=device)
        n = layer_attn_workspace(B, Tq, H, D, Ncap + W) if fused else dense_attn_workspace(B, Tq, H, D, Ncap)
        self.ws = torch.empty(n, dtype=torch.uint8, device=device) if n else None

    def __call__(self, q, q_pos0, Kc, Vc, n_valid, Kr, Vr, raw_pos0, stream=None):
        if self.fused:
            return hca_layer_attn(q, Kc, Vc, n_valid, self.m, Kr, Vr, q_pos0, raw_pos0, self.W, self.scale,
                                  out=self.out, workspace=self.ws, stream=stream)
        hca_dense_attn(q, Kc, Vc, q_pos0, n_valid, self.m, self.scale, O=self.O_h, lse=self.L_h,
                       workspace=self.ws, stream=stream)
        swa_attn(q, Kr, Vr, q_pos0, raw_pos0, self.W, self.scale, O=self.O_w, lse=self.L_w, stream=stream)
        return attn_merge([(self.O_h, self.L_h), (self.O_w, self.L_w)], out=self.out, stream=stream)


class PairDecodePlan:
    """One decode step of an interleaved CSA/HCA layer pair ("딥시크 V4 분석: ...",
    section "주요 인사이트": the two kinds of layer alternate; section "쉽게
    이해하기": 128-token window, CSA pools every 4 tokens, HCA every 128).

    A step appends the new token of each layer to that layer's caches
    (lcc_decode_append: raw row, gate, and the pooled entry of a block the
    token completes, with its indexer key for CSA), then runs the CSA layer
    and the HCA layer with the shared query.  Every decision (does a block
    complete? how many entries are visible?) is taken on the device from
    ``pos``, so a sequence of steps can be captured into one CUDA graph.

    Caches are dicts of caller-owned tensors: ``Kr, Vr`` [B, R, D] bf16,
    ``gate`` [B, R] fp32, ``raw_pos0`` [B] int64, ``Kc, Vc`` [B, Ncap, D] bf16,
    ``n_valid`` [B] int32, and for CSA ``kI`` (bf16 [B, Ncap, DI] or NVFP4
    uint8 [B, Ncap, DI/2]) with ``kI_scale`` for NVFP4.  New tokens are dicts
    with ``k, v`` [B, D] bf16, ``g`` [B] fp32 and, for CSA, ``kI`` (+
    ``kI_scale``): the indexer key of the entry the token completes.
    """

    def __init__(self, B, H, D, Ncap_csa, Ncap_hca, k, W, device="cuda", m_csa=4, m_hca=128, scale=1.0):
        self.m_csa, self.m_hca = m_csa, m_hca
        self.csa = CsaLayerPlan(B, 1, H, D, Ncap_csa, k, W, device=device, m=m_csa, scale=scale)
        self.hca = HcaLayerPlan(B, 1, H, D, Ncap_hca, W, device=device, m=m_hca, scale=scale)

    def __call__(self, pos, q, qI, w, csa_new, hca_new, csa_cache, hca_cache, stream=None):
        c, h = csa_cache, hca_cache
        decode_append(self.m_csa, csa_new["k"], csa_new["v"], csa_new["g"], pos, c["Kr"], c["Vr"], c["gate"],
                      c["raw_pos0"], c["Kc"], c["Vc"], c["n_valid"], kI_new=csa_new.get("kI"), kI=c["kI"],
                      kI_scale_new=csa_new.get("kI_scale"), kI_scale=c.get("kI_scale"), stream=stream)
        decode_append(self.m_hca, hca_new["k"], hca_new["v"], hca_new["g"], pos, h["Kr"], h["Vr"], h["gate"],
                      h["raw_pos0"], h["Kc"], h["Vc"], h["n_valid"], stream=stream)
        oc = self.csa(q, qI, w, pos, c["kI"], c["n_valid"], c["Kc"], c["Vc"], c["Kr"], c["Vr"], c["raw_pos0"],
                      kI_scale=c.get("kI_scale"), stream=stream)
        oh = self.hca(q, pos, h["Kc"], h["Vc"], h["n_valid"], h["Kr"], h["Vr"], h["raw_pos0"], stream=stream)
        return oc, oh


class SwaReplayPlan:
    """SWA bounded replay of a CSA/HCA layer pair (the DeepSeek V4.1 Flash post,
    SWA Bounded Replay passage): when a paused session's 128-token window state
    has been dropped, the compressed caches are kept and only the last R input
    tokens are replayed -- an R-token prefill chunk of each layer against its
    kept caches, with a raw buffer that holds just the replayed tokens
    (raw_pos0 = the first replayed position).  The last replayed query then
    sees its full window again, so the state after the replay equals the state
    before the window was dropped.

    Caches as in PairDecodePlan, except that ``Kr, Vr`` [B, R, D] hold the
    replayed tokens' raw K/V; queries are [B, R, H, D] (indexer [B, R, HI, DI],
    weights [B, R, HI]); ``pos0`` [B] int64 is the first replayed position.
    """

    def __init__(self, B, R, H, D, Ncap_csa, Ncap_hca, k, W, device="cuda", m_csa=4, m_hca=128, scale=1.0):
        self.csa = CsaLayerPlan(B, R, H, D, Ncap_csa, k, W, device=device, m=m_csa, scale=scale)
        self.hca = HcaLayerPlan(B, R, H, D, Ncap_hca, W, device=device, m=m_hca, scale=scale)

    def __call__(self, pos0, q, qI, w, csa_cache, hca_cache, stream=None):
        c, h = csa_cache, hca_cache
        oc = self.csa(q, qI, w, pos0, c["kI"], c["n_valid"], c["Kc"], c["Vc"], c["Kr"], c["Vr"], pos0,
                      kI_scale=c.get("kI_scale"), stream=stream)
        oh = self.hca(q, pos0, h["Kc"], h["Vc"], h["n_valid"], h["Kr"], h["Vr"], pos0, stream=stream)
        return oc, oh


class Csa2GroupPlan:
    """A group of CSA layers that share one index (CSA2, the DeepSeek V4.1 Flash
    post: a full-mode layer reads the context and keeps the notes, re-index
    layers mark their own parts of those notes, reuse layers copy the layer
    before them).

    ``modes``: e.g. ("full", "reindex", "reuse"); the first must be "full".
    A full layer runs the lightning indexer over every visible entry, keeps
    its n_notes best entries as the group's notes (lcc_lightning_index_topk)
    and attends to its own top-k, which is the top-k of its notes under its
    own query (lcc_lightning_reindex_topk); a re-index layer scores only the
    notes with its own indexer query; a reuse layer attends to the previous
    layer's entries and runs no indexer.  Every layer attends to its own
    compressed cache and window (lcc_csa_layer_attn).  The indexer keys kI are
    the full layer's.
    """

    def __init__(self, modes, B, Tq, H, D, Ncap, k, W, n_notes, device="cuda", m=4, scale=1.0):
        if not modes or modes[0] != "full":
            raise ValueError("the first layer of a group works in full mode")
        self.modes, self.k, self.W, self.m, self.scale, self.n_notes = tuple(modes), k, W, m, scale, n_notes
        i32 = dict(dtype=torch.int32, device=device)
        self.notes = torch.empty((B, Tq, n_notes), **i32)
        self.idx = []
        for mode in self.modes:
            self.idx.append(self.idx[-1] if mode == "reuse" else torch.empty((B, Tq, k), **i32))
        self.out = [torch.empty((B, Tq, H, D), dtype=torch.bfloat16, device=device) for _ in self.modes]
        self.ws_index = torch.empty(max(16, index_topk_workspace(B, Tq, Ncap, n_notes)), dtype=torch.uint8,
                                    device=device)
        n = layer_attn_workspace(B, Tq, H, D, k + W)
        self.ws_attn = torch.empty(n, dtype=torch.uint8, device=device) if n else None

    def __call__(self, qs, qIs, ws, q_pos0, kI, n_valid, caches, raw_pos0, kI_scale=None, stream=None):
        """qs / qIs / ws: per layer (qIs[l], ws[l] unused for reuse layers); caches:
        per layer dicts with Kc, Vc, Kr, Vr.  Returns the layers' bf16 outputs."""
        for l, mode in enumerate(self.modes):
            if mode == "full":
                lightning_index_topk(qIs[l], ws[l], q_pos0, kI, n_valid, self.m, self.n_notes, kI_scale=kI_scale,
                                     idx=self.notes, workspace=self.ws_index, stream=stream)
            if mode in ("full", "reindex"):
                lightning_reindex_topk(qIs[l], ws[l], kI, self.notes, self.k, kI_scale=kI_scale, idx=self.idx[l],
                                       stream=stream)
            c = caches[l]
            csa_layer_attn(qs[l], c["Kc"], c["Vc"], self.idx[l], c["Kr"], c["Vr"], q_pos0, raw_pos0, self.W,
                           scale=self.scale, out=self.out[l], workspace=self.ws_attn, stream=stream)
        return self.out
