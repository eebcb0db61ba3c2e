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

from . import (attn_merge, csa_layer, csa_layer_workspace, csa_sparse_attn, dense_attn_workspace, hca_dense_attn,
               hca_layer_attn, index_topk_workspace, layer_attn_workspace, lightning_index_topk, swa_attn)


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
