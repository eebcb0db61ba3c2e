"""Small, fixed cases of single library calls, sized for a profiler capture.

    python profile_cases.py <case> [--queries Q]

Each case builds its inputs with the seeded workload generators (``datagen``),
runs the call twice and synchronises (capture the first launch: ncu flushes
the caches before each replay pass, so its DRAM figures are cold-cache
reads).  A few hundred MB at most are held on the device, so a multi-pass
capture (``ncu --set full``) of one launch finishes in seconds:

    index-topk-prefill   the last Q queries (default 4096) of the 131072-token
                         CSA prefill: indexer with the fused top-k
    hca-prefill-attn     the first Q queries (default 4096) of the HCA prefill
                         chunk: dense compressed entries + window, one softmax
    csa-decode-index     the CSA decode batch (32 x 16384 entries): indexer
                         scores only
    csa-prefill-attn     the first Q queries (default 4096) of the CSA prefill
                         at the end of the 131072-token sequence: 128 selected
                         entries per query + the window, one softmax
    pair-decode-index    the layer-pair decode's CSA indexer at 1M context
                         (4 x 262160 entries, NVFP4 keys): scores only
    csa-decode-topk      the CSA decode batch's indexer + top-k (32 x 16384
                         entries, top-128)
    csa-decode-layer     the CSA decode batch through the layer call:
                         indexer, then top-k + attention in one cluster per
                         query
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import datagen  # noqa: E402
from datagen.workloads import CsaDecode, CsaPrefill, HcaPrefill, PairDecode, T_KI, T_QI, T_W  # noqa: E402

from long_context_compressed_15_b300.layers import CsaLayerPlan  # noqa: E402
from long_context_compressed_15_b300 import (csa_layer_attn, hca_layer_attn, lightning_index_scores,  # noqa: E402
                                             lightning_index_topk, load)


def index_topk_prefill(dev, nq):
    c = CsaPrefill()
    q0 = c.T - nq
    qI = datagen.normal_bf16(c.seed, T_QI, (1, nq, c.HI, c.DI), device=dev)
    w = datagen.uniform_f32(c.seed, T_W, (1, nq, c.HI), device=dev)
    kI = datagen.normal_bf16(c.seed, T_KI, (1, c.N, c.DI), device=dev)
    idx = torch.empty((1, nq, c.k), dtype=torch.int32, device=dev)
    return lambda: lightning_index_topk(qI, w, q0, kI, c.N, c.m, c.k, idx=idx)


def hca_prefill_attn(dev, nq):
    c = HcaPrefill()
    g = c.make(dev, with_q=False)
    q = datagen.normal_bf16(c.seed + 101, 4, (1, nq, c.H, c.D), c.q_scale, device=dev)
    out = torch.empty((1, nq, c.H, c.D), dtype=torch.bfloat16, device=dev)
    return lambda: hca_layer_attn(q, g["Kc"], g["Vc"], c.Ncap, c.m, g["Kr"], g["Vr"], c.q_pos0, c.raw_pos0, c.W,
                                  out=out)


def csa_decode_index(dev, nq):
    c = CsaDecode()
    s = c.make(dev)
    pos = torch.full((c.B,), c.q_pos, dtype=torch.int64, device=dev)
    nval = torch.full((c.B,), c.N, dtype=torch.int32, device=dev)
    scores = torch.empty((c.B, 1, c.N), dtype=torch.float32, device=dev)
    return lambda: lightning_index_scores(s["qI"], s["w"], pos, s["kI"], nval, 4, scores=scores)


def csa_prefill_attn(dev, nq):
    c = CsaPrefill()
    t0 = c.T - nq  # the last nq queries of the sequence: every list holds k entries
    q = datagen.normal_bf16(c.seed, 4, (1, nq, c.H, c.D), c.q_scale, device=dev)
    Kc = datagen.normal_bf16(c.seed, 8, (1, c.N, c.D), device=dev)
    Vc = datagen.normal_bf16(c.seed, 9, (1, c.N, c.D), device=dev)
    R = nq + c.W - 1
    Kr = datagen.normal_bf16(c.seed, 10, (1, R, c.D), device=dev)
    Vr = datagen.normal_bf16(c.seed, 11, (1, R, c.D), device=dev)
    # k distinct entries per query spread over the cache: one per stride, at a per-query offset
    stride = c.N // c.k
    off = (torch.arange(nq, device=dev, dtype=torch.int64) * 2654435761) % stride
    idx = (torch.arange(c.k, device=dev, dtype=torch.int64)[None, :] * stride + off[:, None])
    idx = idx.to(torch.int32).reshape(1, nq, c.k)
    out = torch.empty((1, nq, c.H, c.D), dtype=torch.bfloat16, device=dev)
    return lambda: csa_layer_attn(q, Kc, Vc, idx, Kr, Vr, t0, t0 - (c.W - 1), c.W, out=out)


def pair_decode_index(dev, nq):
    c = PairDecode()
    g = c.make(dev)
    pos = torch.full((c.B,), c.ctx, dtype=torch.int64, device=dev)
    scores = torch.empty((c.B, 1, c.Ncap_csa), dtype=torch.float32, device=dev)
    return lambda: lightning_index_scores(g["qI"][0][:, None], g["w"][0][:, None], pos, g["kI_packed"],
                                          c.N_csa, c.m_csa, kI_scale=g["kI_scale"], scores=scores)


def csa_decode_topk(dev, nq):
    c = CsaDecode()
    s = c.make(dev)
    pos = torch.full((c.B,), c.q_pos, dtype=torch.int64, device=dev)
    idx = torch.empty((c.B, 1, c.k), dtype=torch.int32, device=dev)
    return lambda: lightning_index_topk(s["qI"], s["w"], pos, s["kI"], c.N, 4, c.k, idx=idx)


def csa_decode_layer(dev, nq):
    c = CsaDecode()
    s = c.make(dev)
    plan = CsaLayerPlan(c.B, 1, c.H, c.D, c.N, c.k, c.W, device=dev)
    return lambda: plan(s["q"], s["qI"], s["w"], c.q_pos, s["kI"], c.N, s["Kc"], s["Vc"], s["Kr"], s["Vr"],
                        c.raw_pos0)


CASES = {"index-topk-prefill": index_topk_prefill, "hca-prefill-attn": hca_prefill_attn,
         "csa-decode-index": csa_decode_index, "csa-prefill-attn": csa_prefill_attn,
         "pair-decode-index": pair_decode_index, "csa-decode-topk": csa_decode_topk,
         "csa-decode-layer": csa_decode_layer}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--queries", type=int, default=4096)
    args = ap.parse_args(argv)
    load()
    dev = "cuda:0"
    torch.cuda.set_device(0)
    run = CASES[args.case](dev, args.queries)
    for _ in range(2):
        run()
    torch.cuda.synchronize()
    print(f"{args.case}: ok")


if __name__ == "__main__":
    main()
