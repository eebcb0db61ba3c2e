"""fp64 CPU oracle of the hybrid compressed-attention path (CSA + HCA + SWA).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product path (the CUDA library ``liblcc.so`` and its Python binding) never
imports or calls it, and the two share no code, table, header or helper.

It is plain numpy in float64: naive per-query loops, with a matrix product or
a sort as the only library steps.  Every function cites the passage it
follows.  Sources (web pages, cited by title and section):

[HYBRID]  "DeepSeek-V4가 이차적 어텐션 비용 없이 백만 토큰 컨텍스트를 달성하는 방법"
          (How DeepSeek-V4 reaches a million-token context without quadratic
          attention cost), section "두 가지 압축 전략: CSA 및 HCA" (Two compression
          strategies: CSA and HCA).
[VIDEO]   "딥시크 V4 분석: CSA·HCA 어텐션으로 100만 토큰 컨텍스트를 저비용에 구현한 방법"
          (DeepSeek V4 analysis: a 1M-token context at low cost with CSA/HCA
          attention), sections "쉽게 이해하기" (Explained simply) and
          "주요 인사이트" (Key insights).
[THREAD]  "DeepSeek v4 (Flash)는 정말 운영 비용이 엄청나게 저렴한가요?" (Is DeepSeek v4
          Flash really that cheap to run?), section "주요 댓글" (Top comments).
[V41]     The DeepSeek V4.1 Flash post on jjy0501.blogspot.com, passages on the
          lightning indexer / CSA2, the FP4 global KV cache and SWA Bounded
          Replay.

Readings where the pages are silent:
  R1 one fp32 gate logit per token, shared by K and V; the pooled entry is
     stored in bf16 (round to nearest even) and later steps use the stored value;
  R2 entry j (tokens j*m .. j*m+m-1) is visible to the query at position t
     iff j*m + m - 1 <= t;
  R3 indexer score s = sum_h w_h * ReLU(q_I,h . k_I); k_I is an input per entry;
  R4 top-k orders by (score desc, index asc), keeps min(k, visible), pads -1;
  R5 the window holds positions max(0, t-W+1) .. t (the query's own token
     included) that are present in the raw buffer;
  R6 branches merge by log-sum-exp; an empty branch has lse = -inf, O = 0;
  R7 NVFP4: e2m1 value times the e4m3 scale of its group of 16, element 2i in
     the low nibble of byte i, no per-tensor scale;
  R8 queries of workloads whose query scale is unstated are N(0,1)/sqrt(128)
     with softmax scale 1;
  R9 decode windows: the CSA decode window is the W raw tokens ending at the
     query; in the layer-pair decode each layer keeps its own raw buffer,
     caches and (CSA) indexer keys, both attend with the shared query, the
     step-s token sits at raw row W+s (position ctx+s), and a block that the
     token completes (position+1 divisible by m) is pooled from raw rows
     W+s+1-m .. W+s into entry (ctx+s+1)/m - 1 before that step attends;
     an HCA prefill chunk starting at position ctx (a multiple of m) sees the
     W-1 raw tokens before it plus itself, and its blocks are pooled from raw
     row W-1 onward into entries ctx/m, ctx/m + 1, ...;
  R10 the 2048-token prefill pools its CSA and HCA entries from the same raw
     K/V and gates;
  R11 the query / KV prologue: RMSNorm (x / sqrt(mean(x^2) + eps) * gain)
     over the head dimension of each query head and of the K and V rows,
     then rotary embedding of the last d_rope channels of q and k (pairs
     (c, c + d_rope/2), angle pos * base^(-2i/d_rope), base 10000); V is
     not rotated;
  R12 CSA2 index sharing: a full-mode layer keeps the n_notes best entries
     by its own indexer score as the group's notes and attends to its own
     top-k; a re-index layer scores only the notes, with its own indexer
     query and weights against the same indexer keys, and attends to its
     top-k among them; a reuse layer attends to the entries the layer before
     it selected; each layer attends to its own compressed cache;
  R16 the indexer computes in FP4: its query is quantised to NVFP4 by R7's
     rule (per group of 16: scale = e4m3 nearest to amax/6, elements = e2m1
     nearest to x/scale, ties to even, saturating) and its keys are NVFP4;
     the head weights stay fp32.

Parity unpinned: the pages print no worked numeric example and no model
dimensions, so the model-level figures (27% of V3.2's per-token FLOPs, ~10%
of its KV cache) cannot be reproduced, and R1, R3 (score form) and the query
distribution are fixed by this implementation rather than by the pages.
Every function below is pinned by closed forms, brute force or library
special cases in tests/test_oracle_pins.py.
"""
from .formats import (bf16_to_f64, f64_to_bf16_bits, round_bf16, e2m1_value,
                      e4m3_value, nvfp4_decode, nvfp4_quantize, nearest_code)
from .method import (pool_weights, pool_exact, pool, visible_count, index_scores,
                     index_scores_fp4, topk_select, attend, window_positions, merge, rms_norm, rope_partial,
                     qkv_prologue)
from . import runs

__all__ = [
    "bf16_to_f64", "f64_to_bf16_bits", "round_bf16", "e2m1_value", "e4m3_value",
    "nvfp4_decode", "nvfp4_quantize", "nearest_code", "index_scores_fp4", "pool_weights", "pool_exact", "pool", "visible_count",
    "index_scores", "topk_select", "attend", "window_positions", "merge", "rms_norm",
    "rope_partial", "qkv_prologue", "runs",
]
