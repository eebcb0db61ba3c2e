// Decode-step update of one layer's caches: the new token's raw K, V and
// gate logit join the layer's raw buffer and, when the token completes a
// block of m tokens, the block is pooled into its compressed entry (with the
// arithmetic of the compression kernels, so an entry pooled here equals the
// one lcc_csa_compress / lcc_hca_compress would write) and the visible-entry
// count moves on.  Sources: "딥시크 V4 분석: ...", section "쉽게 이해하기"
// (the window holds the most recent 128 tokens; CSA pools every 4 tokens,
// HCA every 128); "DeepSeek-V4가 이차적 어텐션 비용 없이 ...", section "두 가지
// 압축 전략: CSA 및 HCA" (softmax-weighted pooling of consecutive tokens).
//
// One CTA per sequence; positions, raw offsets and counts are read on the
// device, so a step captured in a CUDA graph needs no host decision.
#pragma once
#include "pool.cuh"

namespace lcc {

struct AppendArgs {
  const bf16* k_new;       // [B, D]
  const bf16* v_new;       // [B, D]
  const float* g_new;      // [B]
  const int64_t* pos;      // [B] position of the new token
  const int64_t* raw_pos0; // [B] position of raw row 0
  bf16* Kr;                // raw rows, batch stride r_bs elements, row stride D
  bf16* Vr;
  float* gate_r;           // raw gate logits, batch stride g_bs
  int64_t r_bs, g_bs;
  int Rcap;
  bf16* Kc;                // compressed entries, batch stride c_bs, row stride D
  bf16* Vc;
  int64_t c_bs;
  int Ncap;
  int32_t* n_valid;        // [B]
  const uint8_t* kI_new;   // optional [B, kI_bytes]: indexer key of the entry the token completes
  uint8_t* kI;             // [B, Ncap, kI_bytes]
  int kI_bytes;
  const uint8_t* kIs_new;  // optional NVFP4 scales [B, kIs_bytes]
  uint8_t* kIs;            // [B, Ncap, kIs_bytes]
  int kIs_bytes;
};

template <int M, int D>
__global__ void __launch_bounds__(256) k_decode_append(AppendArgs a) {
  constexpr int LPR = D / 8;  // 16-byte chunks per row
  const int b = blockIdx.x;
  const int64_t pos = __ldg(a.pos + b);
  const int64_t r = pos - __ldg(a.raw_pos0 + b);
  if (pos < 0 || r < 0 || r >= a.Rcap) {  // uniform across the CTA
    if (threadIdx.x == 0) record_error(DEV_ERR_RANGE, static_cast<unsigned>(b));
    return;
  }
  if (threadIdx.x < 2 * LPR) {
    const int isV = threadIdx.x / LPR, col = (threadIdx.x % LPR) * 8;
    const uint4 v = ld16<true>((isV ? a.v_new : a.k_new) + static_cast<int64_t>(b) * D + col);
    *reinterpret_cast<uint4*>((isV ? a.Vr : a.Kr) + b * a.r_bs + r * D + col) = v;
  }
  if (threadIdx.x == 0) a.gate_r[b * a.g_bs + r] = __ldg(a.g_new + b);
  if ((pos + 1) % M != 0) return;  // no block completes
  const int64_t j = (pos + 1) / M - 1;
  const int64_t r0 = r - (M - 1);
  if (r0 < 0 || j >= a.Ncap) {
    if (threadIdx.x == 0) record_error(DEV_ERR_RANGE, static_cast<unsigned>(b));
    return;
  }
  __syncthreads();  // the new row and gate are visible to every thread of the CTA
  const float* g = a.gate_r + b * a.g_bs + r0;
  const bf16* K = a.Kr + b * a.r_bs + r0 * D;
  const bf16* V = a.Vr + b * a.r_bs + r0 * D;
  bf16* Kc = a.Kc + b * a.c_bs + j * D;
  bf16* Vc = a.Vc + b * a.c_bs + j * D;
  if constexpr (M <= 16) {
    if (threadIdx.x < 2 * LPR) pool_block_small<M, D, false>(g, K, V, Kc, Vc, threadIdx.x);
  } else {
    __shared__ PoolLargeSmem<M, D> sm;
    pool_block_large<M, D, false>(g, K, V, Kc, Vc, sm);
  }
  if (a.kI_new) {
    const int64_t e = static_cast<int64_t>(b) * a.Ncap + j;
    for (int i = threadIdx.x; i < a.kI_bytes; i += blockDim.x)
      a.kI[e * a.kI_bytes + i] = a.kI_new[static_cast<int64_t>(b) * a.kI_bytes + i];
    if (a.kIs_new)
      for (int i = threadIdx.x; i < a.kIs_bytes; i += blockDim.x)
        a.kIs[e * a.kIs_bytes + i] = a.kIs_new[static_cast<int64_t>(b) * a.kIs_bytes + i];
  }
  if (threadIdx.x == 0) a.n_valid[b] = static_cast<int32_t>(j + 1);
}

}  // namespace lcc
