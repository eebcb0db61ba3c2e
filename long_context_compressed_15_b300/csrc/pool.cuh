// Softmax-weighted pooling of m consecutive tokens' K and V into one
// compressed entry (CSA m=4, HCA m=128).  Source: "DeepSeek-V4가 이차적 어텐션
// 비용 없이 백만 토큰 컨텍스트를 달성하는 방법", section "두 가지 압축 전략: CSA 및 HCA";
// "딥시크 V4 분석: ...", section "쉽게 이해하기" (learned per-token contribution).
//
// HBM-bound stream: every byte of K, V and the gates is read once with
// 16-byte vector loads and every entry written once.  Accumulation is fp32;
// the stored entry is rounded to bf16 (nearest even).
#pragma once
#include "common.cuh"

namespace lcc {

struct PoolArgs {
  const bf16* K;
  const bf16* V;
  const float* gate;
  int B, nblk;
  int64_t kv_bs, g_bs;
  bf16* Kc;
  bf16* Vc;
  int64_t c_bs;
};

__device__ __forceinline__ void fma8(float (&acc)[8], float a, uint4 v) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(p[i]);
    acc[2 * i] = fmaf(a, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(a, f.y, acc[2 * i + 1]);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&acc)[8]) {
  uint4 o;
  o.x = pack_bf16(acc[0], acc[1]);
  o.y = pack_bf16(acc[2], acc[3]);
  o.z = pack_bf16(acc[4], acc[5]);
  o.w = pack_bf16(acc[6], acc[7]);
  return o;
}

// Small blocks (m <= 16): each (half-)warp pools one block.  Lanes
// [0, D/8) read K rows, lanes [D/8, D/4) read V rows, 16 bytes per lane.
template <int M, int D>
__global__ void __launch_bounds__(256) k_pool_small(PoolArgs a) {
  constexpr int LPR = D / 8;          // lanes per row (16-byte chunks)
  constexpr int LPB = 2 * LPR;        // lanes per block (K and V)
  constexpr int BPW = 32 / LPB;       // blocks per warp
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / LPB, isV = (lane / LPR) & 1, col = (lane % LPR) * 8;
  const int b = blockIdx.y;
  const int64_t blk = (static_cast<int64_t>(blockIdx.x) * 8 + warp) * BPW + sub;
  if (blk >= a.nblk) return;
  const float* g = a.gate + b * a.g_bs + blk * M;
  float gv[M];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < M; ++i) { gv[i] = __ldg(g + i); mx = fmaxf(mx, gv[i]); }
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < M; ++i) { gv[i] = expf(gv[i] - mx); sum += gv[i]; }
  const float inv = 1.0f / sum;
  const bf16* src = (isV ? a.V : a.K) + b * a.kv_bs + blk * M * D + col;
  uint4 v[M];
#pragma unroll
  for (int i = 0; i < M; ++i) v[i] = __ldg(reinterpret_cast<const uint4*>(src + i * D));
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < M; ++i) fma8(acc, gv[i] * inv, v[i]);
  bf16* dst = (isV ? a.Vc : a.Kc) + b * a.c_bs + blk * D + col;
  *reinterpret_cast<uint4*>(dst) = pack8(acc);
}

// Large blocks (m >= 32): one CTA of 256 threads per block.  Each warp
// covers token slots with its K-half and V-half lanes; partial sums meet in
// shared memory.
template <int M, int D>
__global__ void __launch_bounds__(256) k_pool_large(PoolArgs a) {
  constexpr int LPR = D / 8;
  constexpr int LPB = 2 * LPR;
  constexpr int SPW = 32 / LPB;       // token slots per warp
  constexpr int SLOTS = 8 * SPW;      // token slots per CTA
  static_assert(M % SLOTS == 0, "block size must be a multiple of the slot count");
  __shared__ float s_g[M];
  __shared__ float s_stat[2];
  __shared__ float s_part[SLOTS][2 * D];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = warp * SPW + lane / LPB, isV = (lane / LPR) & 1, col = (lane % LPR) * 8;
  const int b = blockIdx.y;
  const int64_t blk = blockIdx.x;
  const float* g = a.gate + b * a.g_bs + blk * M;
  for (int i = threadIdx.x; i < M; i += 256) s_g[i] = __ldg(g + i);
  __syncthreads();
  if (warp == 0) {
    float mx = -INFINITY;
    for (int i = lane; i < M; i += 32) mx = fmaxf(mx, s_g[i]);
    mx = warp_max(mx);
    float sum = 0.f;
    for (int i = lane; i < M; i += 32) sum += expf(s_g[i] - mx);
    sum = warp_sum(sum);
    if (lane == 0) { s_stat[0] = mx; s_stat[1] = 1.0f / sum; }
  }
  __syncthreads();
  const float mx = s_stat[0], inv = s_stat[1];
  const bf16* src = (isV ? a.V : a.K) + b * a.kv_bs + blk * M * D + col;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  constexpr int PER = M / SLOTS;
  constexpr int UNR = PER < 8 ? PER : 8;
  for (int i0 = 0; i0 < PER; i0 += UNR) {
    uint4 v[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) v[u] = __ldg(reinterpret_cast<const uint4*>(src + ((i0 + u) * SLOTS + slot) * D));
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int tok = (i0 + u) * SLOTS + slot;
      fma8(acc, expf(s_g[tok] - mx) * inv, v[u]);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) s_part[slot][isV * D + col + e] = acc[e];
  __syncthreads();
  for (int c = threadIdx.x; c < 2 * D / 8; c += 256) {
    float o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int s = 0; s < SLOTS; ++s)
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] += s_part[s][c * 8 + e];
    const int which = (c * 8) / D, cc = (c * 8) % D;
    bf16* dst = (which ? a.Vc : a.Kc) + b * a.c_bs + blk * D + cc;
    *reinterpret_cast<uint4*>(dst) = pack8(o);
  }
}

}  // namespace lcc
