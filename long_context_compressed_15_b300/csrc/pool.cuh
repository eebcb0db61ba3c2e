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
  // device positions (optional): row 0 of sequence b is token tok0[b], a
  // multiple of m; block j goes to entry tok0[b]/m + j if below Ncap, and
  // n_valid[b] (optional) is raised to the entries present
  const int64_t* tok0;
  int32_t* n_valid;
  int Ncap;
};

// Entry of block 0 of sequence b (-1: the sequence is skipped).  With device
// positions, the first CTA of the sequence also raises n_valid and reports a
// misaligned position.
template <int M>
__device__ __forceinline__ int64_t pool_entry0(const PoolArgs& a, int b, bool first_cta) {
  if (!a.tok0) return 0;
  const int64_t t0 = __ldg(a.tok0 + b);
  if (t0 < 0 || t0 % M != 0) {
    if (first_cta && threadIdx.x == 0) record_error(DEV_ERR_POS, static_cast<unsigned>(b));
    return -1;
  }
  const int64_t e0 = t0 / M;
  if (first_cta && threadIdx.x == 0 && a.n_valid) {
    const int64_t top = e0 + a.nblk < a.Ncap ? e0 + a.nblk : a.Ncap;
    if (top > 0) atomicMax(a.n_valid + b, static_cast<int>(top));
  }
  return e0;
}

__device__ __forceinline__ void fma8(float (&acc)[8], float a, uint4 v) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(p[i]);
    acc[2 * i] = fmaf(a, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(a, f.y, acc[2 * i + 1]);
  }
}

// 16-byte load: through the read-only path (RO) when nothing the kernel
// writes can alias the source, else a plain coherent load.
template <bool RO>
__device__ __forceinline__ uint4 ld16(const bf16* p) {
  if constexpr (RO) return __ldg(reinterpret_cast<const uint4*>(p));
  else return *reinterpret_cast<const uint4*>(p);
}
template <bool RO>
__device__ __forceinline__ float ldf(const float* p) {
  if constexpr (RO) return __ldg(p);
  else return *p;
}

__device__ __forceinline__ uint4 pack8(const float (&acc)[8]) {
  uint4 o;
  o.x = pack_bf16(acc[0], acc[1]);
  o.y = pack_bf16(acc[2], acc[3]);
  o.z = pack_bf16(acc[4], acc[5]);
  o.w = pack_bf16(acc[6], acc[7]);
  return o;
}

// Pool one block of M <= 16 tokens with the lanes [sub*LPB, sub*LPB + LPB)
// of a warp: lanes [0, D/8) of the group read K rows, lanes [D/8, D/4) V
// rows, 16 bytes per lane.  g: the block's M gate logits; K/V: its first
// token row; Kc/Vc: the entry.
template <int M, int D, bool RO>
__device__ __forceinline__ void pool_block_small(const float* g, const bf16* K, const bf16* V, bf16* Kc, bf16* Vc,
                                                 int lane_in_group) {
  constexpr int LPR = D / 8;
  const int isV = lane_in_group / LPR, col = (lane_in_group % LPR) * 8;
  float gv[M];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < M; ++i) { gv[i] = ldf<RO>(g + i); mx = fmaxf(mx, gv[i]); }
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < M; ++i) { gv[i] = expf(gv[i] - mx); sum += gv[i]; }
  const float inv = 1.0f / sum;
  const bf16* src = (isV ? V : K) + col;
  uint4 v[M];
#pragma unroll
  for (int i = 0; i < M; ++i) v[i] = ld16<RO>(src + i * D);
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < M; ++i) fma8(acc, gv[i] * inv, v[i]);
  *reinterpret_cast<uint4*>((isV ? Vc : Kc) + col) = pack8(acc);
}

// Small blocks (m <= 16): each (half-)warp pools NB blocks, every block's
// loads issued before any arithmetic, so that each lane keeps NB * M 16-byte
// loads in flight; the arithmetic is pool_block_small's.
template <int M, int D, int NB>
__global__ void __launch_bounds__(256, 2) k_pool_small(PoolArgs a) {
  constexpr int LPB = 2 * (D / 8);    // lanes per block (K and V)
  constexpr int BPW = 32 / LPB;       // blocks per warp and pass
  constexpr int LPR = D / 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / LPB, li = lane % LPB;
  const int isV = li / LPR, col = (li % LPR) * 8;
  const int b = blockIdx.y;
  const int64_t e0 = pool_entry0<M>(a, b, blockIdx.x == 0);
  if (e0 < 0) return;
  // block j goes to entry e0 + j; blocks at or past `lim` fall beyond Ncap
  bf16* const dst0 = (isV ? a.Vc : a.Kc) + b * a.c_bs + e0 * D + col;
  const int64_t lim = a.tok0 ? a.Ncap - e0 : a.nblk;
  // the CTA's NB passes cover 8 * BPW * NB consecutive blocks
  const int64_t blk0 = static_cast<int64_t>(blockIdx.x) * 8 * BPW * NB + warp * BPW + sub;
  uint4 v[NB][M];
  float gv[NB][M];
#pragma unroll
  for (int n = 0; n < NB; ++n) {
    const int64_t blk = blk0 + static_cast<int64_t>(n) * 8 * BPW;
    if (blk < a.nblk) {
      const bf16* src = (isV ? a.V : a.K) + b * a.kv_bs + blk * M * D + col;
      const float* g = a.gate + b * a.g_bs + blk * M;
#pragma unroll
      for (int i = 0; i < M; ++i) {
        v[n][i] = ld16<true>(src + i * D);
        gv[n][i] = __ldg(g + i);
      }
    }
  }
#pragma unroll
  for (int n = 0; n < NB; ++n) {
    const int64_t blk = blk0 + static_cast<int64_t>(n) * 8 * BPW;
    if (blk >= a.nblk) break;
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < M; ++i) mx = fmaxf(mx, gv[n][i]);
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < M; ++i) { gv[n][i] = expf(gv[n][i] - mx); sum += gv[n][i]; }
    const float inv = 1.0f / sum;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < M; ++i) fma8(acc, gv[n][i] * inv, v[n][i]);
    if (blk < lim) *reinterpret_cast<uint4*>(dst0 + blk * D) = pack8(acc);
  }
}

// Shared memory of pool_block_large.
template <int M, int D>
struct PoolLargeSmem {
  static constexpr int SLOTS = 8 * (32 / (2 * (D / 8)));   // token slots per CTA
  float g[M];
  float stat[2];
  float part[SLOTS][2 * D];
};

// Pool one block of M >= 32 tokens with a whole CTA of 256 threads.  Each
// warp covers token slots with its K-half and V-half lanes; partial sums
// meet in shared memory.  Every thread of the CTA must call it.
template <int M, int D, bool RO>
__device__ __forceinline__ void pool_block_large(const float* g, const bf16* K, const bf16* V, bf16* Kc, bf16* Vc,
                                                 PoolLargeSmem<M, D>& sm) {
  constexpr int LPR = D / 8;
  constexpr int LPB = 2 * LPR;
  constexpr int SPW = 32 / LPB;       // token slots per warp
  constexpr int SLOTS = PoolLargeSmem<M, D>::SLOTS;
  static_assert(M % SLOTS == 0, "block size must be a multiple of the slot count");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = warp * SPW + lane / LPB, isV = (lane / LPR) & 1, col = (lane % LPR) * 8;
  for (int i = threadIdx.x; i < M; i += 256) sm.g[i] = ldf<RO>(g + i);
  __syncthreads();
  if (warp == 0) {
    float mx = -INFINITY;
    for (int i = lane; i < M; i += 32) mx = fmaxf(mx, sm.g[i]);
    mx = warp_max(mx);
    float sum = 0.f;
    for (int i = lane; i < M; i += 32) sum += expf(sm.g[i] - mx);
    sum = warp_sum(sum);
    if (lane == 0) { sm.stat[0] = mx; sm.stat[1] = 1.0f / sum; }
  }
  __syncthreads();
  const float mx = sm.stat[0], inv = sm.stat[1];
  const bf16* src = (isV ? V : K) + col;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  constexpr int PER = M / SLOTS;
  constexpr int UNR = PER < 8 ? PER : 8;
  for (int i0 = 0; i0 < PER; i0 += UNR) {
    uint4 v[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) v[u] = ld16<RO>(src + ((i0 + u) * SLOTS + slot) * D);
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int tok = (i0 + u) * SLOTS + slot;
      fma8(acc, expf(sm.g[tok] - mx) * inv, v[u]);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) sm.part[slot][isV * D + col + e] = acc[e];
  __syncthreads();
  for (int c = threadIdx.x; c < 2 * D / 8; c += 256) {
    float o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int s = 0; s < SLOTS; ++s)
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] += sm.part[s][c * 8 + e];
    const int which = (c * 8) / D, cc = (c * 8) % D;
    *reinterpret_cast<uint4*>((which ? Vc : Kc) + cc) = pack8(o);
  }
}

// Large blocks (m >= 32): one CTA of 256 threads per block.
template <int M, int D>
__global__ void __launch_bounds__(256) k_pool_large(PoolArgs a) {
  __shared__ PoolLargeSmem<M, D> sm;
  const int b = blockIdx.y;
  const int64_t blk = blockIdx.x;
  const int64_t e0 = pool_entry0<M>(a, b, blk == 0);
  if (e0 < 0 || (a.tok0 && e0 + blk >= a.Ncap)) return;  // uniform across the CTA
  pool_block_large<M, D, true>(a.gate + b * a.g_bs + blk * M, a.K + b * a.kv_bs + blk * M * D,
                         a.V + b * a.kv_bs + blk * M * D, a.Kc + b * a.c_bs + (e0 + blk) * D,
                         a.Vc + b * a.c_bs + (e0 + blk) * D, sm);
}

}  // namespace lcc
