// Log-sum-exp combination of attention partials: the branch merge of a
// layer (window + CSA sparse, or window + HCA dense) and the reduction of
// key-range splits of one branch.  Both compute, per row,
//   L = log sum_b exp(lse_b),  O = sum_b exp(lse_b - L) O_b,
// which equals one softmax over the union of the partials' key sets
// ("DeepSeek-V4가 이차적 어텐션 비용 없이 ...", section "두 가지 압축 전략: CSA 및 HCA":
// the window branch runs in parallel with the compressed one).
#pragma once
#include "common.cuh"

namespace lcc {

struct MergeArgs {
  const float* O[4];
  const float* lse[4];
  int nb;
  int64_t rows;
  int D;
  bf16* out;       // nullable
  float* out_f32;  // nullable
  float* lse_out;  // nullable
};

// One warp per row; lane owns D/32 consecutive floats.
template <int D>
__global__ void __launch_bounds__(256) k_merge(MergeArgs a) {
  constexpr int PER = D / 32;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.rows) return;
  float l[4];
  float L = -INFINITY;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    l[b] = b < a.nb ? __ldg(a.lse[b] + row) : -INFINITY;
    L = fmaxf(L, l[b]);
  }
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float tot = 0.f;
  if (L != -INFINITY) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      if (b >= a.nb || l[b] == -INFINITY) continue;
      const float w = expf(l[b] - L);
      tot += w;
      const float* src = a.O[b] + row * D + lane * PER;
      if constexpr (PER == 4) {
        float4 v = __ldg(reinterpret_cast<const float4*>(src));
        acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
        acc[2] = fmaf(w, v.z, acc[2]); acc[3] = fmaf(w, v.w, acc[3]);
      } else {
        float2 v = __ldg(reinterpret_cast<const float2*>(src));
        acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
      }
    }
  }
  const float inv = tot > 0.f ? 1.0f / tot : 0.f;
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] *= inv;
  if (a.out) {
    bf16* dst = a.out + row * D + lane * PER;
    if constexpr (PER == 4) {
      uint2 o;
      o.x = pack_bf16(acc[0], acc[1]);
      o.y = pack_bf16(acc[2], acc[3]);
      *reinterpret_cast<uint2*>(dst) = o;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0], acc[1]);
    }
  }
  if (a.out_f32) {
    float* dst = a.out_f32 + row * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) dst[e] = acc[e];
  }
  if (a.lse_out && lane == 0) a.lse_out[row] = (L == -INFINITY) ? -INFINITY : L + logf(tot);
}

// Splits whose partial rows the combine requests together with the lse values
// (one round of loads); decode calls split their keys at most this many ways.
constexpr int kCombineFirstSplits = 24;

// Reduction of `nsplit` key-range partials stored [nsplit][rows][D] and
// [nsplit][rows] into O [rows][D] fp32 and/or out [rows][D] bf16, and lse
// [rows] (each output optional).
template <int D>
__global__ void __launch_bounds__(256) k_split_combine(const float* __restrict__ Op, const float* __restrict__ lp,
                                                       int nsplit, int64_t rows, float* __restrict__ O,
                                                       float* __restrict__ lse, bf16* __restrict__ out) {
  constexpr int PER = D / 32;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_wait();  // the partials come from the split attention kernel
  if (row >= rows) return;
  // the first CH splits' partial rows are requested together with every
  // split's lse (lane s holds splits s, s+32, ...): for up to CH splits the
  // reduction waits on one round of loads
  constexpr int CH = kCombineFirstSplits;
  const float ls0 = lane < nsplit ? __ldg(lp + static_cast<int64_t>(lane) * rows + row) : -INFINITY;
  const int n0 = min(CH, nsplit);
  float x0[CH][PER];
#pragma unroll
  for (int u = 0; u < CH; ++u) {
    const bool in = u < n0;  // an empty split's partial is written as zeros
    const float* src = Op + (static_cast<int64_t>(u) * rows + row) * D + lane * PER;
    if constexpr (PER == 4) {
      const float4 v = in ? __ldg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
      x0[u][0] = v.x; x0[u][1] = v.y; x0[u][2] = v.z; x0[u][3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < PER; ++e) x0[u][e] = in ? __ldg(src + e) : 0.f;
    }
  }
  float L = ls0;
  for (int s = lane + 32; s < nsplit; s += 32) L = fmaxf(L, __ldg(lp + static_cast<int64_t>(s) * rows + row));
  L = warp_max(L);
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float tot = 0.f;
  if (L != -INFINITY) {
    const float wl0 = ls0 == -INFINITY ? 0.f : expf(ls0 - L);
#pragma unroll
    for (int u = 0; u < CH; ++u) {
      const float w = __shfl_sync(0xffffffffu, wl0, u);
      if (u < n0) {
        tot += w;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, x0[u][e], acc[e]);
      }
    }
    // further splits, 32 at a time (lane s holds split s0 + s)
    for (int s0 = CH; s0 < nsplit; s0 += 32) {
      const int sl = s0 + lane;
      const float ls = sl < nsplit ? __ldg(lp + static_cast<int64_t>(sl) * rows + row) : -INFINITY;
      const float wl = ls == -INFINITY ? 0.f : expf(ls - L);
      const int n = min(32, nsplit - s0);
      // partial rows are independent loads: up to 16 vector loads in flight per lane
      for (int j = 0; j < n; j += 16) {
        float wj[16];
        float x[16][PER];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          wj[u] = __shfl_sync(0xffffffffu, wl, (j + u) & 31);
          const bool in = j + u < n;
          const float* src = Op + (static_cast<int64_t>(s0 + j + u) * rows + row) * D + lane * PER;
          if constexpr (PER == 4) {
            const float4 v = in ? __ldg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
            x[u][0] = v.x; x[u][1] = v.y; x[u][2] = v.z; x[u][3] = v.w;
          } else {
#pragma unroll
            for (int e = 0; e < PER; ++e) x[u][e] = in ? __ldg(src + e) : 0.f;
          }
          if (!in) wj[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          tot += wj[u];
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[e] = fmaf(wj[u], x[u][e], acc[e]);
        }
      }
    }
  }
  const float inv = tot > 0.f ? 1.0f / tot : 0.f;
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] *= inv;
  if (O) {
    float* dst = O + row * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) dst[e] = acc[e];
  }
  if (out) {
    bf16* dst = out + row * D + lane * PER;
    if constexpr (PER == 4) {
      uint2 o;
      o.x = pack_bf16(acc[0], acc[1]);
      o.y = pack_bf16(acc[2], acc[3]);
      *reinterpret_cast<uint2*>(dst) = o;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0], acc[1]);
    }
  }
  if (lse && lane == 0) lse[row] = (L == -INFINITY) ? -INFINITY : L + logf(tot);
}

}  // namespace lcc
