// Query / KV prologue of the path: RMS normalisation of every query head row
// and of the shared K and V rows, then rotary position embedding of the last
// d_rope channels of q and k.  Source: "DeepSeek-V4가 이차적 어텐션 비용 없이 ...",
// section "두 가지 압축 전략: CSA 및 HCA" (both mechanisms use MQA with shared
// KV projections, query and KV normalisation and partial RoPE).
//
// HBM-bound elementwise pass: one CTA per token reads its H query rows and its
// K and V rows once (8-byte loads, all of a warp's rows in flight before any
// arithmetic) and writes them once.  The d_rope/2 rotation angles of the token
// are formed once per CTA: the angle pos * base^(-2i/d_rope) is reduced modulo
// 2*pi in double precision (exact enough at positions up to 2^40) and its
// sine and cosine are taken in single precision on the reduced angle.
#pragma once
#include "common.cuh"

namespace lcc {

struct PrologueArgs {
  const bf16* q;      // [B, T, H, D]
  const bf16* k;      // [B, T, D]
  const bf16* v;      // [B, T, D] or null
  bf16* q_out;
  bf16* k_out;
  bf16* v_out;
  const float* gq;    // [D] gains
  const float* gk;
  const float* gv;
  const int64_t* pos0;  // [B]
  int B, T, H;
  float eps;
  int d_rope;
  double log2_base;
};

template <int D>
__global__ void __launch_bounds__(256) k_qkv_prologue(PrologueArgs a) {
  constexpr int E = D / 32;        // channels per lane
  constexpr int MAXR = 17;         // rows per warp: (128 heads + K + V) / 8 warps, rounded up
  __shared__ float s_cos[D / 2], s_sin[D / 2];
  const int64_t tok = blockIdx.x;  // b * T + t
  const int b = static_cast<int>(tok / a.T), t = static_cast<int>(tok % a.T);
  const int half = a.d_rope / 2;
  if (static_cast<int>(threadIdx.x) < half) {
    const int64_t p = __ldg(a.pos0 + b) + t;
    const double inv_freq = exp2(-2.0 * static_cast<double>(threadIdx.x) / a.d_rope * a.log2_base);
    double ang = static_cast<double>(p) * inv_freq;
    ang -= 6.283185307179586 * rint(ang * 0.15915494309189535);
    float sn, cs;
    sincosf(static_cast<float>(ang), &sn, &cs);
    s_cos[threadIdx.x] = cs;
    s_sin[threadIdx.x] = sn;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrows = a.H + 1 + (a.v ? 1 : 0);
  // where this lane's channels sit in the rotary part (if at all) and its partner lane
  const int c0 = lane * E;                        // first channel of the lane
  const int rot0 = D - a.d_rope;                  // first rotated channel
  const bool in_rot = c0 >= rot0;
  const bool first_half = c0 < D - half;
  const int partner = in_rot ? (first_half ? lane + half / E : lane - half / E) : lane;
  using Vec = typename std::conditional<E == 4, uint2, uint32_t>::type;
  Vec raw[MAXR];
#pragma unroll
  for (int u = 0; u < MAXR; ++u) {
    const int r = warp + 8 * u;
    if (r < nrows) {
      const bf16* src = r < a.H ? a.q + (tok * a.H + r) * D : (r == a.H ? a.k : a.v) + tok * D;
      raw[u] = __ldg(reinterpret_cast<const Vec*>(src + c0));
    }
  }
#pragma unroll
  for (int u = 0; u < MAXR; ++u) {
    const int r = warp + 8 * u;
    if (r >= nrows) break;  // uniform across the warp
    float x[E];
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
#pragma unroll
    for (int e = 0; e < E / 2; ++e) {
      const float2 f = __bfloat1622float2(h2[e]);
      x[2 * e] = f.x;
      x[2 * e + 1] = f.y;
    }
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(x[e], x[e], ss);
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / D + a.eps);
    const float* g = r < a.H ? a.gq : (r == a.H ? a.gk : a.gv);
    float y[E];
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = x[e] * inv * __ldg(g + c0 + e);
    if (r <= a.H) {  // q and k rows are rotated, v rows are not
      float yp[E];
#pragma unroll
      for (int e = 0; e < E; ++e) yp[e] = __shfl_sync(0xffffffffu, y[e], partner);
      if (in_rot) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = (c0 + e - rot0) % half;
          const float cs = s_cos[i], sn = s_sin[i];
          y[e] = first_half ? y[e] * cs - yp[e] * sn : y[e] * cs + yp[e] * sn;
        }
      }
    }
    Vec o;
    uint32_t* o32 = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int e = 0; e < E / 2; ++e) o32[e] = pack_bf16(y[2 * e], y[2 * e + 1]);
    bf16* dst = r < a.H ? a.q_out + (tok * a.H + r) * D : (r == a.H ? a.k_out : a.v_out) + tok * D;
    *reinterpret_cast<Vec*>(dst + c0) = o;
  }
}

}  // namespace lcc
