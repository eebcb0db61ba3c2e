// Re-index mode of CSA2 index sharing: a layer scores only the candidate
// entries another layer selected (its "notes") with its own indexer query and
// weights, and keeps its top-k among them.  Source: the DeepSeek V4.1 Flash
// post (jjy0501.blogspot.com), CSA2 passage (full / re-index / reuse modes:
// a re-index layer uses the full layer's notes as they are and marks what
// matters for its own task).
//
// One CTA per query.  The candidate key rows are gathered with 16-byte loads
// (bf16 rows of DI*2 bytes, or NVFP4 rows of DI/2 bytes plus DI/16 e4m3
// scales, decoded exactly), scored in fp32 against the query held in shared
// memory, and turned into 64-bit keys (score key << 32 | ~index, so that equal
// scores order by lower index).  A bitonic sort in shared memory finds the
// k-th key; the winners are then written in the candidates' list order, which
// is ascending index order.
#pragma once
#include "common.cuh"

namespace lcc {

struct ReindexArgs {
  const bf16* qI;         // [B, Tq, HI, DI]
  const float* w;         // [B, Tq, HI]
  int B, Tq;
  const void* kI;         // [B, Ncap, DI] bf16 or [B, Ncap, DI/2] e2m1 pairs
  const uint8_t* kIs;     // NVFP4 scales [B, Ncap, DI/16] or null
  int Ncap;
  const int32_t* cand;    // [B, Tq, n_cand]: ascending entries, then -1
  int n_cand, k;
  int32_t* idx;           // [B, Tq, k]
  float* score;           // optional [B, Tq, k]
};

template <int HI, int DI, bool FP4, int NT, int CAP>
__global__ void __launch_bounds__(NT) k_reindex_topk(ReindexArgs a) {
  static_assert((CAP & (CAP - 1)) == 0 && CAP >= NT, "CAP: a power of two >= NT");
  __shared__ float s_q[HI][DI];
  __shared__ float s_w[HI];
  __shared__ unsigned long long s_sort[CAP];
  __shared__ unsigned long long s_list[CAP];
  __shared__ int s_wsum[NT / 32];
  const int64_t row = blockIdx.x;
  const int b = static_cast<int>(row / a.Tq);
  for (int u = threadIdx.x; u < HI * DI; u += NT)
    s_q[u / DI][u % DI] = __bfloat162float(a.qI[row * HI * DI + u]);
  if (threadIdx.x < HI) s_w[threadIdx.x] = a.w[row * HI + threadIdx.x];
  __syncthreads();
  const int32_t* cand = a.cand + row * a.n_cand;
  for (int c = threadIdx.x; c < CAP; c += NT) {
    unsigned long long key = 0;  // 0 = no candidate (no finite score maps below it)
    const int j = c < a.n_cand ? __ldg(cand + c) : -1;
    if (j >= a.Ncap) record_error(DEV_ERR_INDEX, static_cast<unsigned>(c));
    if (j >= 0 && j < a.Ncap) {
      const int64_t e = static_cast<int64_t>(b) * a.Ncap + j;
      float kv[DI];
      if constexpr (FP4) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.kI) + e * (DI / 2));
        const uint8_t* sc = a.kIs + e * (DI / 16);
#pragma unroll
        for (int v = 0; v < DI / 32; ++v) {
          const uint4 p = __ldg(src + v);
          const uint32_t wds[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
          for (int g = 0; g < 2; ++g) {           // two groups of 16 elements per 16 bytes
            const uint32_t s2 = e4m3_to_f16x2_bcast(__ldg(sc + v * 2 + g));
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t word = wds[g * 2 + u];
#pragma unroll
              for (int by = 0; by < 4; ++by) {
                const uint32_t h2 = hmul2_u32(e2m1x2_to_f16x2(word >> (8 * by)), s2);
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
                const int c0 = v * 32 + g * 16 + u * 8 + by * 2;
                kv[c0] = f.x;
                kv[c0 + 1] = f.y;
              }
            }
          }
        }
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const bf16*>(a.kI) + e * DI);
#pragma unroll
        for (int v = 0; v < DI / 8; ++v) {
          const uint4 p = __ldg(src + v);
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&p);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 f = __bfloat1622float2(h[u]);
            kv[v * 8 + 2 * u] = f.x;
            kv[v * 8 + 2 * u + 1] = f.y;
          }
        }
      }
      float s = 0.f;
#pragma unroll
      for (int h = 0; h < HI; ++h) {
        float d = 0.f;
#pragma unroll
        for (int x = 0; x < DI; ++x) d = fmaf(s_q[h][x], kv[x], d);
        s = fmaf(s_w[h], fmaxf(d, 0.f), s);
      }
      key = (static_cast<unsigned long long>(f32_to_key(s)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(j));
    }
    s_sort[c] = key;
    s_list[c] = key;
  }
  __syncthreads();
  // bitonic sort, descending
  for (int size = 2; size <= CAP; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < CAP; i += NT) {
        const int p = i ^ stride;
        if (p > i) {
          const unsigned long long x = s_sort[i], y = s_sort[p];
          const bool desc = (i & size) == 0;
          if (desc ? x < y : x > y) { s_sort[i] = y; s_sort[p] = x; }
        }
      }
      __syncthreads();
    }
  }
  unsigned long long thr = s_sort[a.k - 1];
  if (thr == 0) thr = 1;  // fewer than k candidates: keep them all
  // winners in list order (ascending index), compacted by warp ballots
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int base = 0;
  int32_t* out_i = a.idx + row * a.k;
  float* out_s = a.score ? a.score + row * a.k : nullptr;
  for (int c0 = 0; c0 < CAP; c0 += NT) {
    const int c = c0 + threadIdx.x;
    const unsigned long long key = s_list[c];
    const bool win = key >= thr;
    const unsigned bal = __ballot_sync(0xffffffffu, win);
    if (lane == 0) s_wsum[warp] = __popc(bal);
    __syncthreads();
    int off = base;
    for (int u = 0; u < warp; ++u) off += s_wsum[u];
    int tot = 0;
    for (int u = 0; u < NT / 32; ++u) tot += s_wsum[u];
    if (win) {
      const int p = off + __popc(bal & ((1u << lane) - 1u));
      if (p < a.k) {
        out_i[p] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull));
        if (out_s) out_s[p] = key_to_f32(static_cast<uint32_t>(key >> 32));
      }
    }
    base += tot;
    __syncthreads();
  }
  for (int p = base + threadIdx.x; p < a.k; p += NT) {
    out_i[p] = -1;
    if (out_s) out_s[p] = -INFINITY;
  }
}

}  // namespace lcc
