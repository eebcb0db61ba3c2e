// Lightning-indexer scores: s[q, j] = sum_h w[q,h] * max(0, qI[q,h,:] . kI[j,:])
// for every visible compressed entry j.  Source: "DeepSeek-V4가 이차적 어텐션
// 비용 없이 ...", section "두 가지 압축 전략: CSA 및 HCA" (a light indexer, run
// in FP4, scores the compressed entries for each query and keeps the top-k);
// the DeepSeek V4.1 Flash post (keys kept in FP4).
//
// The dot products form a dense contraction [entries x DI] . [DI x (q,h)],
// so they run on the tensor pipe (m16n8k16: 16 entries x 8 (query, head)
// columns per MMA), which frees the FP32 pipe for the ReLU-weighted head sum.
// Key rows are loaded straight from HBM into MMA fragments with 16-byte
// loads: because a dot product does not depend on the order of its terms,
// the same permutation of the DI dimension is applied to both operands so
// that every thread reads contiguous 16-byte chunks of one key row and of
// one query head.
//
// NVFP4 keys (e2m1 values, one e4m3 scale per 16 elements): each thread
// owns one 16-element group of a row; values are converted to fp16 and
// multiplied by the group scale (both steps exact: an e2m1 x e4m3 product
// has at most 6 significant bits), and the indexer query is rounded to fp16.
#pragma once
#include "common.cuh"

namespace lcc {

struct IndexArgs {
  const bf16* qI;   // [B, Tq, HI, DI]
  const float* w;   // [B, Tq, HI]
  int B, Tq;
  const int64_t* q_pos0;
  const void* kI;        // bf16 [B, Ncap, DI] or uint8 [B, Ncap, DI/2]
  const uint8_t* kIs;    // uint8 [B, Ncap, DI/16] (NVFP4)
  const int32_t* n_valid;
  int Ncap, m;
  int q0, nq;            // query chunk [q0, q0+nq)
  float* scores;         // [nq, Ncap] for this chunk (row = (b, i - q0) flattened as b*nq + i-q0)
  uint32_t* gmax;        // optional [B*nq, g_stride]: key of the largest score of each 16-entry group
  int g_stride;
  int* counters;         // optional [2, B*nq]: zeroed here for the top-k kernel that follows
};

// Each CTA: 4 warps x 64 entries; NQ queries (n-tiles of 8 (query, head) columns).
template <int HI, int DI, bool FP4, int NQ>
__global__ void __launch_bounds__(128) k_index_score(IndexArgs a) {
  static_assert(8 % HI == 0, "HI must divide 8");
  constexpr int QPT = 8 / HI;           // queries per n-tile
  constexpr int NTILE = NQ / QPT;       // n-tiles per CTA
  constexpr int ENT = 256;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c4 = lane & 3;
  const int b = blockIdx.z;
  const int qbase = a.q0 + blockIdx.y * NQ;  // first query of this CTA
  const int64_t pos0 = __ldg(a.q_pos0 + b);
  const int nval = __ldg(a.n_valid + b);
  // largest visible count among this CTA's queries (queries are causal)
  const int qlast = min(qbase + NQ, a.q0 + a.nq) - 1;
  const int vis_max = visible_entries(pos0 + qlast, a.m, nval, a.Ncap);
  const int e_cta = blockIdx.x * ENT;
  pdl_trigger();  // the top-k that follows may start launching (it waits for this grid)
  if (a.counters && blockIdx.x == 0 && threadIdx.x < NQ) {
    const int qq = qbase + threadIdx.x;
    if (qq < a.q0 + a.nq && qq < a.Tq) {
      const int64_t r = static_cast<int64_t>(b) * a.nq + (qq - a.q0);
      a.counters[r] = 0;
      a.counters[static_cast<int64_t>(a.B) * a.nq + r] = 0;
    }
  }
  if (e_cta >= vis_max) return;

  // ---- B fragments: indexer queries, permuted to match the key loads ----
  constexpr int NKS = DI / 16;
  uint32_t bq[NTILE][NKS][2];
  float wv[NTILE][2];
#pragma unroll
  for (int nt = 0; nt < NTILE; ++nt) {
    const int col = g;  // this thread's n column within the tile
    const int qq = qbase + nt * QPT + col / HI, hh = col % HI;
    const bool qv = qq < a.q0 + a.nq && qq < a.Tq;
    const bf16* qp = a.qI + ((static_cast<int64_t>(b) * a.Tq + (qv ? qq : 0)) * HI + hh) * DI;
    if (!FP4) {
#pragma unroll
      for (int ch = 0; ch < DI / 32; ++ch) {
        uint4 v = qv ? __ldg(reinterpret_cast<const uint4*>(qp + ch * 32 + c4 * 8)) : make_uint4(0, 0, 0, 0);
        bq[nt][2 * ch][0] = v.x; bq[nt][2 * ch][1] = v.y;
        bq[nt][2 * ch + 1][0] = v.z; bq[nt][2 * ch + 1][1] = v.w;
      }
    } else {
      // dims 16*c4 .. 16*c4+15 of head hh, converted to fp16
      uint4 v0 = qv ? __ldg(reinterpret_cast<const uint4*>(qp + 16 * c4)) : make_uint4(0, 0, 0, 0);
      uint4 v1 = qv ? __ldg(reinterpret_cast<const uint4*>(qp + 16 * c4 + 8)) : make_uint4(0, 0, 0, 0);
      uint32_t w8[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w8[i]));
        __half2 hv = __floats2half2_rn(f.x, f.y);
        w8[i] = *reinterpret_cast<uint32_t*>(&hv);
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) { bq[nt][s][0] = w8[2 * s]; bq[nt][s][1] = w8[2 * s + 1]; }
    }
    // head weights of the two columns this thread's accumulators hold
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int colw = 2 * c4 + e;
      const int qw = qbase + nt * QPT + colw / HI, hw = colw % HI;
      const bool ok = qw < a.q0 + a.nq && qw < a.Tq;
      wv[nt][e] = ok ? __ldg(a.w + (static_cast<int64_t>(b) * a.Tq + qw) * HI + hw) : 0.f;
    }
  }

  // ---- this warp's 64 entries: 4 m-tiles of 16 ----
#pragma unroll 1
  for (int mt = 0; mt < 4; ++mt) {
    const int e0 = e_cta + warp * 64 + mt * 16;
    if (e0 >= vis_max) break;
    const int rowA = e0 + g, rowB = e0 + g + 8;
    const bool okA = rowA < a.Ncap, okB = rowB < a.Ncap;
    uint32_t af[NKS][4];
    if (!FP4) {
      const bf16* kb = reinterpret_cast<const bf16*>(a.kI) + static_cast<int64_t>(b) * a.Ncap * DI;
#pragma unroll
      for (int ch = 0; ch < DI / 32; ++ch) {
        uint4 va = okA ? __ldg(reinterpret_cast<const uint4*>(kb + static_cast<int64_t>(rowA) * DI + ch * 32 + c4 * 8))
                       : make_uint4(0, 0, 0, 0);
        uint4 vb = okB ? __ldg(reinterpret_cast<const uint4*>(kb + static_cast<int64_t>(rowB) * DI + ch * 32 + c4 * 8))
                       : make_uint4(0, 0, 0, 0);
        af[2 * ch][0] = va.x; af[2 * ch][1] = vb.x; af[2 * ch][2] = va.y; af[2 * ch][3] = vb.y;
        af[2 * ch + 1][0] = va.z; af[2 * ch + 1][1] = vb.z; af[2 * ch + 1][2] = va.w; af[2 * ch + 1][3] = vb.w;
      }
    } else {
      static_assert(!FP4 || DI == 64, "NVFP4 keys need DI = 64");
      const uint8_t* kp = reinterpret_cast<const uint8_t*>(a.kI) + static_cast<int64_t>(b) * a.Ncap * (DI / 2);
      const uint8_t* ks = a.kIs + static_cast<int64_t>(b) * a.Ncap * (DI / 16);
      uint2 pa = okA ? __ldg(reinterpret_cast<const uint2*>(kp + static_cast<int64_t>(rowA) * 32 + 8 * c4)) : make_uint2(0, 0);
      uint2 pb = okB ? __ldg(reinterpret_cast<const uint2*>(kp + static_cast<int64_t>(rowB) * 32 + 8 * c4)) : make_uint2(0, 0);
      const uint32_t sa = e4m3_to_f16x2_bcast(okA ? __ldg(ks + static_cast<int64_t>(rowA) * 4 + c4) : 0u);
      const uint32_t sb = e4m3_to_f16x2_bcast(okB ? __ldg(ks + static_cast<int64_t>(rowB) * 4 + c4) : 0u);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint32_t wa = s < 2 ? pa.x : pa.y, wb = s < 2 ? pb.x : pb.y;
        const int sh = (s & 1) * 16;
        af[s][0] = hmul2_u32(e2m1x2_to_f16x2(wa >> sh), sa);
        af[s][2] = hmul2_u32(e2m1x2_to_f16x2(wa >> (sh + 8)), sa);
        af[s][1] = hmul2_u32(e2m1x2_to_f16x2(wb >> sh), sb);
        af[s][3] = hmul2_u32(e2m1x2_to_f16x2(wb >> (sh + 8)), sb);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NTILE; ++nt) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < NKS; ++s) {
        if (FP4) mma_f16(acc, af[s], bq[nt][s][0], bq[nt][s][1]);
        else mma_bf16(acc, af[s], bq[nt][s][0], bq[nt][s][1]);
      }
      // ReLU, head weights, sum over the query's heads (lanes of the quad)
      float sA = wv[nt][0] * fmaxf(acc[0], 0.f) + wv[nt][1] * fmaxf(acc[1], 0.f);
      float sB = wv[nt][0] * fmaxf(acc[2], 0.f) + wv[nt][1] * fmaxf(acc[3], 0.f);
      if (HI >= 4) { sA += __shfl_xor_sync(0xffffffffu, sA, 1); sB += __shfl_xor_sync(0xffffffffu, sB, 1); }
      if (HI >= 8) { sA += __shfl_xor_sync(0xffffffffu, sA, 2); sB += __shfl_xor_sync(0xffffffffu, sB, 2); }
      if ((c4 & (HI / 2 - 1)) == 0) {
        const int qq = qbase + nt * QPT + (2 * c4) / HI;
        if (qq < a.q0 + a.nq && qq < a.Tq) {
          float* dst = a.scores + (static_cast<int64_t>(b) * a.nq + (qq - a.q0)) * a.Ncap;
          const int vis = visible_entries(pos0 + qq, a.m, nval, a.Ncap);
          if (rowA < vis) dst[rowA] = sA;
          if (rowB < vis) dst[rowB] = sB;
        }
      }
      if (a.gmax && HI == 8) {
        // group maximum over the m-tile's 16 entries (one query per n-tile when HI = 8)
        const int qq = qbase + nt;
        const bool qok = qq < a.q0 + a.nq && qq < a.Tq;
        const int vis = qok ? visible_entries(pos0 + qq, a.m, nval, a.Ncap) : 0;
        uint32_t key = max(rowA < vis ? f32_to_key(sA) : 0u, rowB < vis ? f32_to_key(sB) : 0u);
        key = __reduce_max_sync(0xffffffffu, key);
        if (lane == 0 && qok && e0 < vis)
          a.gmax[(static_cast<int64_t>(b) * a.nq + (qq - a.q0)) * a.g_stride + (e0 >> 4)] = key;
      }
    }
  }
}

}  // namespace lcc
