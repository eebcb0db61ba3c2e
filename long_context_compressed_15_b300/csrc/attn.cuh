// Multi-query attention of H query heads over a set of shared K/V rows,
// flash-style (online softmax, fp32 accumulation, bf16 operands), with three
// key sources:
//   GATHER  CSA sparse branch: the k entries of the query's index list;
//   RANGE   HCA dense branch: every compressed entry visible at the query;
//   WINDOW  sliding-window branch: raw rows of positions t-W+1 .. t.
// Source: "DeepSeek-V4가 이차적 어텐션 비용 없이 ...", section "두 가지 압축 전략:
// CSA 및 HCA" (MQA with shared KV projections; CSA attends over the selected
// top-k entries, HCA densely over all entries, the window branch over recent
// raw tokens).
//
// Rows of a CTA are (query, head) pairs: for MQA all heads of one query
// share the keys, so one K/V tile in shared memory serves ROWS rows.  Warps
// own 16 rows each and use the warp-level m16n8k16 MMA; K/V tiles of 64
// keys are double-buffered with cp.async.  gridDim.z splits the key range
// (decode); partials are then reduced by k_split_combine.
#pragma once
#include "common.cuh"

namespace lcc {

enum AttnMode { ATT_GATHER = 0, ATT_RANGE = 1, ATT_WINDOW = 2 };

struct AttnArgs {
  const bf16* q;
  int B, Tq, H;
  float scale_log2;  // scale * log2(e)
  const int64_t* q_pos0;
  const bf16* K;
  const bf16* V;
  int64_t kv_bs;  // elements between batches
  int64_t kv_rs;  // elements between rows
  int Ncap;       // rows available per batch
  const int32_t* idx;
  int k;
  const int32_t* n_valid;
  int m;
  const int64_t* raw_pos0;
  int W;
  float* O;
  float* lse;
  int nsplit;
  int64_t rows_total;  // B*Tq*H: stride between split partials
};

template <int D, int ROWS>
struct AttnSmem {
  static constexpr int KT = 64;
  static constexpr size_t q_bytes = size_t(ROWS) * D * 2;
  static constexpr size_t kv_bytes = size_t(2) * KT * D * 2;  // one of K or V, two stages
  static constexpr size_t key_bytes = size_t(2) * KT * 4;
  static constexpr size_t total = q_bytes + 2 * kv_bytes + key_bytes;
};

template <int MODE>
__device__ __forceinline__ void attn_row_bounds(const AttnArgs& a, int b, int qi, bool valid, int& lo, int& hi) {
  lo = 0;
  hi = 0;
  if (!valid) return;
  if (MODE == ATT_GATHER) {
    hi = a.k;
    return;
  }
  const int64_t t = __ldg(a.q_pos0 + b) + qi;
  if (MODE == ATT_RANGE) {
    hi = visible_entries(t, a.m, __ldg(a.n_valid + b), a.Ncap);
  } else {
    const int64_t rp0 = __ldg(a.raw_pos0 + b);
    int64_t plo = t - a.W + 1;
    if (plo < 0) plo = 0;
    int64_t l = plo - rp0, h = t - rp0 + 1;
    if (l < 0) l = 0;
    if (h > a.Ncap) h = a.Ncap;
    if (h < l) h = l;
    lo = static_cast<int>(l);
    hi = static_cast<int>(h);
  }
}

template <int D, int ROWS, int MODE>
__global__ void __launch_bounds__(ROWS * 2) k_attn(AttnArgs a) {
  constexpr int NT = ROWS * 2;
  constexpr int KT = 64;
  constexpr int CPR = D / 8;  // 16-byte chunks per row
  constexpr int NKS = D / 16;  // k-steps of Q.K
  constexpr int NDT = D / 8;   // dim tiles of O
  using S = AttnSmem<D, ROWS>;
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = reinterpret_cast<bf16*>(smem + S::q_bytes);
  bf16* sV = reinterpret_cast<bf16*>(smem + S::q_bytes + S::kv_bytes);
  int* sKey = reinterpret_cast<int*>(smem + S::q_bytes + 2 * S::kv_bytes);
  __shared__ int s_lo, s_hi;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c4 = lane & 3;
  const int b = blockIdx.y, z = blockIdx.z;

  // ---- row -> (query, head) ----
  int qi_cta = 0, h0 = 0;
  int64_t fr0 = 0;
  if (MODE == ATT_GATHER) {
    const int hblocks = (a.H + ROWS - 1) / ROWS;
    qi_cta = blockIdx.x / hblocks;
    h0 = (blockIdx.x % hblocks) * ROWS;
  } else {
    fr0 = static_cast<int64_t>(blockIdx.x) * ROWS;
  }
  auto row_qh = [&](int r, int& qi, int& h) -> bool {
    if (MODE == ATT_GATHER) {
      qi = qi_cta;
      h = h0 + r;
      return h < a.H && qi < a.Tq;
    }
    const int64_t fr = fr0 + r;
    qi = static_cast<int>(fr / a.H);
    h = static_cast<int>(fr % a.H);
    return qi < a.Tq;
  };

  if (tid == 0) { s_lo = INT_MAX; s_hi = INT_MIN; }
  __syncthreads();
  const int rA = warp * 16 + g, rB = rA + 8;
  int qA, hA, qB, hB, loA, hiA, loB, hiB;
  const bool vA = row_qh(rA, qA, hA), vB = row_qh(rB, qB, hB);
  attn_row_bounds<MODE>(a, b, qA, vA, loA, hiA);
  attn_row_bounds<MODE>(a, b, qB, vB, loB, hiB);
  if (c4 == 0) {
    if (vA && hiA > loA) { atomicMin(&s_lo, loA); atomicMax(&s_hi, hiA); }
    if (vB && hiB > loB) { atomicMin(&s_lo, loB); atomicMax(&s_hi, hiB); }
  }
  __syncthreads();
  int z_lo = 0, z_hi = 0;
  if (s_hi > s_lo) {
    const int len = s_hi - s_lo;
    const int per = ((len + a.nsplit - 1) / a.nsplit + KT - 1) / KT * KT;
    z_lo = s_lo + z * per;
    z_hi = min(s_hi, z_lo + per);
  }
  const int ntiles = z_hi > z_lo ? (z_hi - z_lo + KT - 1) / KT : 0;

  // ---- async loads ----
  const int64_t qrow_base = MODE == ATT_GATHER ? (static_cast<int64_t>(b) * a.Tq + qi_cta) : 0;
  for (int u = tid; u < ROWS * CPR; u += NT) {
    const int r = u / CPR, cc = u % CPR;
    int qi, h;
    const bool v = row_qh(r, qi, h);
    const bf16* src = a.q + ((static_cast<int64_t>(b) * a.Tq + (v ? qi : 0)) * a.H + (v ? h : 0)) * D + cc * 8;
    cp_async16(smem_u32(sQ + r * D + ((cc ^ (r & 7)) * 8)), src, v ? 16 : 0);
  }
  auto load_kv = [&](int j0, int st) {
    for (int u = tid; u < 2 * KT * CPR; u += NT) {
      const int which = u / (KT * CPR), rem = u % (KT * CPR);
      const int kk = rem / CPR, cc = rem % CPR;
      const int j = j0 + kk;
      int e = -1;
      if (j < z_hi) {
        if (MODE == ATT_GATHER) {
          e = __ldg(a.idx + qrow_base * a.k + j);
          if (e >= a.Ncap || e < -1) {
            record_error(DEV_ERR_INDEX, static_cast<unsigned>(j));
            e = -1;
          }
        } else {
          e = j;
        }
      }
      const bf16* base = which ? a.V : a.K;
      const bf16* src = base + (e >= 0 ? (b * a.kv_bs + static_cast<int64_t>(e) * a.kv_rs + cc * 8) : 0);
      bf16* dst = (which ? sV : sK) + st * KT * D + kk * D + ((cc ^ (kk & 7)) * 8);
      cp_async16(smem_u32(dst), src, e >= 0 ? 16 : 0);
      if (which == 0 && cc == 0) sKey[st * KT + kk] = e;
    }
  };
  if (ntiles > 0) load_kv(z_lo, 0);
  cp_async_commit();

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float oacc[NDT][4];
#pragma unroll
  for (int n = 0; n < NDT; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
  uint32_t qf[NKS][4];

  for (int t = 0; t < ntiles; ++t) {
    const int st = t & 1;
    const int j0 = z_lo + t * KT;
    if (t + 1 < ntiles) {
      load_kv(j0 + KT, st ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (t == 0) {
#pragma unroll
      for (int ks = 0; ks < NKS; ++ks) {
        const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int cc = 2 * ks + (lane >> 4);
        ldsm_x4(smem_u32(sQ + r * D + ((cc ^ (r & 7)) * 8)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
      }
    }
    const bf16* tK = sK + st * KT * D;
    const bf16* tV = sV + st * KT * D;
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < NKS; ++ks) {
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int key = 16 * p + (lane & 7) + ((lane >> 4) & 1) * 8;
        const int cc = 2 * ks + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(tK + key * D + ((cc ^ (key & 7)) * 8)), b0, b1, b2, b3);
        mma_bf16(s[2 * p], qf[ks], b0, b1);
        mma_bf16(s[2 * p + 1], qf[ks], b2, b3);
      }
    }
    // mask, scale, row max
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kk = 8 * n + 2 * c4 + (e & 1);
        const int jg = j0 + kk;
        const bool keyok = sKey[st * KT + kk] >= 0;
        const bool ok = keyok && (e < 2 ? (jg >= loA && jg < hiA) : (jg >= loB && jg < hiB));
        const float v = ok ? s[n][e] * a.scale_log2 : -INFINITY;
        s[n][e] = v;
        if (e < 2) mx0 = fmaxf(mx0, v); else mx1 = fmaxf(mx1, v);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float base0 = mn0 == -INFINITY ? 0.f : mn0, base1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = exp2f(m0 - base0), al1 = exp2f(m1 - base1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      s[n][0] = exp2f(s[n][0] - base0);
      s[n][1] = exp2f(s[n][1] - base0);
      s[n][2] = exp2f(s[n][2] - base1);
      s[n][3] = exp2f(s[n][3] - base1);
      rs0 += s[n][0] + s[n][1];
      rs1 += s[n][2] + s[n][3];
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
#pragma unroll
    for (int n = 0; n < NDT; ++n) {
      oacc[n][0] *= al0; oacc[n][1] *= al0;
      oacc[n][2] *= al1; oacc[n][3] *= al1;
    }
    // O += P V
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * ks][0], s[2 * ks][1]);
      pa[1] = pack_bf16(s[2 * ks][2], s[2 * ks][3]);
      pa[2] = pack_bf16(s[2 * ks + 1][0], s[2 * ks + 1][1]);
      pa[3] = pack_bf16(s[2 * ks + 1][2], s[2 * ks + 1][3]);
#pragma unroll
      for (int p = 0; p < NDT / 2; ++p) {
        const int key = 16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int cc = 2 * p + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(tV + key * D + ((cc ^ (key & 7)) * 8)), b0, b1, b2, b3);
        mma_bf16(oacc[2 * p], pa, b0, b1);
        mma_bf16(oacc[2 * p + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // ---- epilogue ----
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const float LN2 = 0.6931471805599453f;
  auto grow = [&](int qi, int h) -> int64_t { return (static_cast<int64_t>(b) * a.Tq + qi) * a.H + h; };
  const int64_t zoff = static_cast<int64_t>(z) * a.rows_total;
  if (vA) {
    const int64_t r = zoff + grow(qA, hA);
    float* o = a.O + r * D;
#pragma unroll
    for (int n = 0; n < NDT; ++n)
      *reinterpret_cast<float2*>(o + 8 * n + 2 * c4) = make_float2(oacc[n][0] * inv0, oacc[n][1] * inv0);
    if (c4 == 0) a.lse[r] = l0 > 0.f ? (m0 + log2f(l0)) * LN2 : -INFINITY;
  }
  if (vB) {
    const int64_t r = zoff + grow(qB, hB);
    float* o = a.O + r * D;
#pragma unroll
    for (int n = 0; n < NDT; ++n)
      *reinterpret_cast<float2*>(o + 8 * n + 2 * c4) = make_float2(oacc[n][2] * inv1, oacc[n][3] * inv1);
    if (c4 == 0) a.lse[r] = l1 > 0.f ? (m1 + log2f(l1)) * LN2 : -INFINITY;
  }
}

}  // namespace lcc
