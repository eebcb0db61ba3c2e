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
//
// WIN2 appends the window branch as a second key source of the same
// softmax: the tiles of the compressed source are followed by the tiles of
// the raw window rows, and one online-softmax state runs over both.  One
// softmax over the union of the two key lists equals the log-sum-exp merge
// of the two branches, so a whole CSA layer (sparse + window) or HCA layer
// (dense + window) comes out of one pass, written as bf16.
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
  // second key source (window rows) for WIN2 kernels
  const bf16* K2;
  const bf16* V2;
  int64_t kv2_bs, kv2_rs;
  int Ncap2;
  bf16* out_bf16;      // if set (and nsplit == 1): the result as bf16 instead of fp32 O
};

template <int D, int ROWS>
struct AttnSmem {
  static constexpr int KT = 64;
  static constexpr size_t q_bytes = size_t(ROWS) * D * 2;
  static constexpr size_t kv_bytes = size_t(2) * KT * D * 2;  // one of K or V, two stages
  static constexpr size_t key_bytes = size_t(2) * KT * 4;
  static constexpr size_t total = q_bytes + 2 * kv_bytes + key_bytes;
};

__device__ __forceinline__ void window_bounds(const AttnArgs& a, int b, int qi, int nrows, int& lo, int& hi) {
  const int64_t t = __ldg(a.q_pos0 + b) + qi;
  const int64_t rp0 = __ldg(a.raw_pos0 + b);
  int64_t plo = t - a.W + 1;
  if (plo < 0) plo = 0;
  int64_t l = plo - rp0, h = t - rp0 + 1;
  if (l < 0) l = 0;
  if (h > nrows) h = nrows;
  if (h < l) h = l;
  lo = static_cast<int>(l);
  hi = static_cast<int>(h);
}

template <int MODE>
__device__ __forceinline__ void attn_row_bounds(const AttnArgs& a, int b, int qi, bool valid, int& lo, int& hi) {
  lo = 0;
  hi = 0;
  if (!valid) return;
  if (MODE == ATT_GATHER) {
    hi = a.k;
    return;
  }
  if (MODE == ATT_RANGE) {
    hi = visible_entries(__ldg(a.q_pos0 + b) + qi, a.m, __ldg(a.n_valid + b), a.Ncap);
  } else {
    window_bounds(a, b, qi, a.Ncap, lo, hi);
  }
}

// One warp, 16 query rows (this lane holds rows g and g+8 of its quad
// layout) against one KT-key tile of K/V in shared memory (rows of D bf16,
// 16-byte chunks XOR-swizzled by key & 7).  Keys with keyv[kk] < 0 or with
// tile position j0+kk outside a row's [lo, hi) are masked.  Online softmax in
// the log2 domain: m = running max of scale*log2(e)*q.k, l = running sum of
// 2^(z - m), oacc = unnormalised output.
// Element offset of 16-byte chunk cc of key row `key` in a K/V tile.  Plain
// layout: rows of D elements, chunks XOR-swizzled by key & 7.  Split layout
// (what TMA writes with 128-byte swizzling from tensor maps whose box is 64
// columns wide): the tile is stored as D/64 halves of KT rows x 128 bytes,
// chunk c of a half at position c ^ (key & 7) -- the same swizzle per half.
template <int D, int KT, bool SPLIT>
__device__ __forceinline__ int kv_off(int key, int cc) {
  if constexpr (SPLIT) return (cc >> 3) * KT * 64 + key * 64 + (((cc & 7) ^ (key & 7)) * 8);
  else return key * D + ((cc ^ (key & 7)) * 8);
}

template <int D, int KT = 64, bool SPLIT = false>
__device__ __forceinline__ void attn_tile_step(const uint32_t (&qf)[D / 16][4], const bf16* tK, const bf16* tV,
                                               const int* keyv, int j0, int lA, int hA, int lB, int hB,
                                               float scale_log2, float& m0, float& m1, float& l0, float& l1,
                                               float (&oacc)[D / 8][4]) {
  constexpr int NKS = D / 16, NDT = D / 8, NN = KT / 8;
  static_assert(KT % 16 == 0, "tiles of whole 16-key steps");
  const int lane = threadIdx.x & 31, c4 = lane & 3;
  float s[NN][4];
#pragma unroll
  for (int n = 0; n < NN; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < NKS; ++ks) {
#pragma unroll
    for (int p = 0; p < KT / 16; ++p) {
      const int key = 16 * p + (lane & 7) + ((lane >> 4) & 1) * 8;
      const int cc = 2 * ks + ((lane >> 3) & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(smem_u32(tK + kv_off<D, KT, SPLIT>(key, cc)), b0, b1, b2, b3);
      mma_bf16(s[2 * p], qf[ks], b0, b1);
      mma_bf16(s[2 * p + 1], qf[ks], b2, b3);
    }
  }
  // mask, scale, row max
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int n = 0; n < NN; ++n) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int kk = 8 * n + 2 * c4 + (e & 1);
      const int jg = j0 + kk;
      const bool keyok = keyv[kk] >= 0;
      const bool ok = keyok && (e < 2 ? (jg >= lA && jg < hA) : (jg >= lB && jg < hB));
      const float v = ok ? s[n][e] * scale_log2 : -INFINITY;
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
  for (int n = 0; n < NN; ++n) {
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
  for (int ks = 0; ks < KT / 16; ++ks) {
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
      ldsm_x4_t(smem_u32(tV + kv_off<D, KT, SPLIT>(key, cc)), b0, b1, b2, b3);
      mma_bf16(oacc[2 * p], pa, b0, b1);
      mma_bf16(oacc[2 * p + 1], pa, b2, b3);
    }
  }
}

template <int D, int ROWS, int MODE, bool WIN2>
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
  __shared__ int s_lo, s_hi, s_lo2, s_hi2;

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

  if (tid == 0) { s_lo = INT_MAX; s_hi = INT_MIN; s_lo2 = INT_MAX; s_hi2 = INT_MIN; }
  __syncthreads();
  const int rA = warp * 16 + g, rB = rA + 8;
  int qA, hA, qB, hB, loA, hiA, loB, hiB;
  int wloA = 0, whiA = 0, wloB = 0, whiB = 0;
  const bool vA = row_qh(rA, qA, hA), vB = row_qh(rB, qB, hB);
  attn_row_bounds<MODE>(a, b, qA, vA, loA, hiA);
  attn_row_bounds<MODE>(a, b, qB, vB, loB, hiB);
  if (WIN2) {
    if (vA) window_bounds(a, b, qA, a.Ncap2, wloA, whiA);
    if (vB) window_bounds(a, b, qB, a.Ncap2, wloB, whiB);
  }
  if (c4 == 0) {
    if (vA && hiA > loA) { atomicMin(&s_lo, loA); atomicMax(&s_hi, hiA); }
    if (vB && hiB > loB) { atomicMin(&s_lo, loB); atomicMax(&s_hi, hiB); }
    if (WIN2 && vA && whiA > wloA) { atomicMin(&s_lo2, wloA); atomicMax(&s_hi2, whiA); }
    if (WIN2 && vB && whiB > wloB) { atomicMin(&s_lo2, wloB); atomicMax(&s_hi2, whiB); }
  }
  __syncthreads();
  // the key tiles of source 1 followed by those of source 2; split z takes a contiguous run
  const int T1 = s_hi > s_lo ? (s_hi - s_lo + KT - 1) / KT : 0;
  const int T2 = (WIN2 && s_hi2 > s_lo2) ? (s_hi2 - s_lo2 + KT - 1) / KT : 0;
  const int per_z = (T1 + T2 + a.nsplit - 1) / a.nsplit;
  const int t_first = z * per_z;
  const int ntiles = max(0, min(T1 + T2, t_first + per_z) - t_first);
  auto tile_start = [&](int tt, int& src, int& j0, int& jend) {
    if (tt < T1) { src = 0; j0 = s_lo + tt * KT; jend = s_hi; }
    else { src = 1; j0 = s_lo2 + (tt - T1) * KT; jend = s_hi2; }
  };

  // ---- async loads ----
  const int64_t qrow_base = MODE == ATT_GATHER ? (static_cast<int64_t>(b) * a.Tq + qi_cta) : 0;
  for (int u = tid; u < ROWS * CPR; u += NT) {
    const int r = u / CPR, cc = u % CPR;
    int qi, h;
    const bool v = row_qh(r, qi, h);
    const bf16* src = a.q + ((static_cast<int64_t>(b) * a.Tq + (v ? qi : 0)) * a.H + (v ? h : 0)) * D + cc * 8;
    cp_async16(smem_u32(sQ + r * D + ((cc ^ (r & 7)) * 8)), src, v ? 16 : 0);
  }
  // Thread tid copies 16-byte chunk (tid % CPR) of key rows tid / CPR + r * RPI:
  // all its row indices are resolved (gathered) first, then all copies issue.
  constexpr int RPI = NT / CPR;    // key rows covered per pass
  constexpr int NPASS = KT / RPI;
  static_assert(NT % CPR == 0 && KT % RPI == 0, "copy layout");
  auto load_kv = [&](int tt, int st) {
    int src_id, j0, jend;
    tile_start(tt, src_id, j0, jend);
    const int cc = tid % CPR, kk0 = tid / CPR;
    int ev[NPASS];
#pragma unroll
    for (int r = 0; r < NPASS; ++r) {
      const int j = j0 + kk0 + r * RPI;
      int e = -1;
      if (j < jend) {
        if (MODE == ATT_GATHER && src_id == 0) {
          e = __ldg(a.idx + qrow_base * a.k + j);
          if (e >= a.Ncap || e < -1) {
            record_error(DEV_ERR_INDEX, static_cast<unsigned>(j));
            e = -1;
          }
        } else {
          e = j;
        }
      }
      ev[r] = e;
    }
    const bf16* Kb = src_id == 0 ? a.K + b * a.kv_bs : a.K2 + b * a.kv2_bs;
    const bf16* Vb = src_id == 0 ? a.V + b * a.kv_bs : a.V2 + b * a.kv2_bs;
    const int64_t rs = src_id == 0 ? a.kv_rs : a.kv2_rs;
#pragma unroll
    for (int r = 0; r < NPASS; ++r) {
      const int kk = kk0 + r * RPI, e = ev[r];
      const int64_t off = e >= 0 ? static_cast<int64_t>(e) * rs + cc * 8 : 0;
      const int so = st * KT * D + kk * D + ((cc ^ (kk & 7)) * 8);
      cp_async16(smem_u32(sK + so), Kb + off, e >= 0 ? 16 : 0);
      cp_async16(smem_u32(sV + so), Vb + off, e >= 0 ? 16 : 0);
      if (cc == 0) sKey[st * KT + kk] = e;
    }
  };
  pdl_trigger();
  pdl_wait();  // index lists (and anything else) from the previous kernel are complete
  if (ntiles > 0) load_kv(t_first, 0);
  cp_async_commit();

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float oacc[NDT][4];
#pragma unroll
  for (int n = 0; n < NDT; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
  uint32_t qf[NKS][4];

  for (int t = 0; t < ntiles; ++t) {
    const int st = t & 1;
    int src_id, j0, jend;
    tile_start(t_first + t, src_id, j0, jend);
    const int lA = src_id ? wloA : loA, hA_ = src_id ? whiA : hiA;
    const int lB = src_id ? wloB : loB, hB_ = src_id ? whiB : hiB;
    if (t + 1 < ntiles) {
      load_kv(t_first + t + 1, st ^ 1);
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
    attn_tile_step<D>(qf, sK + st * KT * D, sV + st * KT * D, sKey + st * KT, j0, lA, hA_, lB, hB_, a.scale_log2,
                      m0, m1, l0, l1, oacc);
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
  const bool to_bf16 = a.out_bf16 != nullptr && a.nsplit == 1;
  if (vA) {
    const int64_t r = zoff + grow(qA, hA);
    if (to_bf16) {
      bf16* o = a.out_bf16 + r * D;
#pragma unroll
      for (int n = 0; n < NDT; ++n)
        *reinterpret_cast<uint32_t*>(o + 8 * n + 2 * c4) = pack_bf16(oacc[n][0] * inv0, oacc[n][1] * inv0);
    } else {
      float* o = a.O + r * D;
#pragma unroll
      for (int n = 0; n < NDT; ++n)
        *reinterpret_cast<float2*>(o + 8 * n + 2 * c4) = make_float2(oacc[n][0] * inv0, oacc[n][1] * inv0);
    }
    if (c4 == 0 && a.lse) a.lse[r] = l0 > 0.f ? (m0 + log2f(l0)) * LN2 : -INFINITY;
  }
  if (vB) {
    const int64_t r = zoff + grow(qB, hB);
    if (to_bf16) {
      bf16* o = a.out_bf16 + r * D;
#pragma unroll
      for (int n = 0; n < NDT; ++n)
        *reinterpret_cast<uint32_t*>(o + 8 * n + 2 * c4) = pack_bf16(oacc[n][2] * inv1, oacc[n][3] * inv1);
    } else {
      float* o = a.O + r * D;
#pragma unroll
      for (int n = 0; n < NDT; ++n)
        *reinterpret_cast<float2*>(o + 8 * n + 2 * c4) = make_float2(oacc[n][2] * inv1, oacc[n][3] * inv1);
    }
    if (c4 == 0 && a.lse) a.lse[r] = l1 > 0.f ? (m1 + log2f(l1)) * LN2 : -INFINITY;
  }
}


// ---------------------------------------------------------------------------
// Short key lists (a decode step of a CSA layer: k selected entries plus the
// window): one CTA per (query, 16 heads).  Its NW warps share the 16 query
// rows and split the key tiles of the concatenated list (compressed source,
// then window rows); each warp runs the online softmax over its tiles, then
// the warps' (m, l, O) states are combined in shared memory and the layer
// output is written as bf16.  No partials leave the CTA.
template <int D, int NW, int KT>
struct WsplitSmem {
  static constexpr size_t q_bytes = size_t(16) * D * 2;
  static constexpr size_t kv_bytes = size_t(KT) * D * 2;          // one of K or V, one warp
  static constexpr size_t tile_bytes = (2 * kv_bytes + KT * 4 + 127) / 128 * 128;  // K, V, key ids of a warp
  static constexpr int CS = D + 8;  // combine row stride (floats): conflict-free float2 stores of the MMA layout
  static constexpr size_t comb_bytes = size_t(NW) * 16 * (CS + 2) * 4;
  static constexpr size_t work = NW * tile_bytes > comb_bytes ? NW * tile_bytes : comb_bytes;
  static constexpr size_t total = q_bytes + work;
};

template <int D, int MODE, bool WIN2, int NW, int KT>
__global__ void __launch_bounds__(NW * 32) k_attn_wsplit(AttnArgs a) {
  constexpr int CPR = D / 8;
  constexpr int NKS = D / 16, NDT = D / 8;
  using S = WsplitSmem<D, NW, KT>;
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  uint8_t* work = smem + S::q_bytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c4 = lane & 3;
  const int hblocks = (a.H + 15) / 16;
  const int qi = blockIdx.x / hblocks, h0 = (blockIdx.x % hblocks) * 16;
  const int b = blockIdx.y;
  bf16* sK = reinterpret_cast<bf16*>(work + warp * S::tile_bytes);
  bf16* sV = reinterpret_cast<bf16*>(work + warp * S::tile_bytes + S::kv_bytes);
  int* sKey = reinterpret_cast<int*>(work + warp * S::tile_bytes + 2 * S::kv_bytes);

  // key ranges (every row of the CTA is the same query)
  int lo1, hi1, lo2 = 0, hi2 = 0;
  attn_row_bounds<MODE>(a, b, qi, true, lo1, hi1);
  if (WIN2) window_bounds(a, b, qi, a.Ncap2, lo2, hi2);
  const int T1 = hi1 > lo1 ? (hi1 - lo1 + KT - 1) / KT : 0;
  const int T2 = (WIN2 && hi2 > lo2) ? (hi2 - lo2 + KT - 1) / KT : 0;
  const int64_t qrow = static_cast<int64_t>(b) * a.Tq + qi;

  // queries of the 16 heads (zeros for heads >= H)
  for (int u = tid; u < 16 * CPR; u += NW * 32) {
    const int r = u / CPR, cc = u % CPR;
    const bool v = h0 + r < a.H;
    const bf16* src = a.q + (qrow * a.H + (v ? h0 + r : 0)) * D + cc * 8;
    cp_async16(smem_u32(sQ + r * D + ((cc ^ (r & 7)) * 8)), src, v ? 16 : 0);
  }
  cp_async_commit();

  // one tile into this warp's buffers: lane covers chunk (lane % CPR) of rows lane / CPR + r * RPW
  constexpr int RPW = 32 / CPR;
  constexpr int NPASS = KT / RPW;
  auto load_tile = [&](int tt) {
    const bool w = tt >= T1;
    const int j0 = w ? lo2 + (tt - T1) * KT : lo1 + tt * KT;
    const int jend = w ? hi2 : hi1;
    const int cc = lane % CPR, kk0 = lane / CPR;
    int ev[NPASS];
#pragma unroll
    for (int r = 0; r < NPASS; ++r) {
      const int j = j0 + kk0 + r * RPW;
      int e = -1;
      if (j < jend) {
        if (MODE == ATT_GATHER && !w) {
          e = __ldg(a.idx + qrow * a.k + j);
          if (e >= a.Ncap || e < -1) {
            record_error(DEV_ERR_INDEX, static_cast<unsigned>(j));
            e = -1;
          }
        } else {
          e = j;
        }
      }
      ev[r] = e;
    }
    const bf16* Kb = w ? a.K2 + b * a.kv2_bs : a.K + b * a.kv_bs;
    const bf16* Vb = w ? a.V2 + b * a.kv2_bs : a.V + b * a.kv_bs;
    const int64_t rs = w ? a.kv2_rs : a.kv_rs;
#pragma unroll
    for (int r = 0; r < NPASS; ++r) {
      const int kk = kk0 + r * RPW, e = ev[r];
      const int64_t off = e >= 0 ? static_cast<int64_t>(e) * rs + cc * 8 : 0;
      const int so = kk * D + ((cc ^ (kk & 7)) * 8);
      cp_async16(smem_u32(sK + so), Kb + off, e >= 0 ? 16 : 0);
      cp_async16(smem_u32(sV + so), Vb + off, e >= 0 ? 16 : 0);
      if (cc == 0) sKey[kk] = e;
    }
    cp_async_commit();
    return j0;
  };

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float oacc[NDT][4];
#pragma unroll
  for (int n = 0; n < NDT; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
  uint32_t qf[NKS][4];
  int j0 = 0;
  pdl_trigger();
  // window rows are inputs of the call; index lists may come from the previous kernel
  if (warp < T1 + T2 && warp >= T1) j0 = load_tile(warp);
  pdl_wait();
  if (warp < T1) j0 = load_tile(warp);
  cp_async_wait<0>();
  __syncthreads();  // queries visible to every warp
#pragma unroll
  for (int ks = 0; ks < NKS; ++ks) {
    const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int cc = 2 * ks + (lane >> 4);
    ldsm_x4(smem_u32(sQ + r * D + ((cc ^ (r & 7)) * 8)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
  }
  for (int tt = warp; tt < T1 + T2; tt += NW) {
    if (tt != warp) {
      __syncwarp();
      j0 = load_tile(tt);
      cp_async_wait<0>();
    }
    __syncwarp();
    const bool w = tt >= T1;
    attn_tile_step<D, KT>(qf, sK, sV, sKey, j0, w ? lo2 : lo1, w ? hi2 : hi1, w ? lo2 : lo1, w ? hi2 : hi1,
                          a.scale_log2, m0, m1, l0, l1, oacc);
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // ---- combine the warps' states ----
  __syncthreads();  // all tiles consumed: the work area becomes the combine area
  constexpr int CS = S::CS;
  float* cO = reinterpret_cast<float*>(work);                    // [NW][16][CS]
  float* cM = cO + NW * 16 * CS;                                 // [NW][16]
  float* cL = cM + NW * 16;                                      // [NW][16]
#pragma unroll
  for (int n = 0; n < NDT; ++n) {
    *reinterpret_cast<float2*>(cO + (warp * 16 + g) * CS + 8 * n + 2 * c4) = make_float2(oacc[n][0], oacc[n][1]);
    *reinterpret_cast<float2*>(cO + (warp * 16 + g + 8) * CS + 8 * n + 2 * c4) = make_float2(oacc[n][2], oacc[n][3]);
  }
  if (c4 == 0) {
    cM[warp * 16 + g] = m0; cL[warp * 16 + g] = l0;
    cM[warp * 16 + g + 8] = m1; cL[warp * 16 + g + 8] = l1;
  }
  __syncthreads();
  constexpr int TPR = NW * 32 / 16;      // threads per row
  constexpr int DPT = D / TPR;           // dims per thread
  static_assert(DPT % 2 == 0, "bf16 pairs");
  const int r = tid / TPR, d0 = (tid % TPR) * DPT;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) M = fmaxf(M, cM[w * 16 + r]);
  float L = 0.f, wt[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    wt[w] = (M == -INFINITY || cL[w * 16 + r] == 0.f) ? 0.f : exp2f(cM[w * 16 + r] - M);
    L += wt[w] * cL[w * 16 + r];
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  if (h0 + r < a.H) {
    const int64_t orow = qrow * a.H + h0 + r;
    bf16* o = a.out_bf16 + orow * D + d0;
    // each thread reads its DPT consecutive floats of every warp's row as one vector
    float x[DPT];
#pragma unroll
    for (int d = 0; d < DPT; ++d) x[d] = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* src = cO + (w * 16 + r) * CS + d0;
      if constexpr (DPT == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        x[0] = fmaf(wt[w], v.x, x[0]); x[1] = fmaf(wt[w], v.y, x[1]);
        x[2] = fmaf(wt[w], v.z, x[2]); x[3] = fmaf(wt[w], v.w, x[3]);
      } else {
#pragma unroll
        for (int d = 0; d < DPT; d += 2) {
          const float2 v = *reinterpret_cast<const float2*>(src + d);
          x[d] = fmaf(wt[w], v.x, x[d]); x[d + 1] = fmaf(wt[w], v.y, x[d + 1]);
        }
      }
    }
#pragma unroll
    for (int d = 0; d < DPT; d += 2) *reinterpret_cast<uint32_t*>(o + d) = pack_bf16(x[d] * inv, x[d + 1] * inv);
    if (a.lse && tid % TPR == 0) a.lse[orow] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
}

}  // namespace lcc
