// CSA layer attention for decode-sized calls with the selected entries
// gathered by TMA.  Source: "DeepSeek-V4가 이차적 어텐션 비용 없이 ...", section
// "두 가지 압축 전략: CSA 및 HCA" (each query attends with MQA to its top-k
// compressed entries; a sliding-window branch over the most recent raw tokens
// runs in parallel -- here one softmax over the union of the two key lists).
//
// The structure is k_attn_wsplit's: one CTA per (query, 16 heads), NW warps
// that split the key tiles of the concatenated list (selected entries, then
// window rows), an online softmax per warp, the warps' states combined in
// shared memory, bf16 out.  What differs is how a selected-entry tile
// arrives: lanes 0..KT/4-1 of the warp each read four entry numbers of the
// index list and issue TMA tile::gather4 copies (four rows per copy, one per
// 64-column half of K and of V) from tensor maps whose box is one 64-column
// row, swizzled by 128 bytes; the warp waits on its own mbarrier (bounded).
// The window rows, which are inputs of the call rather than products of the
// top-k, are loaded with cp.async before the programmatic-launch wait.
#pragma once
#include "attn.cuh"
#include "attn_gather_tc.cuh"

namespace lcc {

template <int NW, int KT, int NB = 1>
struct WsplitTmaSmem {
  static constexpr int D = 128;
  static constexpr size_t q_bytes = 16 * D * 2;                           // 4 KB, 1024-aligned region
  static constexpr size_t tile_bytes = size_t(2) * KT * D * 2;            // K and V of one warp tile
  static constexpr int CS = D + 8;
  static constexpr size_t comb_bytes = size_t(NW) * 16 * (CS + 2) * 4;
  static constexpr size_t work = NW * NB * tile_bytes > comb_bytes ? NW * NB * tile_bytes : comb_bytes;
  static constexpr size_t off_work = (q_bytes + 1023) / 1024 * 1024;
  static constexpr size_t off_keys = off_work + (work + 1023) / 1024 * 1024;
  static constexpr size_t off_bars = off_keys + NW * NB * KT * 4;
  static constexpr size_t total = off_bars + NW * 8 + 1024;               // + alignment slack
};

// The attention of query qi of sequence b for heads h0 .. h0+15 by one CTA
// of NW warps; smem is the CTA's 1024-aligned WsplitTmaSmem area.  The index
// list comes from global memory (a.idx) or, with SIDX, from shared memory
// (sidx[0..k)).  between() runs after the window rows and queries are
// requested and before the index list is read: it waits for whatever
// produces the list.
//
// NB = 2 (every warp holds one selected-entry tile and one window tile, the
// caller guarantees T1, T2 <= NW): a warp's window tile is requested before
// between() and attended while its selected rows are still being gathered.
template <int NW, int KT, bool SIDX, int NB = 1, class Between>
__device__ __forceinline__ void attn_wsplit_tma_body(const CUtensorMap* tmK, const CUtensorMap* tmV,
                                                     const AttnArgs& a, uint8_t* smem, int qi, int h0, int b,
                                                     const int* sidx, Between& between) {
  constexpr int D = 128, CPR = D / 8, NKS = D / 16, NDT = D / 8;
  static_assert(KT % 4 == 0 && KT / 4 <= 32, "four rows per gather, one lane per gather");
  static_assert(NB == 1 || NB == 2, "one or two tile buffers per warp");
  using S = WsplitTmaSmem<NW, KT, NB>;
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  uint8_t* work = smem + S::off_work;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c4 = lane & 3;
  auto buf_k = [&](int bi) { return reinterpret_cast<bf16*>(work + (warp * NB + bi) * S::tile_bytes); };
  auto buf_key = [&](int bi) { return reinterpret_cast<int*>(smem + S::off_keys) + (warp * NB + bi) * KT; };
  bf16* sK = buf_k(0);
  bf16* sV = sK + KT * D;
  int* sKey = buf_key(0);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + S::off_bars) + warp;

  int lo2 = 0, hi2 = 0;
  window_bounds(a, b, qi, a.Ncap2, lo2, hi2);
  const int T1 = (a.k + KT - 1) / KT;
  const int T2 = hi2 > lo2 ? (hi2 - lo2 + KT - 1) / KT : 0;
  const int64_t qrow = static_cast<int64_t>(b) * a.Tq + qi;

  if (lane == 0) {
    tc::mbar_init(bar, 1);
    tc::fence_barrier_init();
  }
  __syncwarp();
  // queries of the 16 heads (zeros for heads >= H)
  for (int u = tid; u < 16 * CPR; u += NW * 32) {
    const int r = u / CPR, cc = u % CPR;
    const bool v = h0 + r < a.H;
    const bf16* src = a.q + (qrow * a.H + (v ? h0 + r : 0)) * D + cc * 8;
    cp_async16(smem_u32(sQ + r * D + ((cc ^ (r & 7)) * 8)), src, v ? 16 : 0);
  }
  cp_async_commit();

  // a window tile (plain layout) into this warp's buffers with cp.async
  constexpr int RPW = 32 / CPR;
  constexpr int NPASS = KT / RPW;
  auto load_window = [&](int tt) {
    const int j0 = lo2 + (tt - T1) * KT;
    const int cc = lane % CPR, kk0 = lane / CPR;
    const bf16* Kb = a.K2 + b * a.kv2_bs;
    const bf16* Vb = a.V2 + b * a.kv2_bs;
#pragma unroll
    for (int r = 0; r < NPASS; ++r) {
      const int kk = kk0 + r * RPW, j = j0 + kk;
      const int e = j < hi2 ? j : -1;
      const int64_t off = e >= 0 ? static_cast<int64_t>(e) * a.kv2_rs + cc * 8 : 0;
      const int so = kk * D + ((cc ^ (kk & 7)) * 8);
      cp_async16(smem_u32(sK + so), Kb + off, e >= 0 ? 16 : 0);
      cp_async16(smem_u32(sV + so), Vb + off, e >= 0 ? 16 : 0);
      if (cc == 0) sKey[kk] = e;
    }
    cp_async_commit();
    return j0;
  };
  // a selected-entry tile (split layout) by TMA gather4: lane l < KT/4 takes list slots 4l .. 4l+3
  int tma_uses = 0;
  auto load_gather = [&](int tt) {
    const int j0 = tt * KT;
    int rows[4] = {0, 0, 0, 0};
    if (lane < KT / 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + 4 * lane + u;
        int e = -1;
        if (j < a.k) {
          e = SIDX ? sidx[j] : __ldg(a.idx + qrow * a.k + j);
          if (e >= a.Ncap || e < -1) {
            record_error(DEV_ERR_INDEX, static_cast<unsigned>(j));
            e = -1;
          }
        }
        sKey[4 * lane + u] = e;
        rows[u] = b * a.Ncap + (e >= 0 ? e : 0);  // an empty slot fetches entry 0, masked later
      }
    }
    if (lane == 0) tc::mbar_arrive_expect_tx(bar, KT * D * 2 * 2);
    __syncwarp();
    if (lane < KT / 4) {
      uint8_t* kb = reinterpret_cast<uint8_t*>(sK);
      uint8_t* vb = reinterpret_cast<uint8_t*>(sV);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int dst = h * KT * 128 + 4 * lane * 128;
        gtc::tma_gather4(kb + dst, tmK, bar, h * 64, rows[0], rows[1], rows[2], rows[3]);
        gtc::tma_gather4(vb + dst, tmV, bar, h * 64, rows[0], rows[1], rows[2], rows[3]);
      }
    }
    return j0;
  };

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float oacc[NDT][4];
#pragma unroll
  for (int n = 0; n < NDT; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
  uint32_t qf[NKS][4];
  int j0 = 0;
  pdl_trigger();
  if constexpr (NB == 2) {
    int jw = 0;
    sK = buf_k(1);
    sV = sK + KT * D;
    sKey = buf_key(1);
    if (warp < T2) jw = load_window(T1 + warp);  // an input of the call: requested before the wait
    between();
    sK = buf_k(0);
    sV = sK + KT * D;
    sKey = buf_key(0);
    if (warp < T1) j0 = load_gather(warp);
    cp_async_wait<0>();
    __syncthreads();  // queries visible to every warp
#pragma unroll
    for (int ks = 0; ks < NKS; ++ks) {
      const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int cc = 2 * ks + (lane >> 4);
      ldsm_x4(smem_u32(sQ + r * D + ((cc ^ (r & 7)) * 8)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }
    if (warp < T2)  // the window tile first, while the gather is in flight
      attn_tile_step<D, KT, false>(qf, buf_k(1), buf_k(1) + KT * D, buf_key(1), jw, lo2, hi2, lo2, hi2,
                                   a.scale_log2, m0, m1, l0, l1, oacc);
    if (warp < T1) {
      tc::mbar_wait(bar, 0, 31);  // bounded; a timeout is recorded for lcc_sync_status
      __syncwarp();
      attn_tile_step<D, KT, true>(qf, buf_k(0), buf_k(0) + KT * D, buf_key(0), j0, 0, a.k, 0, a.k, a.scale_log2,
                                  m0, m1, l0, l1, oacc);
    }
  }
  // window rows are inputs of the call; index lists come later
  if (NB == 1 && warp < T1 + T2 && warp >= T1) j0 = load_window(warp);
  if constexpr (NB == 1) between();
  if (NB == 1 && warp < T1) j0 = load_gather(warp);
  if constexpr (NB == 1) {
    cp_async_wait<0>();
    __syncthreads();  // queries visible to every warp
#pragma unroll
    for (int ks = 0; ks < NKS; ++ks) {
      const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int cc = 2 * ks + (lane >> 4);
      ldsm_x4(smem_u32(sQ + r * D + ((cc ^ (r & 7)) * 8)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }
  }
  for (int tt = warp; NB == 1 && tt < T1 + T2; tt += NW) {
    const bool gath = tt < T1;
    if (tt != warp) {
      __syncwarp();
      j0 = gath ? load_gather(tt) : load_window(tt);
    }
    if (gath) {
      tc::mbar_wait(bar, tma_uses & 1, 31);  // bounded; a timeout is recorded for lcc_sync_status
      ++tma_uses;
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    if (gath)
      attn_tile_step<D, KT, true>(qf, sK, sV, sKey, j0, 0, a.k, 0, a.k, a.scale_log2, m0, m1, l0, l1, oacc);
    else
      attn_tile_step<D, KT, false>(qf, sK, sV, sKey, j0, lo2, hi2, lo2, hi2, a.scale_log2, m0, m1, l0, l1, oacc);
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
    float x[DPT];
#pragma unroll
    for (int d = 0; d < DPT; ++d) x[d] = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* src = cO + (w * 16 + r) * CS + d0;
#pragma unroll
      for (int d = 0; d < DPT; d += 2) {
        const float2 v = *reinterpret_cast<const float2*>(src + d);
        x[d] = fmaf(wt[w], v.x, x[d]); x[d + 1] = fmaf(wt[w], v.y, x[d + 1]);
      }
    }
#pragma unroll
    for (int d = 0; d < DPT; d += 2) *reinterpret_cast<uint32_t*>(o + d) = pack_bf16(x[d] * inv, x[d + 1] * inv);
    if (a.lse && tid % TPR == 0) a.lse[orow] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
}

template <int NW, int KT, int NB = 1>
__global__ void __launch_bounds__(NW * 32) k_attn_wsplit_tma(const __grid_constant__ CUtensorMap tmK,
                                                             const __grid_constant__ CUtensorMap tmV, AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  const int hblocks = (a.H + 15) / 16;
  const int qi = blockIdx.x / hblocks, h0 = (blockIdx.x % hblocks) * 16;
  auto wait_lists = []() { pdl_wait(); };  // index lists may come from the previous kernel
  attn_wsplit_tma_body<NW, KT, false, NB>(&tmK, &tmV, a, smem, qi, h0, static_cast<int>(blockIdx.y), nullptr,
                                          wait_lists);
}

}  // namespace lcc
