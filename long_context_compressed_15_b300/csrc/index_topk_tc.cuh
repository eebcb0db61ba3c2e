// Lightning-indexer scores with the top-k fused into the epilogue (prefill
// form).  Source: "DeepSeek-V4가 이차적 어텐션 비용 없이 ...", section "두 가지
// 압축 전략: CSA 및 HCA" (a light indexer scores the compressed entries for
// each query and keeps the top-k, typically about 128).
//
// Prefill form with the top-k fused into the epilogue: no scores leave the
// CTA.  Entries arrive in increasing index order, so for every query the CTA
// keeps a candidate buffer (key, index) and a threshold theta = the k-th
// largest key kept so far; an entry enters the buffer only if its key is
// strictly greater (a later entry with an equal key has a higher index and
// loses every tie).  A buffer that could overflow within the next tile is
// compacted by one warp to its exact top-k, which raises theta.  At the end
// each query's top-k is written in ascending index order.
#pragma once
#include "index_tc.cuh"

namespace lcc {

namespace ftk {

// k-th largest of the warp's keys held as v[i] = key of element lane + 32*i
// (0 for none), by a bitwise radix select.
template <int CAPQ>
__device__ __forceinline__ uint32_t warp_kth(const uint32_t (&v)[CAPQ / 32], int k) {
  uint32_t prefix = 0u;
  int need = k;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t hi_mask = bit == 31 ? 0u : ~((2u << bit) - 1u);
    int c = 0;
#pragma unroll
    for (int i = 0; i < CAPQ / 32; ++i) c += ((v[i] & hi_mask) == prefix) && ((v[i] >> bit) & 1u);
    c = __reduce_add_sync(0xffffffffu, c);
    if (c >= need) prefix |= 1u << bit;
    else need -= c;
  }
  return prefix;
}

// Keep the top-k of a query's buffer (key desc, index asc); returns the new
// count (min(n, k)) and sets *theta to the k-th key when n >= k.  One warp.
// Every register array is indexed by compile-time constants (unrolled
// loops), so it stays in registers.
template <int CAPQ>
__device__ __forceinline__ int warp_compact(uint32_t* keys, int32_t* ids, int n, int k, uint32_t* theta) {
  constexpr int V = CAPQ / 32;
  const int lane = threadIdx.x & 31;
  if (n <= k) return n;
  uint32_t v[V];
  int32_t id[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < n ? keys[e] : 0u;
    id[i] = e < n ? ids[e] : 0x7FFFFFFF;
  }
  const uint32_t T = warp_kth<CAPQ>(v, k);
  int gt = 0, eq = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) { gt += v[i] > T; eq += v[i] == T; }
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  const int need_eq = k - gt;
  // which of my entries are kept: keys above T, and the need_eq lowest indices
  // among keys equal to T (counted from the buffer itself; only when some
  // ties must be dropped, which needs exactly equal scores)
  uint32_t keepm = 0u;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    bool keep = v[i] > T;
    if (v[i] == T) {
      if (eq == need_eq) {
        keep = true;
      } else {
        int before = 0;
        for (int e2 = 0; e2 < n; ++e2) before += (keys[e2] == T) && (ids[e2] < id[i]);
        keep = before < need_eq;
      }
    }
    keepm |= (keep ? 1u : 0u) << i;
  }
  __syncwarp();  // every lane has read the buffer before it is overwritten
  int out = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const bool keep = (keepm >> i) & 1u;
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int p = out + __popc(m & ((1u << lane) - 1u));
      keys[p] = v[i];
      ids[p] = id[i];
    }
    out += __popc(m);
  }
  __syncwarp();
  if (lane == 0) *theta = T;
  return k;
}

}  // namespace ftk

struct IndexTopkTcArgs {
  const bf16* qI;
  const float* w;
  int B, Tq;
  const int64_t* q_pos0;
  const int32_t* n_valid;
  int Ncap, m, k;
  int32_t* idx;      // [B, Tq, k]
  float* score;      // optional [B, Tq, k]
};

template <int HI, int DI, int NQ, int STAGES>
struct IndexTopkTcCfg {
  using Base = IndexTcCfg<HI, DI, NQ, STAGES>;
  // candidate slots per query (128 KB of buffers in all) and the number of
  // tiles between buffer checks: a buffer is compacted once it could not
  // take SYNC more tiles
  static constexpr int CAPQ = NQ <= 16 ? 1024 : 512;
  static constexpr int SYNC = NQ <= 16 ? 4 : 2;
  static constexpr int OFF_KEYS = (Base::OFF_BAR + Base::NBAR * 8 + 64 + 1023) / 1024 * 1024;
  static constexpr int OFF_IDS = OFF_KEYS + NQ * CAPQ * 4;
  static constexpr int OFF_ST = OFF_IDS + NQ * CAPQ * 4;   // theta[NQ], cnt[NQ]
  static constexpr int SMEM = OFF_ST + NQ * 8 + 1024;
};

// Threads: warp 0 TMA, warp 1 TMEM allocation + MMA, warps 2..9 epilogue.
// Epilogue warp e reads TMEM lanes 32*(e%4).. (its warp id mod 4) and owns
// the queries of half e/4 (NQ/2 queries, NQ*HI/2 accumulator columns).
template <int HI, int DI, int NQ, int STAGES>
__global__ void __launch_bounds__(320, 1) k_index_topk_tc(const __grid_constant__ CUtensorMap tmap_k, IndexTopkTcArgs a) {
  using C = IndexTcCfg<HI, DI, NQ, STAGES>;
  using X = IndexTopkTcCfg<HI, DI, NQ, STAGES>;
  constexpr int NEPI = 256;              // epilogue threads
  constexpr int QH = NQ / 2;             // queries per epilogue half
  constexpr int COLS = QH * HI;          // accumulator columns per half (64)
  static_assert(C::NREAL == C::N && COLS % 32 == 0, "whole 32-column loads");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  float* sW = reinterpret_cast<float*>(smem + C::OFF_W);
  int* sVis = reinterpret_cast<int*>(smem + C::OFF_VIS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint32_t* sKeys = reinterpret_cast<uint32_t*>(smem + X::OFF_KEYS);  // [NQ][CAPQ]
  int32_t* sIds = reinterpret_cast<int32_t*>(smem + X::OFF_IDS);      // [NQ][CAPQ]
  uint32_t* sTheta = reinterpret_cast<uint32_t*>(smem + X::OFF_ST);   // [NQ]
  int* sCnt = reinterpret_cast<int*>(smem + X::OFF_ST + NQ * 4);      // [NQ]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  // heavy (late) query groups first: they see the most entries
  const int grp = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);
  const int qg0 = grp * NQ;
  const int qend = min(qg0 + NQ, a.Tq);
  const int64_t pos0 = __ldg(a.q_pos0 + b);
  const int nval = __ldg(a.n_valid + b);
  const int vis_max = visible_entries(pos0 + qend - 1, a.m, nval, a.Ncap);
  const int vis_min = visible_entries(pos0 + qg0, a.m, nval, a.Ncap);
  const int ntiles = (vis_max + C::TILE - 1) / C::TILE;
  const int k = a.k;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) { tc::mbar_init(full + i, 1); tc::mbar_init(empty + i, 1); }
    for (int i = 0; i < 2; ++i) { tc::mbar_init(tfull + i, 1); tc::mbar_init(tempty + i, NEPI); }
    *s_abort = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  const int row0 = b * a.Ncap;
  if (warp == 0 && lane == 0 && ntiles > 0) {
    tc::tma_prefetch_desc(&tmap_k);
    for (int t = 0; t < min(STAGES, ntiles); ++t) {
      tc::mbar_arrive_expect_tx(full + t, C::A_BYTES);
      tc::tma_load_2d(sA + t * C::A_BYTES, &tmap_k, full + t, 0, row0 + t * C::TILE);
    }
  }
  if (warp == 1) tc::tmem_alloc(s_tmem, C::TMEM_COLS);
  if (warp >= 2) {
    const int t = threadIdx.x - 64;
    constexpr int CPR = DI / 8;
    for (int u = t; u < C::N * CPR; u += NEPI) {
      const int n = u / CPR, c = u % CPR;
      const int qq = qg0 + n / HI, hh = n % HI;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (qq < qend)
        v = __ldg(reinterpret_cast<const uint4*>(a.qI + ((static_cast<int64_t>(b) * a.Tq + qq) * HI + hh) * DI) + c);
      const int sw = C::ROWB == 128 ? (c ^ (n & 7)) : (c ^ ((n & 7) >> 1));
      *reinterpret_cast<uint4*>(sB + (n >> 3) * C::SBO + (n & 7) * C::ROWB + sw * 16) = v;
    }
    for (int u = t; u < NQ * HI; u += NEPI) {
      const int qq = qg0 + u / HI;
      sW[u] = qq < qend ? __ldg(a.w + (static_cast<int64_t>(b) * a.Tq + qq) * HI + u % HI) : 0.f;
    }
    for (int u = t; u < NQ; u += NEPI) {
      const int qq = qg0 + u;
      sVis[u] = qq < qend ? visible_entries(pos0 + qq, a.m, nval, a.Ncap) : 0;
      sTheta[u] = 0u;
      sCnt[u] = 0;
    }
    tc::fence_proxy_async_smem();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    int issued = min(STAGES, ntiles);
    if (lane == 0) {
      for (int t = STAGES; t < ntiles; ++t) {
        const int s = t % STAGES;
        if (*s_abort || !tc::mbar_wait(empty + s, ((t / STAGES) & 1) ^ 1, 21)) { *s_abort = 1; break; }
        tc::mbar_arrive_expect_tx(full + s, C::A_BYTES);
        tc::tma_load_2d(sA + s * C::A_BYTES, &tmap_k, full + s, 0, row0 + t * C::TILE);
        issued = t + 1;
      }
      for (int t = max(0, issued - STAGES); t < issued; ++t)
        tc::mbar_wait(full + t % STAGES, (t / STAGES) & 1, 22);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % STAGES, acc = t & 1;
        if (*s_abort || !tc::mbar_wait(tempty + acc, ((t >> 1) & 1) ^ 1, 23)) { *s_abort = 1; break; }
        if (*s_abort || !tc::mbar_wait(full + s, (t / STAGES) & 1, 24)) { *s_abort = 1; break; }
        tc::tc_fence_after();
        const uint32_t d = tmem + acc * C::N;
#pragma unroll
        for (int kk = 0; kk < DI / 16; ++kk) {
          const uint64_t ad = tc::smem_desc(a_base + s * C::A_BYTES + kk * 32, 16, C::SBO, C::SWZ);
          const uint64_t bd = tc::smem_desc(b_base + kk * 32, 16, C::SBO, C::SWZ);
          tc::mma_f16_ss(d, ad, bd, C::IDESC, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(empty + s);
        tc::mma_commit(tfull + acc);
        issued = t + 1;
      }
      if (issued > 0) tc::mbar_wait(tfull + ((issued - 1) & 1), ((issued - 1) >> 1) & 1, 25);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue + streaming top-k
    const int ew = warp - 2;        // epilogue warp 0..7
    const int quarter = warp & 3;   // TMEM lanes 32*quarter .. +31
    const int half = ew >> 2;       // queries [half*QH, half*QH + QH)
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + half * COLS;
    // this warp's queries: head weights and visible counts are fixed for the
    // CTA, thresholds change only at buffer checks -- all kept in registers
    // the threshold test runs on floats: key(s) > key(theta) <=> s > f(theta)
    // with f(0) = -inf (no threshold yet); keys are formed only for entries taken
    const float4* sW4 = reinterpret_cast<const float4*>(sW) + half * QH * HI / 4;  // broadcast reads
    int visr[QH];
    float thf[QH];
#pragma unroll
    for (int j = 0; j < QH; ++j) {
      visr[j] = sVis[half * QH + j];
      thf[j] = -INFINITY;
    }
    for (int t = 0; t < ntiles; ++t) {
      const int acc = t & 1;
      // After a failed wait a warp keeps looping without work (later waits are
      // skipped), so the eight epilogue warps still meet at every named barrier.
      const bool wok = __all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(tfull + acc, (t >> 1) & 1, 26));
      if (!wok) *s_abort = 1;
      if (wok) {
      tc::tc_fence_after();
      float v[COLS];
#pragma unroll
      for (int c = 0; c < COLS / 32; ++c) {
        float x[32];
        tc::tmem_ld32(lane_addr + acc * C::N + c * 32, x);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[c * 32 + i] = x[i];
      }
      tc::tmem_wait_ld();
      tc::tc_fence_before();
      tc::mbar_arrive(tempty + acc);  // the accumulator is in registers: the next MMA may start
      const int entry = t * C::TILE + quarter * 32 + lane;
      const bool all_vis = (t + 1) * C::TILE <= vis_min;  // every query sees the whole tile
      float sc[QH];
      bool any = false;
#pragma unroll
      for (int j = 0; j < QH; ++j) {
        float s = 0.f;
#pragma unroll
        for (int h4 = 0; h4 < HI / 4; ++h4) {
          const float4 wv = sW4[j * HI / 4 + h4];
          s = fmaf(wv.x, fmaxf(v[j * HI + 4 * h4 + 0], 0.f), s);
          s = fmaf(wv.y, fmaxf(v[j * HI + 4 * h4 + 1], 0.f), s);
          s = fmaf(wv.z, fmaxf(v[j * HI + 4 * h4 + 2], 0.f), s);
          s = fmaf(wv.w, fmaxf(v[j * HI + 4 * h4 + 3], 0.f), s);
        }
        sc[j] = (all_vis || entry < visr[j]) ? s : -INFINITY;
        any |= sc[j] > thf[j];
      }
      if (__any_sync(0xffffffffu, any)) {  // some entry of this warp passes a threshold
#pragma unroll
        for (int j = 0; j < QH; ++j) {
          const int qi = half * QH + j;
          const bool take = sc[j] > thf[j];
          const unsigned msk = __ballot_sync(0xffffffffu, take);
          if (msk) {
            const int leader = __ffs(msk) - 1;
            int base = 0;
            if (lane == leader) base = atomicAdd(sCnt + qi, __popc(msk));
            base = __shfl_sync(0xffffffffu, base, leader);
            if (take) {
              const int slot = base + __popc(msk & ((1u << lane) - 1u));
              if (slot < X::CAPQ) {  // cannot fail: buffers keep room for SYNC whole tiles
                sKeys[qi * X::CAPQ + slot] = f32_to_key(sc[j]);
                sIds[qi * X::CAPQ + slot] = entry;
              }
            }
          }
        }
      }
      }  // wok
      if ((t + 1) % X::SYNC == 0 || t + 1 == ntiles) {
        // every append so far is in place; shrink buffers that could overflow before the next check
        tc::named_sync(1, NEPI);
        for (int qi = ew; qi < NQ && !*s_abort; qi += 8) {
          const int n = sCnt[qi];
          if (n > X::CAPQ - X::SYNC * C::TILE) {
            const int nk =
                ftk::warp_compact<X::CAPQ>(sKeys + qi * X::CAPQ, sIds + qi * X::CAPQ, n, k, sTheta + qi);
            if (lane == 0) sCnt[qi] = nk;
          }
        }
        tc::named_sync(1, NEPI);
#pragma unroll
        for (int j = 0; j < QH; ++j) {
          const uint32_t th = sTheta[half * QH + j];
          thf[j] = th == 0u ? -INFINITY : key_to_f32(th);
        }
      }
    }
    // ---- final: exact top-k of every query, in ascending index order ----
    for (int qi = ew; qi < NQ; qi += 8) {
      const int q = qg0 + qi;
      if (q >= qend) continue;
      int n = sCnt[qi];
      if (*s_abort) n = 0;
      uint32_t* kq = sKeys + qi * X::CAPQ;
      int32_t* iq = sIds + qi * X::CAPQ;
      n = ftk::warp_compact<X::CAPQ>(kq, iq, n, k, sTheta + qi);
      __syncwarp();
      int32_t* oi = a.idx + (static_cast<int64_t>(b) * a.Tq + q) * k;
      float* os = a.score ? a.score + (static_cast<int64_t>(b) * a.Tq + q) * k : nullptr;
      for (int c = lane; c < k; c += 32) {
        if (c < n) {
          const int32_t me = iq[c];
          int p = 0;
          for (int d = 0; d < n; ++d) p += iq[d] < me;
          oi[p] = me;
          if (os) os[p] = key_to_f32(kq[c]);
        } else {
          oi[c] = -1;
          if (os) os[c] = -INFINITY;
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace lcc
