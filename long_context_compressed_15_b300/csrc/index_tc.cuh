// Lightning-indexer scores on the 5th-generation tensor cores:
//   s[q, j] = sum_h w[q,h] * max(0, qI[q,h,:] . kI[j,:])
// for every visible compressed entry j.  Source: "DeepSeek-V4가 이차적 어텐션
// 비용 없이 ...", section "두 가지 압축 전략: CSA 및 HCA" (a light indexer scores
// the compressed entries for each query and keeps the top-k).
//
// The contraction kI[entries x DI] . qI^T[DI x (query, head)] runs as
// tcgen05.mma with M = 128 entries per tile and N = NQ*HI (query, head)
// columns, so that one TMEM lane holds every head of every query for one
// entry and the ReLU-weighted head sum needs no cross-thread traffic.
// Roles (192 threads):
//   warp 0      TMA producer: streams 128-entry key tiles into a ring of
//               STAGES swizzled shared-memory buffers;
//   warp 1      allocates TMEM, issues the MMAs (one thread) into two
//               accumulator buffers, releases key buffers through
//               tcgen05.commit;
//   warps 2..5  epilogue: TMEM -> registers, ReLU, head weights, head sum,
//               coalesced score stores.  Also stage the indexer queries (B
//               operand) and head weights once per CTA.
#pragma once
#include "tc.cuh"

namespace lcc {

struct IndexTcArgs {
  const bf16* qI;   // [B, Tq, HI, DI]
  const float* w;   // [B, Tq, HI]
  int B, Tq;
  const int64_t* q_pos0;
  const int32_t* n_valid;
  int Ncap, m;
  int q0, nq;       // query chunk [q0, q0 + nq)
  int tiles_per_split;
  float* scores;    // [B * nq, Ncap]: row (b, i - q0)
  uint32_t* gmax;   // optional [B * nq, g_stride]: key of the largest score of each 32-entry group
  int g_stride;
  int* counters;    // optional [2, B * nq]: zeroed here for the top-k kernel that follows
};

template <int HI, int DI, int NQ, int STAGES>
struct IndexTcCfg {
  static constexpr int TILE = 128;
  static constexpr int NREAL = NQ * HI;
  static constexpr int N = NREAL < 16 ? 16 : (NREAL + 15) / 16 * 16;
  static_assert(N <= 256, "at most 256 MMA columns");
  static constexpr int ROWB = DI * 2;                   // bytes per key row
  static constexpr uint64_t SWZ = ROWB == 128 ? tc::SW_128B : tc::SW_64B;
  static constexpr uint32_t SBO = 8 * ROWB;             // one 8-row swizzle atom
  static constexpr int A_BYTES = TILE * ROWB;
  static constexpr int B_BYTES = N * ROWB;
  static constexpr int TMEM_COLS = (2 * N <= 32) ? 32 : (2 * N <= 64) ? 64 : (2 * N <= 128) ? 128
                                   : (2 * N <= 256) ? 256 : 512;
  // shared memory carve-up (1024-byte aligned operand buffers)
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_W = OFF_B + (B_BYTES + 1023) / 1024 * 1024;
  static constexpr int OFF_VIS = OFF_W + (NQ * HI * 4 + 15) / 16 * 16;
  static constexpr int OFF_BAR = OFF_VIS + (NQ * 4 + 15) / 16 * 16;
  static constexpr int NBAR = 2 * STAGES + 4;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;  // + alignment slack
  static constexpr uint32_t IDESC = tc::idesc_f16(128, N, true);
};

template <int HI, int DI, int NQ, int STAGES>
__global__ void __launch_bounds__(192, 1) k_index_tc(const __grid_constant__ CUtensorMap tmap_k, IndexTcArgs a) {
  using C = IndexTcCfg<HI, DI, NQ, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  float* sW = reinterpret_cast<float*>(smem + C::OFF_W);
  int* sVis = reinterpret_cast<int*>(smem + C::OFF_VIS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;                 // [STAGES] key tile landed
  uint64_t* empty = bars + STAGES;       // [STAGES] key tile consumed by the MMA
  uint64_t* tfull = bars + 2 * STAGES;   // [2] accumulator ready
  uint64_t* tempty = bars + 2 * STAGES + 2;  // [2] accumulator drained
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  // launched as a programmatic dependent of whatever ran before on the
  // stream: nothing is read before that grid has completed
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int qg0 = a.q0 + blockIdx.y * NQ;                   // first query of this CTA
  const int qend = min(qg0 + NQ, a.q0 + a.nq);              // one past the last
  const int64_t pos0 = __ldg(a.q_pos0 + b);
  const int nval = __ldg(a.n_valid + b);
  const int vis_max = visible_entries(pos0 + qend - 1, a.m, nval, a.Ncap);
  const int ntiles_vis = (vis_max + C::TILE - 1) / C::TILE;
  const int t_lo = blockIdx.x * a.tiles_per_split;
  const int t_hi = min(t_lo + a.tiles_per_split, ntiles_vis);
  if (t_lo >= t_hi) return;  // uniform across the CTA
  const int ntiles = t_hi - t_lo;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) { tc::mbar_init(full + i, 1); tc::mbar_init(empty + i, 1); }
    for (int i = 0; i < 2; ++i) { tc::mbar_init(tfull + i, 1); tc::mbar_init(tempty + i, 128); }
    *s_abort = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  const int row0 = b * a.Ncap + t_lo * C::TILE;
  if (warp == 0 && lane == 0) {
    // start streaming keys before the rest of the set-up
    tc::tma_prefetch_desc(&tmap_k);
    for (int t = 0; t < min(STAGES, ntiles); ++t) {
      tc::mbar_arrive_expect_tx(full + t, C::A_BYTES);
      tc::tma_load_2d(sA + t * C::A_BYTES, &tmap_k, full + t, 0, row0 + t * C::TILE);
    }
  }
  if (warp == 1) tc::tmem_alloc(s_tmem, C::TMEM_COLS);
  if (warp >= 2) {
    // B operand: row n = (query n / HI, head n % HI), K-major, swizzled like the TMA tiles
    const int t = threadIdx.x - 64;
    constexpr int CPR = DI / 8;  // 16-byte chunks per row
    for (int u = t; u < C::N * CPR; u += 128) {
      const int n = u / CPR, c = u % CPR;
      const int qq = qg0 + n / HI, hh = n % HI;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (n < C::NREAL && qq < qend)
        v = __ldg(reinterpret_cast<const uint4*>(a.qI + ((static_cast<int64_t>(b) * a.Tq + qq) * HI + hh) * DI) + c);
      const int sw = C::ROWB == 128 ? (c ^ (n & 7)) : (c ^ ((n & 7) >> 1));
      *reinterpret_cast<uint4*>(sB + (n >> 3) * C::SBO + (n & 7) * C::ROWB + sw * 16) = v;
    }
    for (int u = t; u < NQ * HI; u += 128) {
      const int qq = qg0 + u / HI;
      sW[u] = qq < qend ? __ldg(a.w + (static_cast<int64_t>(b) * a.Tq + qq) * HI + u % HI) : 0.f;
    }
    for (int u = t; u < NQ; u += 128) {
      const int qq = qg0 + u;
      sVis[u] = qq < qend ? visible_entries(pos0 + qq, a.m, nval, a.Ncap) : 0;
      if (a.counters && blockIdx.x == 0 && qq < qend) {
        const int64_t r = static_cast<int64_t>(b) * a.nq + (qq - a.q0);
        a.counters[r] = 0;
        a.counters[static_cast<int64_t>(a.B) * a.nq + r] = 0;
      }
    }
    tc::fence_proxy_async_smem();  // generic-proxy writes of B -> visible to the tensor core
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_trigger();  // the top-k that follows may start launching (it waits for this grid)

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    int issued = min(STAGES, ntiles);
    if (lane == 0) {
      for (int t = STAGES; t < ntiles; ++t) {
        const int s = t % STAGES;
        if (*s_abort || !tc::mbar_wait(empty + s, ((t / STAGES) & 1) ^ 1, 1)) { *s_abort = 1; break; }
        tc::mbar_arrive_expect_tx(full + s, C::A_BYTES);
        tc::tma_load_2d(sA + s * C::A_BYTES, &tmap_k, full + s, 0, row0 + t * C::TILE);
        issued = t + 1;
      }
      // copies still in flight must land before the CTA may exit
      for (int t = max(0, issued - STAGES); t < issued; ++t)
        tc::mbar_wait(full + t % STAGES, (t / STAGES) & 1, 2);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % STAGES, acc = t & 1;
        if (*s_abort || !tc::mbar_wait(tempty + acc, ((t >> 1) & 1) ^ 1, 3)) { *s_abort = 1; break; }
        if (*s_abort || !tc::mbar_wait(full + s, (t / STAGES) & 1, 4)) { *s_abort = 1; break; }
        tc::tc_fence_after();
        const uint32_t d = tmem + acc * C::N;
#pragma unroll
        for (int k = 0; k < DI / 16; ++k) {
          const uint64_t ad = tc::smem_desc(a_base + s * C::A_BYTES + k * 32, 16, C::SBO, C::SWZ);
          const uint64_t bd = tc::smem_desc(b_base + k * 32, 16, C::SBO, C::SWZ);
          tc::mma_f16_ss(d, ad, bd, C::IDESC, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(empty + s);
        tc::mma_commit(tfull + acc);
        issued = t + 1;
      }
      if (issued > 0) tc::mbar_wait(tfull + ((issued - 1) & 1), ((issued - 1) >> 1) & 1, 5);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    for (int t = 0; t < ntiles; ++t) {
      const int acc = t & 1;
      // the TMEM loads below are warp-collective: leave the loop as a whole warp
      if (!__all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(tfull + acc, (t >> 1) & 1, 6))) {
        *s_abort = 1;
        break;
      }
      tc::tc_fence_after();
      const int entry = (t_lo + t) * C::TILE + quarter * 32 + lane;
      constexpr int QPC = 8 / HI < 1 ? 1 : 8 / HI;  // queries per 8-column load
      constexpr int NCH = (C::NREAL + 7) / 8;
#pragma unroll 4
      for (int ch = 0; ch < NCH; ++ch) {
        float v[8];
        tc::tmem_ld8(lane_addr + acc * C::N + ch * 8, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int qq = 0; qq < QPC; ++qq) {
          const int qi = ch * QPC + qq;
          const int q = qg0 + qi;
          if (qi < NQ && q < qend) {  // uniform across the warp
            float s = 0.f;
#pragma unroll
            for (int h = 0; h < HI; ++h) s = fmaf(sW[qi * HI + h], fmaxf(v[qq * HI + h], 0.f), s);
            const int vis = sVis[qi];
            const int64_t r = static_cast<int64_t>(b) * a.nq + (q - a.q0);
            if (entry < vis) a.scores[r * a.Ncap + entry] = s;
            if (a.gmax) {
              const uint32_t key = __reduce_max_sync(0xffffffffu, entry < vis ? f32_to_key(s) : 0u);
              const int g0 = entry - lane;
              if (lane == 0 && g0 < vis) a.gmax[r * a.g_stride + (g0 >> 5)] = key;
            }
          }
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(tempty + acc);
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
