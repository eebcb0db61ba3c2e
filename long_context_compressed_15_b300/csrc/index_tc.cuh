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
  const uint8_t* kI_fp4;   // NVFP4 keys [B, Ncap, DI/2] (k_index_tc_fp4 only)
  const uint8_t* kI_scale; // their e4m3 scales [B, Ncap, DI/16]
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
  static constexpr int NBAR = 2 * STAGES + 8;          // full, empty, up to 4 accumulators ready / drained
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;  // + alignment slack
  static constexpr uint32_t IDESC = tc::idesc_f16(128, N, true);
};

template <int HI, int DI, int NQ, int STAGES>
__global__ void __maxnreg__(48) k_index_tc(const __grid_constant__ CUtensorMap tmap_k, IndexTcArgs a) {
  using C = IndexTcCfg<HI, DI, NQ, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  float* sW = reinterpret_cast<float*>(smem + C::OFF_W);
  int* sVis = reinterpret_cast<int*>(smem + C::OFF_VIS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;                 // [STAGES] key tile landed
  uint64_t* empty = bars + STAGES;       // [STAGES] key tile consumed by the MMA
  // accumulators in TMEM: four when they are narrow (the MMA may run three tiles
  // ahead of the epilogue), two at N = 128 (three CTAs per SM share 512 columns)
  constexpr int NACC = C::N <= 64 ? 4 : 2;
  constexpr uint32_t TMEM_COLS = NACC * C::N <= 32 ? 32 : NACC * C::N <= 64 ? 64 : NACC * C::N <= 128 ? 128 : 256;
  static_assert(NACC * C::N <= 256 && (2 * STAGES + 2 * NACC) * 8 + 8 <= C::NBAR * 8 + 16, "TMEM / barrier room");
  uint64_t* tfull = bars + 2 * STAGES;   // [NACC] accumulator ready
  uint64_t* tempty = tfull + NACC;       // [NACC] accumulator drained
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(tempty + NACC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // set-up that reads nothing a previous kernel may write (barriers, TMEM
  // columns, the tensor map's descriptor) runs before the launch wait, so it
  // overlaps the previous kernel when this CTA is launched early
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) { tc::mbar_init(full + i, 1); tc::mbar_init(empty + i, 1); }
    for (int i = 0; i < NACC; ++i) { tc::mbar_init(tfull + i, 1); tc::mbar_init(tempty + i, 128); }
    *s_abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) tc::tma_prefetch_desc(&tmap_k);
  if (warp == 1) tc::tmem_alloc(s_tmem, TMEM_COLS);
  // launched as a programmatic dependent of whatever ran before on the
  // stream: nothing else is read before that grid has completed
  pdl_wait();
  const int b = blockIdx.z;
  const int qg0 = a.q0 + blockIdx.y * NQ;                   // first query of this CTA
  const int qend = min(qg0 + NQ, a.q0 + a.nq);              // one past the last
  const int64_t pos0 = __ldg(a.q_pos0 + b);
  const int nval = __ldg(a.n_valid + b);
  const int vis_max = visible_entries(pos0 + qend - 1, a.m, nval, a.Ncap);
  const int ntiles_vis = (vis_max + C::TILE - 1) / C::TILE;
  const int t_lo = blockIdx.x * a.tiles_per_split;
  const int t_hi = min(t_lo + a.tiles_per_split, ntiles_vis);
  if (t_lo >= t_hi) {  // uniform across the CTA: give the TMEM columns back
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc::tc_fence_after();
      tc::tmem_dealloc(*s_tmem, TMEM_COLS);
    }
    return;
  }
  const int ntiles = t_hi - t_lo;

  __syncthreads();  // barriers initialised
  const int row0 = b * a.Ncap + t_lo * C::TILE;
  const int drop = warp == 0 && lane == 0 ? *static_cast<volatile int*>(&tc::g_test_drop_tile) : -1;
  if (warp == 0 && lane == 0) {
    // start streaming keys before the rest of the set-up
    for (int t = 0; t < min(STAGES, ntiles); ++t) {
      if (t == drop) continue;  // test hook: this tile's barrier never completes
      tc::mbar_arrive_expect_tx(full + t, C::A_BYTES);
      tc::tma_load_2d(sA + t * C::A_BYTES, &tmap_k, full + t, 0, row0 + t * C::TILE);
    }
  }
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
        issued = t + 1;
        if (t == drop) continue;
        tc::mbar_arrive_expect_tx(full + s, C::A_BYTES);
        tc::tma_load_2d(sA + s * C::A_BYTES, &tmap_k, full + s, 0, row0 + t * C::TILE);
      }
      // copies still in flight must land before the CTA may exit (a dropped
      // tile's wait runs out instead: nothing of it is in flight)
      for (int t = max(0, issued - STAGES); t < issued; ++t)
        if (t != drop) tc::mbar_wait(full + t % STAGES, (t / STAGES) & 1, 2);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % STAGES, acc = t % NACC;
        if (*s_abort || !tc::mbar_wait(tempty + acc, ((t / NACC) & 1) ^ 1, 3)) { *s_abort = 1; break; }
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
      if (issued > 0) tc::mbar_wait(tfull + ((issued - 1) % NACC), ((issued - 1) / NACC) & 1, 5);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    for (int t = 0; t < ntiles; ++t) {
      const int acc = t % NACC;
      // the TMEM loads below are warp-collective: leave the loop as a whole warp
      if (!__all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(tfull + acc, (t / NACC) & 1, 6))) {
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
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}


// ---------------------------------------------------------------------------
// NVFP4 keys on the tensor cores.  The keys stream as packed e2m1 pairs (32
// bytes per entry) plus one e4m3 scale per 16 elements (4 bytes per entry):
// 36 bytes instead of 128.  Roles (320 threads):
//   warp 0      producer: bulk copies of 128-entry packed tiles (4 KB) and
//               their scales (512 B) into a ring of raw buffers;
//   warp 1      TMEM allocation; one thread issues tcgen05.mma (kind::f16,
//               fp16 operands) from a ring of converted buffers;
//   warps 2..5  epilogue as k_index_tc; they also stage the indexer queries;
//   warps 6..9  converters: one thread per entry of a tile expands its 64
//               values to fp16 -- e2m1 -> fp16 (cvt) times the group's
//               e4m3 scale (exact: the product has at most 6 significant
//               bits and lies within fp16's normal range) -- into the
//               128-byte-swizzled K-major layout of the MMA's A operand.
// The indexer query is bf16, which fp16 cannot hold as it stands (8 exponent
// bits against 5).  Each (query, head) row is multiplied by the power of two
// that brings its largest element just under 2^15, which makes every element
// within a factor 2^31 of that largest one exact in fp16, and the head weight
// is multiplied by the inverse power: a power-of-two scale commutes with fp32
// rounding, so ReLU(2^s q.k) * (2^-s w) equals ReLU(q.k) * w exactly.
template <int DI>
struct IndexTcFp4Cfg {
  static constexpr int TILE = 128;
  static constexpr int PACK_BYTES = TILE * DI / 2;      // packed values of a tile
  static constexpr int RAW_BYTES = PACK_BYTES + TILE * DI / 16;   // + their scales
  static constexpr int ROWB = DI * 2;                   // converted row (fp16)
  static constexpr int A_BYTES = TILE * ROWB;
};

template <int HI, int DI, int NQ, int SR, int SC>
struct IndexTcFp4Smem {
  using F = IndexTcFp4Cfg<DI>;
  using C = IndexTcCfg<HI, DI, NQ, 1>;
  static constexpr int N = C::N;
  static constexpr int OFF_A = 0;                                      // SC converted tiles
  static constexpr int OFF_B = OFF_A + SC * F::A_BYTES;                // queries (fp16, scaled)
  static constexpr int OFF_RAW = OFF_B + (C::B_BYTES + 1023) / 1024 * 1024;
  static constexpr int OFF_W = OFF_RAW + SR * F::RAW_BYTES;
  static constexpr int OFF_VIS = OFF_W + (NQ * HI * 4 + 15) / 16 * 16;
  static constexpr int OFF_BAR = OFF_VIS + (NQ * 4 + 15) / 16 * 16;
  // accumulators: four narrow ones (N <= 64), else two (two CTAs per SM share 512 columns)
  static constexpr int NACC = N <= 64 ? 4 : 2;
  static constexpr uint32_t TMEM_COLS = NACC * N <= 32 ? 32 : NACC * N <= 64 ? 64 : NACC * N <= 128 ? 128 : 256;
  static constexpr int NBAR = 2 * SR + 2 * SC + 2 * NACC;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
  static constexpr uint32_t IDESC = tc::idesc_f16(128, N, false);     // fp16 x fp16 -> fp32
  static constexpr uint32_t SBO = 8 * F::ROWB;
};

template <int HI, int DI, int NQ, int SR, int SC>
__global__ void __launch_bounds__(320, 2) k_index_tc_fp4(IndexTcArgs a) {
  using F = IndexTcFp4Cfg<DI>;
  using S = IndexTcFp4Smem<HI, DI, NQ, SR, SC>;
  using C = IndexTcCfg<HI, DI, NQ, 1>;
  static_assert(DI == 64, "NVFP4 keys: DI = 64 (one 128-byte swizzle row per converted entry)");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint8_t* sA = smem + S::OFF_A;
  uint8_t* sB = smem + S::OFF_B;
  uint8_t* sRaw = smem + S::OFF_RAW;
  float* sW = reinterpret_cast<float*>(smem + S::OFF_W);
  int* sVis = reinterpret_cast<int*>(smem + S::OFF_VIS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  uint64_t* rfull = bars;                    // [SR] packed tile landed
  uint64_t* rempty = bars + SR;              // [SR] packed tile read by the converters
  uint64_t* cfull = bars + 2 * SR;           // [SC] converted tile written
  uint64_t* cempty = bars + 2 * SR + SC;     // [SC] converted tile consumed by the MMA
  constexpr int NACC = S::NACC;
  uint64_t* tfull = bars + 2 * SR + 2 * SC;  // [NACC] accumulator ready
  uint64_t* tempty = tfull + NACC;           // [NACC] accumulator drained
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + S::NBAR);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int qg0 = a.q0 + blockIdx.y * NQ;
  const int qend = min(qg0 + NQ, a.q0 + a.nq);
  const int64_t pos0 = __ldg(a.q_pos0 + b);
  const int nval = __ldg(a.n_valid + b);
  const int vis_max = visible_entries(pos0 + qend - 1, a.m, nval, a.Ncap);
  const int ntiles_vis = (vis_max + F::TILE - 1) / F::TILE;
  const int t_lo = blockIdx.x * a.tiles_per_split;
  const int t_hi = min(t_lo + a.tiles_per_split, ntiles_vis);
  if (t_lo >= t_hi) return;  // uniform across the CTA
  const int ntiles = t_hi - t_lo;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SR; ++i) { tc::mbar_init(rfull + i, 1); tc::mbar_init(rempty + i, 128); }
    for (int i = 0; i < SC; ++i) { tc::mbar_init(cfull + i, 128); tc::mbar_init(cempty + i, 1); }
    for (int i = 0; i < NACC; ++i) { tc::mbar_init(tfull + i, 1); tc::mbar_init(tempty + i, 128); }
    *s_abort = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  const int64_t row_base = static_cast<int64_t>(b) * a.Ncap;   // entry row of this batch's entry 0
  // rows of tile t (CTA-local), the last one possibly partial
  auto tile_rows = [&](int t) { return min(F::TILE, a.Ncap - (t_lo + t) * F::TILE); };
  // bytes of tile t's scales that one bulk copy moves (a multiple of 16; the
  // scales of the last 1..3 rows of a ragged final tile are read directly)
  // (none when this batch's scale rows do not start on a 16-byte boundary)
  const bool scale_bulk = ((reinterpret_cast<uintptr_t>(a.kI_scale) + row_base * (DI / 16)) & 15) == 0;
  auto scale_bytes = [&](int t) {
    return scale_bulk ? static_cast<uint32_t>(tile_rows(t)) * (DI / 16) & ~15u : 0u;
  };
  auto issue = [&](int t) {
    const int s = t % SR;
    const uint32_t bytes = static_cast<uint32_t>(tile_rows(t)) * (DI / 2), sbytes = scale_bytes(t);
    tc::mbar_arrive_expect_tx(rfull + s, bytes + sbytes);
    const int64_t e0 = row_base + static_cast<int64_t>(t_lo + t) * F::TILE;
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(sRaw + s * F::RAW_BYTES)), "l"(a.kI_fp4 + e0 * (DI / 2)), "r"(bytes),
        "r"(smem_u32(rfull + s))
        : "memory");
    if (sbytes)
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
          ::"r"(smem_u32(sRaw + s * F::RAW_BYTES + F::PACK_BYTES)), "l"(a.kI_scale + e0 * (DI / 16)),
          "r"(sbytes), "r"(smem_u32(rfull + s))
          : "memory");
  };
  if (warp == 0 && lane == 0)
    for (int t = 0; t < min(SR, ntiles); ++t) issue(t);
  if (warp == 1) tc::tmem_alloc(s_tmem, S::TMEM_COLS);
  if (warp >= 2 && warp < 6) {
    // B operand: row n = (query n / HI, head n % HI), fp16 after a power-of-two
    // scale, K-major, swizzled like the converted tiles; head weight times the
    // inverse scale
    const int t = threadIdx.x - 64;
    for (int n = t; n < C::N; n += 128) {
      const int qq = qg0 + n / HI, hh = n % HI;
      const bool live = n < C::NREAL && qq < qend;
      uint4 v[DI / 8];
      int emax = 0;
#pragma unroll
      for (int c = 0; c < DI / 8; ++c) {
        v[c] = live ? __ldg(reinterpret_cast<const uint4*>(a.qI + ((static_cast<int64_t>(b) * a.Tq + qq) * HI + hh) *
                                                                      DI) + c)
                    : make_uint4(0, 0, 0, 0);
        const uint32_t wd[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          emax = max(emax, static_cast<int>((wd[u] >> 7) & 0xFF));
          emax = max(emax, static_cast<int>((wd[u] >> 23) & 0xFF));
        }
      }
      // 2^sc brings the largest element to [2^14, 2^15) (rows of values below
      // 2^-112 stay below that range: 2^sc must remain a finite float)
      const int sc = emax == 0 ? 0 : min(141 - emax, 126);
      const float up = ldexpf(1.0f, sc);
#pragma unroll
      for (int c = 0; c < DI / 8; ++c) {
        const uint32_t wd[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
        uint32_t o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[u]));
          __half2 h = __floats2half2_rn(f.x * up, f.y * up);
          o[u] = *reinterpret_cast<uint32_t*>(&h);
        }
        const int sw = c ^ (n & 7);
        *reinterpret_cast<uint4*>(sB + (n >> 3) * S::SBO + (n & 7) * F::ROWB + sw * 16) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
      if (n < NQ * HI)
        sW[n] = live ? __ldg(a.w + (static_cast<int64_t>(b) * a.Tq + qq) * HI + hh) * ldexpf(1.0f, -sc) : 0.f;
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
    tc::fence_proxy_async_smem();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_trigger();

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    int issued = min(SR, ntiles);
    if (lane == 0) {
      for (int t = SR; t < ntiles; ++t) {
        const int s = t % SR;
        if (*s_abort || !tc::mbar_wait(rempty + s, ((t / SR) & 1) ^ 1, 11)) { *s_abort = 1; break; }
        issue(t);
        issued = t + 1;
      }
      for (int t = max(0, issued - SR); t < issued; ++t) tc::mbar_wait(rfull + t % SR, (t / SR) & 1, 12);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int c = t % SC, acc = t % NACC;
        if (*s_abort || !tc::mbar_wait(tempty + acc, ((t / NACC) & 1) ^ 1, 13)) { *s_abort = 1; break; }
        if (*s_abort || !tc::mbar_wait(cfull + c, (t / SC) & 1, 14)) { *s_abort = 1; break; }
        tc::tc_fence_after();
        const uint32_t d = tmem + acc * C::N;
#pragma unroll
        for (int k = 0; k < DI / 16; ++k) {
          const uint64_t ad = tc::smem_desc(a_base + c * F::A_BYTES + k * 32, 16, S::SBO, tc::SW_128B);
          const uint64_t bd = tc::smem_desc(b_base + k * 32, 16, S::SBO, tc::SW_128B);
          tc::mma_f16_ss(d, ad, bd, S::IDESC, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(cempty + c);
        tc::mma_commit(tfull + acc);
        issued = t + 1;
      }
      if (issued > 0) tc::mbar_wait(tfull + ((issued - 1) % NACC), ((issued - 1) / NACC) & 1, 15);
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ---------------------------------------------------------- converters
    const int r = threadIdx.x - 192;                // entry row within a tile
    for (int t = 0; t < ntiles; ++t) {
      const int s = t % SR, c = t % SC;
      const int64_t e = row_base + static_cast<int64_t>(t_lo + t) * F::TILE + r;
      const bool live = r < tile_rows(t);
      const bool copied = static_cast<uint32_t>(r) * (DI / 16) < scale_bytes(t);
      if (!__all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(rfull + s, (t / SR) & 1, 16))) { *s_abort = 1; break; }
      const uint32_t scales =
          copied ? *reinterpret_cast<const uint32_t*>(sRaw + s * F::RAW_BYTES + F::PACK_BYTES + r * (DI / 16))
                 : (live ? __ldg(reinterpret_cast<const uint32_t*>(a.kI_scale + e * (DI / 16))) : 0u);
      if (!__all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(cempty + c, ((t / SC) & 1) ^ 1, 17))) {
        *s_abort = 1;
        break;
      }
      uint4 p0 = make_uint4(0, 0, 0, 0), p1 = p0;
      if (live) {
        p0 = *reinterpret_cast<const uint4*>(sRaw + s * F::RAW_BYTES + r * (DI / 2));
        p1 = *reinterpret_cast<const uint4*>(sRaw + s * F::RAW_BYTES + r * (DI / 2) + 16);
      }
      tc::mbar_arrive(rempty + s);
      const uint32_t wd[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      uint8_t* dst = sA + c * F::A_BYTES + (r >> 3) * S::SBO + (r & 7) * F::ROWB;
      uint32_t sb[4];  // scale of elements 16g .. 16g+15, both halves
      e4m3x4_to_f16x2_bcast(scales, sb);
#pragma unroll
      for (int ch = 0; ch < DI / 8; ++ch) {       // one packed word = 8 elements = one 16-byte fp16 chunk
        uint32_t h[4];
        e2m1x8_to_f16x2x4(wd[ch], h);
        const uint32_t s2 = sb[ch >> 1];
        uint4 o;
        o.x = hmul2_u32(h[0], s2);
        o.y = hmul2_u32(h[1], s2);
        o.z = hmul2_u32(h[2], s2);
        o.w = hmul2_u32(h[3], s2);
        *reinterpret_cast<uint4*>(dst + ((ch ^ (r & 7)) * 16)) = o;
      }
      tc::fence_proxy_async_smem();   // generic writes -> visible to the tensor core
      tc::mbar_arrive(cfull + c);
    }
  } else {
    // ---------------------------------------------------------- epilogue (warps 2..5)
    const int quarter = warp & 3;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    for (int t = 0; t < ntiles; ++t) {
      const int acc = t % NACC;
      if (!__all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(tfull + acc, (t / NACC) & 1, 18))) {
        *s_abort = 1;
        break;
      }
      tc::tc_fence_after();
      const int entry = (t_lo + t) * F::TILE + quarter * 32 + lane;
      constexpr int QPC = 8 / HI < 1 ? 1 : 8 / HI;
      constexpr int NCH = (C::NREAL + 7) / 8;
      static_assert(NCH % 2 == 0, "columns in pairs of 8-column chunks");
#pragma unroll 2
      for (int ch2 = 0; ch2 < NCH; ch2 += 2) {
        // two 8-column chunks per TMEM round trip
        float v16[16];
        tc::tmem_ld16(lane_addr + acc * C::N + ch2 * 8, v16);
        tc::tmem_wait_ld();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int ch = ch2 + half;
          const float* v = v16 + half * 8;
#pragma unroll
          for (int qq = 0; qq < QPC; ++qq) {
            const int qi = ch * QPC + qq;
            const int q = qg0 + qi;
            if (qi < NQ && q < qend) {
              float sc = 0.f;
#pragma unroll
              for (int h = 0; h < HI; ++h) sc = fmaf(sW[qi * HI + h], fmaxf(v[qq * HI + h], 0.f), sc);
              const int vis = sVis[qi];
              const int64_t rr = static_cast<int64_t>(b) * a.nq + (q - a.q0);
              if (entry < vis) a.scores[rr * a.Ncap + entry] = sc;
              if (a.gmax) {
                const uint32_t key = __reduce_max_sync(0xffffffffu, entry < vis ? f32_to_key(sc) : 0u);
                const int g0 = entry - lane;
                if (lane == 0 && g0 < vis) a.gmax[rr * a.g_stride + (g0 >> 5)] = key;
              }
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
    tc::tmem_dealloc(tmem, S::TMEM_COLS);
  }
}

}  // namespace lcc
