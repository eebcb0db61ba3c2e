// Multi-query flash attention on the 5th-generation tensor cores for long
// query blocks (prefill): HCA dense attention over the visible compressed
// entries and/or the sliding window over raw rows, one online softmax over
// both key sources.  Source: "DeepSeek-V4가 이차적 어텐션 비용 없이 ...", section
// "두 가지 압축 전략: CSA 및 HCA" (MQA with shared KV; HCA attends densely over
// all compressed entries; a window branch runs in parallel).
//
// A CTA owns 128 consecutive (query, head) rows of one sequence -- with 64
// heads that is two queries -- and walks 128-key tiles of the compressed
// source then of the window:
//   warp 4 (TMA)      Q once; K and V tiles (two 64-column swizzled halves
//                     each) into two-stage rings; a K stage is released by
//                     its Q K^T, a V stage by its P V, so the next K tile
//                     streams in while the softmax still runs;
//   warp 5 (MMA)      S[t] = Q K[t]^T into one of two TMEM buffers, then
//                     O += P[t-1] V[t-1] (P from one of two shared-memory
//                     buffers, V as an MN-major operand), O in TMEM;
//   warps 0..3        one thread per row (= TMEM lane): read S, row maximum
//                     (masking only tiles that cross the row's key range),
//                     online softmax in the log2 domain with the scale folded
//                     into one FMA per score, write P (bf16, swizzled) for
//                     the tensor core; at the end O / l to global memory.
// The running maximum is only raised (and O, l rescaled) when a tile's
// maximum exceeds it by more than 8 (a factor 256): P stays <= 2^8, exact
// in the final normalisation, and O is rarely touched.
#pragma once
#include "tc.cuh"
#include "attn.cuh"

namespace lcc {

struct AttnTcArgs {
  int B, Tq, H;
  float scale_log2;
  const int64_t* q_pos0;
  int mode1;          // key source 1: ATT_RANGE (visible entries) or ATT_WINDOW (raw rows); -1 none
  int Ncap1;          // rows per batch of source 1
  const int32_t* n_valid;
  int m;
  bool win2;          // window rows as source 2
  int Ncap2;
  const int64_t* raw_pos0;
  int W;
  bf16* out_bf16;     // [B*Tq*H, D] bf16, or
  float* O;           // [B*Tq*H, D] fp32 with
  float* lse;         // [B*Tq*H] (optional with out_bf16)
  int rpt;            // rows per CTA tile: 128, or H (one query's heads) for decode
  int tps;            // key tiles per split (gridDim.z splits the tile list)
  int64_t rows_total; // B*Tq*H: distance between the fp32 partials of two splits
};

template <int D>
struct AttnTcCfg {
  static constexpr int TILE = 128;            // keys per tile; rows per CTA
  static constexpr int STAGES = 2;
  static constexpr int HALF = 128 * 64 * 2;   // one 64-column swizzled half: 16 KB
  static constexpr int OP = (D / 64) * HALF;  // one 128 x D operand
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + OP;
  static constexpr int OFF_V = OFF_K + STAGES * OP;
  static constexpr int OFF_P = OFF_V + STAGES * OP;
  static constexpr int PB = 2 * HALF;                   // one P buffer: 128 rows x 128 keys
  static constexpr int OFF_BAR = OFF_P + 2 * PB;        // two P buffers
  static constexpr int NBAR = 1 + 4 * STAGES + 2 + 2 + 2 + 2 + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 64 + 1024;
  static constexpr uint32_t IDESC_S = tc::idesc_f16(128, 128, true);            // Q K^T
  static constexpr uint32_t IDESC_O = tc::idesc_f16(128, D, true, false, true); // P V, V MN-major
  static constexpr int TMEM_COLS = 512;       // S: 2 x 128, O: D
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK1,
              const __grid_constant__ CUtensorMap tmV1, const __grid_constant__ CUtensorMap tmK2,
              const __grid_constant__ CUtensorMap tmV2, AttnTcArgs a) {
  using C = AttnTcCfg<D>;
  constexpr float TAU = 8.0f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;                  // [STAGES]
  uint64_t* k_empty = k_full + C::STAGES;       // [STAGES]
  uint64_t* v_full = k_empty + C::STAGES;       // [STAGES]
  uint64_t* v_empty = v_full + C::STAGES;       // [STAGES]
  uint64_t* s_full = v_empty + C::STAGES;       // [2]
  uint64_t* s_free = s_full + 2;                // [2]
  uint64_t* p_full = s_free + 2;                // [2]
  uint64_t* p_free = p_full + 2;                // [2]
  uint64_t* o_full = p_free + 2;                // [1]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_rng = reinterpret_cast<int*>(s_tmem + 2);  // lo1, hi1, lo2, hi2

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int64_t rows_b = static_cast<int64_t>(a.Tq) * a.H;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * a.rpt;  // rows past rpt are padding

  // ---- per-row key ranges (softmax threads own one row each) ----
  int lo1 = 0, hi1 = 0, lo2 = 0, hi2 = 0;
  bool row_ok = false;
  if (warp < 4) {
    const int64_t r = row0 + threadIdx.x;
    row_ok = static_cast<int>(threadIdx.x) < a.rpt && r < rows_b;
    if (row_ok) {
      const int qi = static_cast<int>(r / a.H);
      const int64_t t = __ldg(a.q_pos0 + b) + qi;
      if (a.mode1 == ATT_RANGE) {
        hi1 = visible_entries(t, a.m, __ldg(a.n_valid + b), a.Ncap1);
      } else if (a.mode1 == ATT_WINDOW) {
        int64_t plo = t - a.W + 1;
        if (plo < 0) plo = 0;
        const int64_t rp0 = __ldg(a.raw_pos0 + b);
        int64_t l = plo - rp0, h = t - rp0 + 1;
        if (l < 0) l = 0;
        if (h > a.Ncap1) h = a.Ncap1;
        if (h < l) h = l;
        lo1 = static_cast<int>(l);
        hi1 = static_cast<int>(h);
      }
      if (a.win2) {
        int64_t plo = t - a.W + 1;
        if (plo < 0) plo = 0;
        const int64_t rp0 = __ldg(a.raw_pos0 + b);
        int64_t l = plo - rp0, h = t - rp0 + 1;
        if (l < 0) l = 0;
        if (h > a.Ncap2) h = a.Ncap2;
        if (h < l) h = l;
        lo2 = static_cast<int>(l);
        hi2 = static_cast<int>(h);
      }
    }
  }
  if (threadIdx.x == 0) {
    s_rng[0] = INT_MAX; s_rng[1] = INT_MIN; s_rng[2] = INT_MAX; s_rng[3] = INT_MIN;
    tc::mbar_init(q_full, 1);
    for (int i = 0; i < C::STAGES; ++i) {
      tc::mbar_init(k_full + i, 1); tc::mbar_init(k_empty + i, 1);
      tc::mbar_init(v_full + i, 1); tc::mbar_init(v_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) { tc::mbar_init(s_full + i, 1); tc::mbar_init(s_free + i, 128); }
    for (int i = 0; i < 2; ++i) { tc::mbar_init(p_full + i, 128); tc::mbar_init(p_free + i, 1); }
    tc::mbar_init(o_full, 1);
    *s_abort = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (warp < 4 && row_ok) {
    if (hi1 > lo1) { atomicMin(s_rng + 0, lo1); atomicMax(s_rng + 1, hi1); }
    if (hi2 > lo2) { atomicMin(s_rng + 2, lo2); atomicMax(s_rng + 3, hi2); }
  }
  if (warp == 5) tc::tmem_alloc(s_tmem, C::TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int rlo1 = s_rng[0], rhi1 = s_rng[1], rlo2 = s_rng[2], rhi2 = s_rng[3];
  const int T1 = rhi1 > rlo1 ? (rhi1 - rlo1 + 127) / 128 : 0;
  const int T2 = rhi2 > rlo2 ? (rhi2 - rlo2 + 127) / 128 : 0;
  // this split's run of the tile list (tiles of source 1, then of the window)
  const int tt0 = static_cast<int>(blockIdx.z) * a.tps;
  const int ntiles = max(0, min(T1 + T2, tt0 + a.tps) - tt0);
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sP = smem + C::OFF_P;
  const uint32_t tmem_o = tmem + 256;  // columns 256 .. 256 + D - 1

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      tc::tma_prefetch_desc(&tmQ);
      tc::mbar_arrive_expect_tx(q_full, C::OP);
      const int qy = static_cast<int>(static_cast<int64_t>(b) * rows_b + row0);
      for (int h = 0; h < D / 64; ++h) tc::tma_load_2d(sQ + h * C::HALF, &tmQ, q_full, h * 64, qy);
      // K of tile i, then V of tile i - 1: a V stage frees later (after P V)
      // than a K stage (after Q K^T), so K loads run one tile ahead
      auto tile_y = [&](int tg, const CUtensorMap*& mk, const CUtensorMap*& mv) {
        const bool w = tg >= T1;
        mk = w ? &tmK2 : &tmK1;
        mv = w ? &tmV2 : &tmV1;
        return w ? b * a.Ncap2 + rlo2 + (tg - T1) * 128 : b * a.Ncap1 + rlo1 + tg * 128;
      };
      int ik = 0, iv = 0;
      bool pok = true;
      for (int i = 0; pok && i <= ntiles; ++i) {
        const CUtensorMap *mk, *mv;
        if (i < ntiles) {
          const int s = i % C::STAGES;
          if (*s_abort || !tc::mbar_wait(k_empty + s, ((i / C::STAGES) & 1) ^ 1, 11)) { pok = false; break; }
          tc::mbar_arrive_expect_tx(k_full + s, C::OP);
          const int y = tile_y(tt0 + i, mk, mv);
          for (int h = 0; h < D / 64; ++h) tc::tma_load_2d(sK + s * C::OP + h * C::HALF, mk, k_full + s, h * 64, y);
          ik = i + 1;
        }
        if (i > 0) {
          const int u = i - 1, s = u % C::STAGES;
          if (*s_abort || !tc::mbar_wait(v_empty + s, ((u / C::STAGES) & 1) ^ 1, 11)) { pok = false; break; }
          tc::mbar_arrive_expect_tx(v_full + s, C::OP);
          const int y = tile_y(tt0 + u, mk, mv);
          for (int h = 0; h < D / 64; ++h) tc::tma_load_2d(sV + s * C::OP + h * C::HALF, mv, v_full + s, h * 64, y);
          iv = u + 1;
        }
      }
      if (!pok) *s_abort = 1;
      // every copy this CTA started has landed before it may exit
      tc::mbar_wait(q_full, 0, 12);
      for (int t = max(0, ik - C::STAGES); t < ik; ++t) tc::mbar_wait(k_full + t % C::STAGES, (t / C::STAGES) & 1, 12);
      for (int t = max(0, iv - C::STAGES); t < iv; ++t) tc::mbar_wait(v_full + t % C::STAGES, (t / C::STAGES) & 1, 12);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && ntiles > 0) {
      const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK), va = smem_u32(sV), pa = smem_u32(sP);
      bool ok = tc::mbar_wait(q_full, 0, 13);
      for (int t = 0; ok && t <= ntiles; ++t) {
        if (t < ntiles) {
          const int s = t % C::STAGES, sb = t & 1;
          if (*s_abort || !tc::mbar_wait(k_full + s, (t / C::STAGES) & 1, 14) ||
              !tc::mbar_wait(s_free + sb, ((t >> 1) & 1) ^ 1, 15)) { ok = false; break; }
          tc::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::HALF + (kk & 3) * 32;
            tc::mma_f16_ss(tmem + sb * 128, tc::smem_desc(qa + off, 16, 1024, tc::SW_128B),
                           tc::smem_desc(ka + s * C::OP + off, 16, 1024, tc::SW_128B), C::IDESC_S, kk > 0);
          }
          tc::mma_commit(s_full + sb);
          tc::mma_commit(k_empty + s);
        }
        if (t > 0) {
          const int u = t - 1, su = u % C::STAGES;
          const int pb = u & 1;
          if (*s_abort || !tc::mbar_wait(p_full + pb, (u >> 1) & 1, 16) ||
              !tc::mbar_wait(v_full + su, (u / C::STAGES) & 1, 16)) { ok = false; break; }
          tc::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // 128 keys in steps of 16
            const uint32_t poff = (kk >> 2) * C::HALF + (kk & 3) * 32;
            tc::mma_f16_ss(tmem_o, tc::smem_desc(pa + pb * C::PB + poff, 16, 1024, tc::SW_128B),
                           tc::smem_desc(va + su * C::OP + kk * 2048, C::HALF, 1024, tc::SW_128B), C::IDESC_O,
                           (u > 0 || kk > 0) ? 1u : 0u);
          }
          tc::mma_commit(p_free + pb);
          tc::mma_commit(v_empty + su);
        }
      }
      if (!ok) *s_abort = 1;
      tc::mma_commit(o_full);
      tc::mbar_wait(o_full, 0, 17);  // nothing of ours is still running on the tensor core
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (thread = row)
    // tcgen05.ld / st are warp-collective: every branch around them is warp-uniform.
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int r = threadIdx.x;
    const float sc = a.scale_log2;  // > 0 (the host routes other scales elsewhere)
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int sb = t & 1;
      ok = __all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(s_full + sb, (t >> 1) & 1, 18));
      if (!ok) break;
      tc::tc_fence_after();
      float v[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float x[32];
        tc::tmem_ld32(tmem + lane_base + sb * 128 + c * 32, x);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[c * 32 + i] = x[i];
      }
      tc::tmem_wait_ld();
      tc::tc_fence_before();
      tc::mbar_arrive(s_free + sb);
      // row maximum of the raw scores; only a tile that crosses the row's key
      // range is masked (masked scores become -inf, which the positive scale
      // keeps at -inf)
      const int tg = tt0 + t;
      const bool w = tg >= T1;
      const int j0 = w ? rlo2 + (tg - T1) * 128 : rlo1 + tg * 128;
      const int lo = row_ok ? (w ? lo2 : lo1) : 0, hi = row_ok ? (w ? hi2 : hi1) : 0;
      if (j0 < lo || j0 + 128 > hi) {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int j = j0 + c;
          if (j < lo || j >= hi) v[c] = -INFINITY;
        }
      }
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = v[i];
#pragma unroll
      for (int c = 8; c < 128; c += 8)
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], v[c + i]);
#pragma unroll
      for (int i = 0; i < 4; ++i) mx8[i] = fmaxf(mx8[i], mx8[i + 4]);
      const float mx = fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])) * sc;
      const int pb = t & 1;  // P buffer of this tile
      float f = 1.f;
      if (mx > -INFINITY) {
        if (m == -INFINITY) {
          m = mx;  // O and l are still zero
        } else if (mx > m + TAU) {
          f = exp2f(m - mx);
          l *= f;
          m = mx;
        }
      }
      if (__any_sync(0xffffffffu, f != 1.f)) {
        // O is rescaled in place: the previous P V must have completed
        if (t > 0) {
          ok = __all_sync(0xffffffffu,
                          !*s_abort && tc::mbar_wait(p_free + ((t - 1) & 1), ((t - 1) >> 1) & 1, 19));
          if (!ok) break;
        }
        tc::tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tc::tmem_ld32(tmem_o + lane_base + c * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          tc::tmem_st32(tmem_o + lane_base + c * 32, o);
        }
        tc::tmem_wait_st();
      }
      // this P buffer was last read by the P V of tile t - 2
      if (t > 1) {
        ok = __all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(p_free + pb, ((t - 2) >> 1) & 1, 19));
        if (!ok) break;
        tc::tc_fence_after();
      }
      // P = 2^(sc * s - m) as bf16, K-major swizzled rows (two 64-key halves)
      const float nbase = m == -INFINITY ? 0.f : -m;
      float rs8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) rs8[i] = 0.f;
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          p[i] = ex2_approx(fmaf(v[ch * 8 + i], sc, nbase));
          rs8[i] += p[i];
        }
        uint4 pk;
        pk.x = pack_bf16(p[0], p[1]);
        pk.y = pack_bf16(p[2], p[3]);
        pk.z = pack_bf16(p[4], p[5]);
        pk.w = pack_bf16(p[6], p[7]);
        const int half = ch >> 3, c8 = ch & 7;
        uint8_t* dst = sP + pb * C::PB + half * C::HALF + (r >> 3) * 1024 + (r & 7) * 128 + ((c8 ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = pk;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) rs8[i] += rs8[i + 4];
      const float rs = (rs8[0] + rs8[1]) + (rs8[2] + rs8[3]);
      l += rs;
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(p_full + pb);
    }
    // ---- epilogue: O / l ----
    if (ntiles > 0 && ok) ok = __all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(o_full, 0, 20));
    tc::tc_fence_after();
    const int64_t grow = static_cast<int64_t>(b) * rows_b + row0 + r +
                         static_cast<int64_t>(blockIdx.z) * a.rows_total;  // split partials
    const float inv = (ok && l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float o[32];
      if (ntiles > 0 && ok) {  // uniform across the warp
        tc::tmem_ld32(tmem_o + lane_base + c * 32, o);
        tc::tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0.f;
      }
      if (!row_ok) continue;
      if (a.out_bf16) {
        uint4* dst = reinterpret_cast<uint4*>(a.out_bf16 + grow * D + c * 32);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 pk;
          pk.x = pack_bf16(o[q4 * 8 + 0] * inv, o[q4 * 8 + 1] * inv);
          pk.y = pack_bf16(o[q4 * 8 + 2] * inv, o[q4 * 8 + 3] * inv);
          pk.z = pack_bf16(o[q4 * 8 + 4] * inv, o[q4 * 8 + 5] * inv);
          pk.w = pack_bf16(o[q4 * 8 + 6] * inv, o[q4 * 8 + 7] * inv);
          dst[q4] = pk;
        }
      } else {
        float4* dst = reinterpret_cast<float4*>(a.O + grow * D + c * 32);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          dst[q4] = make_float4(o[q4 * 4] * inv, o[q4 * 4 + 1] * inv, o[q4 * 4 + 2] * inv, o[q4 * 4 + 3] * inv);
      }
    }
    if (row_ok && a.lse) a.lse[grow] = (ok && l > 0.f) ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace lcc
