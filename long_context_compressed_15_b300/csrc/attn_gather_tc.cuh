// CSA sparse attention (+ the sliding window, one softmax) on the 5th-
// generation tensor cores for long query blocks (prefill).  Source:
// "DeepSeek-V4가 이차적 어텐션 비용 없이 ...", section "두 가지 압축 전략: CSA 및
// HCA" (each query attends to its top-k compressed entries with MQA; a window
// branch over the most recent raw tokens runs in parallel).
//
// Work items are 128 (query, head) rows of one sequence -- two queries of 64
// heads or one of 128 -- and a persistent CTA walks items blockIdx.x,
// blockIdx.x + gridDim.x, ...  An item's key tiles are one gathered tile per
// 128 selected entries of each of its queries (rows fetched with TMA
// tile::gather4 from tensor maps with one-row boxes; in a tile of query A the
// rows of query B are masked, as are slots marked -1) followed by the window
// tiles (plain TMA tiles of raw rows, shared by the item's queries).
// Roles (192 threads):
//   warp 4 (producer)  Q of each item (one buffer, reloaded once the item's
//                      last Q K^T has run); K and V tiles into two-stage
//                      rings, V one tile behind K (a gathered tile takes
//                      several times as long to land as a window tile, so
//                      neither ring may serialise on it);
//   warp 5 (MMA)       S[g] = Q K[g]^T into one of two TMEM buffers, then
//                      O += P[g-1] V[g-1] into the TMEM accumulator of the
//                      item of tile g-1 (two accumulators: the epilogue of
//                      one item overlaps the next item's tiles);
//   warps 0..3         one thread per row: online softmax in the log2 domain
//                      (as in k_attn_tc), P into one of two buffers, and per
//                      item the epilogue O / l to global memory.
// Every tile counter (K stage, V, S and P buffers) runs over the CTA's whole
// tile sequence, so the pipeline never drains between items.
#pragma once
#include "tc.cuh"

namespace lcc {

namespace gtc {

// Four rows y0..y3 of a 2-D tensor (tensor map with one-row boxes) into four
// consecutive box-sized rows at dst.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y0, int y1,
                                            int y2, int y3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3),
        "r"(smem_u32(bar))
      : "memory");
}

}  // namespace gtc

struct AttnGatherArgs {
  int B, Tq, H;
  float scale_log2;        // scale * log2(e), > 0
  const int64_t* q_pos0;   // [B] (window only)
  const int32_t* idx;      // [B, Tq, k] entries of Kc/Vc, -1 = empty slot
  int k, Ncap;
  int win;                 // window over raw rows as the second key source
  int Rcap;
  const int64_t* raw_pos0; // [B]
  int W;
  bf16* out_bf16;          // [B*Tq*H, D] bf16, or
  float* O;                // [B*Tq*H, D] fp32
  float* lse;              // [B*Tq*H] natural log (optional)
  int tiles_q;             // 128-row items per sequence
};

struct AttnGatherCfg {
  static constexpr int D = 128;
  static constexpr int HALF = 128 * 64 * 2;   // one 64-column swizzled half: 16 KB
  static constexpr int OP = 2 * HALF;         // 128 rows x 128 columns bf16
  static constexpr int OFF_Q = 0;             // one buffer
  static constexpr int OFF_K = 1 * OP;        // two stages
  static constexpr int OFF_V = 3 * OP;        // two stages
  static constexpr int OFF_P = 5 * OP;        // two buffers
  static constexpr int OFF_BAR = 7 * OP;
  static constexpr int NBAR = 23;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 64 + 1024;
  static constexpr uint32_t IDESC_S = tc::idesc_f16(128, 128, true);             // Q K^T
  static constexpr uint32_t IDESC_O = tc::idesc_f16(128, D, true, false, true);  // P V, V MN-major
  static constexpr int TMEM_COLS = 512;       // S: 2 x 128, O: 2 x 128
};

// Geometry of work item `it`.
struct GItem {
  int b, q_first, q_last, tpq, T1, T2, rlo2;
  int64_t row0;
};

__device__ __forceinline__ GItem gather_item(const AttnGatherArgs& a, int it) {
  GItem g;
  g.b = it / a.tiles_q;
  g.row0 = static_cast<int64_t>(it % a.tiles_q) * 128;
  const int64_t rows_b = static_cast<int64_t>(a.Tq) * a.H;
  const int64_t row_end = g.row0 + 128 < rows_b ? g.row0 + 128 : rows_b;
  g.q_first = static_cast<int>(g.row0 / a.H);
  g.q_last = static_cast<int>((row_end - 1) / a.H);
  g.tpq = (a.k + 127) / 128;
  g.T1 = (g.q_last - g.q_first + 1) * g.tpq;
  g.T2 = 0;
  g.rlo2 = 0;
  if (a.win) {  // union of the item's windows (monotone in the position)
    const int64_t p0 = __ldg(a.q_pos0 + g.b), rp0 = __ldg(a.raw_pos0 + g.b);
    int64_t lo = p0 + g.q_first - a.W + 1;
    if (lo < 0) lo = 0;
    lo -= rp0;
    if (lo < 0) lo = 0;
    int64_t hi = p0 + g.q_last - rp0 + 1;
    if (hi > a.Rcap) hi = a.Rcap;
    if (hi > lo) {
      g.rlo2 = static_cast<int>(lo);
      g.T2 = static_cast<int>((hi - lo + 127) / 128);
    }
  }
  return g;
}

__global__ void __launch_bounds__(192, 1)
    k_attn_gather_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKw,
                     const __grid_constant__ CUtensorMap tmVw, AttnGatherArgs a) {
  using C = AttnGatherCfg;
  constexpr int D = C::D;
  constexpr float TAU = 8.0f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;        // [1]
  uint64_t* q_empty = bars + 1;   // [1]
  uint64_t* k_full = bars + 2;    // [2]
  uint64_t* k_empty = bars + 4;   // [2]
  uint64_t* v_full = bars + 6;    // [2]
  uint64_t* v_empty = bars + 8;   // [2]
  // bars + 10 .. : S, P, O and the final MMA barrier
  uint64_t* s_full = bars + 10;   // [2]
  uint64_t* s_free = bars + 12;   // [2]
  uint64_t* p_full = bars + 14;   // [2]
  uint64_t* p_free = bars + 16;   // [2]
  uint64_t* o_full = bars + 18;   // [2]
  uint64_t* o_free = bars + 20;   // [2]
  uint64_t* mma_done = bars + 22; // [1]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sP = smem + C::OFF_P;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    tc::mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(k_full + i, 32);  // one arrival per producer lane
      tc::mbar_init(k_empty + i, 1);
      tc::mbar_init(v_full + i, 32);
      tc::mbar_init(v_empty + i, 1);
      tc::mbar_init(s_full + i, 1);
      tc::mbar_init(s_free + i, 128);
      tc::mbar_init(p_full + i, 128);
      tc::mbar_init(p_free + i, 1);
      tc::mbar_init(o_full + i, 1);
      tc::mbar_init(o_free + i, 128);
    }
    tc::mbar_init(mma_done, 1);
    *s_abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 5) tc::tmem_alloc(s_tmem, C::TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_wait();  // the index lists may come from the kernel launched just before

  const int nitems = a.B * a.tiles_q;
  const int64_t rows_b = static_cast<int64_t>(a.Tq) * a.H;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    // a tile of the CTA's sequence: gathered (rows y[0..3] of this lane, read
    // from the index list when the tile is described, reused for its V) or
    // window (first raw row y[0])
    struct TileRef {
      int y[4];
      bool gathered;
    };
    auto describe = [&](const GItem& gi, int t) {
      TileRef r;
      r.gathered = t < gi.T1;
      if (r.gathered) {
        const int oq = gi.q_first + t / gi.tpq, kb = t % gi.tpq;
        const int32_t* irow = a.idx + (static_cast<int64_t>(gi.b) * a.Tq + oq) * a.k;
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // lane l: rows 4l .. 4l+3 of the tile
          const int c = kb * 128 + 4 * lane + i;
          int e = c < a.k ? __ldg(irow + c) : -1;
          if (e >= a.Ncap || e < -1) {
            record_error(DEV_ERR_INDEX, static_cast<unsigned>(c));
            e = -1;
          }
          r.y[i] = gi.b * a.Ncap + (e >= 0 ? e : 0);  // an empty slot reads row 0 (masked by the softmax)
        }
      } else {
        r.y[0] = gi.b * a.Rcap + gi.rlo2 + (t - gi.T1) * 128;
        r.y[1] = r.y[2] = r.y[3] = 0;
      }
      return r;
    };
    // one K or V tile into dst; every lane arrives once on bar
    auto load = [&](const TileRef& r, bool is_v, uint8_t* dst, uint64_t* bar) {
      if (lane == 0) tc::mbar_arrive_expect_tx(bar, C::OP);
      __syncwarp();
      if (r.gathered) {
        const int rr = 4 * lane;
        const CUtensorMap* m = is_v ? &tmV : &tmK;
#pragma unroll
        for (int h = 0; h < D / 64; ++h)
          gtc::tma_gather4(dst + h * C::HALF + (rr >> 3) * 1024 + (rr & 7) * 128, m, bar, h * 64, r.y[0], r.y[1],
                           r.y[2], r.y[3]);
        if (lane != 0) tc::mbar_arrive(bar);
      } else {
        if (lane == 0) {
          const CUtensorMap* m = is_v ? &tmVw : &tmKw;
          for (int h = 0; h < D / 64; ++h) tc::tma_load_2d(dst + h * C::HALF, m, bar, h * 64, r.y[0]);
        } else {
          tc::mbar_arrive(bar);
        }
      }
    };
    auto wait0 = [&](uint64_t* bar, uint32_t parity, unsigned site) {  // lane 0 waits, the warp follows
      bool okw = true;
      if (lane == 0) okw = !*s_abort && tc::mbar_wait(bar, parity, site);
      return __shfl_sync(0xffffffffu, okw, 0) != 0;
    };
    uint32_t nk = 0, nv = 0, il = 0;
    TileRef prev{};
    bool have_prev = false, pok = true;
    for (int it = blockIdx.x; pok && it < nitems; it += gridDim.x, ++il) {
      const GItem gi = gather_item(a, it);
      if (!wait0(q_empty, (il & 1) ^ 1, 31)) { pok = false; break; }
      if (lane == 0) {
        tc::mbar_arrive_expect_tx(q_full, C::OP);
        const int qy = static_cast<int>(static_cast<int64_t>(gi.b) * rows_b + gi.row0);
        for (int h = 0; h < D / 64; ++h) tc::tma_load_2d(sQ + h * C::HALF, &tmQ, q_full, h * 64, qy);
      }
      const int T = gi.T1 + gi.T2;
      for (int t = 0; t < T; ++t) {
        const TileRef cur = describe(gi, t);
        const int s = nk & 1;
        if (!wait0(k_empty + s, ((nk >> 1) & 1) ^ 1, 32)) { pok = false; break; }
        load(cur, false, sK + s * C::OP, k_full + s);
        ++nk;
        if (have_prev) {  // V one tile behind K
          if (!wait0(v_empty + (nv & 1), ((nv >> 1) & 1) ^ 1, 33)) { pok = false; break; }
          load(prev, true, sV + (nv & 1) * C::OP, v_full + (nv & 1));
          ++nv;
        }
        prev = cur;
        have_prev = true;
      }
    }
    if (pok && have_prev) {  // V of the last tile
      if (wait0(v_empty + (nv & 1), ((nv >> 1) & 1) ^ 1, 33)) {
        load(prev, true, sV + (nv & 1) * C::OP, v_full + (nv & 1));
        ++nv;
      } else {
        pok = false;
      }
    }
    if (!pok && lane == 0) *s_abort = 1;
    // every copy this CTA started has landed before it may exit
    if (lane == 0) {
      if (il > 0) tc::mbar_wait(q_full, (il - 1) & 1, 34);
      for (uint32_t i = nk > 2 ? nk - 2 : 0; i < nk; ++i) tc::mbar_wait(k_full + (i & 1), (i >> 1) & 1, 34);
      for (uint32_t i = nv > 2 ? nv - 2 : 0; i < nv; ++i) tc::mbar_wait(v_full + (i & 1), (i >> 1) & 1, 34);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK), va = smem_u32(sV), pa = smem_u32(sP);
      struct PvRef {
        uint32_t g, il;
        bool first, last;
      };
      bool ok = true;
      auto issue_pv = [&](const PvRef& p) {
        const int pb = p.g & 1, ob = p.il & 1;
        if (*s_abort || !tc::mbar_wait(p_full + pb, (p.g >> 1) & 1, 41) ||
            !tc::mbar_wait(v_full + (p.g & 1), (p.g >> 1) & 1, 42)) {
          ok = false;
          return;
        }
        // the accumulator was last read by the epilogue of item il - 2
        if (p.first && p.il >= 2 && !tc::mbar_wait(o_free + ob, ((p.il >> 1) & 1) ^ 1, 43)) {
          ok = false;
          return;
        }
        tc::tc_fence_after();
        const uint32_t tmem_o = tmem + 256 + ob * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // 128 keys in steps of 16
          const uint32_t poff = (kk >> 2) * C::HALF + (kk & 3) * 32;
          tc::mma_f16_ss(tmem_o, tc::smem_desc(pa + pb * C::OP + poff, 16, 1024, tc::SW_128B),
                         tc::smem_desc(va + (p.g & 1) * C::OP + kk * 2048, C::HALF, 1024, tc::SW_128B), C::IDESC_O,
                         (!p.first || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(p_free + pb);
        tc::mma_commit(v_empty + (p.g & 1));
        if (p.last) tc::mma_commit(o_full + ob);
      };
      uint32_t g = 0, il = 0;
      PvRef prev{};
      bool have_prev = false;
      for (int it = blockIdx.x; ok && it < nitems; it += gridDim.x, ++il) {
        const GItem gi = gather_item(a, it);
        const int T = gi.T1 + gi.T2;
        if (*s_abort || !tc::mbar_wait(q_full, il & 1, 44)) { ok = false; break; }
        for (int t = 0; ok && t < T; ++t, ++g) {
          const int s = g & 1, sb = g & 1;
          if (*s_abort || !tc::mbar_wait(k_full + s, (g >> 1) & 1, 45) ||
              !tc::mbar_wait(s_free + sb, ((g >> 1) & 1) ^ 1, 46)) { ok = false; break; }
          tc::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::HALF + (kk & 3) * 32;
            tc::mma_f16_ss(tmem + sb * 128, tc::smem_desc(qa + off, 16, 1024, tc::SW_128B),
                           tc::smem_desc(ka + s * C::OP + off, 16, 1024, tc::SW_128B), C::IDESC_S, kk > 0);
          }
          tc::mma_commit(s_full + sb);
          tc::mma_commit(k_empty + s);
          if (t == T - 1) tc::mma_commit(q_empty);  // the next item's Q may be loaded
          if (have_prev) issue_pv(prev);  // P V of the previous tile (possibly of the previous item)
          prev = PvRef{g, il, t == 0, t == T - 1};
          have_prev = true;
        }
      }
      if (ok && have_prev) issue_pv(prev);
      if (!ok) *s_abort = 1;
      tc::mma_commit(mma_done);
      tc::mbar_wait(mma_done, 0, 47);  // nothing of ours is still running on the tensor core
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue (thread = row)
    // tcgen05.ld / st are warp-collective: every branch around them is warp-uniform.
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int r = threadIdx.x;
    const float sc = a.scale_log2;
    bool ok = true;
    uint32_t g = 0, il = 0;
    for (int it = blockIdx.x; ok && it < nitems; it += gridDim.x, ++il) {
      const GItem gi = gather_item(a, it);
      const int ob = il & 1;
      const int T = gi.T1 + gi.T2;
      const int64_t row = gi.row0 + r;
      const bool row_ok = row < rows_b;
      const int q = static_cast<int>(row / a.H);  // this row's query
      int lo2 = 0, hi2 = 0;                       // this row's window (raw rows)
      if (a.win && row_ok) {
        const int64_t t_pos = __ldg(a.q_pos0 + gi.b) + q, rp0 = __ldg(a.raw_pos0 + gi.b);
        int64_t l0 = t_pos - a.W + 1;
        if (l0 < 0) l0 = 0;
        l0 -= rp0;
        if (l0 < 0) l0 = 0;
        int64_t h0 = t_pos - rp0 + 1;
        if (h0 > a.Rcap) h0 = a.Rcap;
        if (h0 < l0) h0 = l0;
        lo2 = static_cast<int>(l0);
        hi2 = static_cast<int>(h0);
      }
      float m = -INFINITY, l = 0.f;
      for (int t = 0; t < T; ++t, ++g) {
        const int sb = g & 1;
        // gathered tile: owner query and its occupied slots (loaded before the wait)
        const bool gt = t < gi.T1;
        const bool mine = gt && row_ok && q - gi.q_first == t / gi.tpq;  // warp-uniform (H >= 32)
        int ev[4] = {-1, -1, -1, -1};  // requested now, consumed after S has been read
        if (mine) {
          const int32_t* irow = a.idx + (static_cast<int64_t>(gi.b) * a.Tq + q) * a.k;
          const int kb = t % gi.tpq;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = kb * 128 + lane + 32 * i;
            if (c < a.k) ev[i] = __ldg(irow + c);
          }
        }
        ok = __all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(s_full + sb, (g >> 1) & 1, 48));
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
        // keep mask of the tile's 128 keys for this row
        uint32_t km[4];
        if (gt) {
#pragma unroll
          for (int i = 0; i < 4; ++i) km[i] = mine ? __ballot_sync(0xffffffffu, ev[i] >= 0 && ev[i] < a.Ncap) : 0u;
        } else {
          const int j0 = gi.rlo2 + (t - gi.T1) * 128;
          const int cl = max(0, lo2 - j0), ch = min(128, max(0, hi2 - j0));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int l_i = min(32, max(0, cl - 32 * i)), h_i = min(32, max(0, ch - 32 * i));
            km[i] = static_cast<uint32_t>(((1ull << h_i) - 1ull) & ~((1ull << l_i) - 1ull));
          }
        }
        if ((km[0] & km[1] & km[2] & km[3]) != 0xFFFFFFFFu) {
#pragma unroll
          for (int c = 0; c < 128; ++c) v[c] = ((km[c >> 5] >> (c & 31)) & 1u) ? v[c] : -INFINITY;
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
        float f = 1.f;
        if (mx > -INFINITY) {
          if (m == -INFINITY) {
            m = mx;  // O and l of this item are still zero
          } else if (mx > m + TAU) {
            f = exp2f(m - mx);
            l *= f;
            m = mx;
          }
        }
        if (__any_sync(0xffffffffu, f != 1.f)) {
          // O is rescaled in place: the previous P V of this item must have completed (t > 0 here)
          ok = __all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(p_free + ((g - 1) & 1), ((g - 1) >> 1) & 1, 49));
          if (!ok) break;
          tc::tc_fence_after();
          const uint32_t tmem_o = tmem + 256 + ob * 128;
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
        // this P buffer was last read by the P V of tile g - 2
        if (g > 1) {
          ok = __all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(p_free + sb, ((g - 2) >> 1) & 1, 50));
          if (!ok) break;
          tc::tc_fence_after();
        }
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
          uint8_t* dst = sP + sb * C::OP + half * C::HALF + (r >> 3) * 1024 + (r & 7) * 128 + ((c8 ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) = pk;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) rs8[i] += rs8[i + 4];
        l += (rs8[0] + rs8[1]) + (rs8[2] + rs8[3]);
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        tc::mbar_arrive(p_full + sb);
      }
      if (!ok) break;
      // ---- epilogue of the item: O / l ----
      ok = __all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(o_full + ob, (il >> 1) & 1, 51));
      if (!ok) break;
      tc::tc_fence_after();
      const int64_t grow = static_cast<int64_t>(gi.b) * rows_b + row;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const uint32_t tmem_o = tmem + 256 + ob * 128;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tc::tmem_ld32(tmem_o + lane_base + c * 32, o);
        tc::tmem_wait_ld();
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
      if (row_ok && a.lse) a.lse[grow] = l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
      tc::tc_fence_before();
      tc::mbar_arrive(o_free + ob);
    }
    if (!ok) *s_abort = 1;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace lcc
