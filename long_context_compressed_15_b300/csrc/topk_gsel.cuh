// Exact top-k of a row of indexer scores, one CTA per row, reading only the
// score groups that can hold a winner.  Source: "DeepSeek-V4가 이차적 어텐션
// 비용 없이 ...", section "두 가지 압축 전략: CSA 및 HCA" (the indexer keeps the
// top-k compressed entries per query).
//
// Result (identical to k_topk_thr / k_topk_cluster): the min(k, visible)
// entries with the largest scores, ties to the lower index, in ascending
// index order, padded with -1.
//
// The indexer writes the key of each group's largest score (groups of gs
// consecutive entries).  theta = the k-th largest group maximum is a lower
// bound of the row's k-th largest score, so every winner lies in a group
// whose maximum reaches theta -- at most k groups plus those tied at theta.
// The same holds for the k-th largest maximum over any partition of the
// groups into at least k parts (a lower theta, a few more listed groups).
//   1. the row's group maxima are loaded and theta is selected: a bitonic
//      sort of the group maxima when there are at most NT groups, else of
//      NT partition maxima (thread t: groups t, t+NT, ...);
//   2. the groups whose maximum reaches theta are listed in index order
//      (warp ballots and one scan over the warps' counts);
//   3. only their scores are read, each thread PER consecutive entries of a
//      group (a warp reads whole 128-byte rows), and the scores >= theta are
//      compacted in index order straight from registers (typically little
//      more than k of them); a candidate wins iff fewer than k others beat
//      it (a larger key, or an equal key at a lower index);
//   4. the winners are written in index order (for more than NT candidates:
//      the exact k-th key T by histogram rounds, then every key above T and
//      the lowest-index keys equal to T).
// When more than CAP scores reach theta (massive exact ties) the CTA falls
// back to a bisection over the whole row.
#pragma once
#include "topk_cluster.cuh"

namespace lcc {

template <int NT, int CAP>
__global__ void __launch_bounds__(NT) k_topk_gsel(TopkThrArgs a) {
  static_assert(CAP >= NT && (NT & (NT - 1)) == 0, "the sort needs a power of two and NT words of scratch");
  extern __shared__ __align__(16) uint32_t sm_gsel[];
  __shared__ int s_warp[NT / 32];
  __shared__ uint32_t s_hist[256];
  __shared__ uint32_t s_bc[4];
  const int G_cap = ((a.Ncap + a.gs - 1) / a.gs + 3) & ~3;  // keeps the arrays below 16-byte aligned
  uint32_t* s_g = sm_gsel;                 // [G_cap] group maxima
  int* s_gl = reinterpret_cast<int*>(s_g + G_cap);   // [G_cap] listed groups, index order
  uint32_t* s_ok = reinterpret_cast<uint32_t*>(s_gl + G_cap);  // [CAP] candidate keys, index order
  int32_t* s_oi = reinterpret_cast<int32_t*>(s_ok + CAP);      // [CAP] their entries

  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bc[2] = 0xFFFFFFFFu;
    s_bc[3] = 0u;
  }
  const int row = blockIdx.x;
  const int b = row / a.nq, i = a.q0 + row % a.nq;
  const int k = a.k;
  const float* srow = a.scores + static_cast<int64_t>(row) * a.Ncap;
  const int64_t qpos = __ldg(a.q_pos0 + b) + i;
  const int nval = __ldg(a.n_valid + b);
  const int vis = visible_entries(qpos, a.m, nval, a.Ncap);
  int32_t* oi = a.out_i + (static_cast<int64_t>(b) * a.Tq + i) * k;
  float* os = a.out_s ? a.out_s + (static_cast<int64_t>(b) * a.Tq + i) * k : nullptr;
  pdl_trigger();
  pdl_wait();  // scores and group maxima come from the indexer kernel

  if (vis <= k) {  // every visible entry is selected
    for (int p = tid; p < k; p += NT) {
      oi[p] = p < vis ? p : -1;
      if (os) os[p] = p < vis ? __ldcg(srow + p) : -INFINITY;
    }
    return;
  }
  const int gs = a.gs;
  const int G = (vis + gs - 1) / gs;
  const uint32_t* gm = a.gmax + static_cast<int64_t>(row) * a.g_stride;
  for (int g0 = 0; g0 < G; g0 += 8 * NT) {  // eight loads in flight per thread
    uint32_t gv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int g = g0 + u * NT + tid;
      gv[u] = g < G ? __ldcg(gm + g) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int g = g0 + u * NT + tid;
      if (g < G) s_g[g] = gv[u];
    }
  }
  __syncthreads();
  // 1. theta (0 when fewer than k groups: every group is listed)
  uint32_t theta = 0u;
  if (G >= k) {
    if (G <= NT) {
      theta = block_kth_bitonic<NT>(tid < G ? s_g[tid] : 0u, k, s_ok, s_bc);
    } else if (k <= NT) {
      // theta' = k-th largest of NT partition maxima (thread t: the groups t,
      // t+NT, ...).  k partitions reach theta', so k distinct scores do and
      // theta' is still a lower bound of the row's k-th score; it lists a few
      // more groups than the exact k-th group maximum would
      uint32_t mx = 0u;
      for (int g = tid; g < G; g += NT) mx = max(mx, s_g[g]);
      theta = block_kth_bitonic<NT>(mx, k, s_ok, s_bc);
    } else {
      theta = block_kth_hist<NT>(s_g, G, k, s_hist, s_bc);
    }
  }
  // 2. groups whose maximum reaches theta, in index order: each warp takes
  // 512 consecutive groups of a chunk (ballots over 32 at a time), one scan
  // over the warps' counts places the warps' lists
  int ng = 0;
  {
    constexpr int NWARP = NT / 32, GPW = 512;
    const int lane = tid & 31, warp = tid >> 5;
    for (int g0 = 0; g0 < G; g0 += NWARP * GPW) {
      const int gw = g0 + warp * GPW;
      int cnt = 0;
#pragma unroll 4
      for (int u = 0; u < GPW / 32; ++u) {
        const int g = gw + u * 32 + lane;
        cnt += __popc(__ballot_sync(0xffffffffu, g < G && s_g[g] >= theta));
      }
      if (lane == 0) s_warp[warp] = cnt;
      __syncthreads();
      int base = ng, tot = 0;
#pragma unroll
      for (int w = 0; w < NWARP; ++w) {
        const int c = s_warp[w];
        base += w < warp ? c : 0;
        tot += c;
      }
      if (cnt > 0) {
#pragma unroll 4
        for (int u = 0; u < GPW / 32; ++u) {
          const int g = gw + u * 32 + lane;
          const bool f = g < G && s_g[g] >= theta;
          const unsigned bal = __ballot_sync(0xffffffffu, f);
          if (f) s_gl[base + __popc(bal & ((1u << lane) - 1u))] = g;
          base += __popc(bal);
        }
      }
      ng += tot;
      __syncthreads();  // s_warp is reused
    }
  }
  __syncthreads();
  // 3. the listed groups' scores, NT*PER entries per pass: each thread takes
  // PER consecutive entries of one group (four 16-byte loads), so a warp reads
  // whole 128-byte rows; the scores >= theta are compacted in index order
  // (one block scan per pass)
  constexpr int PER = 16;
  const int C = ng * 32;
  const bool vec = (a.Ncap & 3) == 0 && (reinterpret_cast<uintptr_t>(a.scores) & 15) == 0;
  int M = 0;
  if (gs == 32) {
    for (int c0 = 0; c0 < C && M <= CAP; c0 += NT * PER) {
      const int c = c0 + tid * PER;
      const int e = c < C ? s_gl[c >> 5] * 32 + (c & 31) : vis;
      uint32_t kv[PER];
      if (vec && e + PER <= vis) {
#pragma unroll
        for (int u = 0; u < PER; u += 4) {
          const float4 x = __ldcg(reinterpret_cast<const float4*>(srow + e + u));
          kv[u] = f32_to_key(x.x); kv[u + 1] = f32_to_key(x.y); kv[u + 2] = f32_to_key(x.z); kv[u + 3] = f32_to_key(x.w);
        }
      } else {
#pragma unroll
        for (int u = 0; u < PER; ++u) kv[u] = e + u < vis ? f32_to_key(__ldcg(srow + e + u)) : 0u;
      }
      int n = 0;
#pragma unroll
      for (int u = 0; u < PER; ++u) n += (kv[u] >= theta && kv[u] != 0u) ? 1 : 0;
      int tot;
      int p = M + block_scan_excl<NT>(n, s_warp, &tot);
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        if (kv[u] >= theta && kv[u] != 0u) {
          if (p < CAP) {
            s_ok[p] = kv[u];
            s_oi[p] = e + u;
          }
          ++p;
        }
      }
      M += tot;
    }
  }
  __syncthreads();
  if (gs == 32 && M <= CAP) {
    // M >= k: each of the k best groups (or partitions) has its maximum among them
    if (M <= NT) {
      // the usual case: a candidate wins iff fewer than k others beat it (larger key,
      // or an equal key at a lower index); winners written in index order by one scan
      const uint32_t v = tid < M ? s_ok[tid] : 0u;
      const bool win = tid < M && rank_by_count(s_ok, M, v, tid & ~31, tid) < k;
      int tot;
      const int q = block_scan_excl<NT>(win ? 1 : 0, s_warp, &tot);
      if (win && q < k) {
        oi[q] = s_oi[tid];
        if (os) os[q] = key_to_f32(s_ok[tid]);
      }
      return;
    }
    const uint32_t T = block_kth_hist<NT>(s_ok, M, k, s_hist, s_bc);
    // 4. everything above T, then the lowest-index entries equal to T
    int pk = 0;
    for (int c = tid; c < M; c += NT) pk += (s_ok[c] > T ? 1 : 0) + (s_ok[c] == T ? 0x10000 : 0);
    pk = block_sum<NT>(pk, s_warp);
    const int need_eq = k - (pk & 0xFFFF), n_eq = pk >> 16;
    int eq_seen = 0, out_pos = 0;
    for (int cb = 0; cb < M; cb += NT) {
      const int c = cb + tid;
      const uint32_t key = c < M ? s_ok[c] : 0u;
      bool sel;
      if (n_eq == need_eq) {
        sel = c < M && key >= T;
      } else {
        const bool eq = c < M && key == T;
        int eq_tot;
        const int eq_rank = eq_seen + block_scan_excl<NT>(eq ? 1 : 0, s_warp, &eq_tot);
        eq_seen += eq_tot;
        sel = c < M && (key > T || (eq && eq_rank < need_eq));
      }
      int sel_tot;
      const int q = out_pos + block_scan_excl<NT>(sel ? 1 : 0, s_warp, &sel_tot);
      out_pos += sel_tot;
      if (sel && q < k) {
        oi[q] = s_oi[c];
        if (os) os[q] = key_to_f32(key);
      }
    }
    return;
  }

  // ---- massive ties: exact k-th key by bisection over the whole row ----
  uint32_t T = 0u;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t c = T | (1u << bit);
    int cnt = 0;
    for (int e = tid; e < vis; e += NT) cnt += f32_to_key(__ldcg(srow + e)) >= c;
    if (block_sum<NT>(cnt, s_warp) >= k) T = c;
  }
  int ngt = 0;
  for (int e = tid; e < vis; e += NT) ngt += f32_to_key(__ldcg(srow + e)) > T;
  const int need_eq = k - block_sum<NT>(ngt, s_warp);
  int out_pos = 0, eq_seen = 0;
  for (int eb = 0; eb < vis; eb += NT) {
    const int e = eb + tid;
    const uint32_t key = e < vis ? f32_to_key(__ldcg(srow + e)) : 0u;
    const bool eq = e < vis && key == T;
    int eq_tot;
    const int eq_rank = eq_seen + block_scan_excl<NT>(eq ? 1 : 0, s_warp, &eq_tot);
    eq_seen += eq_tot;
    const bool sel = e < vis && (key > T || (eq && eq_rank < need_eq));
    int sel_tot;
    const int p = out_pos + block_scan_excl<NT>(sel ? 1 : 0, s_warp, &sel_tot);
    out_pos += sel_tot;
    if (sel && p < k) {
      oi[p] = e;
      if (os) os[p] = key_to_f32(key);
    }
  }
}

}  // namespace lcc
