// Exact top-k of a row of indexer scores, one thread-block cluster per row.
// Source: "DeepSeek-V4가 이차적 어텐션 비용 없이 ...", section "두 가지 압축 전략:
// CSA 및 HCA" (the indexer keeps the top-k compressed entries per query).
//
// Result (identical to k_topk_thr): the min(k, visible) entries of the row
// with the largest scores, ties to the lower index, in ascending index
// order, padded with -1.
//
// The same threshold argument as k_topk_thr (theta = k-th largest
// super-group maximum is a lower bound of the k-th largest score), spread
// over the CL CTAs of a cluster so that each SM touches 1/CL of the row and
// of the counting work, and the CTAs exchange through distributed shared
// memory instead of global memory:
//   1. every CTA loads its SEG = NT*PER scores and builds all super-group
//      maxima from the group maxima; CTA r counts the r-th share of them and
//      the owner of the k-th largest writes theta into every CTA;
//   2. every CTA compacts its entries >= theta in index order (its list is
//      complete: SEG entries at most), then gathers all CTAs' keys in rank
//      (= index) order; CTA r counts the r-th share of the candidates and
//      the owner of the exact k-th largest key T writes it into CTA 0;
//   3. CTA 0 writes every candidate above T and the lowest-index candidates
//      equal to T.
// Candidates that do not fit CAP (massive exact ties) fall back to a
// bisection over the row's scores in CTA 0.  Control flow through the
// cluster barriers depends only on per-row values, so every CTA of the
// cluster meets each barrier.
#pragma once
#include "topk_thr.cuh"

namespace lcc {

namespace clu {
__device__ __forceinline__ uint32_t rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ void sync() {
  arrive();
  wait();
}
// Address of the shared variable `p` of CTA `r` of this cluster.
__device__ __forceinline__ uint32_t map(const void* p, uint32_t r) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(r));
  return d;
}
__device__ __forceinline__ void st(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
}  // namespace clu

// The elements vals[s0..s1) that are the k-th largest of vals[0..n) (zero
// padded to a multiple of 128): v with #{x > v} < k <= #{x >= v}.  Each one
// found is stored at shared variable `dst` of the cluster CTAs [r0, r1).
// Every thread of the CTA calls this with the same arguments.
template <int NT>
__device__ __forceinline__ void kth_share(const uint32_t* vals, int n, int k, int s0, int s1, const uint32_t* dst,
                                          uint32_t r0, uint32_t r1) {
  const int ne = s1 - s0;
  if (ne <= 0) return;
  const int tpe = threads_per_elem<NT>(ne);
  const int np4 = (n + 127) / 128 * 32;
  const int groups = NT / tpe, part = threadIdx.x % tpe;
  const uint4* v4 = reinterpret_cast<const uint4*>(vals);
  for (int it = 0; it < (ne + groups - 1) / groups; ++it) {
    const int e = s0 + it * groups + static_cast<int>(threadIdx.x) / tpe;
    const bool real = e < s1;
    const uint32_t v = real ? vals[e] : 0xFFFFFFFFu;
    int gt = 0, ge = 0;
#pragma unroll 4
    for (int w = part; w < np4; w += tpe) {
      const uint4 x = v4[w];
      gt += (x.x > v) + (x.y > v) + (x.z > v) + (x.w > v);
      ge += (x.x >= v) + (x.y >= v) + (x.z >= v) + (x.w >= v);
    }
    for (int o = 1; o < tpe; o <<= 1) {
      gt += __shfl_xor_sync(0xffffffffu, gt, o);
      ge += __shfl_xor_sync(0xffffffffu, ge, o);
    }
    if (real && part == 0 && gt < k && ge >= k)
      for (uint32_t r = r0; r < r1; ++r) clu::st(clu::map(dst, r), v);
  }
}

template <int NT, int PER, int CAP, int MAXG>
struct TopkClSmem {
  static constexpr int SEG = NT * PER;
  static constexpr size_t lk = 0;                                   // this CTA's candidates (keys)
  static constexpr size_t li = lk + SEG * 4;                        // ... and their entries
  static constexpr size_t ck = li + SEG * 4;                        // all candidates' keys (+ zero pad)
  static constexpr size_t ci = ck + (CAP + 128) * 4;                // all candidates' entries (CTA 0)
  static constexpr size_t g = ci + CAP * 4;                         // super-group maxima (+ zero pad)
  static constexpr size_t total = g + (MAXG + 128) * 4;
};

// MAXG: most super-groups (2k); the host routes rows to this kernel only when
// 2k <= MAXG, k * (entries per group) <= CAP and the row fits CL*SEG entries.
template <int NT, int PER, int CAP, int MAXG>
__global__ void __launch_bounds__(NT) k_topk_cluster(TopkThrArgs a) {
  using L = TopkClSmem<NT, PER, CAP, MAXG>;
  constexpr int SEG = L::SEG;
  static_assert(PER % 4 == 0, "4-wide loads");
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* s_lk = reinterpret_cast<uint32_t*>(smem + L::lk);
  int32_t* s_li = reinterpret_cast<int32_t*>(smem + L::li);
  uint32_t* s_ck = reinterpret_cast<uint32_t*>(smem + L::ck);
  int32_t* s_ci = reinterpret_cast<int32_t*>(smem + L::ci);
  uint32_t* s_g = reinterpret_cast<uint32_t*>(smem + L::g);
  __shared__ int s_warp[NT / 32];
  __shared__ uint32_t s_theta, s_T;
  __shared__ int s_cnt;
  __shared__ int s_off[9];

  const int tid = threadIdx.x;
  const uint32_t rk = clu::rank(), CL = clu::size();
  clu::arrive();  // every CTA of the cluster has started before any remote access (wait below)
  const int row = static_cast<int>(blockIdx.x / CL);
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
    if (rk == 0)
      for (int p = tid; p < k; p += NT) {
        oi[p] = p < vis ? p : -1;
        if (os) os[p] = p < vis ? __ldcg(srow + p) : -INFINITY;
      }
    clu::wait();
    return;
  }

  // this CTA's scores
  const int lo = static_cast<int>(rk) * SEG;
  const int e0 = lo + tid * PER;
  const int hi = min(vis, lo + SEG);
  float sv[PER];
  if ((a.Ncap & 3) == 0) {
#pragma unroll
    for (int u = 0; u < PER; u += 4) {
      const float4 v = e0 + u < hi ? __ldcg(reinterpret_cast<const float4*>(srow + e0 + u))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
      sv[u] = v.x; sv[u + 1] = v.y; sv[u + 2] = v.z; sv[u + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < PER; ++u) sv[u] = e0 + u < hi ? __ldcg(srow + e0 + u) : 0.f;
  }

  // super-group maxima (all of them, in every CTA)
  const int G = (vis + a.gs - 1) / a.gs;
  const int f = (G + 2 * k - 1) / (2 * k);
  const int Gs = (G + f - 1) / f;
  const bool use_theta = Gs >= k;
  if (use_theta) {
    const uint32_t* gm = a.gmax + static_cast<int64_t>(row) * a.g_stride;
    const int Gp = (Gs + 127) / 128 * 128;
    for (int s = tid; s < Gp; s += NT) {
      uint32_t mx = 0u;
      if (s < Gs) {
        const int g1 = min(G, (s + 1) * f);
        for (int g = s * f; g < g1; ++g) mx = max(mx, __ldcg(gm + g));
      }
      s_g[s] = mx;
    }
  }
  if (tid == 0) {
    s_theta = 0u;  // fewer than k super-groups: every visible entry is a candidate
    s_T = 0u;
  }
  __syncthreads();
  clu::wait();
  if (use_theta) {
    const int spc = (Gs + static_cast<int>(CL) - 1) / static_cast<int>(CL);
    const int s0 = static_cast<int>(rk) * spc;
    kth_share<NT>(s_g, Gs, k, s0, min(Gs, s0 + spc), &s_theta, 0u, CL);
  }
  clu::sync();  // theta everywhere
  const uint32_t theta = s_theta;

  // this CTA's candidates, in index order
  uint32_t keys[PER];
  int n = 0;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    keys[u] = e0 + u < hi ? f32_to_key(sv[u]) : 0u;
    n += keys[u] >= theta && keys[u] != 0u;
  }
  int tot;
  int pos = block_scan_excl<NT>(n, s_warp, &tot);
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    if (keys[u] >= theta && keys[u] != 0u) {
      s_lk[pos] = keys[u];
      s_li[pos] = e0 + u;
      ++pos;
    }
  }
  if (tid == 0) s_cnt = tot;
  clu::sync();  // every CTA's list and count

  if (tid < static_cast<int>(CL)) s_off[tid + 1] = static_cast<int>(clu::ld(clu::map(&s_cnt, tid)));
  if (tid == 0) s_off[0] = 0;
  __syncthreads();
  if (tid == 0)
    for (uint32_t r = 1; r <= CL; ++r) s_off[r] += s_off[r - 1];
  __syncthreads();
  const int C = s_off[CL];
  const bool ok = C >= k && C <= CAP;
  if (ok) {
    for (int c = tid; c < C; c += NT) {
      uint32_t r = 0;
      while (c >= s_off[r + 1]) ++r;
      const int j = c - s_off[r];
      s_ck[c] = clu::ld(clu::map(s_lk + j, r));
      if (rk == 0) s_ci[c] = static_cast<int32_t>(clu::ld(clu::map(s_li + j, r)));
    }
    for (int c = C + tid; c < (C + 127) / 128 * 128; c += NT) s_ck[c] = 0u;
    __syncthreads();
    const int cpc = (C + static_cast<int>(CL) - 1) / static_cast<int>(CL);
    const int c0 = static_cast<int>(rk) * cpc;
    kth_share<NT>(s_ck, C, k, c0, min(C, c0 + cpc), &s_T, 0u, 1u);
  }
  clu::sync();  // T in CTA 0; no remote access after this point
  if (rk != 0) return;

  if (ok) {
    const uint32_t T = s_T;
    int pk = 0;
    for (int c = tid; c < C; c += NT) pk += (s_ck[c] > T ? 1 : 0) + (s_ck[c] == T ? 0x10000 : 0);
    pk = block_sum<NT>(pk, s_warp);
    const int need_eq = k - (pk & 0xFFFF), n_eq = pk >> 16;
    int eq_seen = 0, out_pos = 0;
    for (int cb = 0; cb < C; cb += NT) {
      const int c = cb + tid;
      const uint32_t key = c < C ? s_ck[c] : 0u;
      bool sel;
      if (n_eq == need_eq) {
        sel = c < C && key >= T;
      } else {
        const bool eq = c < C && key == T;
        int eq_tot;
        const int eq_rank = eq_seen + block_scan_excl<NT>(eq ? 1 : 0, s_warp, &eq_tot);
        eq_seen += eq_tot;
        sel = c < C && (key > T || (eq && eq_rank < need_eq));
      }
      int sel_tot;
      const int p = out_pos + block_scan_excl<NT>(sel ? 1 : 0, s_warp, &sel_tot);
      out_pos += sel_tot;
      if (sel && p < k) {
        oi[p] = s_ci[c];
        if (os) os[p] = key_to_f32(key);
      }
    }
    return;
  }

  // ---- overflow: exact k-th key by bisection over the whole row (CTA 0) ----
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
