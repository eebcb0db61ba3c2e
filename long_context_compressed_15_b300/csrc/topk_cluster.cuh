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
// over the CL CTAs of a cluster so that each SM loads 1/CL of the row:
//   1. every CTA loads its SEG = NT*PER scores, builds all super-group
//      maxima from the group maxima and finds theta itself (the same
//      deterministic selection in every CTA: no exchange);
//   2. every CTA compacts its entries >= theta (a run in index order) and
//      stores it, with its length, into its own CAP/CL-slot region of CTA 0
//      through distributed shared memory; one cluster barrier;
//   3. CTA 0 takes the runs in CTA (= index) order, one candidate per
//      thread, selects the exact k-th largest key T and writes every
//      candidate above T and the lowest-index candidates equal to T.
// Both selections (theta among the super-group maxima, T among the
// candidates) sort up to NT values, one per thread, with a bitonic network
// and take the k-th; larger sets take 256-bin histogram rounds, each
// narrowing the key interval to the bin that holds the k-th value (at most
// four rounds for 32-bit keys).  A run that does not fit its region (massive exact ties) falls back
// to a bisection over the row's scores in CTA 0.  Control flow through the
// cluster barriers depends only on per-row values, so every CTA of the
// cluster meets each barrier.
#pragma once
#include "topk_thr.cuh"

namespace lcc {

// k-th largest of vals[0..n) (1 <= k <= n), returned to every thread of
// the CTA (every thread calls this).  Each round histograms the values in
// the current interval [lo, hi] into 256 bins of width w = ceil((hi-lo+1)/256),
// finds the bin holding the k-th largest of them and narrows the interval to
// it; with w = 1 the bin is a single value.
template <int NT>
__device__ __forceinline__ uint32_t block_kth_hist(const uint32_t* vals, int n, int k, uint32_t* s_hist,
                                                   uint32_t* s_bc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  for (int i = tid; i < n; i += NT) {
    const uint32_t v = vals[i];
    mn = min(mn, v);
    mx = max(mx, v);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  for (int b = tid; b < 256; b += NT) s_hist[b] = 0u;
  if (lane == 0) {
    atomicMin(s_bc + 2, mn);
    atomicMax(s_bc + 3, mx);
  }
  __syncthreads();
  uint32_t lo = s_bc[2], hi = s_bc[3];
  int krem = k;
  while (true) {
    const uint64_t range = static_cast<uint64_t>(hi) - lo + 1;
    const uint32_t w = static_cast<uint32_t>((range + 255) / 256);
    for (int i = tid; i < n; i += NT) {
      const uint32_t v = vals[i];
      if (v >= lo && v <= hi) atomicAdd(s_hist + (v - lo) / w, 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane L owns bins 8L .. 8L+7; suffix sums from the top bin down
      uint32_t h[8], t = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        h[j] = s_hist[lane * 8 + j];
        t += h[j];
      }
      uint32_t above = t;  // inclusive suffix over lanes >= lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, above, o);
        if (lane + o < 32) above += y;
      }
      uint32_t run = above - t;  // values in bins of higher lanes
      int bstar = -1;
      uint32_t ab = 0;
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        if (bstar < 0 && run + h[j] >= static_cast<uint32_t>(krem)) {
          bstar = lane * 8 + j;
          ab = run;
        }
        run += h[j];
      }
      int best = bstar;
#pragma unroll
      for (int o = 16; o; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
      if (bstar == best && bstar >= 0) {
        s_bc[0] = static_cast<uint32_t>(bstar);
        s_bc[1] = ab;
      }
    }
    __syncthreads();
    const uint32_t bs = s_bc[0];
    krem -= static_cast<int>(s_bc[1]);
    const uint32_t nlo = lo + bs * w;
    const uint64_t nhi = static_cast<uint64_t>(nlo) + w - 1;
    hi = nhi < hi ? static_cast<uint32_t>(nhi) : hi;
    lo = nlo;
    if (w == 1u) break;
    for (int b = tid; b < 256; b += NT) s_hist[b] = 0u;
    __syncthreads();
  }
  __syncthreads();  // s_bc and s_hist may be reused after the return
  if (tid == 0) {
    s_bc[2] = 0xFFFFFFFFu;
    s_bc[3] = 0u;
  }
  return lo;
}

// k-th largest (1 <= k <= NT) of the values held one per thread (v; padding
// values must be 0), returned to every thread.  A bitonic sort network over
// the CTA's threads into descending order: partners within a warp exchange
// by shuffles, partners in other warps through shared memory (x: NT words).
// Every stage is a few independent instructions per thread, so the whole
// CTA shares the work instead of one warp walking a long dependent chain.
template <int NT>
__device__ __forceinline__ uint32_t block_kth_bitonic(uint32_t v, int k, uint32_t* x, uint32_t* s_bc) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int kk = 2; kk <= NT; kk <<= 1) {
#pragma unroll
    for (int j = kk >> 1; j > 0; j >>= 1) {
      uint32_t u;
      if (j < 32) {
        u = __shfl_xor_sync(0xffffffffu, v, j);
      } else {
        x[tid] = v;
        __syncthreads();
        u = x[tid ^ j];
        __syncthreads();
      }
      // blocks of kk threads alternate direction; the last merge is descending
      const bool desc = (tid & kk) == 0;
      const bool low = (tid & j) == 0;
      v = (low == desc) ? max(v, u) : min(v, u);
    }
  }
  if (tid == k - 1) s_bc[0] = v;
  __syncthreads();
  const uint32_t r = s_bc[0];
  __syncthreads();
  return r;
}

// k-th largest of vals[0..n) (1 <= k <= n <= 32*PL) by one warp, without
// block barriers: T is built bit by bit from the top as the largest key with
// at least k values >= T (each lane counts its PL values, one warp
// reduction per bit).  Returned to every lane of the calling warp.
template <int PL>
__device__ __forceinline__ uint32_t warp_kth_bits(const uint32_t* vals, int n, int k) {
  const int lane = threadIdx.x & 31;
  uint32_t v[PL];
#pragma unroll
  for (int j = 0; j < PL; ++j) {
    const int i = j * 32 + lane;
    v[j] = i < n ? vals[i] : 0u;
  }
  uint32_t T = 0u;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t c = T | (1u << bit);
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < PL; ++j) cnt += v[j] >= c ? 1 : 0;
    if (static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(cnt))) >= k) T = c;
  }
  return T;
}

// Rank of the value v at position pos among vals[0..n): how many values beat
// it (a larger value, or an equal value at a lower position).  Called by whole
// warps with pos = wb + lane, wb a multiple of 32 (the same in every lane);
// vals 16-byte aligned in shared memory.  Positions below the warp's own
// compare with >=, those above with >, the warp's own 32 one by one; the
// vector loads are warp-wide broadcasts.
__device__ __forceinline__ int rank_by_count(const uint32_t* vals, int n, uint32_t v, int wb, int pos) {
  if (wb >= n) return 0;
  const uint4* v4 = reinterpret_cast<const uint4*>(vals);
  int r0 = 0, r1 = 0;
  const int a4 = wb >> 2;
#pragma unroll 4
  for (int j = 0; j < a4; ++j) {
    const uint4 u = v4[j];
    r0 += (u.x >= v ? 1 : 0) + (u.y >= v ? 1 : 0);
    r1 += (u.z >= v ? 1 : 0) + (u.w >= v ? 1 : 0);
  }
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    const int j = wb + t;
    if (j < n) {
      const uint32_t u = vals[j];
      r0 += (u > v || (u == v && j < pos)) ? 1 : 0;
    }
  }
  const int b = wb + 32, n4 = n >> 2;
#pragma unroll 4
  for (int j = b >> 2; j < n4; ++j) {
    const uint4 u = v4[j];
    r0 += (u.x > v ? 1 : 0) + (u.y > v ? 1 : 0);
    r1 += (u.z > v ? 1 : 0) + (u.w > v ? 1 : 0);
  }
  for (int j = max(b, n4 << 2); j < n; ++j) r0 += vals[j] > v ? 1 : 0;
  return r0 + r1;
}

template <int NT, int PER, int CAP, int MAXG>
struct TopkClSmem {
  static constexpr size_t ck = 0;                   // candidate keys, in arrival order (CTA 0)
  static constexpr size_t ci = ck + CAP * 4;        // ... their entries
  static constexpr size_t ok = ci + CAP * 4;        // candidate keys in index order (CTA 0)
  static constexpr size_t oi = ok + CAP * 4;        // ... their entries
  static constexpr size_t g = oi + CAP * 4;         // super-group maxima
  static constexpr size_t total = g + MAXG * 4;
};

// Where a row's result goes: entry e (and, when wanted, its score) at place p.
struct TopkOut {
  int32_t* oi;
  float* os;
  __device__ __forceinline__ void put(int p, int e) const { oi[p] = e; }
  __device__ __forceinline__ bool scores() const { return os != nullptr; }
  __device__ __forceinline__ void put_score(int p, float v) const { os[p] = v; }
};

// The top-k of one row by the CTAs of a thread-block cluster (every CTA calls
// this with the same row, after the scores and group maxima are visible).
// CTA 0 writes the result through `out`; every CTA returns after the same
// number of cluster barriers.  MAXG: most super-groups (2k); callers route
// rows here only when 2k <= MAXG, k * (entries per group) <= CAP and the row
// fits (CTAs of the cluster) * NT * PER entries.
template <int NT, int PER, int CAP, int MAXG, class Out>
__device__ __forceinline__ void topk_cluster_row(const TopkThrArgs a, uint8_t* smem, int row, const Out out) {
  using L = TopkClSmem<NT, PER, CAP, MAXG>;
  constexpr int SEG = NT * PER;
  static_assert(PER % 4 == 0, "4-wide loads");
  static_assert(NT <= 256 && (NT & (NT - 1)) == 0, "the sorts exchange through s_hist, one word per thread");
  uint32_t* s_ck = reinterpret_cast<uint32_t*>(smem + L::ck);
  int32_t* s_ci = reinterpret_cast<int32_t*>(smem + L::ci);
  uint32_t* s_ok = reinterpret_cast<uint32_t*>(smem + L::ok);
  int32_t* s_oi = reinterpret_cast<int32_t*>(smem + L::oi);
  uint32_t* s_g = reinterpret_cast<uint32_t*>(smem + L::g);
  __shared__ int s_warp[NT / 32];
  __shared__ uint32_t s_hist[256];
  __shared__ uint32_t s_bc[4];
  __shared__ uint32_t s_rc[8];  // CTA 0: length of each CTA's run

  const int tid = threadIdx.x;
  const uint32_t rk = clu::rank(), CL = clu::size();
  if (tid == 0) {  // before the arrive, so that no remote access can precede these
    s_bc[2] = 0xFFFFFFFFu;
    s_bc[3] = 0u;
  }
  clu::arrive();  // every CTA of the cluster has started before any remote access (wait below)
  const int b = row / a.nq, i = a.q0 + row % a.nq;
  const int k = a.k;
  const float* srow = a.scores + static_cast<int64_t>(row) * a.Ncap;
  const int64_t qpos = __ldg(a.q_pos0 + b) + i;
  const int nval = __ldg(a.n_valid + b);
  const int vis = visible_entries(qpos, a.m, nval, a.Ncap);

  if (vis <= k) {  // every visible entry is selected
    clu::wait();  // every CTA has started: `out` may write into their shared memory
    if (rk == 0)
      for (int p = tid; p < k; p += NT) {
        out.put(p, p < vis ? p : -1);
        if (out.scores()) out.put_score(p, p < vis ? __ldcg(srow + p) : -INFINITY);
      }
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

  // theta from the super-group maxima (the same value in every CTA)
  const int G = (vis + a.gs - 1) / a.gs;
  const int f = (G + 2 * k - 1) / (2 * k);
  const int Gs = (G + f - 1) / f;
  uint32_t theta = 0u;  // fewer than k super-groups: every visible entry is a candidate
  if (Gs >= k) {
    const uint32_t* gm = a.gmax + static_cast<int64_t>(row) * a.g_stride;
    if (f == 2 && (reinterpret_cast<uintptr_t>(gm) & 7) == 0 && 2 * Gs <= a.g_stride) {
      // the usual pairing: both groups of a super-group in one 8-byte load
      for (int s = tid; s < Gs; s += NT) {
        const uint2 pr = __ldcg(reinterpret_cast<const uint2*>(gm) + s);
        s_g[s] = 2 * s + 1 < G ? max(pr.x, pr.y) : pr.x;
      }
    } else {
      for (int s = tid; s < Gs; s += NT) {
        uint32_t mx = 0u;
        const int g1 = min(G, (s + 1) * f);
        for (int g = s * f; g < g1; ++g) mx = max(mx, __ldcg(gm + g));
        s_g[s] = mx;
      }
    }
    __syncthreads();
    if (Gs <= NT) {
      theta = block_kth_bitonic<NT>(tid < Gs ? s_g[tid] : 0u, k, s_hist, s_bc);
    } else {
      theta = block_kth_hist<NT>(s_g, Gs, k, s_hist, s_bc);
    }
  }

  // this CTA's run of candidates, stored into its own region of CTA 0 (CAP / CL
  // slots per CTA: the runs lie in CTA order = index order, with no atomics)
  const int RUN = CAP / static_cast<int>(CL);
  uint32_t keys[PER];
  int n = 0;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    keys[u] = e0 + u < hi ? f32_to_key(sv[u]) : 0u;
    n += keys[u] >= theta && keys[u] != 0u;
  }
  int tot;
  int pos = block_scan_excl<NT>(n, s_warp, &tot);
  clu::wait();
  if (tid == 0) clu::st(clu::map(s_rc + rk, 0), static_cast<uint32_t>(tot));
  {
    const uint32_t rck = clu::map(s_ck, 0), rci = clu::map(s_ci, 0);
    const int base = static_cast<int>(rk) * RUN;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      if (keys[u] >= theta && keys[u] != 0u) {
        if (pos < RUN) {
          clu::st(rck + 4u * (base + pos), keys[u]);
          clu::st(rci + 4u * (base + pos), static_cast<uint32_t>(e0 + u));
        }
        ++pos;
      }
    }
  }
  clu::sync();  // CTA 0 holds every run; no remote access after this point
  if (rk != 0) return;

  int C = 0;
  bool fits = true;
  for (uint32_t r = 0; r < CL; ++r) {
    const int rc = static_cast<int>(s_rc[r]);
    C += rc;
    fits = fits && rc <= RUN;
  }
  if (fits && C >= k && C <= NT) {
    // the usual case (a few hundred candidates): candidate t of the concatenated
    // runs in thread t, the exact k-th key T by a bitonic sort, then every key
    // above T and the lowest-index keys equal to T, in index order
    uint32_t v = 0u;
    int ent = -1;
    if (tid < C) {
      int r = 0, pre = 0;
      while (tid >= pre + static_cast<int>(s_rc[r])) pre += static_cast<int>(s_rc[r++]);
      v = s_ck[r * RUN + tid - pre];
      ent = s_ci[r * RUN + tid - pre];
    }
    const uint32_t T = block_kth_bitonic<NT>(v, k, s_hist, s_bc);
    const int pk = block_sum<NT>((v > T ? 1 : 0) + (v == T ? 0x10000 : 0), s_warp);
    const int need_eq = k - (pk & 0xFFFF), n_eq = pk >> 16;
    bool sel;
    if (n_eq == need_eq) {
      sel = tid < C && v >= T;
    } else {
      const bool eq = tid < C && v == T;
      int eq_tot;
      const int eq_rank = block_scan_excl<NT>(eq ? 1 : 0, s_warp, &eq_tot);
      sel = tid < C && (v > T || (eq && eq_rank < need_eq));
    }
    int sel_tot;
    const int p = block_scan_excl<NT>(sel ? 1 : 0, s_warp, &sel_tot);
    if (sel && p < k) {
      out.put(p, ent);
      if (out.scores()) out.put_score(p, key_to_f32(v));
    }
    return;
  }
  if (fits && C >= k) {
    // more candidates than threads: lay the runs out contiguously first
    int off = 0;
    for (uint32_t r = 0; r < CL; ++r) {
      const int rc = static_cast<int>(s_rc[r]);
      for (int c = tid; c < rc; c += NT) {
        s_ok[off + c] = s_ck[r * RUN + c];
        s_oi[off + c] = s_ci[r * RUN + c];
      }
      off += rc;
    }
    __syncthreads();
    uint32_t T;
    if (C <= 512) {  // one warp, no block barriers
      if (tid < 32) {
        const uint32_t t = warp_kth_bits<16>(s_ok, C, k);
        if (tid == 0) s_bc[0] = t;
      }
      __syncthreads();
      T = s_bc[0];
    } else {
      T = block_kth_hist<NT>(s_ok, C, k, s_hist, s_bc);
    }
    int pk = 0;
    for (int c = tid; c < C; c += NT) pk += (s_ok[c] > T ? 1 : 0) + (s_ok[c] == T ? 0x10000 : 0);
    pk = block_sum<NT>(pk, s_warp);
    const int need_eq = k - (pk & 0xFFFF), n_eq = pk >> 16;
    int eq_seen = 0, out_pos = 0;
    for (int cb = 0; cb < C; cb += NT) {
      const int c = cb + tid;
      const uint32_t key = c < C ? s_ok[c] : 0u;
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
        out.put(p, s_oi[c]);
        if (out.scores()) out.put_score(p, key_to_f32(key));
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
      out.put(p, e);
      if (out.scores()) out.put_score(p, key_to_f32(key));
    }
  }
}

// One thread-block cluster per row; the rows of the call are blockIdx.x / (cluster size).
template <int NT, int PER, int CAP, int MAXG>
__global__ void __launch_bounds__(NT) k_topk_cluster(TopkThrArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int row = static_cast<int>(blockIdx.x / clu::size());
  const int b = row / a.nq, i = a.q0 + row % a.nq;
  const int64_t o = (static_cast<int64_t>(b) * a.Tq + i) * a.k;
  pdl_trigger();
  pdl_wait();  // scores and group maxima come from the indexer kernel
  topk_cluster_row<NT, PER, CAP, MAXG>(a, smem, row, TopkOut{a.out_i + o, a.out_s ? a.out_s + o : nullptr});
}

}  // namespace lcc
