// Exact top-k of indexer scores by threshold filtering.  Source: "DeepSeek-V4가
// 이차적 어텐션 비용 없이 ...", section "두 가지 압축 전략: CSA 및 HCA" (the indexer
// keeps the top-k, typically about 128, compressed entries per query).
//
// Result: the min(k, visible) entries of a row with the largest scores, ties
// to the lower index, in ascending index order, padded with -1.
//
// The indexer kernels also write, for every group of `gs` consecutive
// entries of a row, the largest score key of the group.  Any k distinct
// groups contain k distinct entries at least as large as the smallest of
// their maxima, so theta = the k-th largest group maximum is a lower bound
// of the row's k-th largest score: every top-k entry has a key >= theta.
// Groups are merged into at most 2k super-groups first (a super-group's
// maximum is the max of its groups'), which keeps the search small while
// the number of entries at or above theta stays a small multiple of k.
//
// One CTA covers a segment of SEG = NT*PER entries (thread t owns PER
// consecutive entries, requested first).  It finds theta by counting over
// the super-group maxima (v is the k-th largest iff fewer than k values
// exceed v and at least k reach it), compacts the entries >= theta in index
// order (one block scan), finds the exact k-th largest key T among those
// candidates by the same count, and writes, in index order, every candidate
// above T and the lowest-index candidates equal to T.  A row longer than one
// segment is split over several CTAs that store their candidates in
// per-segment regions; the last CTA of the row to finish (atomic ticket)
// gathers the regions in segment order and selects.  When candidates
// overflow (massive exact ties at theta) the selecting CTA finds T by
// bisection over the whole row instead.  The per-row ticket counters are
// zeroed by the indexer kernel that runs just before this one.
#pragma once
#include "common.cuh"

namespace lcc {

struct TopkThrArgs {
  const float* scores;     // row r at scores + r*Ncap
  const uint32_t* gmax;    // row r at gmax + r*g_stride: order-preserving keys of group maxima
  int gs, g_stride;
  int Ncap;
  const int64_t* q_pos0;
  const int32_t* n_valid;
  int m, Tq, q0, nq;
  int k;
  // rows longer than one segment: segment s of row r keeps its candidates at
  // cand_* + (r*nseg + s)*seg_cap and their number at seg_cnt[r*nseg + s]
  uint32_t* cand_key;
  int32_t* cand_idx;
  int* seg_cnt;
  int seg_cap, nseg;
  int* done;               // [rows] CTAs of the row finished
  int32_t* out_i;          // final list of row (b, i) at (b*Tq + i)*k
  float* out_s;            // optional
};

// Exclusive prefix sum over the CTA; *total receives the sum.
template <int NT>
__device__ __forceinline__ int block_scan_excl(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  int pre = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const int t = s_warp[w];
    pre += w < warp ? t : 0;
    tot += t;
  }
  *total = tot;
  return pre + x - v;
}

template <int NT>
__device__ __forceinline__ int block_sum(int v, int* s_warp) {
  int tot;
  (void)block_scan_excl<NT>(v, s_warp, &tot);
  return tot;
}

// Threads that share the counting for one element: the largest power of two
// <= NT / n, between 1 and 32 (a group stays inside one warp).
template <int NT>
__device__ __forceinline__ int threads_per_elem(int n) {
  int t = 1;
  while (t < 32 && 2 * t * n <= NT) t <<= 1;
  return t;
}

// k-th largest of vals[0..n) (1 <= k <= n) by counting: the value v with
// #{x > v} < k <= #{x >= v}.  vals must be zero-padded up to a multiple of
// 128 entries (0 is never counted: every real value here is >= 1).  Every
// thread of the CTA calls this; the result is stored in *out.
template <int NT>
__device__ __forceinline__ void block_kth_largest(const uint32_t* vals, int n, int k, uint32_t* out) {
  const int tpe = threads_per_elem<NT>(n);
  const int np4 = (n + 127) / 128 * 32;  // 4-wide words to scan
  const int groups = NT / tpe, part = threadIdx.x % tpe;
  const uint4* v4 = reinterpret_cast<const uint4*>(vals);
  for (int it = 0; it < (n + groups - 1) / groups; ++it) {
    const int e = it * groups + static_cast<int>(threadIdx.x) / tpe;
    const uint32_t v = e < n ? vals[e] : 0xFFFFFFFFu;
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
    if (e < n && part == 0 && gt < k && ge >= k) *out = v;  // every writer stores the same value
  }
}

template <int NT, int PER, int CAP>
__global__ void __launch_bounds__(NT, 1) k_topk_thr(TopkThrArgs a) {
  constexpr int SEG = NT * PER;
  static_assert(PER % 4 == 0, "4-wide loads");
  __shared__ __align__(16) uint32_t s_ck[CAP + 128];   // candidates, index order (+ zero padding)
  __shared__ __align__(16) int32_t s_ci[CAP];
  __shared__ __align__(16) uint32_t s_g[CAP + 128];    // super-group maxima (+ zero padding)
  __shared__ int s_warp[NT / 32];
  __shared__ uint32_t s_theta, s_T;
  __shared__ int s_last;

  const int tid = threadIdx.x;
  const int row = blockIdx.x, segi = blockIdx.y;
  const int b = row / a.nq, i = a.q0 + row % a.nq;
  const int k = a.k;
  const float* srow = a.scores + static_cast<int64_t>(row) * a.Ncap;
  const int64_t qpos = __ldg(a.q_pos0 + b) + i;   // inputs of the call: ready before the indexer ran
  const int nval = __ldg(a.n_valid + b);
  pdl_trigger();
  pdl_wait();  // scores, group maxima and counters come from the indexer kernel
  // This thread's PER consecutive scores of the segment, requested before
  // anything that depends on the visible count (masked once it is known).
  const int lo = segi * SEG;
  const int e0 = lo + tid * PER;
  const int cap_hi = min(a.Ncap, lo + SEG);
  float sv[PER];
  if ((a.Ncap & 3) == 0) {
#pragma unroll
    for (int u = 0; u < PER; u += 4) {
      const float4 v = e0 + u < cap_hi ? __ldcg(reinterpret_cast<const float4*>(srow + e0 + u))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
      sv[u] = v.x; sv[u + 1] = v.y; sv[u + 2] = v.z; sv[u + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < PER; ++u) sv[u] = e0 + u < cap_hi ? __ldcg(srow + e0 + u) : 0.f;
  }
  const int vis = visible_entries(qpos, a.m, nval, a.Ncap);
  int32_t* oi = a.out_i + (static_cast<int64_t>(b) * a.Tq + i) * k;
  float* os = a.out_s ? a.out_s + (static_cast<int64_t>(b) * a.Tq + i) * k : nullptr;
  const bool multi = vis > SEG;

  if (vis <= k) {  // every visible entry is selected
    if (segi == 0)
      for (int p = tid; p < k; p += NT) {
        oi[p] = p < vis ? p : -1;
        if (os) os[p] = p < vis ? __ldcg(srow + p) : -INFINITY;
      }
    return;
  }
  if (!multi && segi > 0) return;

  const int hi = min(vis, lo + SEG);
  int C = 0;  // candidates in s_ck / s_ci (index order); -1 = overflow
  if (lo < hi) {
    // ---- theta: k-th largest super-group maximum ----
    const int G = (vis + a.gs - 1) / a.gs;
    const int f = (G + 2 * k - 1) / (2 * k);   // groups per super-group
    const int Gs = (G + f - 1) / f;            // super-groups (<= 2k <= CAP)
    if (tid == 0) s_theta = 0u;                // fewer than k groups: every entry is a candidate
    if (Gs >= k) {
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
      __syncthreads();
      block_kth_largest<NT>(s_g, Gs, k, &s_theta);
    }
    __syncthreads();
    const uint32_t theta = s_theta;
    // ---- ordered compaction of the entries >= theta ----
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
        if (pos < CAP) { s_ck[pos] = keys[u]; s_ci[pos] = e0 + u; }
        ++pos;
      }
    }
    C = tot <= CAP ? tot : -1;
    __syncthreads();
  }

  if (multi) {
    // ---- store this segment's candidates; the last CTA of the row gathers them in order ----
    const int64_t rs = static_cast<int64_t>(row) * a.nseg + segi;
    uint32_t* ck = a.cand_key + rs * a.seg_cap;
    int32_t* ci = a.cand_idx + rs * a.seg_cap;
    const int nstore = (C >= 0 && C <= a.seg_cap) ? C : -1;
    for (int u = tid; u < nstore; u += NT) { ck[u] = s_ck[u]; ci[u] = s_ci[u]; }
    if (tid == 0) a.seg_cnt[rs] = nstore;
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const int ticket = atomicAdd(a.done + row, 1);
      s_last = ticket == static_cast<int>(gridDim.y) - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // gather every segment's list, in segment (= index) order
    C = 0;
    for (int sg = 0; sg < a.nseg; ++sg) {
      const int64_t r2 = static_cast<int64_t>(row) * a.nseg + sg;
      const int n2 = __ldcg(a.seg_cnt + r2);
      if (n2 < 0 || C + n2 > CAP) { C = -1; break; }
      for (int u = tid; u < n2; u += NT) {
        s_ck[C + u] = __ldcg(a.cand_key + r2 * a.seg_cap + u);
        s_ci[C + u] = __ldcg(a.cand_idx + r2 * a.seg_cap + u);
      }
      C += n2;
    }
    __syncthreads();
    if (tid == 0) a.done[row] = 0;
  }

  uint32_t T;
  if (C >= k) {
    // ---- exact k-th largest key among the candidates ----
    for (int c = C + tid; c < (C + 127) / 128 * 128; c += NT) s_ck[c] = 0u;
    __syncthreads();
    block_kth_largest<NT>(s_ck, C, k, &s_T);
    __syncthreads();
    T = s_T;
    // counts of keys above T and equal to T, in one reduction (both <= CAP < 2^16)
    int pk = 0;
    for (int c = tid; c < C; c += NT) pk += (s_ck[c] > T ? 1 : 0) + (s_ck[c] == T ? 0x10000 : 0);
    pk = block_sum<NT>(pk, s_warp);
    const int need_eq = k - (pk & 0xFFFF), n_eq = pk >> 16;
    // ---- ordered output: keys > T, and the first need_eq keys == T ----
    int eq_seen = 0, out_pos = 0;
    for (int c0 = 0; c0 < C; c0 += NT) {
      const int c = c0 + tid;
      const uint32_t key = c < C ? s_ck[c] : 0u;
      bool sel;
      if (n_eq == need_eq) {  // every key equal to T is kept (the usual case): one scan
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

  // ---- overflow (or an inconsistent count): exact k-th key by bisection over the whole row ----
  T = 0u;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t c = T | (1u << bit);
    int n = 0;
    for (int e = tid; e < vis; e += NT) n += f32_to_key(__ldcg(srow + e)) >= c;
    if (block_sum<NT>(n, s_warp) >= k) T = c;
  }
  int ngt = 0;
  for (int e = tid; e < vis; e += NT) ngt += f32_to_key(__ldcg(srow + e)) > T;
  const int need_eq = k - block_sum<NT>(ngt, s_warp);
  int out_pos = 0, eq_seen = 0;
  for (int e0 = 0; e0 < vis; e0 += NT) {
    const int e = e0 + tid;
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
