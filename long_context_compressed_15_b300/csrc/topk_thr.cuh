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
// maximum is the max of its groups'), which keeps the sort small while the
// number of entries at or above theta stays a small multiple of k.
//
// Grid (rows, segments): every CTA derives theta for its row, scans its
// segment of the scores and appends the entries with key >= theta to the
// row's candidate list.  The last CTA of a row to finish (atomic ticket)
// sorts the candidates by (score desc, index asc), keeps k, re-sorts them by
// index and writes the row.  If a row has more candidates than the list
// holds (massive exact ties at theta), that CTA instead finds the exact k-th
// key by bisection over the whole row and compacts it in index order.
// Counters are zeroed by the indexer kernel before this kernel runs.
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
  int seg;                 // entries per segment (one CTA)
  uint32_t* cand_key;      // row r at + r*cap
  int32_t* cand_idx;
  int cap;
  int* cnt;                // [rows] candidates appended
  int* done;               // [rows] CTAs finished
  int32_t* out_i;          // final list of row (b, i) at (b*Tq + i)*k
  float* out_s;            // optional
};

template <int NT>
__device__ __forceinline__ int block_sum(int v, int* s_red) {
  v = __reduce_add_sync(0xffffffffu, v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) t += s_red[w];
  return t;
}

// In-place bitonic sort of P (power of two) 64-bit values in shared memory.
template <int NT, bool DESC>
__device__ __forceinline__ void bitonic_sort(unsigned long long* v, int P) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < P / 2; t += NT) {
        const int i = 2 * t - (t & (stride - 1));
        const int j = i + stride;
        const bool up = (i & size) == 0;
        const unsigned long long a = v[i], b = v[j];
        const bool out_of_order = DESC ? (a < b) : (a > b);
        if (out_of_order == up) { v[i] = b; v[j] = a; }
      }
      __syncthreads();
    }
  }
}

template <int NT, int SORTCAP>
__global__ void __launch_bounds__(NT) k_topk_thr(TopkThrArgs a) {
  __shared__ unsigned long long s_v[SORTCAP];
  __shared__ int s_red[NT / 32];
  __shared__ uint32_t s_theta;
  __shared__ int s_last;

  const int tid = threadIdx.x, lane = tid & 31;
  const int row = blockIdx.x, segi = blockIdx.y;
  const int b = row / a.nq, i = a.q0 + row % a.nq;
  const int vis = visible_entries(__ldg(a.q_pos0 + b) + i, a.m, __ldg(a.n_valid + b), a.Ncap);
  const int k = a.k;
  int32_t* oi = a.out_i + (static_cast<int64_t>(b) * a.Tq + i) * k;
  float* os = a.out_s ? a.out_s + (static_cast<int64_t>(b) * a.Tq + i) * k : nullptr;
  const float* srow = a.scores + static_cast<int64_t>(row) * a.Ncap;

  if (vis <= k) {  // every visible entry is selected
    if (segi == 0)
      for (int p = tid; p < k; p += NT) {
        oi[p] = p < vis ? p : -1;
        if (os) os[p] = p < vis ? __ldcg(srow + p) : -INFINITY;
      }
    return;
  }

  const int lo = segi * a.seg, hi = min(vis, lo + a.seg);
  if (lo < hi) {
    // ---- theta: k-th largest super-group maximum ----
    const int G = (vis + a.gs - 1) / a.gs;
    const int f = (G + 2 * k - 1) / (2 * k);          // groups per super-group
    const int Gs = (G + f - 1) / f;                   // super-groups (<= 2k)
    if (tid == 0) s_theta = 0u;
    if (Gs >= k) {
      int P = 1;
      while (P < Gs) P <<= 1;
      const uint32_t* gm = a.gmax + static_cast<int64_t>(row) * a.g_stride;
      for (int s = tid; s < P; s += NT) {
        uint32_t mx = 0u;
        if (s < Gs) {
          const int g1 = min(G, (s + 1) * f);
          for (int g = s * f; g < g1; ++g) mx = max(mx, __ldcg(gm + g));
        }
        s_v[s] = mx;
      }
      __syncthreads();
      bitonic_sort<NT, true>(s_v, P);
      if (tid == 0) s_theta = static_cast<uint32_t>(s_v[k - 1]);
    }
    __syncthreads();
    const uint32_t theta = s_theta;
    // ---- append candidates of this segment ----
    uint32_t* ck = a.cand_key + static_cast<int64_t>(row) * a.cap;
    int32_t* ci = a.cand_idx + static_cast<int64_t>(row) * a.cap;
    for (int e0 = lo; e0 < hi; e0 += NT) {
      const int e = e0 + tid;
      uint32_t key = 0u;
      if (e < hi) key = f32_to_key(__ldcg(srow + e));
      const bool take = e < hi && key >= theta;
      const unsigned mask = __ballot_sync(0xffffffffu, take);
      if (mask) {
        const int leader = __ffs(mask) - 1;
        int base = 0;
        if (lane == leader) base = atomicAdd(a.cnt + row, __popc(mask));
        base = __shfl_sync(0xffffffffu, base, leader);
        const int slot = base + __popc(mask & ((1u << lane) - 1u));
        if (take && slot >= 0 && slot < a.cap) { ck[slot] = key; ci[slot] = e; }
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int ticket = atomicAdd(a.done + row, 1);
    s_last = ticket == static_cast<int>(gridDim.y) - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- the last CTA of the row selects ----
  const int C = atomicAdd(a.cnt + row, 0);
  if (C >= 0 && C <= a.cap && C <= SORTCAP) {
    int P = 1;
    while (P < C) P <<= 1;
    const uint32_t* ck = a.cand_key + static_cast<int64_t>(row) * a.cap;
    const int32_t* ci = a.cand_idx + static_cast<int64_t>(row) * a.cap;
    for (int s = tid; s < P; s += NT) {
      unsigned long long v = 0ull;
      if (s < C) v = (static_cast<unsigned long long>(__ldcg(ck + s)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(__ldcg(ci + s)));
      s_v[s] = v;
    }
    __syncthreads();
    bitonic_sort<NT, true>(s_v, P);  // (key desc, index asc)
    int K2 = 1;
    while (K2 < k) K2 <<= 1;
    // keep the first k, re-key by (index, key) and sort ascending by index
    unsigned long long tmp[(1024 + NT - 1) / NT];
    int c = 0;
    for (int s = tid; s < K2; s += NT, ++c) {
      unsigned long long v = ~0ull;
      if (s < k) {
        const unsigned long long x = s_v[s];
        const uint32_t idx = 0xFFFFFFFFu - static_cast<uint32_t>(x & 0xFFFFFFFFu);
        v = (static_cast<unsigned long long>(idx) << 32) | static_cast<uint32_t>(x >> 32);
      }
      tmp[c] = v;
    }
    __syncthreads();
    c = 0;
    for (int s = tid; s < K2; s += NT, ++c) s_v[s] = tmp[c];
    __syncthreads();
    bitonic_sort<NT, false>(s_v, K2);
    for (int p = tid; p < k; p += NT) {
      const unsigned long long v = s_v[p];
      oi[p] = static_cast<int32_t>(v >> 32);
      if (os) os[p] = key_to_f32(static_cast<uint32_t>(v & 0xFFFFFFFFu));
    }
  } else {
    // ---- overflow: exact k-th key by bisection over the whole row ----
    uint32_t T = 0u;
    for (int bit = 31; bit >= 0; --bit) {
      const uint32_t c = T | (1u << bit);
      int n = 0;
      for (int e = tid; e < vis; e += NT) n += f32_to_key(__ldcg(srow + e)) >= c;
      if (block_sum<NT>(n, s_red) >= k) T = c;
    }
    int ngt = 0;
    for (int e = tid; e < vis; e += NT) ngt += f32_to_key(__ldcg(srow + e)) > T;
    const int need_eq = k - block_sum<NT>(ngt, s_red);
    // ordered compaction: all keys > T, and the first need_eq keys == T by index
    int out_pos = 0, eq_seen = 0;
    for (int e0 = 0; e0 < vis; e0 += NT) {
      const int e = e0 + tid;
      const uint32_t key = e < vis ? f32_to_key(__ldcg(srow + e)) : 0u;
      const bool gt = e < vis && key > T, eq = e < vis && key == T;
      const unsigned meq = __ballot_sync(0xffffffffu, eq);
      // rank of this tie among the CTA's ties of this chunk
      __syncthreads();
      if (lane == 0) s_red[tid >> 5] = __popc(meq);
      __syncthreads();
      int before = 0, tot = 0;
      for (int w = 0; w < NT / 32; ++w) { const int c = s_red[w]; if (w < (tid >> 5)) before += c; tot += c; }
      const int eq_rank = eq_seen + before + __popc(meq & ((1u << lane) - 1u));
      eq_seen += tot;
      const bool sel = gt || (eq && eq_rank < need_eq);
      const unsigned msel = __ballot_sync(0xffffffffu, sel);
      __syncthreads();
      if (lane == 0) s_red[tid >> 5] = __popc(msel);
      __syncthreads();
      int sb = 0, st = 0;
      for (int w = 0; w < NT / 32; ++w) { const int c = s_red[w]; if (w < (tid >> 5)) sb += c; st += c; }
      if (sel) {
        const int p = out_pos + sb + __popc(msel & ((1u << lane) - 1u));
        if (p < k) { oi[p] = e; if (os) os[p] = key_to_f32(key); }
      }
      out_pos += st;
    }
  }
  __syncthreads();
  if (tid == 0) { a.cnt[row] = 0; a.done[row] = 0; }
}

}  // namespace lcc
