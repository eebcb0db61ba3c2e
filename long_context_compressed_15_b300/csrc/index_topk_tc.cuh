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
__device__ __forceinline__ int warp_compact_t(uint32_t* keys, int32_t* ids, int n, int k, uint32_t& T_out);

template <int CAPQ>
__device__ __forceinline__ int warp_compact(uint32_t* keys, int32_t* ids, int n, int k, uint32_t* theta) {
  uint32_t T = 0u;
  const int r = warp_compact_t<CAPQ>(keys, ids, n, k, T);
  if (n > k && (threadIdx.x & 31) == 0) *theta = T;
  return r;
}

// As warp_compact, with the k-th key returned to every lane (when n > k).
template <int CAPQ>
__device__ __forceinline__ int warp_compact_t(uint32_t* keys, int32_t* ids, int n, int k, uint32_t& T_out) {
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
  T_out = T;
  return k;
}

// Shrink a buffer that is filling up without selecting exactly: one warp
// histograms its n keys into 256 bins spread linearly over [min, max] of the
// buffer (a monotone map of the key), finds the highest bin b* such that the
// bins >= b* hold at least k keys, and keeps exactly the keys in those bins,
// in buffer (= index) order.  Every key of the buffer's top-k is kept, and
// the smallest kept key m is a valid threshold for later entries: at least
// k kept keys are >= m and all have lower indices, so a later entry with
// key <= m can never enter the top-k.  Returns the new count (>= min(n, k))
// and sets m_out; falls back to the exact cut when the bins do not separate
// (many equal keys) and the buffer would stay fuller than `room_left`.
// hist: 256 words of shared memory private to the warp.
// With kp > 0 it also sets *p_out to a key that at least kp kept keys reach
// (the smallest kept key of the highest bins holding kp keys; the k-th key
// after an exact cut).
template <int CAPQ>
__device__ __forceinline__ int warp_cut(uint32_t* keys, int32_t* ids, int n, int k, int max_keep, uint32_t* hist,
                                        uint32_t& m_out, int kp = 0, uint32_t* p_out = nullptr) {
  constexpr int V = CAPQ / 32;
  const int lane = threadIdx.x & 31;
  uint32_t v[V];
  int32_t id[V];
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < n ? keys[e] : 0u;
    id[i] = e < n ? ids[e] : 0;
    if (e < n) { lo = min(lo, v[i]); hi = max(hi, v[i]); }
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
#pragma unroll
  for (int j = 0; j < 8; ++j) hist[lane * 8 + j] = 0u;
  __syncwarp();
  const float inv = 256.f / (static_cast<float>(hi - lo) + 1.f);
  uint32_t bins[V / 4 > 0 ? V / 4 : 1];  // four 8-bit bin numbers per word
#pragma unroll
  for (int i = 0; i < V / 4; ++i) bins[i] = 0u;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    const uint32_t bn = min(255u, static_cast<uint32_t>(static_cast<float>(v[i] - lo) * inv));
    bins[i / 4] |= bn << (8 * (i % 4));
    if (e < n) atomicAdd(hist + bn, 1u);
  }
  __syncwarp();
  // highest bin b* whose suffix count reaches k (lane L owns bins 8L .. 8L+7)
  uint32_t h[8], t = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) { h[j] = hist[lane * 8 + j]; t += h[j]; }
  uint32_t above = t;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, above, o);
    if (lane + o < 32) above += y;
  }
  uint32_t run = above - t;
  int bstar = -1, bp = -1;
  uint32_t keep_n = 0;
#pragma unroll
  for (int j = 7; j >= 0; --j) {
    if (bstar < 0 && run + h[j] >= static_cast<uint32_t>(k)) { bstar = lane * 8 + j; keep_n = run + h[j]; }
    if (bp < 0 && run + h[j] >= static_cast<uint32_t>(kp)) bp = lane * 8 + j;
    run += h[j];
  }
  int best = __reduce_max_sync(0xffffffffu, bstar);
  const int bestp = kp > 0 ? __reduce_max_sync(0xffffffffu, bp) : 256;
  const uint32_t kept = __shfl_sync(0xffffffffu, keep_n, __ffs(__ballot_sync(0xffffffffu, bstar == best)) - 1);
  __syncwarp();  // everyone has read the histogram before the next use
  if (best < 0 || static_cast<int>(kept) > max_keep) {
    uint32_t T = 0u;
    const int r = warp_compact_t<CAPQ>(keys, ids, n, k, T);
    m_out = T;
    if (kp > 0) *p_out = T;
    return r;
  }
  int out = 0;
  uint32_t mk = 0xFFFFFFFFu, mp = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    const int bn = static_cast<int>((bins[i / 4] >> (8 * (i % 4))) & 255u);
    const bool keep = e < n && bn >= best;
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int p = out + __popc(m & ((1u << lane) - 1u));
      keys[p] = v[i];
      ids[p] = id[i];
      mk = min(mk, v[i]);
      if (bn >= bestp) mp = min(mp, v[i]);
    }
    out += __popc(m);
  }
  __syncwarp();
  m_out = __reduce_min_sync(0xffffffffu, mk);
  if (kp > 0) *p_out = __reduce_min_sync(0xffffffffu, mp);
  return out;
}


// Highest bin b of a 256-bin histogram (hist, shared memory, 8 bins per
// lane) such that the bins >= b hold at least `need` keys; -1 if none.
__device__ __forceinline__ int hist_top_bin(const uint32_t* hist, int need) {
  const int lane = threadIdx.x & 31;
  uint32_t h[8], t = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) { h[j] = hist[lane * 8 + j]; t += h[j]; }
  uint32_t above = t;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, above, o);
    if (lane + o < 32) above += y;
  }
  uint32_t run = above - t;
  int bstar = -1;
#pragma unroll
  for (int j = 7; j >= 0; --j) {
    if (bstar < 0 && run + h[j] >= static_cast<uint32_t>(need)) bstar = lane * 8 + j;
    run += h[j];
  }
  return __reduce_max_sync(0xffffffffu, bstar);
}

// Output of a kept set stored as four runs [kb[r], kb[r+1]) that are each in
// ascending index order: the entry at p goes to slot sum_r #{entries of run r
// with a lower index} (its own run contributes p - kb[r]), found by
// fixed-step binary searches (runs shorter than 256), two entries per lane in
// flight; slots kb[4] .. k-1 get -1 / -inf.
template <int CAPB>
__device__ __forceinline__ void runs_out(const uint32_t* keys, const int32_t* ids, const int (&kb)[5], int k,
                                         int32_t* oi, float* os) {
  static_assert(CAPB <= 256, "runs shorter than 256");
  const int lane = threadIdx.x & 31;
  const int nk = kb[4];
  for (int p0 = 0; p0 < nk; p0 += 64) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int p = p0 + 32 * h + lane;
      if (p < nk) {
        const int32_t me = ids[p];
        int rank = 0;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int s0 = kb[r], s1 = kb[r + 1];
          int pos = s0;
#pragma unroll
          for (int step = 128; step >= 1; step >>= 1)
            if (pos + step <= s1 && ids[pos + step - 1] < me) pos += step;
          rank += pos - s0;
        }
        oi[rank] = me;
        if (os) os[rank] = key_to_f32(keys[p]);
      }
    }
  }
  for (int o = nk + lane; o < k; o += 32) {
    oi[o] = -1;
    if (os) os[o] = -INFINITY;
  }
}

// Exact top-k (key desc, index asc) of the union of four candidate lists
// that are each in ascending index order (lists r at keys + r*CAPB, counts
// cnt4[r]), written to oi / os in ascending index order and padded with -1
// / -inf up to k.  One warp.  P is a key that the union's k-th largest key
// reaches (0 = none): entries below it are dropped first.  When at most CAPB
// entries remain, they are gathered into one list and selected once (the
// bitwise select starts at the highest bit in which the remaining keys
// differ), and each kept entry finds its output slot by binary searches in
// the other lists.  More than CAPB are first cut to the keys of the highest
// bins of a 256-bin histogram spread linearly over their key range that hold
// at least k of them (a superset of the top-k, in list order); if that still
// leaves more than CAPB (many equal keys), every list is cut to its own top-k
// and the lists are merged one after the other.  The lists' storage is
// overwritten; hist: 256 words of shared memory private to the warp.
template <int CAPB>
__device__ __forceinline__ void union_topk_general(uint32_t* keys, int32_t* ids, const int* cnt4, uint32_t P, int k,
                                                   uint32_t* hist, int32_t* oi, float* os) {
  const int lane = threadIdx.x & 31;
  const unsigned below = (1u << lane) - 1u;
  int c[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {  // drop the entries below P (stable, in place)
    uint32_t* kr = keys + r * CAPB;
    int32_t* ir = ids + r * CAPB;
    const int n = cnt4[r];
    int out = 0;
    for (int e0 = 0; e0 < n; e0 += 32) {
      const int e = e0 + lane;
      uint32_t kv = 0u;
      int32_t iv = 0;
      if (e < n) { kv = kr[e]; iv = ir[e]; }
      const bool keep = e < n && kv >= P;
      const unsigned m = __ballot_sync(0xffffffffu, keep);
      __syncwarp();
      if (keep) { kr[out + __popc(m & below)] = kv; ir[out + __popc(m & below)] = iv; }
      out += __popc(m);
    }
    c[r] = out;
  }
  __syncwarp();
  int ntot = c[0] + c[1] + c[2] + c[3];
  if (ntot > CAPB) {
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
    for (int r = 0; r < 4; ++r)
      for (int e = lane; e < c[r]; e += 32) {
        const uint32_t kv = keys[r * CAPB + e];
        lo = min(lo, kv);
        hi = max(hi, kv);
      }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
#pragma unroll
    for (int j = 0; j < 8; ++j) hist[lane * 8 + j] = 0u;
    __syncwarp();
    const float inv = 256.f / (static_cast<float>(hi - lo) + 1.f);
    auto bin = [&](uint32_t kv) { return min(255u, static_cast<uint32_t>(static_cast<float>(kv - lo) * inv)); };
#pragma unroll
    for (int r = 0; r < 4; ++r)
      for (int e = lane; e < c[r]; e += 32) atomicAdd(hist + bin(keys[r * CAPB + e]), 1u);
    __syncwarp();
    const int best = hist_top_bin(hist, k);
    __syncwarp();
    if (best >= 0) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {  // keep the bins >= best (stable, in place)
        uint32_t* kr = keys + r * CAPB;
        int32_t* ir = ids + r * CAPB;
        const int n = c[r];
        int out = 0;
        for (int e0 = 0; e0 < n; e0 += 32) {
          const int e = e0 + lane;
          uint32_t kv = 0u;
          int32_t iv = 0;
          if (e < n) { kv = kr[e]; iv = ir[e]; }
          const bool keep = e < n && static_cast<int>(bin(kv)) >= best;
          const unsigned m = __ballot_sync(0xffffffffu, keep);
          __syncwarp();
          if (keep) { kr[out + __popc(m & below)] = kv; ir[out + __popc(m & below)] = iv; }
          out += __popc(m);
        }
        c[r] = out;
      }
      __syncwarp();
      ntot = c[0] + c[1] + c[2] + c[3];
    }
  }
  if (ntot > CAPB) {
    // many equal keys: each list down to its own top-k, then merged in turn
    int n = 0;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      uint32_t T;
      const int cr = warp_compact_t<CAPB>(keys + r * CAPB, ids + r * CAPB, c[r], k, T);
      if (r == 0) { n = cr; continue; }
      for (int e0 = 0; e0 < cr; e0 += 32) {  // behind the running top-k (forward copy)
        const int e = e0 + lane;
        uint32_t kv = 0u;
        int32_t iv = 0;
        if (e < cr) { kv = keys[r * CAPB + e]; iv = ids[r * CAPB + e]; }
        __syncwarp();
        if (e < cr) { keys[n + e] = kv; ids[n + e] = iv; }
        __syncwarp();
      }
      n = warp_compact_t<2 * CAPB>(keys, ids, n + cr, k, T);
      __syncwarp();
    }
    for (int o = lane; o < k; o += 32) {
      if (o < n) {
        const int32_t me = ids[o];
        int p = 0;
        for (int d = 0; d < n; ++d) p += ids[d] < me;
        oi[p] = me;
        if (os) os[p] = key_to_f32(keys[o]);
      } else {
        oi[o] = -1;
        if (os) os[o] = -INFINITY;
      }
    }
    return;
  }
  // gather the lists behind list 0 (the destination stays below CAPB, under
  // every later list's storage)
  int b[5];
  b[0] = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) b[r + 1] = b[r] + c[r];
#pragma unroll
  for (int r = 1; r < 4; ++r)
    for (int e = lane; e < c[r]; e += 32) { keys[b[r] + e] = keys[r * CAPB + e]; ids[b[r] + e] = ids[r * CAPB + e]; }
  __syncwarp();
  constexpr int V = CAPB / 32;
  uint32_t v[V];
  int32_t id[V];
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < ntot ? keys[e] : 0u;
    id[i] = e < ntot ? ids[e] : 0x7FFFFFFF;
    if (e < ntot) { lo = min(lo, v[i]); hi = max(hi, v[i]); }
  }
  unsigned km[V];  // ballot of the kept entries of each register slot
  if (ntot > k) {
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    // k-th largest key: bits above the highest one in which lo and hi differ
    // are common to every candidate
    uint32_t T = hi;
    if (lo != hi) {
      const int top = 31 - __clz(lo ^ hi);
      uint32_t prefix = top == 31 ? 0u : hi & ~((2u << top) - 1u);
      int need = k;
      for (int bit = top; bit >= 0; --bit) {
        const uint32_t hm = ~((2u << bit) - 1u);  // bits above `bit` (bit 31: none)
        const uint32_t hmask = bit == 31 ? 0u : hm;
        int cc = 0;
#pragma unroll
        for (int i = 0; i < V; ++i) cc += ((v[i] & hmask) == prefix) && ((v[i] >> bit) & 1u);
        cc = __reduce_add_sync(0xffffffffu, cc);
        if (cc >= need) prefix |= 1u << bit;
        else need -= cc;
      }
      T = prefix;
    }
    int gt = 0, eq = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) { gt += v[i] > T; eq += v[i] == T; }
    gt = __reduce_add_sync(0xffffffffu, gt);
    eq = __reduce_add_sync(0xffffffffu, eq);
    const int need_eq = k - gt;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      bool keep = v[i] > T;
      if (v[i] == T) {
        if (eq == need_eq) {
          keep = true;
        } else {  // only with exactly equal scores: the lowest indices among them
          int before = 0;
          for (int e2 = 0; e2 < ntot; ++e2) before += (keys[e2] == T) && (ids[e2] < id[i]);
          keep = before < need_eq;
        }
      }
      km[i] = __ballot_sync(0xffffffffu, keep);
    }
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) km[i] = __ballot_sync(0xffffffffu, lane + 32 * i < ntot);
  }
  // kept entries, in list order, to the front; kb[r] = first kept of list r
  int kb[5];
#pragma unroll
  for (int r = 0; r < 5; ++r) {
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int lim = min(max(b[r] - 32 * i, 0), 32);
      cnt += __popc(km[i] & (lim == 32 ? 0xffffffffu : (1u << lim) - 1u));
    }
    kb[r] = cnt;
  }
  __syncwarp();  // every lane holds its entries before they are overwritten
  {
    int out = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      if ((km[i] >> lane) & 1u) {
        const int p = out + __popc(km[i] & below);
        keys[p] = v[i];
        ids[p] = id[i];
      }
      out += __popc(km[i]);
    }
  }
  __syncwarp();
  runs_out<CAPB>(keys, ids, kb, k, oi, os);
}


// Exact top-k (key desc, index asc) of the union of four candidate lists
// that are each in ascending index order (list r at keys + r*CAPB, count
// cnt4[r]), written to oi / os in ascending index order and padded with -1
// / -inf up to k.  One warp; hist: 256 words of shared memory private to the
// warp; the lists' storage is overwritten.  P is a key that the union's k-th
// largest key reaches (0 = none).  One read-only pass counts the entries at
// or above P and their key range; a 256-bin histogram spread linearly over
// that range gives the bin that holds the k-th largest key: the entries of
// higher bins are kept, and those of that bin (at most 32 of them) are
// ranked against each other.  The kept entries are gathered list by list,
// so each list stays a run in index order, and every entry finds its output
// slot by binary searches in the other runs.  A bin of more than 32 entries
// (many nearly equal keys) takes the general path.
template <int CAPB>
__device__ __forceinline__ void union_topk_out(uint32_t* keys, int32_t* ids, const int* cnt4, uint32_t P, int k,
                                               uint32_t* hist, int32_t* oi, float* os) {
  constexpr int V = CAPB / 32;
  const int lane = threadIdx.x & 31;
  const unsigned below = (1u << lane) - 1u;
  int ntot = 0;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    int cnt = 0;
    for (int e = lane; e < cnt4[r]; e += 32) {
      const uint32_t kv = keys[r * CAPB + e];
      if (kv >= P) { ++cnt; lo = min(lo, kv); hi = max(hi, kv); }
    }
    ntot += __reduce_add_sync(0xffffffffu, cnt);
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  const bool all = ntot <= k;
  const float inv = 256.f / (static_cast<float>(hi - lo) + 1.f);
  auto bin = [&](uint32_t kv) {
    return static_cast<int>(min(255u, static_cast<uint32_t>(static_cast<float>(kv - lo) * inv)));
  };
  int best = 0, A = 0, Bc = 0;
  if (!all) {
#pragma unroll
    for (int j = 0; j < 8; ++j) hist[lane * 8 + j] = 0u;
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 4; ++r)
      for (int e = lane; e < cnt4[r]; e += 32) {
        const uint32_t kv = keys[r * CAPB + e];
        if (kv >= P) atomicAdd(hist + bin(kv), 1u);
      }
    __syncwarp();
    best = hist_top_bin(hist, k);
    int a = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) a += (lane * 8 + j > best) ? static_cast<int>(hist[lane * 8 + j]) : 0;
    A = __reduce_add_sync(0xffffffffu, a);
    Bc = best >= 0 ? static_cast<int>(hist[best]) : 0;
    __syncwarp();
    if (best < 0 || Bc > 32 || A + Bc > CAPB) {
      union_topk_general<CAPB>(keys, ids, cnt4, P, k, hist, oi, os);
      return;
    }
  }
  // gather the candidates (at or above P and, unless all are kept, in bins
  // >= best), list by list; b[r] = first of list r
  int b[5];
  int out = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const uint32_t* kr = keys + r * CAPB;
    const int32_t* ir = ids + r * CAPB;
    const int n = cnt4[r];
    b[r] = out;
    for (int e0 = 0; e0 < n; e0 += 32) {
      const int e = e0 + lane;
      uint32_t kv = 0u;
      int32_t iv = 0;
      if (e < n) { kv = kr[e]; iv = ir[e]; }
      const bool keep = e < n && kv >= P && (all || bin(kv) >= best);
      const unsigned m = __ballot_sync(0xffffffffu, keep);
      __syncwarp();  // list 0 is compacted in place: the chunk is read before it is overwritten
      if (keep) { keys[out + __popc(m & below)] = kv; ids[out + __popc(m & below)] = iv; }
      out += __popc(m);
    }
  }
  b[4] = out;
  __syncwarp();
  uint32_t v[V];
  int32_t id[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < out ? keys[e] : 0u;
    id[i] = e < out ? ids[e] : 0x7FFFFFFF;
  }
  unsigned km[V];  // ballot of the kept entries of each register slot
  if (!all) {
    // the entries of bin `best` to hist[0 .. Bc) (keys) and hist[32 ..] (indices)
    unsigned bm[V];
    int q = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const bool isb = lane + 32 * i < out && bin(v[i]) == best;
      bm[i] = __ballot_sync(0xffffffffu, isb);
      if (isb) {
        const int slot = q + __popc(bm[i] & below);
        hist[slot] = v[i];
        hist[32 + slot] = static_cast<uint32_t>(id[i]);
      }
      q += __popc(bm[i]);
    }
    __syncwarp();
    const uint32_t mk = lane < Bc ? hist[lane] : 0u;
    const int32_t mi = lane < Bc ? static_cast<int32_t>(hist[32 + lane]) : 0x7FFFFFFF;
    int rank = 0;  // bin entries before this one (key desc, index asc)
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const uint32_t ok = __shfl_sync(0xffffffffu, mk, j);
      const int32_t oj = __shfl_sync(0xffffffffu, mi, j);
      rank += (j < Bc) && (ok > mk || (ok == mk && oj < mi));
    }
    const unsigned win = __ballot_sync(0xffffffffu, lane < Bc && rank < k - A);
    q = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const bool isb = (bm[i] >> lane) & 1u;
      const int slot = q + __popc(bm[i] & below);
      const bool keep = lane + 32 * i < out && (!isb || ((win >> slot) & 1u));
      km[i] = __ballot_sync(0xffffffffu, keep);
      q += __popc(bm[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) km[i] = __ballot_sync(0xffffffffu, lane + 32 * i < out);
  }
  int kb[5];
#pragma unroll
  for (int r = 0; r < 5; ++r) {
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int lim = min(max(b[r] - 32 * i, 0), 32);
      cnt += __popc(km[i] & (lim == 32 ? 0xffffffffu : (1u << lim) - 1u));
    }
    kb[r] = cnt;
  }
  __syncwarp();  // every lane holds its entries before they are overwritten
  {
    int o2 = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      if ((km[i] >> lane) & 1u) {
        const int p = o2 + __popc(km[i] & below);
        keys[p] = v[i];
        ids[p] = id[i];
      }
      o2 += __popc(km[i]);
    }
  }
  __syncwarp();
  runs_out<CAPB>(keys, ids, kb, k, oi, os);
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
  static constexpr int OFF_HIST = OFF_ST + NQ * 8;          // 256 words per epilogue warp
  static constexpr int SMEM = OFF_HIST + 8 * 256 * 4 + 1024;
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
  uint8_t* smem = align_smem_1024(smem_raw);
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
  uint32_t* sHist = reinterpret_cast<uint32_t*>(smem + X::OFF_HIST);  // [8][256]

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
            uint32_t th;
            const int nk = ftk::warp_cut<X::CAPQ>(sKeys + qi * X::CAPQ, sIds + qi * X::CAPQ, n, k,
                                                  X::CAPQ - X::SYNC * C::TILE, sHist + ew * 256, th);
            if (lane == 0) {
              sCnt[qi] = nk;
              sTheta[qi] = th;
            }
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


// ---------------------------------------------------------------------------
// Variant with warp-private candidate buffers (16 queries per CTA, k up to
// CAPB - 32).  Each (query, TMEM lane quadrant) pair has its own buffer,
// threshold and count, owned by the one epilogue warp that reads that
// quadrant's accumulator columns of the query: appends need no atomics and
// compactions no barrier, so the epilogue warps run independently until the
// end.  A quadrant's buffer holds the top-k of the entries of that quadrant
// seen so far (its threshold is the k-th of them, a lower bound of the
// query's k-th); the union of the four buffers therefore contains the
// query's top-k, which one warp selects exactly at the end.  16 epilogue
// warps (four per quadrant, four queries each) keep more loads and
// dependency chains in flight than one warp per SMSP pair.
template <int HI, int DI, int NQ, int STAGES>
struct IndexTopkPwCfg {
  using Base = IndexTcCfg<HI, DI, NQ, STAGES>;
  static constexpr int EW = 16;                    // epilogue warps
  static constexpr int NT = 64 + EW * 32;          // + TMA and MMA warps
  static constexpr int CAPB = 256;                 // slots per (query, quadrant)
  static constexpr int NB = NQ * 4;                // buffers
  static constexpr int OFF_KEYS = (Base::OFF_BAR + Base::NBAR * 8 + 64 + 1023) / 1024 * 1024;
  static constexpr int OFF_IDS = OFF_KEYS + NB * CAPB * 4;
  static constexpr int OFF_CNT = OFF_IDS + NB * CAPB * 4;   // final count of every buffer
  static constexpr int OFF_HIST = OFF_CNT + NB * 4;         // 256 words per epilogue warp
  static constexpr int OFF_PUB = OFF_HIST + EW * 256 * 4;   // published bound of every buffer
  static constexpr int SMEM = OFF_PUB + NB * 4 + 1024;
};

template <int HI, int DI, int NQ, int STAGES>
__global__ void __launch_bounds__(IndexTopkPwCfg<HI, DI, NQ, STAGES>::NT, 1)
    k_index_topk_pw(const __grid_constant__ CUtensorMap tmap_k, IndexTopkTcArgs a) {
  using C = IndexTcCfg<HI, DI, NQ, STAGES>;
  using X = IndexTopkPwCfg<HI, DI, NQ, STAGES>;
  constexpr int EW = X::EW;
  constexpr int NEPI = EW * 32;
  constexpr int G = EW / 4;              // query groups (epilogue warps per quadrant)
  constexpr int QG = NQ / G;             // queries per epilogue warp
  constexpr int COLS = QG * HI;          // accumulator columns per warp
  constexpr int CAPB = X::CAPB;
  static_assert(C::NREAL == C::N && COLS % 32 == 0 && NQ % G == 0, "whole 32-column loads");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  float* sW = reinterpret_cast<float*>(smem + C::OFF_W);
  int* sVis = reinterpret_cast<int*>(smem + C::OFF_VIS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  // NACC accumulators in TMEM (4 x 128 columns = all 512): the MMA can run three
  // tiles ahead of the epilogue, whose per-tile latency is the bottleneck
  constexpr int NACC = 4;
  constexpr uint32_t TMEM_COLS = NACC * C::N;
  static_assert(TMEM_COLS <= 512 && (2 * STAGES + 2 * NACC) * 8 + 8 <= C::NBAR * 8 + 64, "TMEM / barrier room");
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + NACC;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(tempty + NACC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint32_t* sKeys = reinterpret_cast<uint32_t*>(smem + X::OFF_KEYS);  // [NQ][4][CAPB]
  int32_t* sIds = reinterpret_cast<int32_t*>(smem + X::OFF_IDS);      // [NQ][4][CAPB]
  int* sCnt = reinterpret_cast<int*>(smem + X::OFF_CNT);              // [NQ][4]
  uint32_t* sHist = reinterpret_cast<uint32_t*>(smem + X::OFF_HIST);  // [EW][256]
  uint32_t* sPub = reinterpret_cast<uint32_t*>(smem + X::OFF_PUB);    // [NQ][4], 0 = none yet

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
    for (int i = 0; i < NACC; ++i) { tc::mbar_init(tfull + i, 1); tc::mbar_init(tempty + i, NEPI); }
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
  if (warp == 1) tc::tmem_alloc(s_tmem, TMEM_COLS);
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
    }
    for (int u = t; u < X::NB; u += NEPI) sPub[u] = 0u;
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
        const int s = t % STAGES, acc = t % NACC;
        if (*s_abort || !tc::mbar_wait(tempty + acc, ((t / NACC) & 1) ^ 1, 23)) { *s_abort = 1; break; }
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
      if (issued > 0) tc::mbar_wait(tfull + ((issued - 1) % NACC), ((issued - 1) / NACC) & 1, 25);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue + streaming top-k
    const int ew = warp - 2;          // epilogue warp 0..EW-1
    const int quarter = warp & 3;     // TMEM lanes 32*quarter .. +31
    const int grpq = ew >> 2;         // queries [grpq*QG, grpq*QG + QG)
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + grpq * COLS;
    const float4* sW4 = reinterpret_cast<const float4*>(sW) + grpq * QG * HI / 4;  // broadcast reads
    int visr[QG], cnt[QG];
    float thf[QG];  // threshold test on floats: key(s) > key(theta) <=> s > f(theta); -inf = none yet
#pragma unroll
    for (int j = 0; j < QG; ++j) {
      visr[j] = sVis[grpq * QG + j];
      thf[j] = -INFINITY;
      cnt[j] = 0;
    }
    auto buf = [&](int j) { return ((grpq * QG + j) * 4 + quarter) * CAPB; };
    // A second filter shared by the four quadrant warps of a query: at every
    // cut a warp publishes a key that at least ceil(k/4) entries of its
    // buffer reach; the four quadrants together then hold at least k entries
    // at or above the smallest published key, so no entry below it can enter
    // the query's top-k (entries equal to it may, by the index rule, and
    // pass).  It is read at cuts and every 8 tiles; a stale read only gives
    // an older, smaller bound.
    const int kp = (k + 3) / 4;
    auto shared_bound = [&](int j) -> float {
      const volatile uint32_t* P = sPub + (grpq * QG + j) * 4;
      const uint32_t m4 = min(min(P[0], P[1]), min(P[2], P[3]));
      if (m4 <= 1u) return -INFINITY;
      const uint32_t below = m4 - 1u == 0x7FFFFFFFu ? 0x7FFFFFFEu : m4 - 1u;  // skip -0 below +0
      return key_to_f32(below);  // the largest float below the bound: s > it <=> s >= bound
    };
    for (int t = 0; t < ntiles; ++t) {
      const int acc = t % NACC;
      if ((t & 7) == 7) {
#pragma unroll
        for (int j = 0; j < QG; ++j) thf[j] = fmaxf(thf[j], shared_bound(j));
      }
      const bool wok = __all_sync(0xffffffffu, !*s_abort && tc::mbar_wait(tfull + acc, (t / NACC) & 1, 26));
      if (!wok) {
        *s_abort = 1;
        break;
      }
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
      float sc[QG];
      unsigned anyq = 0u;  // bit j: this lane's entry passes query j's threshold
#pragma unroll
      for (int j = 0; j < QG; ++j) {
        // two fp32 chains (even and odd heads) in one packed register pair:
        // each half is an IEEE fma, in the order of the scalar code
        uint64_t s01 = 0ull;
#pragma unroll
        for (int h4 = 0; h4 < HI / 4; ++h4) {
          const float4 wv = sW4[j * HI / 4 + h4];
          s01 = fma_f32x2(pack_f32x2(wv.x, wv.y),
                          pack_f32x2(fmaxf(v[j * HI + 4 * h4 + 0], 0.f), fmaxf(v[j * HI + 4 * h4 + 1], 0.f)), s01);
          s01 = fma_f32x2(pack_f32x2(wv.z, wv.w),
                          pack_f32x2(fmaxf(v[j * HI + 4 * h4 + 2], 0.f), fmaxf(v[j * HI + 4 * h4 + 3], 0.f)), s01);
        }
        float s0, s1;
        unpack_f32x2(s01, s0, s1);
        const float s = s0 + s1;
        sc[j] = (all_vis || entry < visr[j]) ? s : -INFINITY;
        anyq |= (sc[j] > thf[j] ? 1u : 0u) << j;
      }
      const unsigned wq = __reduce_or_sync(0xffffffffu, anyq);  // queries with a taker in this warp
      if (wq) {
#pragma unroll
        for (int j = 0; j < QG; ++j) {
          if (!((wq >> j) & 1u)) continue;  // warp-uniform
          const bool take = (anyq >> j) & 1u;
          const unsigned msk = __ballot_sync(0xffffffffu, take);
          {
            const int bo = buf(j);
            if (take) {
              const int slot = cnt[j] + __popc(msk & ((1u << lane) - 1u));
              sKeys[bo + slot] = f32_to_key(sc[j]);
              sIds[bo + slot] = entry;
            }
            cnt[j] += __popc(msk);
            if (cnt[j] > CAPB - 32) {  // the next tile could overflow: cut to a superset of the top-k
              __syncwarp();
              uint32_t th, pb;
              cnt[j] = ftk::warp_cut<CAPB>(sKeys + bo, sIds + bo, cnt[j], k, CAPB - 32, sHist + ew * 256, th, kp,
                                           &pb);
              if (lane == 0) reinterpret_cast<volatile uint32_t*>(sPub)[bo / CAPB] = pb;
              thf[j] = fmaxf(key_to_f32(th), shared_bound(j));
            }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < QG; ++j)
      if (lane == 0) sCnt[buf(j) / CAPB] = cnt[j];
    tc::named_sync(1, NEPI);
    // ---- final: exact top-k of every query over its four buffers, ascending index order ----
    for (int qi = ew; qi < NQ; qi += EW) {
      const int q = qg0 + qi;
      if (q >= qend) continue;
      const volatile uint32_t* Pq = sPub + qi * 4;
      const uint32_t P = min(min(Pq[0], Pq[1]), min(Pq[2], Pq[3]));
      int c4[4];  // an abandoned run (a wait that gave up) writes padding only
#pragma unroll
      for (int r = 0; r < 4; ++r) c4[r] = *s_abort ? 0 : sCnt[qi * 4 + r];
      ftk::union_topk_out<CAPB>(sKeys + qi * 4 * CAPB, sIds + qi * 4 * CAPB, c4, P, k, sHist + ew * 256,
                                a.idx + (static_cast<int64_t>(b) * a.Tq + q) * k,
                                a.score ? a.score + (static_cast<int64_t>(b) * a.Tq + q) * k : nullptr);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace lcc
