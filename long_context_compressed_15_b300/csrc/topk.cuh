// Exact top-k by radix selection: keeps the k largest scores of a row, ties
// to the lower index, output in ascending index order padded with -1.
// Source: "DeepSeek-V4가 이차적 어텐션 비용 없이 ...", section "두 가지 압축 전략:
// CSA 및 HCA" (the indexer keeps the top-k, typically about 128, entries).
//
// A CTA loads up to CAP (score, index) pairs of one row segment into shared
// memory as order-preserving 32-bit keys, finds the k-th largest key with
// four 8-bit histogram passes, and writes the selected pairs with an
// order-preserving block scan, so ties at the threshold go to the lowest
// indices.  Rows longer than CAP are cut into segments (stage A) whose
// candidate lists are merged by a second launch (stage B).
#pragma once
#include "common.cuh"

namespace lcc {

struct TopkArgs {
  // stage A source: scores of row r at scores + r*Ncap, elements [0, vis)
  const float* scores;
  int Ncap;
  const int64_t* q_pos0;
  const int32_t* n_valid;
  int m, Tq, q0, nq;
  // stage B source: candidates of row r at cand_* + r*ncand
  const float* cand_s;
  const int32_t* cand_i;
  int ncand;
  int k;
  int seg;  // stage A segment length
  // outputs of row r at out_* + r*out_stride (+ segment*k for stage A lists)
  int32_t* out_i;
  float* out_s;
  int64_t out_stride;  // candidate lists: elements between rows
  int final_out;       // 1: write the final list of row (b, i) at out + (b*Tq + i)*k
};

template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int& total, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  int wpre = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const int t = s_warp[w];
    if (w < warp) wpre += t;
    tot += t;
  }
  __syncthreads();
  total = tot;
  return wpre + x - v;
}

// MERGE = false: stage A over row segments of scores; MERGE = true: stage B
// over candidate lists.  CAP elements per CTA, NT threads, E = CAP/NT each.
template <int NT, int CAP, bool MERGE>
__global__ void __launch_bounds__(NT) k_topk(TopkArgs a) {
  constexpr int E = CAP / NT;
  static_assert(E % 4 == 0, "vectorised smem access");
  extern __shared__ __align__(16) uint32_t s_key[];   // CAP keys
  int32_t* s_id = reinterpret_cast<int32_t*>(s_key + CAP);  // CAP ids (MERGE only)
  __shared__ uint32_t s_hist[256];
  __shared__ int s_warp[NT / 32];
  __shared__ uint32_t s_dig, s_above;

  const int tid = threadIdx.x;
  const int row = blockIdx.y;  // flattened (b, i - q0)
  const int segi = blockIdx.x;
  int n = 0, id_base = 0;
  if (!MERGE) {
    const int b = row / a.nq, i = a.q0 + row % a.nq;
    const int vis = visible_entries(__ldg(a.q_pos0 + b) + i, a.m, __ldg(a.n_valid + b), a.Ncap);
    id_base = segi * a.seg;
    n = max(0, min(a.seg, vis - id_base));
    const float* src = a.scores + static_cast<int64_t>(row) * a.Ncap + id_base;
    for (int e = tid; e < CAP; e += NT) s_key[e] = e < n ? f32_to_key(__ldg(src + e)) : 0u;
  } else {
    n = a.ncand;
    const float* cs = a.cand_s + static_cast<int64_t>(row) * a.ncand;
    const int32_t* ci = a.cand_i + static_cast<int64_t>(row) * a.ncand;
    for (int e = tid; e < CAP; e += NT) {
      const int id = e < n ? __ldg(ci + e) : -1;
      s_id[e] = id;
      s_key[e] = id >= 0 ? f32_to_key(__ldg(cs + e)) : 0u;
    }
  }
  __syncthreads();

  // number of real elements
  int cnt_local = 0;
  for (int e = tid; e < CAP; e += NT) cnt_local += s_key[e] != 0u;
  int nreal;
  (void)block_excl_scan<NT>(cnt_local, nreal, s_warp);

  const int k = a.k;
  uint32_t prefix = 0, pmask = 0;
  int need = k;
  bool tie_mode = false;  // threshold key fully resolved, ties need ranking
  bool take_all = nreal <= k;
  if (!take_all) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += NT) s_hist[i] = 0;
      __syncthreads();
      for (int e = tid; e < CAP; e += NT) {
        const uint32_t key = s_key[e];
        if (key != 0u && (key & pmask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        // lane l owns digits 255-8l-7 .. 255-8l (descending order)
        uint32_t c[8];
        uint32_t sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) { c[j] = s_hist[255 - 8 * tid - j]; sum += c[j]; }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += y;
        }
        uint32_t excl = incl - sum;  // elements with a larger digit than this lane's bins
        if (excl < static_cast<uint32_t>(need) && incl >= static_cast<uint32_t>(need)) {
          uint32_t run = excl;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (run < static_cast<uint32_t>(need) && run + c[j] >= static_cast<uint32_t>(need)) {
              s_dig = 255 - 8 * tid - j;
              s_above = run;
            }
            run += c[j];
          }
        }
      }
      __syncthreads();
      const uint32_t d = s_dig;
      need -= static_cast<int>(s_above);
      prefix |= d << shift;
      pmask |= 0xFFu << shift;
      const int cd = static_cast<int>(s_hist[d]);
      __syncthreads();
      if (cd == need) break;  // every element with this prefix is selected
      if (shift == 0) tie_mode = true;
    }
  }

  // ---- ordered compaction ----
  int64_t ooff;
  if (a.final_out) {
    const int b = row / a.nq, i = a.q0 + row % a.nq;
    ooff = (static_cast<int64_t>(b) * a.Tq + i) * k;
  } else {
    ooff = static_cast<int64_t>(row) * a.out_stride + static_cast<int64_t>(segi) * k;
  }
  int32_t* oi = a.out_i + ooff;
  float* os = a.out_s ? a.out_s + ooff : nullptr;
  int out_pos = 0, ties_seen = 0;
  for (int base = 0; base < CAP; base += NT * 4) {
    const int e0 = base + tid * 4;
    const uint4 kv = *reinterpret_cast<const uint4*>(s_key + e0);
    const uint32_t kk[4] = {kv.x, kv.y, kv.z, kv.w};
    bool above[4], eq[4];
    int neq = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t key = kk[j];
      const bool real = key != 0u;
      above[j] = real && (take_all || (key & pmask) > prefix);
      eq[j] = real && !take_all && (key & pmask) == prefix;
      neq += eq[j];
    }
    int tot_eq = 0;
    int tie_rank = 0;
    if (tie_mode) tie_rank = ties_seen + block_excl_scan<NT>(neq, tot_eq, s_warp);
    bool sel[4];
    int nsel = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (tie_mode) {
        sel[j] = above[j] || (eq[j] && tie_rank < need);
        if (eq[j]) ++tie_rank;
      } else {
        sel[j] = above[j] || eq[j];
      }
      nsel += sel[j];
    }
    ties_seen += tot_eq;
    int tot_sel;
    int pos = out_pos + block_excl_scan<NT>(nsel, tot_sel, s_warp);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (sel[j] && pos < k) {
        const int e = e0 + j;
        oi[pos] = MERGE ? s_id[e] : id_base + e;
        if (os) os[pos] = key_to_f32(kk[j]);
        ++pos;
      }
    }
    out_pos += tot_sel;
  }
  for (int p = out_pos + tid; p < k; p += NT) {
    oi[p] = -1;
    if (os) os[p] = -INFINITY;
  }
}

}  // namespace lcc
