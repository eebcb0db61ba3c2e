// CSA layer decode: top-k selection and sparse attention in one thread-block
// cluster per query.  Source: "DeepSeek-V4가 이차적 어텐션 비용 없이 ...",
// section "두 가지 압축 전략: CSA 및 HCA" (the indexer keeps the top-k
// compressed entries per query; the query attends with MQA to those entries
// and, through the sliding-window branch, to the most recent raw tokens).
//
// The result equals the indexer top-k (k_topk_cluster) followed by the
// decode attention (k_attn_wsplit_tma), without the index list's round trip
// through global memory and without a kernel boundary between the two:
//   * the cluster has one CTA per block of 16 heads (CL = H / 16);
//   * every CTA first requests its queries and window rows (inputs of the
//     call, ready before the indexer finishes), then waits for the
//     indexer's scores and runs its share of the cluster top-k
//     (topk_cluster_row: each CTA loads 1/CL of the row);
//   * CTA 0 writes each selected entry to the global index list and, through
//     distributed shared memory, into the index list of every CTA of the
//     cluster; one cluster barrier;
//   * every CTA gathers the selected K/V rows by TMA and runs the attention
//     of its 16 heads (attn_wsplit_tma_body, two 16-key tiles per warp: its
//     window tile is attended while its selected rows are gathered) from its
//     own copy of the list.
#pragma once
#include "attn_decode_tma.cuh"
#include "topk_cluster.cuh"

namespace lcc {

// Writes each selected entry to the global list and to the shared-memory list
// (sidx) of all CTAs of the cluster.
struct TopkOutCluster {
  int32_t* oi;
  float* os;
  const int* sidx;
  uint32_t cl;
  __device__ __forceinline__ void put(int p, int e) const {
    oi[p] = e;
    for (uint32_t r = 0; r < cl; ++r) clu::st(clu::map(sidx + p, r), static_cast<uint32_t>(e));
  }
  __device__ __forceinline__ bool scores() const { return os != nullptr; }
  __device__ __forceinline__ void put_score(int p, float v) const { os[p] = v; }
};

template <int NW, int KT, int PER, int CAP, int MAXG>
struct CsaFusedSmem {
  using A = WsplitTmaSmem<NW, KT, 2>;
  using T = TopkClSmem<NW * 32, PER, CAP, MAXG>;
  static constexpr size_t off_topk = (A::off_bars + NW * 8 + 127) / 128 * 128;
  static constexpr size_t off_idx = off_topk + T::total;
  static constexpr size_t total = off_idx + MAXG / 2 * 4 + 1024;  // + alignment slack
};

// Grid (Tq * CL, B), clusters of CL CTAs along x: CTA rank r of the cluster
// takes heads 16r .. 16r+15 of query blockIdx.x / CL of sequence blockIdx.y.
// t describes the top-k rows of the whole call (nq = Tq, q0 = 0).
template <int NW, int KT, int PER, int CAP, int MAXG>
__global__ void __launch_bounds__(NW * 32) k_csa_decode_fused(const __grid_constant__ CUtensorMap tmK,
                                                              const __grid_constant__ CUtensorMap tmV, AttnArgs a,
                                                              TopkThrArgs t) {
  using S = CsaFusedSmem<NW, KT, PER, CAP, MAXG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  int* sidx = reinterpret_cast<int*>(smem + S::off_idx);
  const uint32_t rk = clu::rank(), CL = clu::size();
  const int qi = static_cast<int>(blockIdx.x / CL), b = static_cast<int>(blockIdx.y);
  const int row = b * t.nq + qi;
  const int64_t o = static_cast<int64_t>(row) * t.k;
  const TopkOutCluster out{t.out_i + o, t.out_s ? t.out_s + o : nullptr, sidx, CL};
  auto select = [&]() {
    pdl_wait();  // scores and group maxima come from the indexer kernel
    topk_cluster_row<NW * 32, PER, CAP, MAXG>(t, smem + S::off_topk, row, out);
    clu::sync();  // CTA 0's list stores are visible in every CTA
  };
  attn_wsplit_tma_body<NW, KT, true, 2>(&tmK, &tmV, a, smem, qi, static_cast<int>(rk) * 16, b, sidx, select);
}

}  // namespace lcc
