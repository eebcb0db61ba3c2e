// Arguments of the lightning-indexer score pass (one query chunk), shared by
// the host code and the tensor-core indexers (index_tc.cuh):
//   s[q, j] = sum_h w[q,h] * max(0, qI[q,h,:] . kI[j,:])
// for every visible compressed entry j.  Source: "DeepSeek-V4가 이차적 어텐션
// 비용 없이 ...", section "두 가지 압축 전략: CSA 및 HCA" (a light indexer, run
// in FP4, scores the compressed entries for each query and keeps the top-k);
// the DeepSeek V4.1 Flash post (keys kept in FP4).
#pragma once
#include "common.cuh"

namespace lcc {

struct IndexArgs {
  const bf16* qI;   // [B, Tq, HI, DI]
  const float* w;   // [B, Tq, HI]
  int B, Tq;
  const int64_t* q_pos0;
  const void* kI;        // bf16 [B, Ncap, DI] or uint8 [B, Ncap, DI/2]
  const uint8_t* kIs;    // uint8 [B, Ncap, DI/16] (NVFP4)
  const int32_t* n_valid;
  int Ncap, m;
  int q0, nq;            // query chunk [q0, q0+nq)
  float* scores;         // [nq, Ncap] for this chunk (row = (b, i - q0) flattened as b*nq + i-q0)
  uint32_t* gmax;        // optional [B*nq, g_stride]: key of the largest score of each 32-entry group
  int g_stride;
  int* counters;         // optional [2, B*nq]: zeroed here for the top-k kernel that follows
};

}  // namespace lcc
