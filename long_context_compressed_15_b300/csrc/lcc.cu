// liblcc.so: C ABI of the hybrid compressed-attention path (declared in
// include/lcc.h).  Host side: argument validation, workspace carving, kernel
// selection and launches.  Every kernel lives in one of the included
// headers; this is the library's only translation unit.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "lcc.h"
#include "common.cuh"
#include "pool.cuh"
#include "merge.cuh"
#include "attn.cuh"
#include "index.cuh"
#include "topk.cuh"

using namespace lcc;

namespace {

thread_local std::string t_last_error;

lcc_status fail(lcc_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

std::atomic<unsigned long long> g_launches{0};

lcc_status launch_check(const char* what) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(LCC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return LCC_OK;
}

// Raise a kernel's dynamic shared-memory limit once per device.
template <typename K>
lcc_status ensure_smem(K kernel, size_t bytes, unsigned long long& done_mask) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(LCC_ERR_CUDA, "cudaGetDevice failed");
  const unsigned long long bit = 1ull << (dev & 63);
  if (done_mask & bit) return LCC_OK;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return fail(LCC_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  done_mask |= bit;
  return LCC_OK;
}

std::mutex g_attr_mu;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ compress
lcc_status compress_impl(int m, const lcc_bf16* K, const lcc_bf16* V, const float* gate, int B, int nblk, int D,
                         int64_t kv_bs, int64_t g_bs, lcc_bf16* Kc, lcc_bf16* Vc, int64_t c_bs, void* stream) {
  const char* name = m == 4 ? "lcc_csa_compress" : "lcc_hca_compress";
  if (B < 0 || nblk < 0) return fail(LCC_ERR_SHAPE, "%s: B=%d n_blocks=%d must be >= 0", name, B, nblk);
  if (B == 0 || nblk == 0) return LCC_OK;
  if (!K || !V || !gate || !Kc || !Vc) return fail(LCC_ERR_ARG, "%s: null pointer", name);
  if (D != 64 && D != 128) return fail(LCC_ERR_SHAPE, "%s: D=%d (supported: 64, 128)", name, D);
  if (!aligned16(K) || !aligned16(V) || !aligned16(Kc) || !aligned16(Vc) || (kv_bs % 8) || (c_bs % 8))
    return fail(LCC_ERR_ALIGN, "%s: K/V/Kc/Vc must be 16-byte aligned and batch strides multiples of 8", name);
  if (B > 1 && (kv_bs < static_cast<int64_t>(nblk) * m * D || c_bs < static_cast<int64_t>(nblk) * D ||
                g_bs < static_cast<int64_t>(nblk) * m))
    return fail(LCC_ERR_SHAPE, "%s: batch strides smaller than one batch's rows", name);
  if (B > 65535) return fail(LCC_ERR_SHAPE, "%s: B=%d too large", name, B);
  PoolArgs a{reinterpret_cast<const bf16*>(K), reinterpret_cast<const bf16*>(V), gate, B, nblk, kv_bs, g_bs,
             reinterpret_cast<bf16*>(Kc), reinterpret_cast<bf16*>(Vc), c_bs};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (m == 4) {
    const int bpw = 32 / (2 * (D / 8));
    dim3 grid((nblk + 8 * bpw - 1) / (8 * bpw), B);
    if (D == 128) k_pool_small<4, 128><<<grid, 256, 0, s>>>(a);
    else k_pool_small<4, 64><<<grid, 256, 0, s>>>(a);
  } else {
    dim3 grid(nblk, B);
    if (D == 128) k_pool_large<128, 128><<<grid, 256, 0, s>>>(a);
    else k_pool_large<128, 64><<<grid, 256, 0, s>>>(a);
  }
  return launch_check(name);
}

// ----------------------------------------------------------------- index/topk
constexpr int kTopkNT = 256;
constexpr int kTopkCap = 8192;  // elements per top-k CTA
constexpr size_t kScoreBudget = size_t(1) << 28;  // score elements per query chunk

int index_chunk(int B, int Tq, int Ncap) {
  int64_t qc = static_cast<int64_t>(kScoreBudget) / (static_cast<int64_t>(B) * Ncap);
  if (qc < 1) qc = 1;
  if (qc > Tq) qc = Tq;
  return static_cast<int>(qc);
}

struct IndexWs {
  size_t scores, cand_s, cand_i, total;
};
IndexWs index_ws(int B, int Tq, int Ncap, int k) {
  IndexWs w{};
  if (B <= 0 || Tq <= 0 || Ncap <= 0 || k <= 0) return w;
  const int qc = index_chunk(B, Tq, Ncap);
  const int64_t rows = static_cast<int64_t>(B) * qc;
  const int nseg = (Ncap + kTopkCap - 1) / kTopkCap;
  w.scores = round_up(rows * Ncap * sizeof(float), 256);
  if (nseg > 1) {
    w.cand_s = round_up(rows * nseg * k * sizeof(float), 256);
    w.cand_i = round_up(rows * nseg * k * sizeof(int32_t), 256);
  }
  w.total = w.scores + w.cand_s + w.cand_i;
  return w;
}

template <int HI, int DI, bool FP4>
lcc_status launch_index_score(const IndexArgs& a, cudaStream_t s) {
  constexpr int QPT = 8 / HI;
  if (a.nq <= QPT) {
    dim3 grid((a.Ncap + 255) / 256, 1, a.B);
    k_index_score<HI, DI, FP4, QPT><<<grid, 128, 0, s>>>(a);
  } else {
    constexpr int NQ = 8 * QPT;
    dim3 grid((a.Ncap + 255) / 256, (a.nq + NQ - 1) / NQ, a.B);
    k_index_score<HI, DI, FP4, NQ><<<grid, 128, 0, s>>>(a);
  }
  return launch_check("k_index_score");
}

unsigned long long g_topk_a_done = 0, g_topk_b_done = 0;

}  // namespace

// ============================================================================
extern "C" {

const char* lcc_last_error(void) { return t_last_error.c_str(); }
const char* lcc_version(void) { return "lcc 0.1 (sm_103a)"; }
uint64_t lcc_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

lcc_status lcc_sync_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(LCC_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_dev_error, sizeof(word));
  if (e != cudaSuccess) return fail(LCC_ERR_CUDA, "reading device error word: %s", cudaGetErrorString(e));
  if (word == 0) return LCC_OK;
  const unsigned int zero = 0;
  cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(zero));
  const unsigned int code = word >> 24, detail = word & 0xFFFFFFu;
  if (code == DEV_ERR_TIMEOUT) return fail(LCC_ERR_TIMEOUT, "device wait gave up (site %u)", detail);
  return fail(LCC_ERR_DEVICE, "index list entry out of range at list position %u", detail);
}

lcc_status lcc_csa_compress(const lcc_bf16* K, const lcc_bf16* V, const float* gate, int B, int n_blocks, int D,
                            int64_t kv_bstride, int64_t gate_bstride, lcc_bf16* Kc, lcc_bf16* Vc, int64_t c_bstride,
                            void* stream) {
  return compress_impl(4, K, V, gate, B, n_blocks, D, kv_bstride, gate_bstride, Kc, Vc, c_bstride, stream);
}

lcc_status lcc_hca_compress(const lcc_bf16* K, const lcc_bf16* V, const float* gate, int B, int n_blocks, int D,
                            int64_t kv_bstride, int64_t gate_bstride, lcc_bf16* Kc, lcc_bf16* Vc, int64_t c_bstride,
                            void* stream) {
  return compress_impl(128, K, V, gate, B, n_blocks, D, kv_bstride, gate_bstride, Kc, Vc, c_bstride, stream);
}

size_t lcc_index_topk_workspace(int B, int Tq, int Ncap, int k) { return index_ws(B, Tq, Ncap, k).total; }

}  // extern "C"

namespace {
lcc_status check_index_args(const char* name, const lcc_bf16* qI, const float* w, int B, int Tq, int HI, int DI,
                            const int64_t* q_pos0, lcc_key_format fmt, const void* kI, const uint8_t* kI_scale,
                            const int32_t* n_valid, int Ncap, int m, const void* out) {
  if (!qI || !w || !q_pos0 || !kI || !n_valid || !out) return fail(LCC_ERR_ARG, "%s: null pointer", name);
  if (fmt != LCC_KEY_BF16 && fmt != LCC_KEY_NVFP4) return fail(LCC_ERR_ARG, "%s: unknown key format %d", name, fmt);
  if (fmt == LCC_KEY_NVFP4 && !kI_scale) return fail(LCC_ERR_ARG, "%s: NVFP4 keys need kI_scale", name);
  if (HI != 4 && HI != 8) return fail(LCC_ERR_SHAPE, "%s: HI=%d (supported: 4, 8)", name, HI);
  if (fmt == LCC_KEY_BF16 && DI != 32 && DI != 64) return fail(LCC_ERR_SHAPE, "%s: DI=%d (bf16: 32, 64)", name, DI);
  if (fmt == LCC_KEY_NVFP4 && (DI != 64 || HI != 8))
    return fail(LCC_ERR_SHAPE, "%s: HI=%d DI=%d (NVFP4 keys: HI=8, DI=64)", name, HI, DI);
  if (m < 1 || Ncap < 1) return fail(LCC_ERR_SHAPE, "%s: m=%d Ncap=%d must be >= 1", name, m, Ncap);
  if (B > 65535) return fail(LCC_ERR_SHAPE, "%s: B=%d too large", name, B);
  if (!aligned16(qI) || !aligned16(kI) || !aligned16(w) || !aligned16(out))
    return fail(LCC_ERR_ALIGN, "%s: qI, w, kI and the output must be 16-byte aligned", name);
  return LCC_OK;
}

lcc_status launch_scores(const IndexArgs& ia, int HI, int DI, lcc_key_format fmt, cudaStream_t s) {
  if (fmt == LCC_KEY_NVFP4) return launch_index_score<8, 64, true>(ia, s);
  if (HI == 8 && DI == 64) return launch_index_score<8, 64, false>(ia, s);
  if (HI == 8 && DI == 32) return launch_index_score<8, 32, false>(ia, s);
  if (HI == 4 && DI == 64) return launch_index_score<4, 64, false>(ia, s);
  return launch_index_score<4, 32, false>(ia, s);
}
}  // namespace

extern "C" {

lcc_status lcc_lightning_index_scores(const lcc_bf16* qI, const float* w, int B, int Tq, int HI, int DI,
                                      const int64_t* q_pos0, lcc_key_format fmt, const void* kI,
                                      const uint8_t* kI_scale, const int32_t* n_valid, int Ncap, int m,
                                      float* scores, void* stream) {
  const char* name = "lcc_lightning_index_scores";
  if (B < 0 || Tq < 0) return fail(LCC_ERR_SHAPE, "%s: B=%d Tq=%d must be >= 0", name, B, Tq);
  if (B == 0 || Tq == 0) return LCC_OK;
  lcc_status st = check_index_args(name, qI, w, B, Tq, HI, DI, q_pos0, fmt, kI, kI_scale, n_valid, Ncap, m, scores);
  if (st != LCC_OK) return st;
  IndexArgs ia{reinterpret_cast<const bf16*>(qI), w, B, Tq, q_pos0, kI, kI_scale, n_valid, Ncap, m, 0, Tq, scores};
  return launch_scores(ia, HI, DI, fmt, static_cast<cudaStream_t>(stream));
}

lcc_status lcc_lightning_index_topk(const lcc_bf16* qI, const float* w, int B, int Tq, int HI, int DI,
                                    const int64_t* q_pos0, lcc_key_format fmt, const void* kI,
                                    const uint8_t* kI_scale, const int32_t* n_valid, int Ncap, int m, int k,
                                    int32_t* idx, float* score, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  const char* name = "lcc_lightning_index_topk";
  if (B < 0 || Tq < 0) return fail(LCC_ERR_SHAPE, "%s: B=%d Tq=%d must be >= 0", name, B, Tq);
  if (B == 0 || Tq == 0) return LCC_OK;
  lcc_status cst = check_index_args(name, qI, w, B, Tq, HI, DI, q_pos0, fmt, kI, kI_scale, n_valid, Ncap, m, idx);
  if (cst != LCC_OK) return cst;
  if (k < 1 || k > 1024) return fail(LCC_ERR_SHAPE, "%s: k=%d (supported: 1..1024)", name, k);
  const int nseg = (Ncap + kTopkCap - 1) / kTopkCap;
  if (nseg > 1 && static_cast<int64_t>(nseg) * k > kTopkCap)
    return fail(LCC_ERR_UNSUPPORTED, "%s: Ncap=%d with k=%d exceeds the two-stage top-k capacity", name, Ncap, k);
  const IndexWs ws = index_ws(B, Tq, Ncap, k);
  if (!workspace || workspace_bytes < ws.total)
    return fail(LCC_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", name, workspace_bytes, ws.total);
  if (!aligned16(workspace)) return fail(LCC_ERR_ALIGN, "%s: workspace must be 16-byte aligned", name);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    lcc_status st = ensure_smem(k_topk<kTopkNT, kTopkCap, false>, kTopkCap * 4, g_topk_a_done);
    if (st != LCC_OK) return st;
    st = ensure_smem(k_topk<kTopkNT, kTopkCap, true>, kTopkCap * 8, g_topk_b_done);
    if (st != LCC_OK) return st;
  }
  char* wsb = static_cast<char*>(workspace);
  float* scores = reinterpret_cast<float*>(wsb);
  float* cand_s = reinterpret_cast<float*>(wsb + ws.scores);
  int32_t* cand_i = reinterpret_cast<int32_t*>(wsb + ws.scores + ws.cand_s);
  const int qc = index_chunk(B, Tq, Ncap);
  for (int q0 = 0; q0 < Tq; q0 += qc) {
    const int nq = qc < Tq - q0 ? qc : Tq - q0;
    IndexArgs ia{reinterpret_cast<const bf16*>(qI), w, B, Tq, q_pos0, kI, kI_scale, n_valid, Ncap, m, q0, nq, scores};
    lcc_status st = launch_scores(ia, HI, DI, fmt, s);
    if (st != LCC_OK) return st;

    TopkArgs ta{};
    ta.scores = scores;
    ta.Ncap = Ncap;
    ta.q_pos0 = q_pos0;
    ta.n_valid = n_valid;
    ta.m = m;
    ta.Tq = Tq;
    ta.q0 = q0;
    ta.nq = nq;
    ta.k = k;
    ta.seg = kTopkCap;
    const int rows = B * nq;
    if (nseg == 1) {
      ta.out_i = idx;
      ta.out_s = score;
      ta.final_out = 1;
      k_topk<kTopkNT, kTopkCap, false><<<dim3(1, rows), kTopkNT, kTopkCap * 4, s>>>(ta);
      if ((st = launch_check("k_topk")) != LCC_OK) return st;
    } else {
      ta.out_i = cand_i;
      ta.out_s = cand_s;
      ta.out_stride = static_cast<int64_t>(nseg) * k;
      ta.final_out = 0;
      k_topk<kTopkNT, kTopkCap, false><<<dim3(nseg, rows), kTopkNT, kTopkCap * 4, s>>>(ta);
      if ((st = launch_check("k_topk")) != LCC_OK) return st;
      TopkArgs tb = ta;
      tb.cand_s = cand_s;
      tb.cand_i = cand_i;
      tb.ncand = nseg * k;
      tb.out_i = idx;
      tb.out_s = score;
      tb.final_out = 1;
      k_topk<kTopkNT, kTopkCap, true><<<dim3(1, rows), kTopkNT, kTopkCap * 8, s>>>(tb);
      if ((st = launch_check("k_topk merge")) != LCC_OK) return st;
    }
  }
  return LCC_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ attention
namespace {

unsigned long long g_attn_done[2][2][3] = {};

template <int D, int ROWS, int MODE>
lcc_status launch_attn(const AttnArgs& a, dim3 grid, cudaStream_t s) {
  const size_t smem = AttnSmem<D, ROWS>::total;
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    lcc_status st = ensure_smem(k_attn<D, ROWS, MODE>, smem, g_attn_done[D == 128][ROWS == 64][MODE]);
    if (st != LCC_OK) return st;
  }
  k_attn<D, ROWS, MODE><<<grid, ROWS * 2, smem, s>>>(a);
  return launch_check("k_attn");
}

template <int MODE>
lcc_status dispatch_attn(const AttnArgs& a, int D, dim3 grid, int rows, cudaStream_t s) {
  if (D == 128) return rows == 64 ? launch_attn<128, 64, MODE>(a, grid, s) : launch_attn<128, 16, MODE>(a, grid, s);
  return rows == 64 ? launch_attn<64, 64, MODE>(a, grid, s) : launch_attn<64, 16, MODE>(a, grid, s);
}

lcc_status check_attn_common(const char* name, const lcc_bf16* q, int B, int Tq, int H, int D, const lcc_bf16* K,
                             const lcc_bf16* V, int64_t rs, int Ncap, const float* O, const float* lse) {
  if (!q || !K || !V || !O || !lse) return fail(LCC_ERR_ARG, "%s: null pointer", name);
  if (D != 64 && D != 128) return fail(LCC_ERR_SHAPE, "%s: D=%d (supported: 64, 128)", name, D);
  if (H < 1 || H > 128 || (H % 8)) return fail(LCC_ERR_SHAPE, "%s: H=%d (supported: multiples of 8 up to 128)", name, H);
  if (Ncap < 0) return fail(LCC_ERR_SHAPE, "%s: Ncap=%d", name, Ncap);
  if (B > 65535) return fail(LCC_ERR_SHAPE, "%s: B=%d too large", name, B);
  if (rs < D || (rs % 8)) return fail(LCC_ERR_ALIGN, "%s: row stride %lld must be >= D and a multiple of 8", name,
                                      static_cast<long long>(rs));
  if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
    return fail(LCC_ERR_ALIGN, "%s: q, K, V and O must be 16-byte aligned", name);
  return LCC_OK;
}

int dense_splits(int B, int Tq, int H, int Ncap) {
  const int64_t rowblocks = static_cast<int64_t>(B) * ((static_cast<int64_t>(Tq) * H + 63) / 64);
  if (rowblocks >= 296) return 1;
  int64_t ns = (296 + rowblocks - 1) / rowblocks;
  const int64_t tiles = (Ncap + 63) / 64;
  if (ns > tiles) ns = tiles;
  if (ns > 128) ns = 128;
  return ns < 1 ? 1 : static_cast<int>(ns);
}

}  // namespace

extern "C" {

lcc_status lcc_csa_sparse_attn(const lcc_bf16* q, int B, int Tq, int H, int D, float scale, const lcc_bf16* Kc,
                               const lcc_bf16* Vc, int64_t kv_rstride, int Ncap, const int32_t* idx, int k, float* O,
                               float* lse, void* stream) {
  const char* name = "lcc_csa_sparse_attn";
  if (B < 0 || Tq < 0) return fail(LCC_ERR_SHAPE, "%s: negative size", name);
  if (B == 0 || Tq == 0) return LCC_OK;
  lcc_status st = check_attn_common(name, q, B, Tq, H, D, Kc, Vc, kv_rstride, Ncap, O, lse);
  if (st != LCC_OK) return st;
  if (!idx) return fail(LCC_ERR_ARG, "%s: null idx", name);
  if (k < 1 || k > 4096) return fail(LCC_ERR_SHAPE, "%s: k=%d (supported: 1..4096)", name, k);
  AttnArgs a{};
  a.q = reinterpret_cast<const bf16*>(q);
  a.B = B; a.Tq = Tq; a.H = H;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.K = reinterpret_cast<const bf16*>(Kc); a.V = reinterpret_cast<const bf16*>(Vc);
  a.kv_bs = static_cast<int64_t>(Ncap) * kv_rstride; a.kv_rs = kv_rstride; a.Ncap = Ncap;
  a.idx = idx; a.k = k;
  a.O = O; a.lse = lse; a.nsplit = 1; a.rows_total = static_cast<int64_t>(B) * Tq * H;
  const int rows = H <= 16 ? 16 : 64;
  const int hblocks = (H + rows - 1) / rows;
  if (static_cast<int64_t>(Tq) * hblocks > 0x7FFFFFFF) return fail(LCC_ERR_SHAPE, "%s: too many queries", name);
  return dispatch_attn<ATT_GATHER>(a, D, dim3(Tq * hblocks, B, 1), rows, static_cast<cudaStream_t>(stream));
}

size_t lcc_dense_attn_workspace(int B, int Tq, int H, int D, int Ncap) {
  if (B <= 0 || Tq <= 0 || H <= 0 || D <= 0 || Ncap <= 0) return 0;
  const int ns = dense_splits(B, Tq, H, Ncap);
  if (ns <= 1) return 0;
  const size_t rows = static_cast<size_t>(B) * Tq * H;
  return round_up(ns * rows * D * sizeof(float), 256) + round_up(ns * rows * sizeof(float), 256);
}

lcc_status lcc_hca_dense_attn(const lcc_bf16* q, int B, int Tq, int H, int D, float scale, const int64_t* q_pos0,
                              const lcc_bf16* Kc, const lcc_bf16* Vc, int64_t kv_rstride, int Ncap,
                              const int32_t* n_valid, int m, float* O, float* lse, void* workspace,
                              size_t workspace_bytes, void* stream) {
  const char* name = "lcc_hca_dense_attn";
  if (B < 0 || Tq < 0) return fail(LCC_ERR_SHAPE, "%s: negative size", name);
  if (B == 0 || Tq == 0) return LCC_OK;
  lcc_status st = check_attn_common(name, q, B, Tq, H, D, Kc, Vc, kv_rstride, Ncap, O, lse);
  if (st != LCC_OK) return st;
  if (!q_pos0 || !n_valid) return fail(LCC_ERR_ARG, "%s: null q_pos0 / n_valid", name);
  if (m < 1) return fail(LCC_ERR_SHAPE, "%s: m=%d", name, m);
  const int64_t rowsT = static_cast<int64_t>(B) * Tq * H;
  const int64_t rblocks = (static_cast<int64_t>(Tq) * H + 63) / 64;
  if (rblocks > 0x7FFFFFFF) return fail(LCC_ERR_SHAPE, "%s: too many queries", name);
  const int ns = dense_splits(B, Tq, H, Ncap);
  const size_t need = lcc_dense_attn_workspace(B, Tq, H, D, Ncap);
  if (ns > 1 && (!workspace || workspace_bytes < need))
    return fail(LCC_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", name, workspace_bytes, need);
  AttnArgs a{};
  a.q = reinterpret_cast<const bf16*>(q);
  a.B = B; a.Tq = Tq; a.H = H;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.q_pos0 = q_pos0;
  a.K = reinterpret_cast<const bf16*>(Kc); a.V = reinterpret_cast<const bf16*>(Vc);
  a.kv_bs = static_cast<int64_t>(Ncap) * kv_rstride; a.kv_rs = kv_rstride; a.Ncap = Ncap;
  a.n_valid = n_valid; a.m = m;
  a.nsplit = ns; a.rows_total = rowsT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ns == 1) {
    a.O = O; a.lse = lse;
    return dispatch_attn<ATT_RANGE>(a, D, dim3(static_cast<unsigned>(rblocks), B, 1), 64, s);
  }
  float* Op = static_cast<float*>(workspace);
  float* lp = reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up(ns * rowsT * D * sizeof(float), 256));
  a.O = Op; a.lse = lp;
  st = dispatch_attn<ATT_RANGE>(a, D, dim3(static_cast<unsigned>(rblocks), B, ns), 64, s);
  if (st != LCC_OK) return st;
  const unsigned g = static_cast<unsigned>((rowsT + 7) / 8);
  if (D == 128) k_split_combine<128><<<g, 256, 0, s>>>(Op, lp, ns, rowsT, O, lse);
  else k_split_combine<64><<<g, 256, 0, s>>>(Op, lp, ns, rowsT, O, lse);
  return launch_check("k_split_combine");
}

lcc_status lcc_swa_attn(const lcc_bf16* q, int B, int Tq, int H, int D, float scale, const int64_t* q_pos0,
                        const lcc_bf16* Kr, const lcc_bf16* Vr, int64_t kv_rstride, int Rcap, const int64_t* raw_pos0,
                        int W, float* O, float* lse, void* stream) {
  const char* name = "lcc_swa_attn";
  if (B < 0 || Tq < 0) return fail(LCC_ERR_SHAPE, "%s: negative size", name);
  if (B == 0 || Tq == 0) return LCC_OK;
  lcc_status st = check_attn_common(name, q, B, Tq, H, D, Kr, Vr, kv_rstride, Rcap, O, lse);
  if (st != LCC_OK) return st;
  if (!q_pos0 || !raw_pos0) return fail(LCC_ERR_ARG, "%s: null q_pos0 / raw_pos0", name);
  if (W < 1 || W > 4096) return fail(LCC_ERR_SHAPE, "%s: W=%d (supported: 1..4096)", name, W);
  const int64_t rblocks = (static_cast<int64_t>(Tq) * H + 63) / 64;
  if (rblocks > 0x7FFFFFFF) return fail(LCC_ERR_SHAPE, "%s: too many queries", name);
  AttnArgs a{};
  a.q = reinterpret_cast<const bf16*>(q);
  a.B = B; a.Tq = Tq; a.H = H;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.q_pos0 = q_pos0;
  a.K = reinterpret_cast<const bf16*>(Kr); a.V = reinterpret_cast<const bf16*>(Vr);
  a.kv_bs = static_cast<int64_t>(Rcap) * kv_rstride; a.kv_rs = kv_rstride; a.Ncap = Rcap;
  a.raw_pos0 = raw_pos0; a.W = W;
  a.O = O; a.lse = lse; a.nsplit = 1; a.rows_total = static_cast<int64_t>(B) * Tq * H;
  return dispatch_attn<ATT_WINDOW>(a, D, dim3(static_cast<unsigned>(rblocks), B, 1), 64,
                                   static_cast<cudaStream_t>(stream));
}

lcc_status lcc_attn_merge(int nb, const float* const* O_parts, const float* const* lse_parts, int64_t rows, int D,
                          lcc_bf16* out, float* out_f32, float* lse_out, void* stream) {
  const char* name = "lcc_attn_merge";
  if (nb < 2 || nb > 4) return fail(LCC_ERR_ARG, "%s: nb=%d (supported: 2..4)", name, nb);
  if (rows < 0) return fail(LCC_ERR_SHAPE, "%s: rows=%lld", name, static_cast<long long>(rows));
  if (rows == 0) return LCC_OK;
  if (!O_parts || !lse_parts) return fail(LCC_ERR_ARG, "%s: null part arrays", name);
  if (D != 64 && D != 128) return fail(LCC_ERR_SHAPE, "%s: D=%d (supported: 64, 128)", name, D);
  if (!out && !out_f32 && !lse_out) return fail(LCC_ERR_ARG, "%s: no output", name);
  MergeArgs a{};
  for (int b = 0; b < nb; ++b) {
    if (!O_parts[b] || !lse_parts[b]) return fail(LCC_ERR_ARG, "%s: null part %d", name, b);
    if (!aligned16(O_parts[b])) return fail(LCC_ERR_ALIGN, "%s: part %d not 16-byte aligned", name, b);
    a.O[b] = O_parts[b];
    a.lse[b] = lse_parts[b];
  }
  if ((out && (reinterpret_cast<uintptr_t>(out) & 7)) || (out_f32 && !aligned16(out_f32)))
    return fail(LCC_ERR_ALIGN, "%s: outputs misaligned", name);
  a.nb = nb; a.rows = rows; a.D = D; a.out = reinterpret_cast<bf16*>(out); a.out_f32 = out_f32; a.lse_out = lse_out;
  const int64_t g = (rows + 7) / 8;
  if (g > 0x7FFFFFFF) return fail(LCC_ERR_SHAPE, "%s: too many rows", name);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (D == 128) k_merge<128><<<static_cast<unsigned>(g), 256, 0, s>>>(a);
  else k_merge<64><<<static_cast<unsigned>(g), 256, 0, s>>>(a);
  return launch_check(name);
}

}  // extern "C"

// ------------------------------------------------------- allocation-free top-k
// Scratch of lcc_lightning_index_topk_noalloc: a fixed device array instead
// of a caller-provided workspace, for callers that cannot allocate.  Host
// code reaches it only through the address cudaGetSymbolAddress returns for
// the current device (the host-side symbol is not a device address).
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
void* g_noalloc_ptr[64] = {};
std::mutex g_noalloc_mu;

lcc_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(LCC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(LCC_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return fail(LCC_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return LCC_OK;
}
}  // namespace

extern "C" lcc_status lcc_lightning_index_topk_noalloc(const lcc_bf16* qI, const float* w, int B, int Tq, int HI,
                                                       int DI, const int64_t* q_pos0, lcc_key_format fmt,
                                                       const void* kI, const uint8_t* kI_scale,
                                                       const int32_t* n_valid, int Ncap, int m, int k, int32_t* idx,
                                                       float* score, void* stream) {
  const char* name = "lcc_lightning_index_topk_noalloc";
  if (B < 0 || Tq < 0) return fail(LCC_ERR_SHAPE, "%s: B=%d Tq=%d must be >= 0", name, B, Tq);
  if (B == 0 || Tq == 0) return LCC_OK;
  lcc_status st = check_index_args(name, qI, w, B, Tq, HI, DI, q_pos0, fmt, kI, kI_scale, n_valid, Ncap, m, idx);
  if (st != LCC_OK) return st;
  if (k < 1 || k > 1024) return fail(LCC_ERR_SHAPE, "%s: k=%d (supported: 1..1024)", name, k);
  const int nseg = (Ncap + kTopkCap - 1) / kTopkCap;
  if (nseg > 1 && static_cast<int64_t>(nseg) * k > kTopkCap)
    return fail(LCC_ERR_UNSUPPORTED, "%s: Ncap=%d with k=%d exceeds the two-stage top-k capacity", name, Ncap, k);
  // bytes one query row of every batch needs: scores + (two-stage) candidate lists
  const size_t per_q_scores = static_cast<size_t>(B) * Ncap * sizeof(float);
  const size_t per_q_cand = nseg > 1 ? static_cast<size_t>(B) * nseg * k * sizeof(float) : 0;
  const size_t per_q = round_up(per_q_scores, 256) + 2 * round_up(per_q_cand, 256);
  if (per_q > kNoAllocScratchBytes)
    return fail(LCC_ERR_WORKSPACE, "%s: one query row needs %zu scratch bytes, the fixed scratch holds %zu", name,
                per_q, kNoAllocScratchBytes);
  int qc = 1;  // largest query chunk whose scores and candidates fit the scratch
  while (qc < Tq) {
    const int nx = qc * 2 < Tq ? qc * 2 : Tq;
    const size_t need = round_up(per_q_scores * nx, 256) + 2 * round_up(per_q_cand * nx, 256);
    if (need > kNoAllocScratchBytes) break;
    qc = nx;
  }
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != LCC_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if ((st = ensure_smem(k_topk<kTopkNT, kTopkCap, false>, kTopkCap * 4, g_topk_a_done)) != LCC_OK) return st;
    if ((st = ensure_smem(k_topk<kTopkNT, kTopkCap, true>, kTopkCap * 8, g_topk_b_done)) != LCC_OK) return st;
  }
  char* base = static_cast<char*>(scratch);
  float* scores = reinterpret_cast<float*>(base);
  const size_t sc_bytes = round_up(per_q_scores * qc, 256);
  const size_t cand_bytes = round_up(per_q_cand * qc, 256);
  float* cand_s = reinterpret_cast<float*>(base + sc_bytes);
  int32_t* cand_i = reinterpret_cast<int32_t*>(base + sc_bytes + cand_bytes);
  for (int q0 = 0; q0 < Tq; q0 += qc) {
    const int nq = qc < Tq - q0 ? qc : Tq - q0;
    IndexArgs ia{reinterpret_cast<const bf16*>(qI), w, B, Tq, q_pos0, kI, kI_scale, n_valid, Ncap, m, q0, nq, scores};
    if ((st = launch_scores(ia, HI, DI, fmt, s)) != LCC_OK) return st;
    TopkArgs ta{};
    ta.scores = scores;
    ta.Ncap = Ncap;
    ta.q_pos0 = q_pos0;
    ta.n_valid = n_valid;
    ta.m = m;
    ta.Tq = Tq;
    ta.q0 = q0;
    ta.nq = nq;
    ta.k = k;
    ta.seg = kTopkCap;
    const int rows = B * nq;
    if (nseg == 1) {
      ta.out_i = idx;
      ta.out_s = score;
      ta.final_out = 1;
      k_topk<kTopkNT, kTopkCap, false><<<dim3(1, rows), kTopkNT, kTopkCap * 4, s>>>(ta);
      if ((st = launch_check("k_topk")) != LCC_OK) return st;
    } else {
      ta.out_i = cand_i;
      ta.out_s = cand_s;
      ta.out_stride = static_cast<int64_t>(nseg) * k;
      ta.final_out = 0;
      k_topk<kTopkNT, kTopkCap, false><<<dim3(nseg, rows), kTopkNT, kTopkCap * 4, s>>>(ta);
      if ((st = launch_check("k_topk")) != LCC_OK) return st;
      TopkArgs tb = ta;
      tb.cand_s = cand_s;
      tb.cand_i = cand_i;
      tb.ncand = nseg * k;
      tb.out_i = idx;
      tb.out_s = score;
      tb.final_out = 1;
      k_topk<kTopkNT, kTopkCap, true><<<dim3(1, rows), kTopkNT, kTopkCap * 8, s>>>(tb);
      if ((st = launch_check("k_topk merge")) != LCC_OK) return st;
    }
  }
  return LCC_OK;
}
