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
#include <utility>

#include "lcc.h"
#include "common.cuh"
#include "pool.cuh"
#include "decode_step.cuh"
#include "prologue.cuh"
#include "reindex.cuh"
#include "nvfp4.cuh"
#include <cmath>
#include <type_traits>
#include "merge.cuh"
#include "attn.cuh"
#include "attn_tc.cuh"
#include "attn_gather_tc.cuh"
#include "attn_decode_tma.cuh"
#include "csa_decode_fused.cuh"
#include "index.cuh"
#include "index_tc.cuh"
#include "index_topk_tc.cuh"
#include "topk_thr.cuh"
#include "topk_cluster.cuh"
#include "topk_gsel.cuh"

#include <cudaTypedefs.h>

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

// Launch `kern` on stream s; with pdl the launch may overlap the tail of the
// previous kernel on the stream (the kernel must pdl_wait() before reading
// anything that kernel writes).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Launch `kern` as clusters of `cx` CTAs along x (grid.x a multiple of cx).
template <typename... KArgs, typename... Args>
cudaError_t launch_kc(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      unsigned cx, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cx;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
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
                         int64_t kv_bs, int64_t g_bs, lcc_bf16* Kc, lcc_bf16* Vc, int64_t c_bs, void* stream,
                         const int64_t* tok0 = nullptr, int32_t* n_valid = nullptr, int Ncap = 0,
                         const char* name = nullptr) {
  if (!name) name = m == 4 ? "lcc_csa_compress" : m == 128 ? "lcc_hca_compress" : "lcc_compress";
  if (m != 1 && m != 4 && m != 128) return fail(LCC_ERR_SHAPE, "%s: m=%d (supported: 1, 4, 128)", name, m);
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
  if (tok0 && Ncap < 1) return fail(LCC_ERR_SHAPE, "%s: Ncap=%d must be >= 1", name, Ncap);
  if (tok0 && B > 1 && c_bs < static_cast<int64_t>(Ncap) * D)
    return fail(LCC_ERR_SHAPE, "%s: entry batch stride smaller than Ncap entries", name);
  PoolArgs a{reinterpret_cast<const bf16*>(K), reinterpret_cast<const bf16*>(V), gate, B, nblk, kv_bs, g_bs,
             reinterpret_cast<bf16*>(Kc), reinterpret_cast<bf16*>(Vc), c_bs, tok0, n_valid, Ncap};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (m <= 4) {
    constexpr int NB = 2;  // blocks per (half-)warp
    const int bpw = 32 / (2 * (D / 8));
    const int64_t per_cta = 8LL * bpw * NB;
    const int64_t gx = (nblk + per_cta - 1) / per_cta;
    if (gx > 0x7FFFFFFF) return fail(LCC_ERR_SHAPE, "%s: too many blocks", name);
    dim3 grid(static_cast<unsigned>(gx), B);
    if (m == 4) {
      if (D == 128) k_pool_small<4, 128, NB><<<grid, 256, 0, s>>>(a);
      else k_pool_small<4, 64, NB><<<grid, 256, 0, s>>>(a);
    } else {  // m = 1: every token is its own entry (softmax over one logit = 1)
      if (D == 128) k_pool_small<1, 128, NB><<<grid, 256, 0, s>>>(a);
      else k_pool_small<1, 64, NB><<<grid, 256, 0, s>>>(a);
    }
  } else {
    dim3 grid(nblk, B);
    if (D == 128) k_pool_large<128, 128><<<grid, 256, 0, s>>>(a);
    else k_pool_large<128, 64><<<grid, 256, 0, s>>>(a);
  }
  return launch_check(name);
}

// ----------------------------------------------------------------- index/topk
constexpr int kTopkNT = 1024;
constexpr int kTopkPer = 16;     // scores per thread: one CTA covers rows of up to 16384 entries
constexpr int kCandCap = 2048;   // candidates one CTA selects from
constexpr int kSegCap = 1024;    // candidates kept per segment of a row longer than one CTA
constexpr int kTopkSeg = kTopkNT * kTopkPer;   // entries per CTA of the threshold top-k
constexpr size_t kScoreBudget = size_t(1) << 28;  // score elements per query chunk

int index_chunk(int B, int Tq, int Ncap) {
  int64_t qc = static_cast<int64_t>(kScoreBudget) / (static_cast<int64_t>(B) * Ncap);
  if (qc < 1) qc = 1;
  if (qc > Tq) qc = Tq;
  return static_cast<int>(qc);
}

int gmax_stride(int Ncap) { return (Ncap + 15) / 16; }
int topk_segments(int Ncap) { return (Ncap + kTopkSeg - 1) / kTopkSeg; }

// Cluster top-k (one cluster of up to 8 CTAs per row): rows of up to
// 8 * kClSeg entries, k up to kClMaxG / 2 with k * (entries per group) <= kClCap.
constexpr int kClNT = 256;
constexpr int kClPer = 8;
constexpr int kClSeg = kClNT * kClPer;
constexpr int kClCap = 4096;
constexpr int kClMaxG = 512;
using ClSmem = TopkClSmem<kClNT, kClPer, kClCap, kClMaxG>;
unsigned long long g_topk_cl_done = 0;

// Group-selected top-k (one CTA per row, reads only the score groups that can
// hold a winner): k up to 256 and rows whose group maxima fit shared memory.
// Rows the cluster top-k takes (up to 16384 entries) go there instead: its
// eight CTAs per row finish sooner than one CTA's serial selection rounds
// (measured on the 32 x 16384 decode batch: 31.7 us against 35.3 us per
// step); longer rows come here, where reading ~k groups instead of the whole
// row wins (262144-entry rows: the layer-pair step 86 us -> 68 us).
// A call with few rows leaves most SMs idle: its rows take 1024-thread CTAs
// (finer partitions for the threshold, twice the loads in flight), which
// finish sooner (4 rows of 262160 entries: 56.2 -> 54.4 us per layer-pair
// step); with many rows the 512-thread CTA is faster (32 rows of 65536: 70.0
// against 72.1 us per step).
constexpr int kGselNT = 512;
constexpr int kGselNTFew = 1024;
constexpr int kGselFewRows = 16;
constexpr int kGselCap = 4096;
unsigned long long g_topk_gsel_done[2] = {};
size_t gsel_smem(int Ncap) { return static_cast<size_t>(((Ncap + 31) / 32 + 3) & ~3) * 8 + kGselCap * 8; }
bool use_gsel(int Ncap, int k) { return k <= 256 && gsel_smem(Ncap) <= 200 * 1024; }

int topk_cluster_ctas(int Ncap, int k, int gs) {
  if (Ncap > 8 * kClSeg || 2 * k > kClMaxG || static_cast<int64_t>(k) * gs > kClCap) return 0;
  return (Ncap + kClSeg - 1) / kClSeg;
}

// Scratch of one query chunk (rows = B * queries in the chunk): scores,
// group maxima, per-row counters and, for rows longer than one top-k
// segment, the per-segment candidate lists.
struct IndexWs {
  size_t scores, gmax, counters, seg_cnt, cand_k, cand_i, total;
};
IndexWs index_ws_rows(int64_t rows, int Ncap) {
  IndexWs w{};
  const int nseg = topk_segments(Ncap);
  w.scores = round_up(rows * Ncap * sizeof(float), 256);
  w.gmax = round_up(rows * gmax_stride(Ncap) * sizeof(uint32_t), 256);
  w.counters = round_up(rows * 2 * sizeof(int), 256);
  if (nseg > 1) {
    w.seg_cnt = round_up(rows * nseg * sizeof(int), 256);
    w.cand_k = round_up(rows * nseg * kSegCap * sizeof(uint32_t), 256);
    w.cand_i = round_up(rows * nseg * kSegCap * sizeof(int32_t), 256);
  }
  w.total = w.scores + w.gmax + w.counters + w.seg_cnt + w.cand_k + w.cand_i;
  return w;
}
IndexWs index_ws(int B, int Tq, int Ncap, int k) {
  if (B <= 0 || Tq <= 0 || Ncap <= 0 || k <= 0) return IndexWs{};
  return index_ws_rows(static_cast<int64_t>(B) * index_chunk(B, Tq, Ncap), Ncap);
}

// ---- TMA tensor maps (driver entry point fetched through the runtime) ----
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over `rows` rows of `cols` elements (row stride `ld`
// elements), box = box_cols x box_rows, with the given swizzle.
lcc_status make_tmap_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld,
                        uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz, const char* what) {
  auto enc = tmap_encoder();
  if (!enc) return fail(LCC_ERR_CUDA, "%s: cuTensorMapEncodeTiled unavailable", what);
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(LCC_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed (%d)", what, int(r));
  return LCC_OK;
}

int g_num_sms = 0;
int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0, n = 148;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) ==
        cudaSuccess)
      g_num_sms = n;
    else
      g_num_sms = 148;
  }
  return g_num_sms;
}

unsigned long long g_index_tc_done[2][2][2] = {};

template <int HI, int DI, int NQ>
lcc_status launch_index_tc_q(const IndexArgs& ia, const CUtensorMap& tm, int bit, cudaStream_t s) {
  constexpr int STAGES = 4;
  using C = IndexTcCfg<HI, DI, NQ, STAGES>;
  auto kern = k_index_tc<HI, DI, NQ, STAGES>;
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    lcc_status st = ensure_smem(kern, C::SMEM, g_index_tc_done[HI == 8][DI == 64][bit]);
    if (st != LCC_OK) return st;
  }
  IndexTcArgs a{ia.qI, ia.w, ia.B, ia.Tq, ia.q_pos0, ia.n_valid, ia.Ncap, ia.m, ia.q0, ia.nq, 0,
                ia.scores, ia.gmax, ia.g_stride, ia.counters};
  const int ngroups = (ia.nq + NQ - 1) / NQ;
  const int tiles = (ia.Ncap + C::TILE - 1) / C::TILE;
  const int64_t base = static_cast<int64_t>(ia.B) * ngroups;
  const int target = 3 * num_sms();
  int nsplit = base >= 2 * num_sms() ? 1 : static_cast<int>((target + base - 1) / base);
  if (nsplit > tiles) nsplit = tiles;
  if (nsplit < 1) nsplit = 1;
  a.tiles_per_split = (tiles + nsplit - 1) / nsplit;
  nsplit = (tiles + a.tiles_per_split - 1) / a.tiles_per_split;
  if (ngroups > 65535) return fail(LCC_ERR_SHAPE, "k_index_tc: %d query groups", ngroups);
  // programmatic dependent launch: the CTAs become resident while the previous
  // kernel on the stream drains and wait for it in griddepcontrol.wait
  launch_k(kern, dim3(nsplit, ngroups, ia.B), dim3(192), C::SMEM, s, true, tm, a);
  return launch_check("k_index_tc");
}

template <int HI, int DI>
lcc_status launch_index_tc(const IndexArgs& ia, cudaStream_t s) {
  CUtensorMap tm;
  lcc_status st = make_tmap_2d(&tm, ia.kI, DI, static_cast<uint64_t>(ia.B) * ia.Ncap, DI, DI, 128,
                               DI == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, "k_index_tc");
  if (st != LCC_OK) return st;
  if (ia.nq * HI <= 16) return launch_index_tc_q<HI, DI, 16 / HI>(ia, tm, 0, s);
  return launch_index_tc_q<HI, DI, 128 / HI>(ia, tm, 1, s);
}

unsigned long long g_index_fp4_done[2] = {};

// NVFP4 keys: tcgen05 indexer fed by bulk copies of the packed tiles and a
// converter warpgroup (k_index_tc_fp4); key-range splits as k_index_tc.
template <int NQ>
lcc_status launch_index_fp4_q(const IndexArgs& ia, int bit, cudaStream_t s) {
  constexpr int HI = 8, DI = 64, SR = 6, SC = 4;
  using Sm = IndexTcFp4Smem<HI, DI, NQ, SR, SC>;
  auto kern = k_index_tc_fp4<HI, DI, NQ, SR, SC>;
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    lcc_status st = ensure_smem(kern, Sm::SMEM, g_index_fp4_done[bit]);
    if (st != LCC_OK) return st;
  }
  IndexTcArgs a{ia.qI, ia.w, ia.B, ia.Tq, ia.q_pos0, ia.n_valid, ia.Ncap, ia.m, ia.q0, ia.nq, 0,
                ia.scores, ia.gmax, ia.g_stride, ia.counters, static_cast<const uint8_t*>(ia.kI), ia.kIs};
  const int ngroups = (ia.nq + NQ - 1) / NQ;
  const int tiles = (ia.Ncap + 127) / 128;
  const int64_t base = static_cast<int64_t>(ia.B) * ngroups;
  const int target = 2 * num_sms();  // one wave at two CTAs per SM
  int nsplit = base >= 2 * num_sms() ? 1 : static_cast<int>((target + base - 1) / base);
  if (nsplit > tiles) nsplit = tiles;
  if (nsplit < 1) nsplit = 1;
  a.tiles_per_split = (tiles + nsplit - 1) / nsplit;
  nsplit = (tiles + a.tiles_per_split - 1) / a.tiles_per_split;
  if (ngroups > 65535) return fail(LCC_ERR_SHAPE, "k_index_tc_fp4: %d query groups", ngroups);
  launch_k(kern, dim3(nsplit, ngroups, ia.B), dim3(320), Sm::SMEM, s, true, a);
  return launch_check("k_index_tc_fp4");
}

lcc_status launch_index_fp4(const IndexArgs& ia, cudaStream_t s) {
  if (ia.nq * 8 <= 16) return launch_index_fp4_q<2>(ia, 0, s);
  return launch_index_fp4_q<16>(ia, 1, s);
}

unsigned long long g_index_topk_tc_done[2][2] = {};
unsigned long long g_index_topk_pw_done[2] = {};
constexpr int kFusedTopkMaxK = 256;

// Prefill: indexer with the streaming top-k in its epilogue (no score buffer).
template <int HI, int DI>
lcc_status launch_index_topk_tc(const lcc_bf16* qI, const float* w, int B, int Tq, const int64_t* q_pos0,
                                const void* kI, const int32_t* n_valid, int Ncap, int m, int k, int32_t* idx,
                                float* score, cudaStream_t s) {
  constexpr int NQ = 128 / HI, STAGES = 3;
  CUtensorMap tm;
  lcc_status st = make_tmap_2d(&tm, kI, DI, static_cast<uint64_t>(B) * Ncap, DI, DI, 128,
                               DI == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, "k_index_topk_tc");
  if (st != LCC_OK) return st;
  IndexTopkTcArgs a{reinterpret_cast<const bf16*>(qI), w, B, Tq, q_pos0, n_valid, Ncap, m, k, idx, score};
  const int groups = (Tq + NQ - 1) / NQ;
  if constexpr (NQ == 16) {
    using P = IndexTopkPwCfg<HI, DI, NQ, STAGES>;
    if (k <= P::CAPB - 32) {  // warp-private candidate buffers
      auto kern = k_index_topk_pw<HI, DI, NQ, STAGES>;
      {
        std::lock_guard<std::mutex> lk(g_attr_mu);
        if ((st = ensure_smem(kern, P::SMEM, g_index_topk_pw_done[DI == 64])) != LCC_OK) return st;
      }
      launch_k(kern, dim3(1, groups, B), dim3(P::NT), P::SMEM, s, false, tm, a);
      return launch_check("k_index_topk_pw");
    }
  }
  using X = IndexTopkTcCfg<HI, DI, NQ, STAGES>;
  auto kern = k_index_topk_tc<HI, DI, NQ, STAGES>;
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if ((st = ensure_smem(kern, X::SMEM, g_index_topk_tc_done[HI == 8][DI == 64])) != LCC_OK) return st;
  }
  launch_k(kern, dim3(1, groups, B), dim3(320), X::SMEM, s, false, tm, a);
  return launch_check("k_index_topk_tc");
}

bool use_fused_topk(lcc_key_format fmt, int Tq, int HI, int k) {
  return fmt == LCC_KEY_BF16 && static_cast<int64_t>(Tq) * HI > 16 && k <= kFusedTopkMaxK &&
         (Tq + 128 / HI - 1) / (128 / HI) <= 65535;
}

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
  if (code == DEV_ERR_RANGE)
    return fail(LCC_ERR_DEVICE, "decode append: the new token of sequence %u falls outside its raw buffer, or the "
                "block it completes outside the raw buffer or the caches", detail);
  if (code == DEV_ERR_POS)
    return fail(LCC_ERR_DEVICE, "compress_at: the first token of sequence %u is negative or not a multiple of m "
                "(the sequence was skipped)", detail);
  return fail(LCC_ERR_DEVICE, "index list entry out of range at list position %u", detail);
}

lcc_status lcc_test_set_wait_fault(uint64_t wait_limit_ns, int drop_tile) {
  unsigned long long lim = wait_limit_ns == 0 ? tc::kWaitLimitNs : static_cast<unsigned long long>(wait_limit_ns);
  if (lim < 1000000ull) lim = 1000000ull;
  if (lim > tc::kWaitLimitNs) lim = tc::kWaitLimitNs;
  const int drop = drop_tile < 0 ? -1 : drop_tile;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(tc::g_wait_limit_ns, &lim, sizeof(lim));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(tc::g_test_drop_tile, &drop, sizeof(drop));
  if (e != cudaSuccess) return fail(LCC_ERR_CUDA, "lcc_test_set_wait_fault: %s", cudaGetErrorString(e));
  return LCC_OK;
}

lcc_status lcc_csa_compress(const lcc_bf16* K, const lcc_bf16* V, const float* gate, int B, int n_blocks, int D,
                            int64_t kv_bstride, int64_t gate_bstride, lcc_bf16* Kc, lcc_bf16* Vc, int64_t c_bstride,
                            void* stream) {
  return compress_impl(4, K, V, gate, B, n_blocks, D, kv_bstride, gate_bstride, Kc, Vc, c_bstride, stream);
}

lcc_status lcc_compress(int m, const lcc_bf16* K, const lcc_bf16* V, const float* gate, int B, int n_blocks, int D,
                        int64_t kv_bstride, int64_t gate_bstride, lcc_bf16* Kc, lcc_bf16* Vc, int64_t c_bstride,
                        void* stream) {
  return compress_impl(m, K, V, gate, B, n_blocks, D, kv_bstride, gate_bstride, Kc, Vc, c_bstride, stream);
}

lcc_status lcc_compress_at(int m, const lcc_bf16* K, const lcc_bf16* V, const float* gate, int B, int n_tokens,
                           int D, int64_t kv_bstride, int64_t gate_bstride, const int64_t* tok0, lcc_bf16* Kc,
                           lcc_bf16* Vc, int Ncap, int64_t c_bstride, int32_t* n_valid, void* stream) {
  const char* name = "lcc_compress_at";
  if (!tok0) return fail(LCC_ERR_ARG, "%s: null tok0", name);
  if (m < 1 || n_tokens < 0) return fail(LCC_ERR_SHAPE, "%s: m=%d n_tokens=%d", name, m, n_tokens);
  return compress_impl(m, K, V, gate, B, n_tokens / m, D, kv_bstride, gate_bstride, Kc, Vc, c_bstride, stream, tok0,
                       n_valid, Ncap, name);
}

lcc_status lcc_hca_compress(const lcc_bf16* K, const lcc_bf16* V, const float* gate, int B, int n_blocks, int D,
                            int64_t kv_bstride, int64_t gate_bstride, lcc_bf16* Kc, lcc_bf16* Vc, int64_t c_bstride,
                            void* stream) {
  return compress_impl(128, K, V, gate, B, n_blocks, D, kv_bstride, gate_bstride, Kc, Vc, c_bstride, stream);
}

size_t lcc_index_topk_workspace(int B, int Tq, int Ncap, int k) { return index_ws(B, Tq, Ncap, k).total; }

lcc_status lcc_qkv_prologue(const lcc_bf16* q, const lcc_bf16* k, const lcc_bf16* v, int B, int T, int H, int D,
                            const float* gamma_q, const float* gamma_k, const float* gamma_v, float eps, int d_rope,
                            float rope_base, const int64_t* pos0, lcc_bf16* q_out, lcc_bf16* k_out, lcc_bf16* v_out,
                            void* stream) {
  const char* name = "lcc_qkv_prologue";
  if (B < 0 || T < 0) return fail(LCC_ERR_SHAPE, "%s: B=%d T=%d must be >= 0", name, B, T);
  if (B == 0 || T == 0) return LCC_OK;
  if (!q || !k || !q_out || !k_out || !gamma_q || !gamma_k || !pos0) return fail(LCC_ERR_ARG, "%s: null pointer", name);
  if ((v == nullptr) != (v_out == nullptr) || (v && !gamma_v))
    return fail(LCC_ERR_ARG, "%s: v, v_out and gamma_v go together", name);
  if (D != 64 && D != 128) return fail(LCC_ERR_SHAPE, "%s: D=%d (supported: 64, 128)", name, D);
  if (H < 1 || H > 128) return fail(LCC_ERR_SHAPE, "%s: H=%d (supported: 1..128)", name, H);
  if (d_rope < 0 || d_rope > D || (d_rope % 16))
    return fail(LCC_ERR_SHAPE, "%s: d_rope=%d (a multiple of 16, at most D)", name, d_rope);
  if (!(eps >= 0.f) || !(rope_base > 1.f) || !std::isfinite(rope_base))
    return fail(LCC_ERR_ARG, "%s: eps must be >= 0 and rope_base > 1", name);
  if (!aligned16(q) || !aligned16(k) || !aligned16(q_out) || !aligned16(k_out) || (v && (!aligned16(v) ||
      !aligned16(v_out))))
    return fail(LCC_ERR_ALIGN, "%s: q, k, v and outputs must be 16-byte aligned", name);
  const int64_t toks = static_cast<int64_t>(B) * T;
  if (toks > 0x7FFFFFFF) return fail(LCC_ERR_SHAPE, "%s: too many tokens", name);
  PrologueArgs a{};
  a.q = reinterpret_cast<const bf16*>(q); a.k = reinterpret_cast<const bf16*>(k); a.v = reinterpret_cast<const bf16*>(v);
  a.q_out = reinterpret_cast<bf16*>(q_out); a.k_out = reinterpret_cast<bf16*>(k_out);
  a.v_out = reinterpret_cast<bf16*>(v_out);
  a.gq = gamma_q; a.gk = gamma_k; a.gv = gamma_v; a.pos0 = pos0;
  a.B = B; a.T = T; a.H = H; a.eps = eps; a.d_rope = d_rope; a.log2_base = std::log2(static_cast<double>(rope_base));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (D == 128) k_qkv_prologue<128><<<static_cast<unsigned>(toks), 256, 0, s>>>(a);
  else k_qkv_prologue<64><<<static_cast<unsigned>(toks), 256, 0, s>>>(a);
  return launch_check(name);
}

lcc_status lcc_decode_append(int m, int B, int D, const lcc_bf16* k_new, const lcc_bf16* v_new, const float* g_new,
                             const int64_t* pos, lcc_bf16* Kr, lcc_bf16* Vr, float* gate_r, int64_t r_bstride,
                             int64_t g_bstride, int Rcap, const int64_t* raw_pos0, lcc_bf16* Kc, lcc_bf16* Vc,
                             int64_t c_bstride, int Ncap, int32_t* n_valid, lcc_key_format fmt, int DI,
                             const void* kI_new, const uint8_t* kI_scale_new, void* kI, uint8_t* kI_scale,
                             void* stream) {
  const char* name = "lcc_decode_append";
  if (B < 0) return fail(LCC_ERR_SHAPE, "%s: B=%d", name, B);
  if (B == 0) return LCC_OK;
  if (m != 1 && m != 4 && m != 128) return fail(LCC_ERR_SHAPE, "%s: m=%d (supported: 1, 4, 128)", name, m);
  if (D != 64 && D != 128) return fail(LCC_ERR_SHAPE, "%s: D=%d (supported: 64, 128)", name, D);
  if (!k_new || !v_new || !g_new || !pos || !Kr || !Vr || !gate_r || !raw_pos0 || !Kc || !Vc || !n_valid)
    return fail(LCC_ERR_ARG, "%s: null pointer", name);
  if (Rcap < 1 || Ncap < 1) return fail(LCC_ERR_SHAPE, "%s: Rcap=%d Ncap=%d must be >= 1", name, Rcap, Ncap);
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(Kr) || !aligned16(Vr) || !aligned16(Kc) ||
      !aligned16(Vc) || (r_bstride % 8) || (c_bstride % 8))
    return fail(LCC_ERR_ALIGN, "%s: K/V buffers must be 16-byte aligned and batch strides multiples of 8", name);
  if (B > 1 && (r_bstride < static_cast<int64_t>(Rcap) * D || c_bstride < static_cast<int64_t>(Ncap) * D ||
                g_bstride < Rcap))
    return fail(LCC_ERR_SHAPE, "%s: batch strides smaller than one batch's rows", name);
  AppendArgs a{};
  a.k_new = reinterpret_cast<const bf16*>(k_new); a.v_new = reinterpret_cast<const bf16*>(v_new); a.g_new = g_new;
  a.pos = pos; a.raw_pos0 = raw_pos0;
  a.Kr = reinterpret_cast<bf16*>(Kr); a.Vr = reinterpret_cast<bf16*>(Vr); a.gate_r = gate_r;
  a.r_bs = r_bstride; a.g_bs = g_bstride; a.Rcap = Rcap;
  a.Kc = reinterpret_cast<bf16*>(Kc); a.Vc = reinterpret_cast<bf16*>(Vc); a.c_bs = c_bstride; a.Ncap = Ncap;
  a.n_valid = n_valid;
  if (kI_new) {
    if (!kI) return fail(LCC_ERR_ARG, "%s: kI_new given without kI", name);
    if (fmt == LCC_KEY_BF16) {
      if (DI != 32 && DI != 64) return fail(LCC_ERR_SHAPE, "%s: DI=%d (bf16 keys: 32, 64)", name, DI);
      a.kI_bytes = DI * 2;
    } else if (fmt == LCC_KEY_NVFP4) {
      if (DI != 64) return fail(LCC_ERR_SHAPE, "%s: DI=%d (NVFP4 keys: 64)", name, DI);
      if (!kI_scale_new || !kI_scale) return fail(LCC_ERR_ARG, "%s: NVFP4 keys need their scales", name);
      a.kI_bytes = DI / 2;
      a.kIs_new = kI_scale_new; a.kIs = kI_scale; a.kIs_bytes = DI / 16;
    } else {
      return fail(LCC_ERR_ARG, "%s: unknown key format %d", name, fmt);
    }
    a.kI_new = static_cast<const uint8_t*>(kI_new);
    a.kI = static_cast<uint8_t*>(kI);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 grid(static_cast<unsigned>(B));
  if (m == 1) {
    if (D == 128) k_decode_append<1, 128><<<grid, 256, 0, s>>>(a); else k_decode_append<1, 64><<<grid, 256, 0, s>>>(a);
  } else if (m == 4) {
    if (D == 128) k_decode_append<4, 128><<<grid, 256, 0, s>>>(a); else k_decode_append<4, 64><<<grid, 256, 0, s>>>(a);
  } else {
    if (D == 128) k_decode_append<128, 128><<<grid, 256, 0, s>>>(a);
    else k_decode_append<128, 64><<<grid, 256, 0, s>>>(a);
  }
  return launch_check(name);
}

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
  if (fmt == LCC_KEY_NVFP4 && (reinterpret_cast<uintptr_t>(kI_scale) & 3))
    return fail(LCC_ERR_ALIGN, "%s: kI_scale must be 4-byte aligned", name);
  return LCC_OK;
}

lcc_status launch_scores(const IndexArgs& ia, int HI, int DI, lcc_key_format fmt, cudaStream_t s) {
  if (fmt == LCC_KEY_NVFP4) return launch_index_fp4(ia, s);
  if (HI == 8 && DI == 64) return launch_index_tc<8, 64>(ia, s);
  if (HI == 8 && DI == 32) return launch_index_tc<8, 32>(ia, s);
  if (HI == 4 && DI == 64) return launch_index_tc<4, 64>(ia, s);
  return launch_index_tc<4, 32>(ia, s);
}

// Indexer + top-k over queries [0, Tq) in chunks of qc queries, with the
// chunk scratch at `scratch` (index_ws_rows(B*qc, Ncap) bytes).
lcc_status run_index_topk(const lcc_bf16* qI, const float* w, int B, int Tq, int HI, int DI, const int64_t* q_pos0,
                          lcc_key_format fmt, const void* kI, const uint8_t* kI_scale, const int32_t* n_valid,
                          int Ncap, int m, int k, int32_t* idx, float* score, void* scratch, int qc,
                          cudaStream_t s) {
  if (use_fused_topk(fmt, Tq, HI, k)) {
    if (HI == 8 && DI == 64) return launch_index_topk_tc<8, 64>(qI, w, B, Tq, q_pos0, kI, n_valid, Ncap, m, k, idx, score, s);
    if (HI == 8 && DI == 32) return launch_index_topk_tc<8, 32>(qI, w, B, Tq, q_pos0, kI, n_valid, Ncap, m, k, idx, score, s);
    if (HI == 4 && DI == 64) return launch_index_topk_tc<4, 64>(qI, w, B, Tq, q_pos0, kI, n_valid, Ncap, m, k, idx, score, s);
    return launch_index_topk_tc<4, 32>(qI, w, B, Tq, q_pos0, kI, n_valid, Ncap, m, k, idx, score, s);
  }
  const IndexWs ws = index_ws_rows(static_cast<int64_t>(B) * qc, Ncap);
  char* base = static_cast<char*>(scratch);
  float* scores = reinterpret_cast<float*>(base);
  base += ws.scores;
  uint32_t* gmax = reinterpret_cast<uint32_t*>(base);
  base += ws.gmax;
  int* counters = reinterpret_cast<int*>(base);
  base += ws.counters;
  int* seg_cnt = reinterpret_cast<int*>(base);
  base += ws.seg_cnt;
  uint32_t* cand_k = reinterpret_cast<uint32_t*>(base);
  base += ws.cand_k;
  int32_t* cand_i = reinterpret_cast<int32_t*>(base);
  const int nseg = topk_segments(Ncap);
  for (int q0 = 0; q0 < Tq; q0 += qc) {
    const int nq = qc < Tq - q0 ? qc : Tq - q0;
    IndexArgs ia{reinterpret_cast<const bf16*>(qI), w, B, Tq, q_pos0, kI, kI_scale, n_valid, Ncap, m, q0, nq,
                 scores, gmax, gmax_stride(Ncap), counters};
    lcc_status st = launch_scores(ia, HI, DI, fmt, s);
    if (st != LCC_OK) return st;
    TopkThrArgs ta{};
    ta.scores = scores;
    ta.gmax = gmax;
    ta.gs = 32;  // both tensor-core indexers write one maximum per 32 entries
    ta.g_stride = gmax_stride(Ncap);
    ta.Ncap = Ncap;
    ta.q_pos0 = q_pos0;
    ta.n_valid = n_valid;
    ta.m = m;
    ta.Tq = Tq;
    ta.q0 = q0;
    ta.nq = nq;
    ta.k = k;
    ta.cand_key = cand_k;
    ta.cand_idx = cand_i;
    ta.seg_cnt = seg_cnt;
    ta.seg_cap = kSegCap;
    ta.nseg = nseg;
    ta.done = counters;
    ta.out_i = idx;
    ta.out_s = score;
    const int64_t rows = static_cast<int64_t>(B) * nq;
    if (rows > 0x7FFFFFFF / 8) return fail(LCC_ERR_SHAPE, "top-k: %lld rows", static_cast<long long>(rows));
    const int cl = topk_cluster_ctas(Ncap, k, ta.gs);
    if (cl == 0 && use_gsel(Ncap, k)) {
      const bool few = rows <= kGselFewRows;
      auto kern = few ? k_topk_gsel<kGselNTFew, kGselCap> : k_topk_gsel<kGselNT, kGselCap>;
      const size_t smem = gsel_smem(Ncap);
      {
        std::lock_guard<std::mutex> lk(g_attr_mu);
        if ((st = ensure_smem(kern, 200 * 1024, g_topk_gsel_done[few])) != LCC_OK) return st;
      }
      launch_k(kern, dim3(static_cast<unsigned>(rows)), dim3(few ? kGselNTFew : kGselNT), smem, s, true, ta);
      if ((st = launch_check("k_topk_gsel")) != LCC_OK) return st;
      continue;
    }
    if (cl > 0) {
      auto kern = k_topk_cluster<kClNT, kClPer, kClCap, kClMaxG>;
      {
        std::lock_guard<std::mutex> lk(g_attr_mu);
        if ((st = ensure_smem(kern, ClSmem::total, g_topk_cl_done)) != LCC_OK) return st;
      }
      launch_kc(kern, dim3(static_cast<unsigned>(rows * cl)), dim3(kClNT), ClSmem::total, s, true,
                static_cast<unsigned>(cl), ta);
      if ((st = launch_check("k_topk_cluster")) != LCC_OK) return st;
      continue;
    }
    launch_k(k_topk_thr<kTopkNT, kTopkPer, kCandCap>, dim3(static_cast<unsigned>(rows), nseg), dim3(kTopkNT), 0, s,
             true, ta);
    if ((st = launch_check("k_topk_thr")) != LCC_OK) return st;
  }
  return LCC_OK;
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
  IndexArgs ia{reinterpret_cast<const bf16*>(qI), w, B, Tq, q_pos0, kI, kI_scale, n_valid, Ncap, m, 0, Tq, scores,
               nullptr, 0, nullptr};
  return launch_scores(ia, HI, DI, fmt, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {
template <int HI, int DI, bool FP4, int CAP>
lcc_status launch_reindex(const ReindexArgs& a, cudaStream_t s) {
  constexpr int NT = 128;
  k_reindex_topk<HI, DI, FP4, NT, CAP><<<static_cast<unsigned>(static_cast<int64_t>(a.B) * a.Tq), NT, 0, s>>>(a);
  return launch_check("k_reindex_topk");
}
template <int HI, int DI, bool FP4>
lcc_status launch_reindex_cap(const ReindexArgs& a, cudaStream_t s) {
  if (a.n_cand <= 256) return launch_reindex<HI, DI, FP4, 256>(a, s);
  if (a.n_cand <= 512) return launch_reindex<HI, DI, FP4, 512>(a, s);
  return launch_reindex<HI, DI, FP4, 1024>(a, s);
}
}  // namespace

extern "C" {

lcc_status lcc_lightning_reindex_topk(const lcc_bf16* qI, const float* w, int B, int Tq, int HI, int DI,
                                      lcc_key_format fmt, const void* kI, const uint8_t* kI_scale, int Ncap,
                                      const int32_t* cand, int n_cand, int k, int32_t* idx, float* score,
                                      void* stream) {
  const char* name = "lcc_lightning_reindex_topk";
  if (B < 0 || Tq < 0) return fail(LCC_ERR_SHAPE, "%s: B=%d Tq=%d must be >= 0", name, B, Tq);
  if (B == 0 || Tq == 0) return LCC_OK;
  if (!qI || !w || !kI || !cand || !idx) return fail(LCC_ERR_ARG, "%s: null pointer", name);
  if (fmt != LCC_KEY_BF16 && fmt != LCC_KEY_NVFP4) return fail(LCC_ERR_ARG, "%s: unknown key format %d", name, fmt);
  if (fmt == LCC_KEY_NVFP4 && !kI_scale) return fail(LCC_ERR_ARG, "%s: NVFP4 keys need kI_scale", name);
  if (HI != 4 && HI != 8) return fail(LCC_ERR_SHAPE, "%s: HI=%d (supported: 4, 8)", name, HI);
  if (fmt == LCC_KEY_BF16 && DI != 32 && DI != 64) return fail(LCC_ERR_SHAPE, "%s: DI=%d (bf16: 32, 64)", name, DI);
  if (fmt == LCC_KEY_NVFP4 && (DI != 64 || HI != 8))
    return fail(LCC_ERR_SHAPE, "%s: HI=%d DI=%d (NVFP4 keys: HI=8, DI=64)", name, HI, DI);
  if (Ncap < 1) return fail(LCC_ERR_SHAPE, "%s: Ncap=%d", name, Ncap);
  if (n_cand < 1 || n_cand > 1024 || k < 1 || k > n_cand)
    return fail(LCC_ERR_SHAPE, "%s: n_cand=%d k=%d (1 <= k <= n_cand <= 1024)", name, n_cand, k);
  if (static_cast<int64_t>(B) * Tq > 0x7FFFFFFF) return fail(LCC_ERR_SHAPE, "%s: too many queries", name);
  if (!aligned16(kI) || !aligned16(qI)) return fail(LCC_ERR_ALIGN, "%s: qI and kI must be 16-byte aligned", name);
  ReindexArgs a{};
  a.qI = reinterpret_cast<const bf16*>(qI); a.w = w; a.B = B; a.Tq = Tq;
  a.kI = kI; a.kIs = kI_scale; a.Ncap = Ncap; a.cand = cand; a.n_cand = n_cand; a.k = k;
  a.idx = idx; a.score = score;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fmt == LCC_KEY_NVFP4) return launch_reindex_cap<8, 64, true>(a, s);
  if (HI == 8 && DI == 64) return launch_reindex_cap<8, 64, false>(a, s);
  if (HI == 8 && DI == 32) return launch_reindex_cap<8, 32, false>(a, s);
  if (HI == 4 && DI == 64) return launch_reindex_cap<4, 64, false>(a, s);
  return launch_reindex_cap<4, 32, false>(a, s);
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
  const IndexWs ws = index_ws(B, Tq, Ncap, k);
  if (!workspace || workspace_bytes < ws.total)
    return fail(LCC_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", name, workspace_bytes, ws.total);
  if (!aligned16(workspace)) return fail(LCC_ERR_ALIGN, "%s: workspace must be 16-byte aligned", name);
  return run_index_topk(qI, w, B, Tq, HI, DI, q_pos0, fmt, kI, kI_scale, n_valid, Ncap, m, k, idx, score, workspace,
                        index_chunk(B, Tq, Ncap), static_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ------------------------------------------------------------------ attention
namespace {

unsigned long long g_attn_done[2][2][3][2] = {};

template <int D, int ROWS, int MODE, bool WIN2>
lcc_status launch_attn(const AttnArgs& a, dim3 grid, cudaStream_t s, bool pdl) {
  const size_t smem = AttnSmem<D, ROWS>::total;
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    lcc_status st = ensure_smem(k_attn<D, ROWS, MODE, WIN2>, smem, g_attn_done[D == 128][ROWS == 64][MODE][WIN2]);
    if (st != LCC_OK) return st;
  }
  launch_k(k_attn<D, ROWS, MODE, WIN2>, grid, dim3(ROWS * 2), smem, s, pdl, a);
  return launch_check("k_attn");
}

template <int MODE, bool WIN2 = false>
lcc_status dispatch_attn(const AttnArgs& a, int D, dim3 grid, int rows, cudaStream_t s, bool pdl = false) {
  if (D == 128)
    return rows == 64 ? launch_attn<128, 64, MODE, WIN2>(a, grid, s, pdl)
                      : launch_attn<128, 16, MODE, WIN2>(a, grid, s, pdl);
  return rows == 64 ? launch_attn<64, 64, MODE, WIN2>(a, grid, s, pdl) : launch_attn<64, 16, MODE, WIN2>(a, grid, s, pdl);
}

template <int D>
lcc_status launch_combine(const float* Op, const float* lp, int ns, int64_t rows, float* O, float* lse, bf16* out,
                          cudaStream_t s) {
  const unsigned g = static_cast<unsigned>((rows + 7) / 8);
  launch_k(k_split_combine<D>, dim3(g), dim3(256), 0, s, true, Op, lp, ns, rows, O, lse, out);
  return launch_check("k_split_combine");
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

// Key-range splits for a call with `rowblocks` CTAs per split and `keys`
// keys per row: enough CTAs to cover the SMs twice, at least one 64-key
// tile per split.
int splits_for(int64_t rowblocks, int64_t keys) {
  const int64_t target = 2 * num_sms();
  if (rowblocks >= target) return 1;
  int64_t ns = (target + rowblocks - 1) / rowblocks;
  const int64_t tiles = (keys + 63) / 64;
  if (ns > tiles) ns = tiles;
  if (ns > 128) ns = 128;
  return ns < 1 ? 1 : static_cast<int>(ns);
}

size_t split_ws_bytes(int ns, int64_t rows, int D) {
  if (ns <= 1) return 0;
  return round_up(ns * rows * D * sizeof(float), 256) + round_up(ns * rows * sizeof(float), 256);
}

// ---- tensor-core attention for long query blocks (prefill) ----
unsigned long long g_attn_tc_done = 0;

// Worth the tensor-core kernel: D = 128 and enough 128-row blocks to fill the GPU.
// The tensor-core kernels fold the (positive, finite) scale into the
// exponent after the row maximum; other scales take the legacy path.
bool tc_scale_ok(float scale) { return scale > 0.f && scale < 3.0e38f; }

bool use_attn_tc(int B, int Tq, int H, int D, float scale) {
  return D == 128 && tc_scale_ok(scale) &&
         static_cast<int64_t>(B) * ((static_cast<int64_t>(Tq) * H + 127) / 128) >= num_sms();
}

// CSA sparse attention (+ window) on the tensor cores: H = 64 or 128 (whole
// queries per 128-row item), enough items for every SM, 32-bit row numbers.
unsigned long long g_attn_gather_done = 0;

bool use_gather_tc(int B, int Tq, int H, int D, float scale, int Ncap, int Rcap) {
  const int64_t items = static_cast<int64_t>(B) * ((static_cast<int64_t>(Tq) * H + 127) / 128);
  return D == 128 && (H == 64 || H == 128) && tc_scale_ok(scale) && Ncap > 0 && items >= num_sms() &&
         items <= 0x7FFFFFFF && static_cast<int64_t>(B) * Ncap < (int64_t(1) << 31) &&
         static_cast<int64_t>(B) * Rcap < (int64_t(1) << 31) &&
         static_cast<int64_t>(B) * Tq * H < (int64_t(1) << 31);
}

lcc_status launch_attn_gather_tc(AttnGatherArgs a, const bf16* q, const bf16* Kc, const bf16* Vc, int64_t kv_rs,
                                 const bf16* Kr, const bf16* Vr, int64_t r_rs, cudaStream_t s, bool pdl) {
  using Cf = AttnGatherCfg;
  constexpr int D = Cf::D;
  CUtensorMap tq, tk, tv, tkw, tvw;
  const uint64_t qrows = static_cast<uint64_t>(a.B) * a.Tq * a.H;
  lcc_status st = make_tmap_2d(&tq, q, D, qrows, D, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "k_attn_gather_tc q");
  if (st != LCC_OK) return st;
  const uint64_t r1 = static_cast<uint64_t>(a.B) * a.Ncap;
  // gathered rows: one-row boxes (tile::gather4 fetches four rows per copy)
  if ((st = make_tmap_2d(&tk, Kc, D, r1, kv_rs, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B, "k_attn_gather_tc K")) != LCC_OK)
    return st;
  if ((st = make_tmap_2d(&tv, Vc, D, r1, kv_rs, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B, "k_attn_gather_tc V")) != LCC_OK)
    return st;
  if (a.win) {
    const uint64_t r2 = static_cast<uint64_t>(a.B) * (a.Rcap > 0 ? a.Rcap : 1);
    if ((st = make_tmap_2d(&tkw, Kr, D, r2, r_rs, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "k_attn_gather_tc Kw")) !=
        LCC_OK)
      return st;
    if ((st = make_tmap_2d(&tvw, Vr, D, r2, r_rs, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "k_attn_gather_tc Vw")) !=
        LCC_OK)
      return st;
  } else {
    tkw = tk;
    tvw = tv;
  }
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if ((st = ensure_smem(k_attn_gather_tc, Cf::SMEM, g_attn_gather_done)) != LCC_OK) return st;
  }
  a.tiles_q = static_cast<int>((static_cast<int64_t>(a.Tq) * a.H + 127) / 128);
  const int64_t items = static_cast<int64_t>(a.B) * a.tiles_q;
  const unsigned grid = static_cast<unsigned>(items < num_sms() ? items : num_sms());
  launch_k(k_attn_gather_tc, dim3(grid), dim3(192), Cf::SMEM, s, pdl, tq, tk, tv, tkw, tvw, a);
  return launch_check("k_attn_gather_tc");
}

// src1 (K1/V1, rows kv_rs1 apart, Ncap1 per batch) and optional window src2.
lcc_status launch_attn_tc(AttnTcArgs a, const bf16* q, const bf16* K1, const bf16* V1, int64_t kv_rs1,
                          const bf16* K2, const bf16* V2, int64_t kv_rs2, int nsplit, cudaStream_t s, bool pdl) {
  constexpr int D = 128;
  using Cf = AttnTcCfg<D>;
  CUtensorMap tq, tk1, tv1, tk2, tv2;
  const uint64_t qrows = static_cast<uint64_t>(a.B) * a.Tq * a.H;
  lcc_status st = make_tmap_2d(&tq, q, D, qrows, D, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "k_attn_tc q");
  if (st != LCC_OK) return st;
  const uint64_t r1 = static_cast<uint64_t>(a.B) * (a.Ncap1 > 0 ? a.Ncap1 : 1);
  if ((st = make_tmap_2d(&tk1, K1, D, r1, kv_rs1, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "k_attn_tc K")) != LCC_OK)
    return st;
  if ((st = make_tmap_2d(&tv1, V1, D, r1, kv_rs1, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "k_attn_tc V")) != LCC_OK)
    return st;
  if (a.win2) {
    const uint64_t r2 = static_cast<uint64_t>(a.B) * (a.Ncap2 > 0 ? a.Ncap2 : 1);
    if ((st = make_tmap_2d(&tk2, K2, D, r2, kv_rs2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "k_attn_tc Kw")) != LCC_OK)
      return st;
    if ((st = make_tmap_2d(&tv2, V2, D, r2, kv_rs2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "k_attn_tc Vw")) != LCC_OK)
      return st;
  } else {
    tk2 = tk1;
    tv2 = tv1;
  }
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if ((st = ensure_smem(k_attn_tc<D>, Cf::SMEM, g_attn_tc_done)) != LCC_OK) return st;
  }
  if (a.rpt <= 0) a.rpt = 128;
  if (a.tps <= 0) a.tps = 0x3FFFFFFF;
  const int64_t gx = (static_cast<int64_t>(a.Tq) * a.H + a.rpt - 1) / a.rpt;
  if (gx > 0x7FFFFFFF) return fail(LCC_ERR_SHAPE, "k_attn_tc: too many rows");
  launch_k(k_attn_tc<D>, dim3(static_cast<unsigned>(gx), a.B, nsplit), dim3(192), Cf::SMEM, s, pdl, tq, tk1, tv1, tk2,
           tv2, a);
  return launch_check("k_attn_tc");
}

// Decode-sized calls on the tensor cores: one query's H <= 128 heads per CTA
// tile (the rest of the 128-row MMA is padding), the key tiles split across
// CTAs, fp32 partials combined to the output.  Returns LCC_ERR_UNSUPPORTED
// when this path does not apply (the caller then uses another kernel).
size_t tc_decode_ws(int B, int Tq, int H, int D, int64_t keys, int* nsplit_out, int* tps_out) {
  const int64_t tiles = (keys + 127) / 128;
  const int64_t ctas = static_cast<int64_t>(B) * Tq;
  int64_t ns = (num_sms() + ctas - 1) / ctas;
  if (ns > kCombineFirstSplits) ns = kCombineFirstSplits;  // the combine then needs one round of loads
  if (ns > tiles) ns = tiles;
  if (ns < 1) ns = 1;
  const int64_t tps = (tiles + ns - 1) / ns;
  ns = (tiles + tps - 1) / tps;
  if (nsplit_out) *nsplit_out = static_cast<int>(ns);
  if (tps_out) *tps_out = static_cast<int>(tps);
  const int64_t rows = static_cast<int64_t>(B) * Tq * H;
  return ns > 1 ? round_up(ns * rows * D * sizeof(float), 256) + round_up(ns * rows * sizeof(float), 256) : 0;
}

lcc_status tc_decode_attn(AttnTcArgs t, int D, int64_t keys, const bf16* q, const bf16* K1, const bf16* V1,
                          int64_t rs1, const bf16* K2, const bf16* V2, int64_t rs2, bf16* out, float* O, float* lse,
                          void* workspace, size_t workspace_bytes, cudaStream_t s, const char* name) {
  int ns = 1, tps = 1;
  const size_t need = tc_decode_ws(t.B, t.Tq, t.H, D, keys, &ns, &tps);
  if (ns > 1 && (!workspace || workspace_bytes < need))
    return fail(LCC_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", name, workspace_bytes, need);
  const int64_t rowsT = static_cast<int64_t>(t.B) * t.Tq * t.H;
  t.rpt = t.H;
  t.tps = tps;
  t.rows_total = rowsT;
  if (ns == 1) {
    t.out_bf16 = out;
    t.O = O;
    t.lse = lse;
    return launch_attn_tc(t, q, K1, V1, rs1, K2, V2, rs2, 1, s, false);
  }
  float* Op = static_cast<float*>(workspace);
  float* lp = reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up(ns * rowsT * D * sizeof(float), 256));
  t.out_bf16 = nullptr;
  t.O = Op;
  t.lse = lp;
  lcc_status st = launch_attn_tc(t, q, K1, V1, rs1, K2, V2, rs2, ns, s, false);
  if (st != LCC_OK) return st;
  return launch_combine<128>(Op, lp, ns, rowsT, O, lse, out, s);
}

unsigned long long g_wsplit_done[2][2] = {};
constexpr int kWsplitWarps = 8;
constexpr int kWsplitTile = 32;   // keys per warp tile

// Short key lists with few (query, 16-head) groups: warps of one CTA split
// the key tiles and combine in shared memory (no workspace, one launch).
template <int MODE>
bool use_wsplit(int64_t groups16, int64_t keys) {
  return groups16 <= 4 * num_sms() && (keys + kWsplitTile - 1) / kWsplitTile <= 4 * kWsplitWarps;
}

template <int D, int MODE>
lcc_status launch_wsplit(const AttnArgs& a, unsigned gx, cudaStream_t s, bool pdl) {
  const size_t smem = WsplitSmem<D, kWsplitWarps, kWsplitTile>::total;
  auto kern = k_attn_wsplit<D, MODE, true, kWsplitWarps, kWsplitTile>;
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    lcc_status st = ensure_smem(kern, smem, g_wsplit_done[D == 128][MODE]);
    if (st != LCC_OK) return st;
  }
  launch_k(kern, dim3(gx, a.B), dim3(kWsplitWarps * 32), smem, s, pdl, a);
  return launch_check("k_attn_wsplit");
}

// CSA layer decode with the selected entries gathered by TMA (D = 128).
unsigned long long g_wsplit_tma_done = 0;
// Lists of at most 8 x 16 selected entries and window rows: every warp takes
// one 16-key tile of each (the window tile attended while the selected rows
// are gathered); longer lists: 32-key tiles walked in turn.
template <int KT, int NB>
lcc_status launch_wsplit_tma_k(const AttnArgs& a, unsigned gx, cudaStream_t s, bool pdl, unsigned long long& done) {
  using Sm = WsplitTmaSmem<kWsplitWarps, KT, NB>;
  CUtensorMap tk, tv;
  const uint64_t rows = static_cast<uint64_t>(a.B) * a.Ncap;
  lcc_status st = make_tmap_2d(&tk, a.K, 128, rows, a.kv_rs, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B, "k_attn_wsplit_tma K");
  if (st != LCC_OK) return st;
  if ((st = make_tmap_2d(&tv, a.V, 128, rows, a.kv_rs, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B, "k_attn_wsplit_tma V")) !=
      LCC_OK)
    return st;
  auto kern = k_attn_wsplit_tma<kWsplitWarps, KT, NB>;
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if ((st = ensure_smem(kern, Sm::total, done)) != LCC_OK) return st;
  }
  launch_k(kern, dim3(gx, a.B), dim3(kWsplitWarps * 32), Sm::total, s, pdl, tk, tv, a);
  return launch_check("k_attn_wsplit_tma");
}
unsigned long long g_wsplit_tma2_done = 0;
lcc_status launch_wsplit_tma(const AttnArgs& a, unsigned gx, cudaStream_t s, bool pdl) {
  constexpr int KT2 = 16;
  if (a.k <= kWsplitWarps * KT2 && a.W <= kWsplitWarps * KT2)
    return launch_wsplit_tma_k<KT2, 2>(a, gx, s, pdl, g_wsplit_tma2_done);
  return launch_wsplit_tma_k<kWsplitTile, 1>(a, gx, s, pdl, g_wsplit_tma_done);
}

// One pass over (compressed source ++ window rows) -> bf16 layer output.
template <int MODE>
lcc_status layer_attn_impl(const char* name, AttnArgs a, int D, int64_t rowblocks, unsigned gx, int rows_per_cta,
                           int64_t keys, lcc_bf16* out, float* lse_out, void* workspace, size_t workspace_bytes,
                           cudaStream_t s, bool pdl = false) {
  const int64_t groups16 = static_cast<int64_t>(a.B) * a.Tq * ((a.H + 15) / 16);
  if (use_wsplit<MODE>(groups16, keys) && groups16 / a.B <= 0x7FFFFFFF) {
    a.out_bf16 = reinterpret_cast<bf16*>(out);
    a.lse = lse_out;
    const unsigned gw = static_cast<unsigned>(static_cast<int64_t>(a.Tq) * ((a.H + 15) / 16));
    // selected entries by TMA gather (row numbers of the tensor map fit 31 bits)
    if (MODE == ATT_GATHER && D == 128 && static_cast<int64_t>(a.B) * a.Ncap < (int64_t(1) << 31))
      return launch_wsplit_tma(a, gw, s, pdl);
    return D == 128 ? launch_wsplit<128, MODE>(a, gw, s, pdl) : launch_wsplit<64, MODE>(a, gw, s, pdl);
  }
  const int ns = splits_for(rowblocks, keys);
  const int64_t rowsT = static_cast<int64_t>(a.B) * a.Tq * a.H;
  const size_t need = split_ws_bytes(ns, rowsT, D);
  if (ns > 1 && (!workspace || workspace_bytes < need))
    return fail(LCC_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", name, workspace_bytes, need);
  a.nsplit = ns;
  a.rows_total = rowsT;
  if (ns == 1) {
    a.O = nullptr;
    a.lse = lse_out;
    a.out_bf16 = reinterpret_cast<bf16*>(out);
    return dispatch_attn<MODE, true>(a, D, dim3(gx, a.B, 1), rows_per_cta, s, pdl);
  }
  float* Op = static_cast<float*>(workspace);
  float* lp = reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up(ns * rowsT * D * sizeof(float), 256));
  a.O = Op;
  a.lse = lp;
  a.out_bf16 = nullptr;
  lcc_status st = dispatch_attn<MODE, true>(a, D, dim3(gx, a.B, ns), rows_per_cta, s, pdl);
  if (st != LCC_OK) return st;
  bf16* ob = reinterpret_cast<bf16*>(out);
  return D == 128 ? launch_combine<128>(Op, lp, ns, rowsT, nullptr, lse_out, ob, s)
                  : launch_combine<64>(Op, lp, ns, rowsT, nullptr, lse_out, ob, s);
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
  if (use_gather_tc(B, Tq, H, D, scale, Ncap, 0)) {
    AttnGatherArgs g{};
    g.B = B; g.Tq = Tq; g.H = H; g.scale_log2 = a.scale_log2;
    g.idx = idx; g.k = k; g.Ncap = Ncap; g.win = 0;
    g.O = O; g.lse = lse;
    return launch_attn_gather_tc(g, a.q, a.K, a.V, kv_rstride, nullptr, nullptr, 0,
                                 static_cast<cudaStream_t>(stream), false);
  }
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
  if (ns == 1 && use_attn_tc(B, Tq, H, D, scale)) {
    AttnTcArgs t{};
    t.B = B; t.Tq = Tq; t.H = H; t.scale_log2 = a.scale_log2; t.q_pos0 = q_pos0;
    t.mode1 = ATT_RANGE; t.Ncap1 = Ncap; t.n_valid = n_valid; t.m = m;
    t.O = O; t.lse = lse;
    return launch_attn_tc(t, a.q, a.K, a.V, kv_rstride, nullptr, nullptr, 0, 1, s, false);
  }
  if (ns == 1) {
    a.O = O; a.lse = lse;
    return dispatch_attn<ATT_RANGE>(a, D, dim3(static_cast<unsigned>(rblocks), B, 1), 64, s);
  }
  float* Op = static_cast<float*>(workspace);
  float* lp = reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up(ns * rowsT * D * sizeof(float), 256));
  a.O = Op; a.lse = lp;
  st = dispatch_attn<ATT_RANGE>(a, D, dim3(static_cast<unsigned>(rblocks), B, ns), 64, s);
  if (st != LCC_OK) return st;
  return D == 128 ? launch_combine<128>(Op, lp, ns, rowsT, O, lse, nullptr, s)
                  : launch_combine<64>(Op, lp, ns, rowsT, O, lse, nullptr, s);
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
  if (use_attn_tc(B, Tq, H, D, scale)) {
    AttnTcArgs t{};
    t.B = B; t.Tq = Tq; t.H = H; t.scale_log2 = a.scale_log2; t.q_pos0 = q_pos0;
    t.mode1 = ATT_WINDOW; t.Ncap1 = Rcap; t.raw_pos0 = raw_pos0; t.W = W;
    t.O = O; t.lse = lse;
    return launch_attn_tc(t, a.q, a.K, a.V, kv_rstride, nullptr, nullptr, 0, 1, static_cast<cudaStream_t>(stream),
                          false);
  }
  return dispatch_attn<ATT_WINDOW>(a, D, dim3(static_cast<unsigned>(rblocks), B, 1), 64,
                                   static_cast<cudaStream_t>(stream));
}

size_t lcc_layer_attn_workspace(int B, int Tq, int H, int D, int n_keys) {
  if (B <= 0 || Tq <= 0 || H <= 0 || D <= 0 || n_keys <= 0) return 0;
  // the CSA layer's CTAs hold one query (H <= 64 heads), the HCA layer's 64 rows
  const int64_t rb_csa = static_cast<int64_t>(B) * Tq * ((H + 63) / 64);
  const int64_t rb_hca = static_cast<int64_t>(B) * ((static_cast<int64_t>(Tq) * H + 63) / 64);
  const int64_t rb = rb_csa < rb_hca ? rb_csa : rb_hca;
  const size_t legacy = split_ws_bytes(splits_for(rb, n_keys), static_cast<int64_t>(B) * Tq * H, D);
  const size_t tcd = D == 128 ? tc_decode_ws(B, Tq, H, D, n_keys, nullptr, nullptr) : 0;
  return legacy > tcd ? legacy : tcd;
}

}  // extern "C"

namespace {
// ---- CSA decode: top-k and attention in one cluster per query ----
constexpr int kCfPer = 16;  // scores per thread of the top-k (4096 per CTA)
static_assert(kWsplitWarps * 32 == kClNT, "the fused kernel's top-k runs on the attention CTA's threads");
// candidate room of the fused kernel's top-k: typically ~1.5 k scores reach
// theta; more (heavy ties) take the exact bisection fallback.  Kept small so
// that an indexer CTA of the next call fits on the same SM (its launch then
// overlaps this kernel)
constexpr int kCfCap = 1024;
constexpr int kCfTile = 16;  // keys per warp tile: one selected-entry and one window tile per warp
using CfSmem = CsaFusedSmem<kWsplitWarps, kCfTile, kCfPer, kCfCap, kClMaxG>;
unsigned long long g_csa_fused_done = 0;

// Decode-shaped calls whose top-k fits the cluster selection (one CTA per 16
// heads, each loading 4096 scores) and whose attention is the warp-split
// kernel with TMA-gathered rows.
bool use_csa_fused(lcc_key_format fmt, int B, int Tq, int H, int D, int HI, float scale, int Ncap, int k, int Rcap,
                   int W) {
  if (D != 128 || H % 16 != 0 || H < 16 || H > 128) return false;
  const int cl = H / 16;
  const int64_t groups16 = static_cast<int64_t>(B) * Tq * cl;
  return !use_fused_topk(fmt, Tq, HI, k) && Ncap <= cl * kClNT * kCfPer && 2 * k <= kClMaxG &&
         static_cast<int64_t>(k) * 8 <= kCfCap && k <= kWsplitWarps * kCfTile && W <= kWsplitWarps * kCfTile &&
         !use_gather_tc(B, Tq, H, D, scale, Ncap, Rcap) &&
         use_wsplit<ATT_GATHER>(groups16, static_cast<int64_t>(k) + W) &&
         static_cast<int64_t>(B) * Ncap < (int64_t(1) << 31) && static_cast<int64_t>(Tq) * cl <= 0x7FFFFFFF &&
         B <= 65535 && index_chunk(B, Tq, Ncap) >= Tq;
}

lcc_status launch_csa_fused(const AttnArgs& a, const TopkThrArgs& t, int cl, cudaStream_t s) {
  CUtensorMap tk, tv;
  const uint64_t rows = static_cast<uint64_t>(a.B) * a.Ncap;
  lcc_status st = make_tmap_2d(&tk, a.K, 128, rows, a.kv_rs, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B, "k_csa_decode_fused K");
  if (st != LCC_OK) return st;
  if ((st = make_tmap_2d(&tv, a.V, 128, rows, a.kv_rs, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B, "k_csa_decode_fused V")) !=
      LCC_OK)
    return st;
  auto kern = k_csa_decode_fused<kWsplitWarps, kCfTile, kCfPer, kCfCap, kClMaxG>;
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if ((st = ensure_smem(kern, CfSmem::total, g_csa_fused_done)) != LCC_OK) return st;
  }
  launch_kc(kern, dim3(static_cast<unsigned>(a.Tq * cl), static_cast<unsigned>(a.B)), dim3(kWsplitWarps * 32),
            CfSmem::total, s, true, static_cast<unsigned>(cl), tk, tv, a, t);
  return launch_check("k_csa_decode_fused");
}

lcc_status check_csa_attn(const char* name, const lcc_bf16* q, int B, int Tq, int H, int D, const int64_t* q_pos0,
                          const lcc_bf16* Kc, const lcc_bf16* Vc, int64_t kv_rstride, int Ncap, const int32_t* idx,
                          int k, const lcc_bf16* Kr, const lcc_bf16* Vr, int64_t r_rstride, int Rcap,
                          const int64_t* raw_pos0, int W, const lcc_bf16* out) {
  if (!out) return fail(LCC_ERR_ARG, "%s: null out", name);
  const float* dummy = reinterpret_cast<const float*>(out);
  lcc_status st = check_attn_common(name, q, B, Tq, H, D, Kc, Vc, kv_rstride, Ncap, dummy, dummy);
  if (st != LCC_OK) return st;
  st = check_attn_common(name, q, B, Tq, H, D, Kr, Vr, r_rstride, Rcap, dummy, dummy);
  if (st != LCC_OK) return st;
  if (!idx || !q_pos0 || !raw_pos0) return fail(LCC_ERR_ARG, "%s: null idx / q_pos0 / raw_pos0", name);
  if (k < 1 || k > 4096) return fail(LCC_ERR_SHAPE, "%s: k=%d (supported: 1..4096)", name, k);
  if (W < 1 || W > 4096) return fail(LCC_ERR_SHAPE, "%s: W=%d (supported: 1..4096)", name, W);
  return LCC_OK;
}

AttnArgs csa_attn_args(const lcc_bf16* q, int B, int Tq, int H, float scale, const int64_t* q_pos0,
                       const lcc_bf16* Kc, const lcc_bf16* Vc, int64_t kv_rstride, int Ncap, const int32_t* idx, int k,
                       const lcc_bf16* Kr, const lcc_bf16* Vr, int64_t r_rstride, int Rcap, const int64_t* raw_pos0,
                       int W) {
  AttnArgs a{};
  a.q = reinterpret_cast<const bf16*>(q);
  a.B = B; a.Tq = Tq; a.H = H;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.q_pos0 = q_pos0;
  a.K = reinterpret_cast<const bf16*>(Kc); a.V = reinterpret_cast<const bf16*>(Vc);
  a.kv_bs = static_cast<int64_t>(Ncap) * kv_rstride; a.kv_rs = kv_rstride; a.Ncap = Ncap;
  a.idx = idx; a.k = k;
  a.K2 = reinterpret_cast<const bf16*>(Kr); a.V2 = reinterpret_cast<const bf16*>(Vr);
  a.kv2_bs = static_cast<int64_t>(Rcap) * r_rstride; a.kv2_rs = r_rstride; a.Ncap2 = Rcap;
  a.raw_pos0 = raw_pos0; a.W = W;
  return a;
}

lcc_status csa_layer_attn_impl(const char* name, const lcc_bf16* q, int B, int Tq, int H, int D, float scale,
                               const int64_t* q_pos0, const lcc_bf16* Kc, const lcc_bf16* Vc, int64_t kv_rstride,
                               int Ncap, const int32_t* idx, int k, const lcc_bf16* Kr, const lcc_bf16* Vr,
                               int64_t r_rstride, int Rcap, const int64_t* raw_pos0, int W, lcc_bf16* out,
                               float* lse_out, void* workspace, size_t workspace_bytes, void* stream, bool pdl) {
  if (B < 0 || Tq < 0) return fail(LCC_ERR_SHAPE, "%s: negative size", name);
  if (B == 0 || Tq == 0) return LCC_OK;
  lcc_status st = check_csa_attn(name, q, B, Tq, H, D, q_pos0, Kc, Vc, kv_rstride, Ncap, idx, k, Kr, Vr, r_rstride,
                                 Rcap, raw_pos0, W, out);
  if (st != LCC_OK) return st;
  const AttnArgs a = csa_attn_args(q, B, Tq, H, scale, q_pos0, Kc, Vc, kv_rstride, Ncap, idx, k, Kr, Vr, r_rstride,
                                   Rcap, raw_pos0, W);
  if (use_gather_tc(B, Tq, H, D, scale, Ncap, Rcap)) {
    AttnGatherArgs g{};
    g.B = B; g.Tq = Tq; g.H = H; g.scale_log2 = a.scale_log2; g.q_pos0 = q_pos0;
    g.idx = idx; g.k = k; g.Ncap = Ncap;
    g.win = 1; g.Rcap = Rcap; g.raw_pos0 = raw_pos0; g.W = W;
    g.out_bf16 = reinterpret_cast<bf16*>(out); g.lse = lse_out;
    return launch_attn_gather_tc(g, a.q, a.K, a.V, kv_rstride, a.K2, a.V2, r_rstride,
                                 static_cast<cudaStream_t>(stream), pdl);
  }
  const int rows = H <= 16 ? 16 : 64;
  const int hblocks = (H + rows - 1) / rows;
  if (static_cast<int64_t>(Tq) * hblocks > 0x7FFFFFFF) return fail(LCC_ERR_SHAPE, "%s: too many queries", name);
  const int64_t rowblocks = static_cast<int64_t>(B) * Tq * hblocks;
  return layer_attn_impl<ATT_GATHER>(name, a, D, rowblocks, static_cast<unsigned>(Tq * hblocks), rows,
                                     static_cast<int64_t>(k) + W, out, lse_out, workspace, workspace_bytes,
                                     static_cast<cudaStream_t>(stream), pdl);
}
}  // namespace

extern "C" {

lcc_status lcc_csa_layer_attn(const lcc_bf16* q, int B, int Tq, int H, int D, float scale, const int64_t* q_pos0,
                              const lcc_bf16* Kc, const lcc_bf16* Vc, int64_t kv_rstride, int Ncap,
                              const int32_t* idx, int k, const lcc_bf16* Kr, const lcc_bf16* Vr, int64_t r_rstride,
                              int Rcap, const int64_t* raw_pos0, int W, lcc_bf16* out, float* lse_out,
                              void* workspace, size_t workspace_bytes, void* stream) {
  return csa_layer_attn_impl("lcc_csa_layer_attn", q, B, Tq, H, D, scale, q_pos0, Kc, Vc, kv_rstride, Ncap, idx, k,
                             Kr, Vr, r_rstride, Rcap, raw_pos0, W, out, lse_out, workspace, workspace_bytes, stream,
                             false);
}

size_t lcc_csa_layer_workspace(int B, int Tq, int H, int D, int Ncap, int k, int W) {
  if (B <= 0 || Tq <= 0 || H <= 0 || D <= 0 || Ncap <= 0 || k <= 0 || W <= 0) return 0;
  return round_up(index_ws(B, Tq, Ncap, k).total, 256) + lcc_layer_attn_workspace(B, Tq, H, D, k + W);
}

lcc_status lcc_csa_layer(const lcc_bf16* q, const lcc_bf16* qI, const float* w, int B, int Tq, int H, int D, int HI,
                         int DI, float scale, const int64_t* q_pos0, lcc_key_format fmt, const void* kI,
                         const uint8_t* kI_scale, const int32_t* n_valid, const lcc_bf16* Kc, const lcc_bf16* Vc,
                         int64_t kv_rstride, int Ncap, int m, int k, const lcc_bf16* Kr, const lcc_bf16* Vr,
                         int64_t r_rstride, int Rcap, const int64_t* raw_pos0, int W, int32_t* idx, lcc_bf16* out,
                         float* lse_out, void* workspace, size_t workspace_bytes, void* stream) {
  const char* name = "lcc_csa_layer";
  if (B < 0 || Tq < 0) return fail(LCC_ERR_SHAPE, "%s: negative size", name);
  if (B == 0 || Tq == 0) return LCC_OK;
  const size_t need = lcc_csa_layer_workspace(B, Tq, H, D, Ncap, k, W);
  if (!workspace || workspace_bytes < need)
    return fail(LCC_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", name, workspace_bytes, need);
  const size_t ws_index = round_up(index_ws(B, Tq, Ncap, k).total, 256);
  if (use_csa_fused(fmt, B, Tq, H, D, HI, scale, Ncap, k, Rcap, W)) {
    // indexer scores, then one cluster per query selects and attends
    lcc_status st = check_index_args(name, qI, w, B, Tq, HI, DI, q_pos0, fmt, kI, kI_scale, n_valid, Ncap, m, idx);
    if (st != LCC_OK) return st;
    if (!aligned16(workspace)) return fail(LCC_ERR_ALIGN, "%s: workspace must be 16-byte aligned", name);
    if ((st = check_csa_attn(name, q, B, Tq, H, D, q_pos0, Kc, Vc, kv_rstride, Ncap, idx, k, Kr, Vr, r_rstride, Rcap,
                             raw_pos0, W, out)) != LCC_OK)
      return st;
    const IndexWs ws = index_ws_rows(static_cast<int64_t>(B) * Tq, Ncap);
    char* base = static_cast<char*>(workspace);
    float* scores = reinterpret_cast<float*>(base);
    uint32_t* gmax = reinterpret_cast<uint32_t*>(base + ws.scores);
    int* counters = reinterpret_cast<int*>(base + ws.scores + ws.gmax);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    IndexArgs ia{reinterpret_cast<const bf16*>(qI), w, B, Tq, q_pos0, kI, kI_scale, n_valid, Ncap, m, 0, Tq,
                 scores, gmax, gmax_stride(Ncap), counters};
    if ((st = launch_scores(ia, HI, DI, fmt, s)) != LCC_OK) return st;
    TopkThrArgs ta{};
    ta.scores = scores;
    ta.gmax = gmax;
    ta.gs = 32;  // the tensor-core indexers write one maximum per 32 entries
    ta.g_stride = gmax_stride(Ncap);
    ta.Ncap = Ncap;
    ta.q_pos0 = q_pos0;
    ta.n_valid = n_valid;
    ta.m = m;
    ta.Tq = Tq;
    ta.q0 = 0;
    ta.nq = Tq;
    ta.k = k;
    ta.out_i = idx;
    ta.out_s = nullptr;
    AttnArgs a = csa_attn_args(q, B, Tq, H, scale, q_pos0, Kc, Vc, kv_rstride, Ncap, idx, k, Kr, Vr, r_rstride, Rcap,
                               raw_pos0, W);
    a.out_bf16 = reinterpret_cast<bf16*>(out);
    a.lse = lse_out;
    return launch_csa_fused(a, ta, H / 16, s);
  }
  lcc_status st = lcc_lightning_index_topk(qI, w, B, Tq, HI, DI, q_pos0, fmt, kI, kI_scale, n_valid, Ncap, m, k, idx,
                                           nullptr, workspace, ws_index, stream);
  if (st != LCC_OK) return st;
  // the attention follows the top-k kernel on the stream: it may launch early and
  // prefetch the queries and window rows, then wait for the index lists
  return csa_layer_attn_impl(name, q, B, Tq, H, D, scale, q_pos0, Kc, Vc, kv_rstride, Ncap, idx, k, Kr, Vr,
                             r_rstride, Rcap, raw_pos0, W, out, lse_out, static_cast<char*>(workspace) + ws_index,
                             workspace_bytes - ws_index, stream, true);
}

lcc_status lcc_hca_layer_attn(const lcc_bf16* q, int B, int Tq, int H, int D, float scale, const int64_t* q_pos0,
                              const lcc_bf16* Kc, const lcc_bf16* Vc, int64_t kv_rstride, int Ncap,
                              const int32_t* n_valid, int m, const lcc_bf16* Kr, const lcc_bf16* Vr,
                              int64_t r_rstride, int Rcap, const int64_t* raw_pos0, int W, lcc_bf16* out,
                              float* lse_out, void* workspace, size_t workspace_bytes, void* stream) {
  const char* name = "lcc_hca_layer_attn";
  if (B < 0 || Tq < 0) return fail(LCC_ERR_SHAPE, "%s: negative size", name);
  if (B == 0 || Tq == 0) return LCC_OK;
  if (!out) return fail(LCC_ERR_ARG, "%s: null out", name);
  const float* dummy = reinterpret_cast<const float*>(out);
  lcc_status st = check_attn_common(name, q, B, Tq, H, D, Kc, Vc, kv_rstride, Ncap, dummy, dummy);
  if (st != LCC_OK) return st;
  st = check_attn_common(name, q, B, Tq, H, D, Kr, Vr, r_rstride, Rcap, dummy, dummy);
  if (st != LCC_OK) return st;
  if (!q_pos0 || !n_valid || !raw_pos0) return fail(LCC_ERR_ARG, "%s: null q_pos0 / n_valid / raw_pos0", name);
  if (m < 1) return fail(LCC_ERR_SHAPE, "%s: m=%d", name, m);
  if (W < 1 || W > 4096) return fail(LCC_ERR_SHAPE, "%s: W=%d (supported: 1..4096)", name, W);
  const int64_t rblocks = (static_cast<int64_t>(Tq) * H + 63) / 64;
  if (rblocks > 0x7FFFFFFF) return fail(LCC_ERR_SHAPE, "%s: too many queries", name);
  AttnArgs a{};
  a.q = reinterpret_cast<const bf16*>(q);
  a.B = B; a.Tq = Tq; a.H = H;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.q_pos0 = q_pos0;
  a.K = reinterpret_cast<const bf16*>(Kc); a.V = reinterpret_cast<const bf16*>(Vc);
  a.kv_bs = static_cast<int64_t>(Ncap) * kv_rstride; a.kv_rs = kv_rstride; a.Ncap = Ncap;
  a.n_valid = n_valid; a.m = m;
  a.K2 = reinterpret_cast<const bf16*>(Kr); a.V2 = reinterpret_cast<const bf16*>(Vr);
  a.kv2_bs = static_cast<int64_t>(Rcap) * r_rstride; a.kv2_rs = r_rstride; a.Ncap2 = Rcap;
  a.raw_pos0 = raw_pos0; a.W = W;
  if (use_attn_tc(B, Tq, H, D, scale)) {
    AttnTcArgs t{};
    t.B = B; t.Tq = Tq; t.H = H; t.scale_log2 = a.scale_log2; t.q_pos0 = q_pos0;
    t.mode1 = ATT_RANGE; t.Ncap1 = Ncap; t.n_valid = n_valid; t.m = m;
    t.win2 = true; t.Ncap2 = Rcap; t.raw_pos0 = raw_pos0; t.W = W;
    t.out_bf16 = reinterpret_cast<bf16*>(out); t.lse = lse_out;
    return launch_attn_tc(t, a.q, a.K, a.V, kv_rstride, a.K2, a.V2, r_rstride, 1, static_cast<cudaStream_t>(stream),
                          false);
  }
  const int64_t groups16 = static_cast<int64_t>(B) * Tq * ((H + 15) / 16);
  if (D == 128 && H <= 128 && tc_scale_ok(scale) && !use_wsplit<ATT_RANGE>(groups16, static_cast<int64_t>(Ncap) + W)) {
    AttnTcArgs t{};
    t.B = B; t.Tq = Tq; t.H = H; t.scale_log2 = a.scale_log2; t.q_pos0 = q_pos0;
    t.mode1 = ATT_RANGE; t.Ncap1 = Ncap; t.n_valid = n_valid; t.m = m;
    t.win2 = true; t.Ncap2 = Rcap; t.raw_pos0 = raw_pos0; t.W = W;
    return tc_decode_attn(t, D, static_cast<int64_t>(Ncap) + W, a.q, a.K, a.V, kv_rstride, a.K2, a.V2, r_rstride,
                          reinterpret_cast<bf16*>(out), nullptr, lse_out, workspace, workspace_bytes,
                          static_cast<cudaStream_t>(stream), name);
  }
  return layer_attn_impl<ATT_RANGE>(name, a, D, static_cast<int64_t>(B) * rblocks, static_cast<unsigned>(rblocks),
                                    64, static_cast<int64_t>(Ncap) + W, out, lse_out, workspace, workspace_bytes,
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
  // prefill-shaped requests take the indexer with the top-k fused into its
  // epilogue: no scratch at all, so no size limit either
  if (use_fused_topk(fmt, Tq, HI, k))
    return run_index_topk(qI, w, B, Tq, HI, DI, q_pos0, fmt, kI, kI_scale, n_valid, Ncap, m, k, idx, score, nullptr,
                          Tq, static_cast<cudaStream_t>(stream));
  // bytes one query row of every batch needs: scores, group maxima, candidates, counters
  const size_t per_q = index_ws_rows(B, Ncap).total;
  if (per_q > kNoAllocScratchBytes)
    return fail(LCC_ERR_WORKSPACE, "%s: one query row needs %zu scratch bytes, the fixed scratch holds %zu", name,
                per_q, kNoAllocScratchBytes);
  int qc = 1;  // largest query chunk whose scratch fits the array
  while (qc < Tq) {
    const int nx = qc * 2 < Tq ? qc * 2 : Tq;
    if (index_ws_rows(static_cast<int64_t>(B) * nx, Ncap).total > kNoAllocScratchBytes) break;
    qc = nx;
  }
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != LCC_OK) return st;
  return run_index_topk(qI, w, B, Tq, HI, DI, q_pos0, fmt, kI, kI_scale, n_valid, Ncap, m, k, idx, score, scratch, qc,
                        static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ NVFP4
namespace {
lcc_status launch_nvfp4_quant(const lcc_bf16* x, int64_t rows, int D, int64_t ld, uint8_t* packed, uint8_t* scale,
                              lcc_bf16* xq, cudaStream_t s) {
  const int64_t groups = rows * (D / 16);
  if (groups == 0) return LCC_OK;
  Nvfp4QuantArgs a{reinterpret_cast<const bf16*>(x), rows, D / 16, ld, packed, scale, reinterpret_cast<bf16*>(xq)};
  launch_k(k_nvfp4_quant, dim3(static_cast<unsigned>((groups + 255) / 256)), dim3(256), 0, s, false, a);
  return launch_check("k_nvfp4_quant");
}

lcc_status launch_nvfp4_expand(const uint8_t* packed, const uint8_t* scale, int64_t rows, int D, lcc_bf16* out,
                               cudaStream_t s) {
  const int64_t groups = rows * (D / 16);
  if (groups == 0) return LCC_OK;
  Nvfp4ExpandArgs a{packed, scale, rows, D / 16, reinterpret_cast<bf16*>(out)};
  launch_k(k_nvfp4_expand, dim3(static_cast<unsigned>((groups + 255) / 256)), dim3(256), 0, s, true, a);
  return launch_check("k_nvfp4_expand");
}

lcc_status check_nvfp4_shape(const char* name, int64_t rows, int D) {
  if (rows < 0) return fail(LCC_ERR_SHAPE, "%s: rows=%lld must be >= 0", name, static_cast<long long>(rows));
  if (D <= 0 || D % 16) return fail(LCC_ERR_SHAPE, "%s: D=%d must be a positive multiple of 16", name, D);
  if (rows * (D / 16) > 0x7FFFFFFFLL * 256)
    return fail(LCC_ERR_SHAPE, "%s: %lld groups of 16", name, static_cast<long long>(rows * (D / 16)));
  return LCC_OK;
}

// Scratch of the FP4 indexer: the dequantised query, then either the keys
// expanded to bf16 (prefill shapes, fused top-k) or the indexer's chunk scratch.
struct Fp4Ws {
  size_t q, keys, index, total;
};
Fp4Ws fp4_ws(int B, int Tq, int HI, int DI, int Ncap, int k) {
  Fp4Ws w{};
  if (B <= 0 || Tq <= 0 || Ncap <= 0 || k <= 0 || HI <= 0 || DI <= 0) return w;
  w.q = round_up(static_cast<size_t>(B) * Tq * HI * DI * sizeof(bf16), 256);
  if (use_fused_topk(LCC_KEY_BF16, Tq, HI, k))
    w.keys = round_up(static_cast<size_t>(B) * Ncap * DI * sizeof(bf16), 256);
  else
    w.index = index_ws(B, Tq, Ncap, k).total;
  w.total = w.q + w.keys + w.index;
  return w;
}
}  // namespace

extern "C" {

lcc_status lcc_nvfp4_quantize(const lcc_bf16* x, int64_t rows, int D, int64_t ld, uint8_t* packed, uint8_t* scale,
                              lcc_bf16* xq, void* stream) {
  const char* name = "lcc_nvfp4_quantize";
  lcc_status st = check_nvfp4_shape(name, rows, D);
  if (st != LCC_OK) return st;
  if (ld < D) return fail(LCC_ERR_SHAPE, "%s: ld=%lld < D=%d", name, static_cast<long long>(ld), D);
  if (rows == 0) return LCC_OK;
  if (!x) return fail(LCC_ERR_ARG, "%s: x is NULL", name);
  if (!aligned16(x) || (ld * 2) % 16)
    return fail(LCC_ERR_ALIGN, "%s: x and its row stride (ld*2 bytes) must be 16-byte aligned", name);
  if (packed && (reinterpret_cast<uintptr_t>(packed) & 7))
    return fail(LCC_ERR_ALIGN, "%s: packed must be 8-byte aligned", name);
  if (xq && !aligned16(xq)) return fail(LCC_ERR_ALIGN, "%s: xq must be 16-byte aligned", name);
  return launch_nvfp4_quant(x, rows, D, ld, packed, scale, xq, static_cast<cudaStream_t>(stream));
}

lcc_status lcc_nvfp4_dequantize(const uint8_t* packed, const uint8_t* scale, int64_t rows, int D, lcc_bf16* x,
                                void* stream) {
  const char* name = "lcc_nvfp4_dequantize";
  lcc_status st = check_nvfp4_shape(name, rows, D);
  if (st != LCC_OK) return st;
  if (rows == 0) return LCC_OK;
  if (!packed || !scale || !x) return fail(LCC_ERR_ARG, "%s: NULL pointer", name);
  if (reinterpret_cast<uintptr_t>(packed) & 7) return fail(LCC_ERR_ALIGN, "%s: packed must be 8-byte aligned", name);
  if (!aligned16(x)) return fail(LCC_ERR_ALIGN, "%s: x must be 16-byte aligned", name);
  return launch_nvfp4_expand(packed, scale, rows, D, x, static_cast<cudaStream_t>(stream));
}

size_t lcc_fp4_index_topk_workspace(int B, int Tq, int HI, int DI, int Ncap, int k) {
  return fp4_ws(B, Tq, HI, DI, Ncap, k).total;
}

lcc_status lcc_fp4_index_topk(const lcc_bf16* qI, const float* w, int B, int Tq, int HI, int DI,
                              const int64_t* q_pos0, const uint8_t* kI, const uint8_t* kI_scale,
                              const int32_t* n_valid, int Ncap, int m, int k, int32_t* idx, float* score,
                              void* workspace, size_t workspace_bytes, void* stream) {
  const char* name = "lcc_fp4_index_topk";
  if (B < 0 || Tq < 0) return fail(LCC_ERR_SHAPE, "%s: B=%d Tq=%d must be >= 0", name, B, Tq);
  if (B == 0 || Tq == 0) return LCC_OK;
  lcc_status st =
      check_index_args(name, qI, w, B, Tq, HI, DI, q_pos0, LCC_KEY_NVFP4, kI, kI_scale, n_valid, Ncap, m, idx);
  if (st != LCC_OK) return st;
  if (k < 1 || k > 1024) return fail(LCC_ERR_SHAPE, "%s: k=%d (supported: 1..1024)", name, k);
  if (reinterpret_cast<uintptr_t>(kI) & 7) return fail(LCC_ERR_ALIGN, "%s: kI must be 8-byte aligned", name);
  const Fp4Ws ws = fp4_ws(B, Tq, HI, DI, Ncap, k);
  if (!workspace || workspace_bytes < ws.total)
    return fail(LCC_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", name, workspace_bytes, ws.total);
  if (!aligned16(workspace)) return fail(LCC_ERR_ALIGN, "%s: workspace must be 16-byte aligned", name);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(workspace);
  lcc_bf16* qd = reinterpret_cast<lcc_bf16*>(base);
  const int64_t qrows = static_cast<int64_t>(B) * Tq * HI;
  if ((st = launch_nvfp4_quant(qI, qrows, DI, DI, nullptr, nullptr, qd, s)) != LCC_OK) return st;
  if (ws.keys) {
    // prefill shapes: keys expanded once per call, then the fused indexer + top-k
    lcc_bf16* kd = reinterpret_cast<lcc_bf16*>(base + ws.q);
    if ((st = launch_nvfp4_expand(kI, kI_scale, static_cast<int64_t>(B) * Ncap, DI, kd, s)) != LCC_OK) return st;
    return run_index_topk(qd, w, B, Tq, HI, DI, q_pos0, LCC_KEY_BF16, kd, nullptr, n_valid, Ncap, m, k, idx, score,
                          nullptr, Tq, s);
  }
  return run_index_topk(qd, w, B, Tq, HI, DI, q_pos0, LCC_KEY_NVFP4, kI, kI_scale, n_valid, Ncap, m, k, idx, score,
                        base + ws.q, index_chunk(B, Tq, Ncap), s);
}

}  // extern "C"

