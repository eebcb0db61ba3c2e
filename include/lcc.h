/*
 * lcc.h -- C ABI of liblcc.so, the hybrid compressed-attention path
 * (CSA + HCA + sliding window) for NVIDIA B300 (sm_103a).
 *
 * Sources (web pages, cited by title and section):
 *  [HYBRID] "DeepSeek-V4가 이차적 어텐션 비용 없이 백만 토큰 컨텍스트를 달성하는 방법"
 *           (How DeepSeek-V4 reaches a million-token context without quadratic
 *           attention cost), section "두 가지 압축 전략: CSA 및 HCA".
 *  [VIDEO]  "딥시크 V4 분석: CSA·HCA 어텐션으로 100만 토큰 컨텍스트를 저비용에 구현한 방법",
 *           sections "쉽게 이해하기" and "주요 인사이트".
 *  [THREAD] "DeepSeek v4 (Flash)는 정말 운영 비용이 엄청나게 저렴한가요?", section "주요 댓글".
 *  [V41]    DeepSeek V4.1 Flash post (jjy0501.blogspot.com), passages on the
 *           lightning indexer / CSA2, FP4 KV storage and SWA Bounded Replay.
 *
 * Conventions shared by every call
 *  - Tensors are row-major and contiguous unless a stride argument says
 *    otherwise.  Element types: lcc_bf16 = raw bfloat16 bits, float = fp32.
 *  - Every data pointer is a DEVICE pointer on the current CUDA device,
 *    16-byte aligned, owned by the caller.  The library never allocates or
 *    frees device memory and keeps no handles; scratch memory ("workspace")
 *    is passed in by the caller, sized by the matching *_workspace call.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *    validates its arguments on the host, enqueues its kernels on the stream
 *    and returns without synchronising.
 *  - Query i of batch b sits at absolute position q_pos0[b] + i.  Compressed
 *    entry j (ratio m) covers positions j*m .. j*m+m-1 and is visible to the
 *    query at position t iff j*m + m - 1 <= t and j < n_valid[b].  Raw row r
 *    of batch b is position raw_pos0[b] + r.
 *  - Attention outputs are fp32 O [B, Tq, H, D] (already normalised) and the
 *    natural-log softmax normaliser lse [B, Tq, H]; an empty key set gives
 *    O = 0 and lse = -inf.
 *  - Errors: a non-LCC_OK status is returned before anything is enqueued
 *    when an argument is invalid; lcc_last_error() then describes it
 *    (thread-local).  Launch failures return LCC_ERR_CUDA.  Conditions found
 *    on the device (an index out of range) set a device error word that
 *    lcc_sync_status() reports.  No C++ exception crosses this interface.
 */
#ifndef LCC_H_
#define LCC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t lcc_bf16;

typedef enum {
  LCC_OK = 0,
  LCC_ERR_ARG = 1,          /* null pointer or invalid value */
  LCC_ERR_SHAPE = 2,        /* unsupported or inconsistent size */
  LCC_ERR_ALIGN = 3,        /* pointer or stride not 16-byte aligned */
  LCC_ERR_UNSUPPORTED = 4,  /* valid request the library does not implement */
  LCC_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
  LCC_ERR_TIMEOUT = 6,      /* a bounded device-side wait gave up */
  LCC_ERR_DEVICE = 7,       /* a kernel found invalid data (see lcc_last_error) */
  LCC_ERR_WORKSPACE = 8     /* workspace missing or too small */
} lcc_status;

typedef enum { LCC_KEY_BF16 = 0, LCC_KEY_NVFP4 = 1 } lcc_key_format;

/* ---------------------------------------------------------------------- *
 * Compression: softmax-weighted pooling of m consecutive tokens' K and V
 * into one compressed entry.  [HYBRID]: CSA merges 4 consecutive tokens,
 * HCA 128 tokens, into one KV entry by softmax-weighted pooling; [VIDEO]
 * "쉽게 이해하기": each token's contribution is learned.
 *
 * For every batch b and block j < n_blocks, with a_i = softmax over the
 * block's m gate logits:
 *   Kc[b, j, :] = bf16_rne( sum_i a_i * K[b, j*m + i, :] )   (same for V)
 * K, V:   token rows of D bf16; row r of batch b at K + b*kv_bstride + r*D.
 *         Pass a pointer offset to the block's first token to pool a
 *         sub-range (e.g. one freshly completed block of a decode buffer).
 * gate:   one fp32 logit per token; token r of batch b at gate + b*gate_bstride + r.
 * Kc, Vc: entry j of batch b at Kc + b*c_bstride + j*D.
 * D in {64, 128}; kv_bstride, c_bstride multiples of 8 elements.
 * ---------------------------------------------------------------------- */
lcc_status lcc_csa_compress(const lcc_bf16* K, const lcc_bf16* V, const float* gate,
                            int B, int n_blocks, int D,
                            int64_t kv_bstride, int64_t gate_bstride,
                            lcc_bf16* Kc, lcc_bf16* Vc, int64_t c_bstride,
                            void* stream);                      /* m = 4 */
lcc_status lcc_hca_compress(const lcc_bf16* K, const lcc_bf16* V, const float* gate,
                            int B, int n_blocks, int D,
                            int64_t kv_bstride, int64_t gate_bstride,
                            lcc_bf16* Kc, lcc_bf16* Vc, int64_t c_bstride,
                            void* stream);                      /* m = 128 */
/* The same for any supported ratio m in {1, 4, 128}.  m = 1 makes every
 * token its own entry (the softmax over one logit is 1, so Kc = K exactly):
 * the cache of the DSA comparator, whose indexer scores every raw token
 * ([THREAD] "주요 댓글": DSA keeps the full KV and runs the light indexer over
 * all of it, then attends only to the selected tokens). */
lcc_status lcc_compress(int m, const lcc_bf16* K, const lcc_bf16* V, const float* gate,
                        int B, int n_blocks, int D,
                        int64_t kv_bstride, int64_t gate_bstride,
                        lcc_bf16* Kc, lcc_bf16* Vc, int64_t c_bstride,
                        void* stream);
/* Pooling at positions held on the device, for graph-captured prefill
 * chunks.  Rows 0 .. n_tokens-1 of sequence b's K/V/gate buffers are the
 * tokens at positions tok0[b] .. tok0[b]+n_tokens-1; tok0 (device, [B]) must
 * be a non-negative multiple of m.  The n_tokens/m complete blocks are pooled
 * as in lcc_compress into entries tok0[b]/m, tok0[b]/m + 1, ... of Kc/Vc
 * (those at or beyond Ncap are dropped), and n_valid[b] (device, [B]; may be
 * NULL) is raised to min(Ncap, tok0[b]/m + n_tokens/m) if it was below.  A
 * sequence whose tok0 is negative or not a multiple of m is skipped and
 * reported as LCC_ERR_DEVICE by the next lcc_sync_status.  c_bstride must
 * cover Ncap entries when B > 1. */
lcc_status lcc_compress_at(int m, const lcc_bf16* K, const lcc_bf16* V, const float* gate,
                           int B, int n_tokens, int D,
                           int64_t kv_bstride, int64_t gate_bstride, const int64_t* tok0,
                           lcc_bf16* Kc, lcc_bf16* Vc, int Ncap, int64_t c_bstride,
                           int32_t* n_valid, void* stream);

/* ---------------------------------------------------------------------- *
 * Query / KV prologue ([HYBRID]: both mechanisms use MQA with shared KV
 * projections, apply query and KV normalisation and use partial RoPE).  For
 * every token (b, t) at position p = pos0[b] + t:
 *   RMSNorm(x) = x / sqrt(mean_c(x_c^2) + eps) * gamma   (over the D channels)
 *   q_out[b,t,h] = RoPE_p(RMSNorm(q[b,t,h]) with gamma_q)   for every head h
 *   k_out[b,t]   = RoPE_p(RMSNorm(k[b,t])   with gamma_k)
 *   v_out[b,t]   = RMSNorm(v[b,t]) with gamma_v              (no rotation)
 * RoPE_p rotates the last d_rope channels in pairs (c, c + d_rope/2),
 * c = D-d_rope .. D-d_rope/2-1, pair i by the angle p * rope_base^(-2i/d_rope):
 *   (x1, x2) -> (x1 cos - x2 sin, x2 cos + x1 sin); the other channels pass.
 * Arithmetic in fp32 (the angle reduced modulo 2*pi in double precision),
 * outputs rounded to bf16 (nearest even).
 * q: [B, T, H, D] bf16; k, v: [B, T, D] bf16 (v, v_out, gamma_v may all be
 * NULL); gammas: [D] fp32; pos0: [B] int64 device array.  Outputs may alias
 * their inputs (in place).  D in {64, 128}; 1 <= H <= 128; d_rope a multiple
 * of 16 in [0, D]; eps >= 0; rope_base > 1.
 * ---------------------------------------------------------------------- */
lcc_status lcc_qkv_prologue(const lcc_bf16* q, const lcc_bf16* k, const lcc_bf16* v,
                            int B, int T, int H, int D,
                            const float* gamma_q, const float* gamma_k, const float* gamma_v,
                            float eps, int d_rope, float rope_base, const int64_t* pos0,
                            lcc_bf16* q_out, lcc_bf16* k_out, lcc_bf16* v_out, void* stream);

/* ---------------------------------------------------------------------- *
 * Decode-step update of one layer's caches ([VIDEO] "쉽게 이해하기": the
 * window keeps the most recent 128 raw tokens, CSA pools every 4 tokens and
 * HCA every 128; [HYBRID]: an entry is the softmax-weighted pool of m
 * consecutive tokens).  For every sequence b, with t = pos[b] the position of
 * the new token and r = t - raw_pos0[b] its raw row:
 *   Kr[b, r, :] = k_new[b, :], Vr[b, r, :] = v_new[b, :], gate_r[b, r] = g_new[b];
 *   if (t + 1) % m == 0 (the token completes block j = (t + 1)/m - 1):
 *     Kc/Vc[b, j, :] = softmax-weighted pool of raw rows r-m+1 .. r, computed
 *       exactly as lcc_csa_compress / lcc_hca_compress compute it;
 *     kI[b, j] = kI_new[b] (and the NVFP4 scales), when kI_new is not NULL;
 *     n_valid[b] = j + 1.
 * Positions, raw offsets and counts live in device memory and every decision
 * is taken on the device, so the call can sit in a captured CUDA graph; the
 * caller advances pos between steps and passes the same pos as q_pos0 to the
 * step's attention calls (the new token is the query).
 * m in {1, 4, 128} (m = 1: every token is its own entry); D in {64, 128}.
 * k_new, v_new: [B, D] bf16; g_new: [B] fp32; pos, raw_pos0: [B] int64.
 * Kr, Vr: [B, Rcap, D] bf16 (batch stride r_bstride elements, rows D apart);
 * gate_r: [B, Rcap] fp32 (batch stride g_bstride); Kc, Vc: [B, Ncap, D] bf16
 * (batch stride c_bstride); n_valid: [B] int32, written.
 * kI_new (optional): [B, DI] bf16 (LCC_KEY_BF16) or [B, DI/2] uint8 with
 * kI_scale_new [B, DI/16] (LCC_KEY_NVFP4): the indexer key of the entry the
 * token completes -- an input, like every indexer key (read only when a
 * block completes); kI / kI_scale: the layer's key store [B, Ncap, ...].
 * A position outside [raw_pos0, raw_pos0 + Rcap), a block whose first token
 * is no longer in the raw buffer, or an entry j >= Ncap skips that sequence
 * and sets the device error word (lcc_sync_status: LCC_ERR_DEVICE).
 * ---------------------------------------------------------------------- */
lcc_status lcc_decode_append(int m, int B, int D,
                             const lcc_bf16* k_new, const lcc_bf16* v_new, const float* g_new,
                             const int64_t* pos,
                             lcc_bf16* Kr, lcc_bf16* Vr, float* gate_r,
                             int64_t r_bstride, int64_t g_bstride, int Rcap,
                             const int64_t* raw_pos0,
                             lcc_bf16* Kc, lcc_bf16* Vc, int64_t c_bstride, int Ncap,
                             int32_t* n_valid,
                             lcc_key_format fmt, int DI, const void* kI_new, const uint8_t* kI_scale_new,
                             void* kI, uint8_t* kI_scale,
                             void* stream);

/* ---------------------------------------------------------------------- *
 * Lightning indexer + top-k.  [HYBRID]: a light indexer running in FP4
 * scores the compressed entries against the query and keeps the top-k
 * (typically about 128) for the expensive attention; [THREAD] "주요 댓글":
 * it picks the likely-relevant candidates before full attention.
 *
 * Score of visible entry j for query (b, i) at position t:
 *   s = sum_h w[b,i,h] * max(0, qI[b,i,h,:] . kI[b,j,:])
 * idx[b,i,:] receives the min(k, visible) entries with the largest s, ties
 * to the lower index, in ascending index order, padded with -1.  score (if
 * not NULL) receives their scores (fp32, -inf for padding).
 *
 * qI:  [B, Tq, HI, DI] bf16; w: [B, Tq, HI] fp32.
 * kI:  LCC_KEY_BF16:  [B, Ncap, DI] bf16, kI_scale unused (NULL);
 *      LCC_KEY_NVFP4: [B, Ncap, DI/2] uint8 e2m1 pairs (element 2c in the
 *      low nibble of byte c) and kI_scale [B, Ncap, DI/16] uint8 e4m3, one
 *      scale per 16 consecutive elements.  ([V41]: keys kept in FP4.)
 * q_pos0, n_valid: device arrays [B] (int64, int32).
 * HI in {4, 8}; DI in {32, 64} (NVFP4: DI = 64); 1 <= k <= 1024; Ncap >= 1.
 * workspace: at least lcc_index_topk_workspace(B, Tq, Ncap, k) bytes.
 * With NVFP4 keys the tensor cores multiply fp16 operands: the keys expand
 * to fp16 exactly (e2m1 x e4m3), and each (query, head) row of qI is scaled
 * by the power of two that puts its largest element just under 2^15, with
 * the head weight scaled by the inverse; every element within a factor 2^31
 * of its row's largest is then exact, so the scores equal those of the bf16
 * queries (a power-of-two scale commutes with the fp32 rounding).
 * ---------------------------------------------------------------------- */
size_t lcc_index_topk_workspace(int B, int Tq, int Ncap, int k);
lcc_status lcc_lightning_index_topk(const lcc_bf16* qI, const float* w,
                                    int B, int Tq, int HI, int DI,
                                    const int64_t* q_pos0,
                                    lcc_key_format fmt, const void* kI, const uint8_t* kI_scale,
                                    const int32_t* n_valid, int Ncap, int m, int k,
                                    int32_t* idx, float* score,
                                    void* workspace, size_t workspace_bytes,
                                    void* stream);

/* Re-index mode of CSA2 index sharing ([V41], the CSA2 passage: a full-mode
 * layer keeps the notes -- the entries that matter -- and a re-index layer
 * uses those notes as they are, adding its own marks for its own task).  For
 * every query (b, i), only the candidate entries cand[b, i, :] (another
 * layer's selection: ascending entry numbers, then -1 padding) are scored,
 *   s = sum_h w[b,i,h] * max(0, qI[b,i,h,:] . kI[b,j,:]),
 * and the k best (ties to the lower index) are written to idx[b, i, :] in
 * ascending index order, padded with -1 when fewer than k candidates exist;
 * score (optional) receives their scores (fp32, -inf for padding).
 * Layouts and key formats as lcc_lightning_index_topk (the keys are the
 * full-mode layer's); 1 <= k <= n_cand <= 1024.  A candidate >= Ncap sets
 * the device error word and is skipped.  No workspace.
 * The reuse mode needs no call: the layer passes the previous layer's idx to
 * its attention (lcc_csa_layer_attn). */
lcc_status lcc_lightning_reindex_topk(const lcc_bf16* qI, const float* w, int B, int Tq, int HI, int DI,
                                      lcc_key_format fmt, const void* kI, const uint8_t* kI_scale, int Ncap,
                                      const int32_t* cand, int n_cand, int k,
                                      int32_t* idx, float* score, void* stream);

/* Indexer scores only: scores[b, i, j] = s for every visible entry j of
 * query (b, i) (entries past the visible count are left untouched).
 * scores: [B, Tq, Ncap] fp32.  Other arguments as lcc_lightning_index_topk. */
lcc_status lcc_lightning_index_scores(const lcc_bf16* qI, const float* w,
                                      int B, int Tq, int HI, int DI,
                                      const int64_t* q_pos0,
                                      lcc_key_format fmt, const void* kI, const uint8_t* kI_scale,
                                      const int32_t* n_valid, int Ncap, int m,
                                      float* scores, void* stream);

/* Allocation-free variant of lcc_lightning_index_topk.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory -- code running while a stream is captured into a CUDA graph
 * (an allocation there is not capturable), plugin-style hosts that hand a
 * routine only its input and output buffers, and decode loops that must not
 * touch an allocator between steps.  Same arguments and results as
 * lcc_lightning_index_topk, minus the workspace: the scratch lives in a
 * fixed 8 MiB array inside the library (8388608 bytes of device memory that
 * every GPU loading the library keeps until the process exits).
 *  - Requests with bf16 keys, Tq*HI > 16 and k <= 256 (prefill shapes) run
 *    the indexer with the top-k fused into its epilogue, which needs no
 *    scratch: they have no size limit and leave the array untouched.
 *  - Other requests are processed in query chunks sized to that array; one
 *    whose single query row needs more than 8 MiB (per batch row: Ncap*4
 *    bytes of scores, ceil(Ncap/16)*4 bytes of group maxima, 8 bytes of
 *    counters and, when Ncap > 16384, ceil(Ncap/16384)*(4 + 8192) bytes of
 *    candidate lists; each array rounded up to 256 bytes) is rejected with
 *    LCC_ERR_WORKSPACE before anything is enqueued.
 *  - The first call on each device looks up the array's device address
 *    (and sets kernel attributes); make that first call before any stream
 *    capture begins.
 *  - All calls share the one array and it keeps the last call's contents;
 *    nothing in it needs to start at zero.  Calls whose kernels overlap on
 *    the GPU (different streams, or different host threads) race on it:
 *    serialise them.
 *  - It never calls cudaMalloc, cudaFree or any allocating routine. */
lcc_status lcc_lightning_index_topk_noalloc(const lcc_bf16* qI, const float* w,
                                            int B, int Tq, int HI, int DI,
                                            const int64_t* q_pos0,
                                            lcc_key_format fmt, const void* kI, const uint8_t* kI_scale,
                                            const int32_t* n_valid, int Ncap, int m, int k,
                                            int32_t* idx, float* score, void* stream);

/* ---------------------------------------------------------------------- *
 * NVFP4 quantisation ([HYBRID]: the lightning indexer computes in FP4; [V41]:
 * the global KV cache is kept in FP4).  Row layout as the NVFP4 indexer keys:
 * e2m1 codes, element 2c in the low nibble of byte c, one e4m3 scale per 16
 * consecutive elements.  Each group of 16 is quantised as
 *   scale  = the e4m3 value nearest to amax/6 (ties to even, saturating at 448);
 *   code_i = the e2m1 value nearest to x_i/scale (ties to even, saturating
 *            at 6) with x_i's sign; magnitude 0 is stored as +0 and a zero
 *            scale stores all-zero codes.
 * The decisions are exact (no rounding step can move a value across a
 * boundary), so the codes are unique for every finite bf16 input; inputs must
 * be finite.
 *
 * lcc_nvfp4_quantize: x [rows, D] bf16 with rows ld elements apart (ld >= D,
 * ld*2 a multiple of 16 bytes, x 16-byte aligned); D a positive multiple of
 * 16.  Outputs, each optional (NULL skips it): packed [rows, D/2] uint8
 * (8-byte aligned), scale [rows, D/16] uint8, xq [rows, D] bf16 = the
 * dequantised values (16-byte aligned; exact: every e2m1 x e4m3 product is a
 * bf16 value).  The caller owns every buffer; nothing is allocated.
 * lcc_nvfp4_dequantize: packed/scale as above, contiguous rows -> x [rows, D]
 * bf16 (exact).
 * ---------------------------------------------------------------------- */
lcc_status lcc_nvfp4_quantize(const lcc_bf16* x, int64_t rows, int D, int64_t ld,
                              uint8_t* packed, uint8_t* scale, lcc_bf16* xq, void* stream);
lcc_status lcc_nvfp4_dequantize(const uint8_t* packed, const uint8_t* scale, int64_t rows, int D,
                                lcc_bf16* x, void* stream);

/* The lightning indexer in FP4 ([HYBRID], section "두 가지 압축 전략: CSA 및
 * HCA": the indexer computes in FP4).  As lcc_lightning_index_topk with NVFP4
 * keys, but the indexer query is first quantised to NVFP4 by
 * lcc_nvfp4_quantize's rule (per (query, head) row, groups of 16): the score
 * of entry j is
 *   s = sum_h w[b,i,h] * max(0, Q(qI[b,i,h,:]) . kI[b,j,:])
 * with Q the quantise-dequantise map and both vectors in their exact NVFP4
 * values; the head weights stay fp32.  Products of two NVFP4 values are exact
 * in fp32, so the result equals the block-scaled FP4 contraction up to the
 * order of the fp32 sums.
 * kI [B, Ncap, DI/2] uint8 (8-byte aligned), kI_scale [B, Ncap, DI/16];
 * HI = 8, DI = 64; other arguments as lcc_lightning_index_topk.
 * workspace: at least lcc_fp4_index_topk_workspace(B, Tq, HI, DI, Ncap, k)
 * bytes, 16-byte aligned.  Prefill shapes (Tq*HI > 16, k <= 256) expand the
 * keys to bf16 in the workspace once per call (36 bytes read and 128 written
 * per entry) and run the tensor-core indexer with the top-k fused into its
 * epilogue; other shapes run the NVFP4-key indexer on the quantised query. */
size_t lcc_fp4_index_topk_workspace(int B, int Tq, int HI, int DI, int Ncap, int k);
lcc_status lcc_fp4_index_topk(const lcc_bf16* qI, const float* w, int B, int Tq, int HI, int DI,
                              const int64_t* q_pos0, const uint8_t* kI, const uint8_t* kI_scale,
                              const int32_t* n_valid, int Ncap, int m, int k,
                              int32_t* idx, float* score,
                              void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------- *
 * CSA sparse attention: MQA (all H heads share one K/V row, [HYBRID]) over
 * the k entries idx[b,i,:] of the compressed cache; entries < 0 are skipped.
 *   z_h,j = scale * q[b,i,h,:] . Kc[b,idx_j,:];  lse = log sum_j e^z;
 *   O[b,i,h,:] = sum_j softmax(z)_j Vc[b,idx_j,:]
 * q: [B, Tq, H, D] bf16; Kc, Vc: [B, Ncap, D] bf16 with rows kv_rstride
 * elements apart (D for separate tensors, 2*D when K and V rows interleave);
 * idx: [B, Tq, k] int32, each entry in [-1, Ncap).  H in {8, 16, ..., 128},
 * D in {64, 128}, 1 <= k <= 4096.
 * ---------------------------------------------------------------------- */
lcc_status lcc_csa_sparse_attn(const lcc_bf16* q, int B, int Tq, int H, int D, float scale,
                               const lcc_bf16* Kc, const lcc_bf16* Vc, int64_t kv_rstride, int Ncap,
                               const int32_t* idx, int k,
                               float* O, float* lse, void* stream);

/* ---------------------------------------------------------------------- *
 * HCA dense attention over every visible compressed entry ([HYBRID]: dense
 * attention over the ~8000 entries a 1M-token context leaves at m=128).
 * Keys of query (b, i): entries j < min(n_valid[b], (q_pos0[b]+i+1)/m).
 * Layouts as lcc_csa_sparse_attn.  Decode-sized calls split the key range
 * across CTAs and need lcc_dense_attn_workspace(...) bytes of workspace.
 * ---------------------------------------------------------------------- */
size_t lcc_dense_attn_workspace(int B, int Tq, int H, int D, int Ncap);
lcc_status lcc_hca_dense_attn(const lcc_bf16* q, int B, int Tq, int H, int D, float scale,
                              const int64_t* q_pos0,
                              const lcc_bf16* Kc, const lcc_bf16* Vc, int64_t kv_rstride, int Ncap,
                              const int32_t* n_valid, int m,
                              float* O, float* lse,
                              void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------- *
 * Sliding-window attention over raw tokens ([HYBRID]: a window branch runs
 * in parallel to keep local detail; [VIDEO]: the most recent 128 tokens).
 * Keys of the query at position t: positions max(0, t-W+1) .. t that the raw
 * buffer holds, i.e. rows r = p - raw_pos0[b] with 0 <= r < Rcap.
 * Kr, Vr: [B, Rcap, D] bf16 (rows kv_rstride apart).  1 <= W <= 4096.
 * ---------------------------------------------------------------------- */
lcc_status lcc_swa_attn(const lcc_bf16* q, int B, int Tq, int H, int D, float scale,
                        const int64_t* q_pos0,
                        const lcc_bf16* Kr, const lcc_bf16* Vr, int64_t kv_rstride, int Rcap,
                        const int64_t* raw_pos0, int W,
                        float* O, float* lse, void* stream);

/* ---------------------------------------------------------------------- *
 * Whole layers in one pass ([HYBRID]: the window branch runs in parallel
 * with the compressed one; [VIDEO] "주요 인사이트": CSA and HCA layers
 * alternate).  The result is the softmax attention over the union of the
 * compressed keys and the window keys, which equals the log-sum-exp merge
 * (lcc_attn_merge) of the two branches:
 *   lcc_csa_layer_attn  keys = entries idx[b,i,:] of Kc/Vc  ++ window rows
 *   lcc_hca_layer_attn  keys = visible entries of Kc/Vc     ++ window rows
 * out: [B, Tq, H, D] bf16 (round to nearest even); lse_out (optional, may be
 * NULL): [B, Tq, H] fp32 natural-log normaliser of the union.
 * Compressed and window arguments as in lcc_csa_sparse_attn /
 * lcc_hca_dense_attn and lcc_swa_attn (Kr/Vr rows r_rstride elements apart,
 * Rcap rows per batch).  Calls with few rows split the key list across CTAs
 * and need lcc_layer_attn_workspace(B, Tq, H, D, n_keys) bytes of workspace,
 * n_keys = k + W (CSA layer) or Ncap + W (HCA layer); 0 means none.
 * ---------------------------------------------------------------------- */
size_t lcc_layer_attn_workspace(int B, int Tq, int H, int D, int n_keys);
lcc_status lcc_csa_layer_attn(const lcc_bf16* q, int B, int Tq, int H, int D, float scale,
                              const int64_t* q_pos0,
                              const lcc_bf16* Kc, const lcc_bf16* Vc, int64_t kv_rstride, int Ncap,
                              const int32_t* idx, int k,
                              const lcc_bf16* Kr, const lcc_bf16* Vr, int64_t r_rstride, int Rcap,
                              const int64_t* raw_pos0, int W,
                              lcc_bf16* out, float* lse_out,
                              void* workspace, size_t workspace_bytes, void* stream);
lcc_status lcc_hca_layer_attn(const lcc_bf16* q, int B, int Tq, int H, int D, float scale,
                              const int64_t* q_pos0,
                              const lcc_bf16* Kc, const lcc_bf16* Vc, int64_t kv_rstride, int Ncap,
                              const int32_t* n_valid, int m,
                              const lcc_bf16* Kr, const lcc_bf16* Vr, int64_t r_rstride, int Rcap,
                              const int64_t* raw_pos0, int W,
                              lcc_bf16* out, float* lse_out,
                              void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------- *
 * A whole CSA layer in one call: lcc_lightning_index_topk (writes idx) then
 * lcc_csa_layer_attn on the selected entries and the window.  The library
 * knows the order of its kernels here, so the attention is launched as a
 * programmatic dependent of the top-k: it may start while the top-k runs,
 * reads the queries and window rows early and waits for the index lists.
 * Decode-shaped calls (H a multiple of 16 up to 128, D = 128, Ncap <=
 * (H/16) * 4096, k <= 128, a few query rows) go further: after the indexer,
 * one thread-block cluster per query (one CTA per 16 heads) selects the
 * top-k and attends, the index list passed between its CTAs on chip; the
 * index lists are identical to the two calls', the outputs equal up to
 * rounding (the attention walks the keys in 16-key tiles).
 * Arguments as the two calls; idx [B, Tq, k] int32 is written; workspace:
 * at least lcc_csa_layer_workspace(B, Tq, H, D, Ncap, k, W) bytes.
 * ---------------------------------------------------------------------- */
size_t lcc_csa_layer_workspace(int B, int Tq, int H, int D, int Ncap, int k, int W);
lcc_status lcc_csa_layer(const lcc_bf16* q, const lcc_bf16* qI, const float* w,
                         int B, int Tq, int H, int D, int HI, int DI, float scale,
                         const int64_t* q_pos0,
                         lcc_key_format fmt, const void* kI, const uint8_t* kI_scale,
                         const int32_t* n_valid,
                         const lcc_bf16* Kc, const lcc_bf16* Vc, int64_t kv_rstride, int Ncap, int m, int k,
                         const lcc_bf16* Kr, const lcc_bf16* Vr, int64_t r_rstride, int Rcap,
                         const int64_t* raw_pos0, int W,
                         int32_t* idx, lcc_bf16* out, float* lse_out,
                         void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------- *
 * Branch merge by log-sum-exp: with L = log sum_b exp(lse_b),
 *   out = sum_b exp(lse_b - L) * O_b  (bf16, round to nearest even),
 *   lse_out = L (optional).
 * Equal to one softmax over the union of the branches' key lists.
 * O_parts / lse_parts: HOST arrays of nb device pointers, each [rows, D] /
 * [rows] fp32, rows = B*Tq*H.  2 <= nb <= 4.  out_f32 (optional, may be
 * NULL) receives the fp32 result as well.
 * ---------------------------------------------------------------------- */
lcc_status lcc_attn_merge(int nb, const float* const* O_parts, const float* const* lse_parts,
                          int64_t rows, int D,
                          lcc_bf16* out, float* out_f32, float* lse_out, void* stream);

/* ---------------------------------------------------------------------- *
 * Utilities.
 * ---------------------------------------------------------------------- */
const char* lcc_last_error(void);          /* thread-local text of the last failure */
const char* lcc_version(void);
/* Number of kernels this library has enqueued since it was loaded (all
 * devices and streams; a launch captured into a CUDA graph counts once). */
uint64_t lcc_launch_count(void);
/* Synchronise `stream`, then report (and clear) the device error word. */
lcc_status lcc_sync_status(void* stream);

/* TEST HOOK (not part of the computation; no page describes it).  Every
 * device-side wait of the tensor-core kernels is bounded; this lets a test
 * make one run out without faulting or hanging anything.
 *  wait_limit_ns: limit of every bounded wait on the current device; 0
 *      restores the default of 2 s; values are clamped to [1 ms, 2 s], so a
 *      kernel winding down still waits long enough for its own copies and
 *      MMAs in flight.
 *  drop_tile: >= 0 makes the decode indexer (lcc_lightning_index_scores and
 *      the score pass of lcc_lightning_index_topk) skip loading the key tile
 *      with that CTA-local number, so the waits for it run out: the call
 *      then leaves its scores unspecified and lcc_sync_status() returns
 *      LCC_ERR_TIMEOUT.  -1 restores normal operation.
 * Synchronises the device first; call it only between steps, never while
 * another thread is launching work.  Returns LCC_ERR_CUDA if the device
 * cannot be reached. */
lcc_status lcc_test_set_wait_fault(uint64_t wait_limit_ns, int drop_tile);

#ifdef __cplusplus
}
#endif
#endif /* LCC_H_ */
