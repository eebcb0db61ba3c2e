// NVFP4 for the indexer: quantisation of the indexer query and expansion of
// NVFP4 rows to bf16.  Source: "DeepSeek-V4가 이차적 어텐션 비용 없이 ...",
// section "두 가지 압축 전략: CSA 및 HCA" (the lightning indexer computes in FP4),
// and the DeepSeek V4.1 Flash post (the global KV cache kept in FP4).
//
// NVFP4 row layout: e2m1 codes, element 2i in the low nibble of byte i, and
// one e4m3 scale per 16 consecutive elements.  Quantisation of a group of 16:
//   scale  = the e4m3 value nearest to amax / 6 (ties to even, saturating at 448);
//   code_i = the e2m1 value nearest to x_i / scale (ties to even, saturating
//            at 6), with the sign of x_i; magnitude 0 is stored as +0, and a
//            zero scale stores all-zero codes.
// The element decisions are taken without rounding: x_i is compared with the
// midpoints mu * scale of the e2m1 grid, and each mu * scale (mu has at most
// three significant bits, scale four) is exact in fp32.  amax / 6 is rounded
// once in fp32 before its conversion to e4m3; for bf16 inputs it is never
// within 2^-9 (relative) of an e4m3 rounding boundary unless it lies on one,
// so the conversion picks the same value as an exact quotient would.
// Every e2m1 x e4m3 product has at most six significant bits and lies in
// [2^-10, 2688]: the expansion to bf16 (or fp16) is exact.
//
// Both kernels are HBM-bound elementwise passes, one thread per group of 16:
// quantisation reads 32 bytes and writes 8 + 1 (+ 32 dequantised) bytes;
// expansion reads 8 + 1 bytes and writes 32.
#pragma once
#include "common.cuh"

namespace lcc {

struct Nvfp4QuantArgs {
  const bf16* x;      // [rows, D], row stride ld elements
  int64_t rows;
  int gpr;            // groups of 16 per row (D / 16)
  int64_t ld;
  uint8_t* packed;    // [rows, D/2] or null
  uint8_t* scale;     // [rows, D/16] or null
  bf16* xq;           // [rows, D] dequantised values, or null
};

// e4m3 byte -> float (exact).
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  const uint32_t h2 = e4m3_to_f16x2_bcast(byte);
  return __low2float(*reinterpret_cast<const __half2*>(&h2));
}

// Positive float -> e4m3 byte, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t float_to_e4m3_satfinite(float v) {
  uint16_t pair;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;\n" : "=h"(pair) : "f"(v));
  return pair & 0xFFu;
}

// 8 e2m1 codes (a 32-bit word, element 2j in the low nibble of byte j) times
// the group scale -> 8 bf16 as four bf16x2 words (exact).
__device__ __forceinline__ void e2m1x8_scaled_to_bf16(uint32_t word, uint32_t s2, uint32_t (&o)[4]) {
  uint32_t h[4];
  e2m1x8_to_f16x2x4(word, h);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t p = hmul2_u32(h[j], s2);   // exact in fp16
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&p));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    o[j] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

__global__ void __launch_bounds__(256) k_nvfp4_quant(Nvfp4QuantArgs a) {
  const int64_t gi = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (gi >= a.rows * a.gpr) return;
  const int64_t r = gi / a.gpr;
  const int g = static_cast<int>(gi - r * a.gpr);
  const uint4* src = reinterpret_cast<const uint4*>(a.x + r * a.ld + g * 16);
  const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
  const uint32_t wd[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float f[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[j]));
    f[2 * j] = p.x;
    f[2 * j + 1] = p.y;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
  const uint32_t sb = float_to_e4m3_satfinite(amax / 6.0f);
  const float s = e4m3_to_float(sb);
  // midpoints of the e2m1 grid {0, .5, 1, 1.5, 2, 3, 4, 6}, scaled; at a
  // midpoint the even code wins, hence > below even codes and >= below odd ones
  const float t0 = 0.25f * s, t1 = 0.75f * s, t2 = 1.25f * s, t3 = 1.75f * s, t4 = 2.5f * s, t5 = 3.5f * s,
              t6 = 5.0f * s;
  uint32_t code[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float x = fabsf(f[i]);
    uint32_t mag = (x > t0) + (x >= t1) + (x > t2) + (x >= t3) + (x > t4) + (x >= t5) + (x > t6);
    if (sb == 0u) mag = 0u;
    const uint32_t c = mag | ((f[i] < 0.f && mag != 0u) ? 8u : 0u);
    code[i >> 3] |= c << (4 * (i & 7));
  }
  if (a.packed)
    *reinterpret_cast<uint2*>(a.packed + r * (a.gpr * 8) + g * 8) = make_uint2(code[0], code[1]);
  if (a.scale) a.scale[r * a.gpr + g] = static_cast<uint8_t>(sb);
  if (a.xq) {
    const uint32_t s2 = e4m3_to_f16x2_bcast(sb);
    uint32_t lo[4], hi[4];
    e2m1x8_scaled_to_bf16(code[0], s2, lo);
    e2m1x8_scaled_to_bf16(code[1], s2, hi);
    uint4* dst = reinterpret_cast<uint4*>(a.xq + r * (static_cast<int64_t>(a.gpr) * 16) + g * 16);
    dst[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    dst[1] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  }
}

struct Nvfp4ExpandArgs {
  const uint8_t* packed;   // [rows, D/2]
  const uint8_t* scale;    // [rows, D/16]
  int64_t rows;
  int gpr;
  bf16* out;               // [rows, D]
};

// Expansion of NVFP4 rows to bf16.  With pdl the launch may overlap the
// previous kernel; the rows are read only after its results are visible.
__global__ void __launch_bounds__(256) k_nvfp4_expand(Nvfp4ExpandArgs a) {
  pdl_wait();
  pdl_trigger();
  const int64_t gi = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (gi >= a.rows * a.gpr) return;
  const uint2 p = __ldg(reinterpret_cast<const uint2*>(a.packed) + gi);
  const uint32_t s2 = e4m3_to_f16x2_bcast(__ldg(a.scale + gi));
  uint32_t lo[4], hi[4];
  e2m1x8_scaled_to_bf16(p.x, s2, lo);
  e2m1x8_scaled_to_bf16(p.y, s2, hi);
  uint4* dst = reinterpret_cast<uint4*>(a.out + gi * 16);
  dst[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  dst[1] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
}

}  // namespace lcc
