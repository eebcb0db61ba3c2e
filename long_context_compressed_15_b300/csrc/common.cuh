// Shared device helpers for liblcc: bf16/fp16 packing, legacy-MMA and
// ldmatrix wrappers, cp.async, and the device error word.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lcc {

typedef __nv_bfloat16 bf16;

// Device error word: the first error a kernel records wins.  Layout:
// bits 31..24 = code, bits 23..0 = detail (a kernel id or an index).
__device__ unsigned int g_dev_error = 0;

enum DevErr : unsigned int {
  DEV_ERR_INDEX = 1,    // an index list entry was outside [-1, Ncap)
  DEV_ERR_TIMEOUT = 2,  // a bounded wait gave up
  DEV_ERR_RANGE = 3,    // a decode append fell outside its raw buffer or caches (detail: sequence)
  DEV_ERR_POS = 4,      // a pooling position was negative or not a multiple of m (detail: sequence)
};

__device__ __forceinline__ void record_error(unsigned int code, unsigned int detail) {
  atomicCAS(&g_dev_error, 0u, (code << 24) | (detail & 0xFFFFFFu));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The first 1024-byte boundary at or after `raw` (the start of a dynamic
// shared-memory array).  Offsetting the pointer itself, rather than rounding
// its integer value, keeps it visibly a shared-memory pointer, so accesses
// through it compile to shared-memory instructions instead of generic ones.
__device__ __forceinline__ uint8_t* align_smem_1024(uint8_t* raw) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(raw));
  return raw + ((1024u - (a & 1023u)) & 1023u);
}

// ---- cp.async (16-byte, zero-fill when src_bytes == 0) ----
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// ---- ldmatrix ----
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// ---- warp-level MMA m16n8k16, fp32 accumulate ----
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x by the SFU's approximate base-2 exponential (PTX ex2.approx.ftz.f32):
// relative error about 2^-22, -inf -> +0, results below 2^-126 flushed to 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two e2m1 values (one byte, element 2c in the low nibble) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low8) {
  uint32_t out;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " mov.b32 {b0, b1, b2, b3}, %1;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n}\n"
      : "=r"(out) : "r"(byte_in_low8));
  return out;
}
// The four e2m1 pairs of a 32-bit word -> four f16x2 (exact), byte j -> h[j]
// (low nibble -> low half), without shifting the word.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t word, uint32_t (&h)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      " cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      " cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(word));
}
// Four e4m3 bytes -> four f16x2, each with both halves equal to one byte's
// value (exact): two paired conversions, then each half duplicated.
__device__ __forceinline__ void e4m3x4_to_f16x2_bcast(uint32_t four, uint32_t (&s)[4]) {
  uint32_t lo, hi;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(lo) : "h"(static_cast<uint16_t>(four & 0xFFFFu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(hi) : "h"(static_cast<uint16_t>(four >> 16)));
  s[0] = __byte_perm(lo, 0u, 0x1010);
  s[1] = __byte_perm(lo, 0u, 0x3232);
  s[2] = __byte_perm(hi, 0u, 0x1010);
  s[3] = __byte_perm(hi, 0u, 0x3232);
}
// One e4m3 byte -> f16x2 with both halves equal to its value (exact).
__device__ __forceinline__ uint32_t e4m3_to_f16x2_bcast(uint32_t byte) {
  uint32_t out;
  uint16_t two = static_cast<uint16_t>((byte & 0xFF) | ((byte & 0xFF) << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(out) : "h"(two));
  return out;
}
// Two fp32 values in one 64-bit register pair (low half first) and the
// packed fma on such pairs: each half is an IEEE fma rounded to nearest.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t x, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Order-preserving map of fp32 to uint32 (larger float -> larger key);
// -0 is folded onto +0 so that equal scores compare equal.  Key 0 never
// arises from a non-NaN float and marks "no element".
__device__ __forceinline__ uint32_t f32_to_key(float f) {
  if (f == 0.0f) f = 0.0f;
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_f32(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the previous kernel on its stream is still
// running; pdl_wait() blocks until that kernel has completed and its memory
// writes are visible (it returns at once for a normally launched kernel).
// pdl_trigger() lets the next kernel on the stream start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Thread-block cluster helpers: rank and size, the cluster barrier (split
// arrive / wait), and loads, stores and atomics on another CTA's shared
// memory through its cluster address.
namespace clu {
__device__ __forceinline__ uint32_t rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ void sync() {
  arrive();
  wait();
}
// Address of the shared variable `p` of CTA `r` of this cluster.
__device__ __forceinline__ uint32_t map(const void* p, uint32_t r) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(r));
  return d;
}
__device__ __forceinline__ void st(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t atom_add(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}
}  // namespace clu

// Visible compressed entries for the query at absolute position t.
__device__ __forceinline__ int visible_entries(int64_t t, int m, int n_valid, int Ncap) {
  int64_t v = (t + 1) / m;
  if (v > n_valid) v = n_valid;
  if (v > Ncap) v = Ncap;
  return v < 0 ? 0 : static_cast<int>(v);
}

}  // namespace lcc
