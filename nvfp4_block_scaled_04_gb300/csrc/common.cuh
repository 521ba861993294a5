// Device helpers shared by the NVFP4 kernels (sm_103a).
//
// Conversions use the Blackwell cvt instructions for the narrow formats
// (e2m1x2 <-> f16x2 / f32, e4m3x2 <-> f16x2 / f32); the GPU tests check them
// against the CPU oracle on tie, saturation and signed-zero vectors.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nvfp4.h"

#define NVFP4_DEV __device__ __forceinline__

namespace nvfp4 {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Padded geometry of the MMA scale layout: rows to 128, scale columns to 4.
inline int64_t mma_scale_rows(int64_t rows) { return ceil_div(rows, 128) * 128; }
inline int64_t mma_scale_cols(int64_t K) { return ceil_div(K / 16, 4) * 4; }

// GPU-scope acquire-release fence for the last-arrival reductions: a
// thread's global writes before it are visible to any thread that observes
// (through the arrival counter) a write of this CTA after it, and reads
// after it see every write published that way before the counter value
// this CTA observed.
NVFP4_DEV void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// ------------------------------------------------------------ conversions

// Eight packed e2m1 codes -> four f16x2 words (byte b -> out[b]); the low
// nibble of each byte lands in the low half.
NVFP4_DEV void e2m1x8_to_f16x2(uint32_t v, uint32_t (&out)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(v));
}

// Two E4M3 codes (low byte first) -> f16x2 (exact: every E4M3 value is a
// normal f16).
NVFP4_DEV uint32_t e4m3x2_to_f16x2(uint32_t v16) {
  uint32_t out;
  asm("{\n\t.reg .b16 s;\n\t"
      "cvt.u16.u32 s, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, s;\n\t}"
      : "=r"(out)
      : "r"(v16));
  return out;
}

// fp32 >= 0 -> E4M3 code, round to nearest even, saturating to 448.
NVFP4_DEV uint32_t f32_to_e4m3(float v) {
  uint32_t out;
  asm("{\n\t.reg .b16 s;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 s, %2, %1;\n\t"
      "cvt.u32.u16 %0, s;\n\t}"
      : "=r"(out)
      : "f"(v), "f"(0.0f));
  return out & 0xFFu;
}

// E4M3 code (0..0x7E) -> fp32 value, from the bit fields (exact).
NVFP4_DEV float e4m3_to_f32(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
  if (e == 0) return __int2float_rn(static_cast<int>(m)) * 0.001953125f;  // m/8 * 2^-6
  return __uint_as_float(((e + 120u) << 23) | (m << 20));                 // (1+m/8) 2^(e-7)
}

// Eight fp32 -> eight e2m1 codes, element j in nibble j (round to nearest
// even, saturating at 6; a negative value that rounds to zero keeps its sign).
NVFP4_DEV uint32_t f32x8_to_e2m1x8(const float (&v)[8]) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return out;
}

// Two non-negative fp32 -> packed e2m1 magnitudes (a in the low nibble,
// b in the high nibble), nearest-even, saturating to 6.
NVFP4_DEV uint32_t f32x2_to_e2m1x2(float a, float b) {
  uint32_t out;
  asm("{\n\t.reg .b8 s;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 s, %2, %1;\n\t"
      "cvt.u32.u8 %0, s;\n\t}"
      : "=r"(out)
      : "f"(a), "f"(b));
  return out & 0xFFu;
}

NVFP4_DEV uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// f16x2 with both halves equal to the low / high half of v.
NVFP4_DEV uint32_t dup_lo(uint32_t v) { return __byte_perm(v, 0, 0x1010); }
NVFP4_DEV uint32_t dup_hi(uint32_t v) { return __byte_perm(v, 0, 0x3232); }

NVFP4_DEV float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// fp32 -> bf16 bits, round to nearest even (finite inputs).
NVFP4_DEV uint32_t f32_to_bf16_bits(float f) {
  uint32_t r;
  asm("{\n\t.reg .b16 h;\n\tcvt.rn.bf16.f32 h, %1;\n\tcvt.u32.u16 %0, h;\n\t}" : "=r"(r) : "f"(f));
  return r;
}

NVFP4_DEV uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

NVFP4_DEV uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

// Orderable key of a float: larger float -> larger unsigned.
NVFP4_DEV uint32_t float_order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
NVFP4_DEV float float_from_order_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// --------------------------------------------------------------- memory

// Streaming 16-byte load that bypasses L1 allocation (weights are read once).
NVFP4_DEV uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
NVFP4_DEV uint32_t ld_stream_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

NVFP4_DEV uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- tensor core

// D += A * B for one m16n8k16 tile, f16 inputs, fp32 accumulators.
NVFP4_DEV void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// --------------------------------------------------------------- clusters

NVFP4_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

NVFP4_DEV void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Load a float from the shared memory of CTA `rank` of this cluster, at the
// same offset as the local shared address `saddr`.
NVFP4_DEV float ld_dsmem_f32(uint32_t saddr, uint32_t rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(saddr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

}  // namespace nvfp4
