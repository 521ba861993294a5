// The per-16-element block step of the NVFP4 quantiser, shared by the
// quantiser kernel and the GEMM epilogues that emit NVFP4 directly, so that
// every producer of NVFP4 takes the same decisions bit for bit:
//   sb    = amax_block / (s_t * 6) -> E4M3, nearest even, saturating at 448
//   q     = x / (e4m3(sb) * s_t)   -> e2m1, nearest even, saturating at 6
// in fp32 with IEEE division and multiplication (no contraction into FMA),
// the sign of x kept on a code whose magnitude rounds to zero, a zero block
// scale forcing zero codes. Format: 4-bit e2m1 values with one 8-bit float
// scale per 16 elements (Serving Qwen3.8-27B in 4-bit with a masked
// speculative decoding head, "What the artifact is").
#pragma once

#include "common.cuh"

namespace nvfp4 {

// Packed fp32 pair multiply (both halves rounded to nearest even).
NVFP4_DEV uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
NVFP4_DEV uint64_t f32_pair(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
// Four fp32 pairs (elements 2j, 2j + 1) -> eight e2m1 codes, element j in
// nibble j (nearest even, saturating at 6, sign kept on a zero magnitude).
NVFP4_DEV uint32_t e2m1x8_of_pairs(uint64_t p0, uint64_t p1, uint64_t p2, uint64_t p3) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .f32 a0, a1, a2, a3, a4, a5, a6, a7;\n\t"
      "mov.b64 {a0, a1}, %1;\n\tmov.b64 {a2, a3}, %2;\n\tmov.b64 {a4, a5}, %3;\n\tmov.b64 {a6, a7}, %4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, a1, a0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, a3, a2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, a5, a4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, a7, a6;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "l"(p0), "l"(p1), "l"(p2), "l"(p3));
  return out;
}

// The sixteen codes of one block (two words, element j of each half in nibble
// j). A code is RNE_e2m1(fl(x / den)) with the sign of x kept on a zero
// magnitude, and depends only on which side of the e2m1 rounding midpoints
// the quotient lies. With r = RN(1/den), rh = RN(r (1 + 2^-20)) > 1/den and
// rl = RN(r (1 - 2^-20)) < 1/den, so RN(|x| rl) <= fl(|x| / den) <= RN(|x| rh)
// (rounding is monotone), and the code magnitude is monotone in the value:
// where the products with rl and rh give the same codes, those are the codes
// of the exact quotients. Otherwise (a quotient at or next to a midpoint) the
// sixteen quotients are formed by IEEE division.
// rh, rl are the two brackets of 1 / den (rh = rl = 0: none, divide).
NVFP4_DEV uint2 e2m1x16_r(const float (&v)[16], float den, float rh, float rl) {
  if (rh != 0.f) {
    const uint64_t RH = f32_pair(rh, rh), RL = f32_pair(rl, rl);
    uint64_t ph[8], pl[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint64_t xv = f32_pair(v[2 * e], v[2 * e + 1]);
      ph[e] = mul_f32x2(xv, RH);
      pl[e] = mul_f32x2(xv, RL);
    }
    const uint32_t h0 = e2m1x8_of_pairs(ph[0], ph[1], ph[2], ph[3]), h1 = e2m1x8_of_pairs(ph[4], ph[5], ph[6], ph[7]);
    const uint32_t l0 = e2m1x8_of_pairs(pl[0], pl[1], pl[2], pl[3]), l1 = e2m1x8_of_pairs(pl[4], pl[5], pl[6], pl[7]);
    if (h0 == l0 && h1 == l1) return make_uint2(h0, h1);
  }
  uint2 out;
  float q[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) q[j] = __fdiv_rn(v[j], den);
  out.x = f32x8_to_e2m1x8(q);
#pragma unroll
  for (int j = 0; j < 8; ++j) q[j] = __fdiv_rn(v[8 + j], den);
  out.y = f32x8_to_e2m1x8(q);
  return out;
}

// The brackets of 1 / den used by e2m1x16_r: rh > 1 / den > rl (exactly),
// or zeros when den is too small or too large for them.
NVFP4_DEV void recip_brackets(float den, float& rh, float& rl) {
  if (den > 1e-30f && den < 1e30f) {
    const float r = __frcp_rn(den);
    rh = __fmul_rn(r, 1.0f + 0x1p-20f);
    rl = __fmul_rn(r, 1.0f - 0x1p-20f);
  } else {
    rh = rl = 0.f;
  }
}

NVFP4_DEV uint2 e2m1x16(const float (&v)[16], float den) {
  float rh, rl;
  recip_brackets(den, rh, rl);
  return e2m1x16_r(v, den, rh, rl);
}

// E4M3 code of fl(ab / d) (ab >= 0): RN(ab rdl) <= fl(ab / d) <= RN(ab rdh)
// for brackets rdl < 1 / d < rdh (recip_brackets), and the E4M3 rounding is
// monotone, so equal codes of the two products are the code of the quotient;
// otherwise (or without brackets) IEEE division.
NVFP4_DEV uint32_t block_scale_code(float ab, float d, float rdh, float rdl) {
  if (rdh != 0.f) {
    const uint32_t h = f32_to_e4m3(__fmul_rn(ab, rdh)), l = f32_to_e4m3(__fmul_rn(ab, rdl));
    if (h == l) return h;
  }
  return f32_to_e4m3(__fdiv_rn(ab, d));
}

// Per tensor scale, the block step's constants for every E4M3 block-scale
// code c (0x00 .. 0x7F; 0x7F is never produced): den[c] = fl(e4m3(c) * s_t)
// and the brackets of 1 / den[c]. Built once per CTA in shared memory, they
// replace a decode, a multiply and a reciprocal per block.
struct QuantTables {
  float den[128];
  float rh[128];
  float rl[128];
};

NVFP4_DEV void quant_tables_init(QuantTables& tb, float st) {
  for (int c = threadIdx.x; c < 128; c += blockDim.x) {
    const float den = __fmul_rn(e4m3_to_f32(static_cast<uint32_t>(c)), st);
    tb.den[c] = den;
    recip_brackets(den, tb.rh[c], tb.rl[c]);
  }
}

// quant_block16 with the block's largest magnitude already known (ab) and the
// scale-code brackets and tables of the tensor scale: the same decisions.
NVFP4_DEV uint32_t quant_block16_tab(const float (&v)[16], float ab, float d, float rdh, float rdl,
                                     const QuantTables& tb, uint2& codes) {
  const uint32_t sc = block_scale_code(ab, d, rdh, rdl);
  codes = sc != 0 ? e2m1x16_r(v, tb.den[sc], tb.rh[sc], tb.rl[sc]) : make_uint2(0u, 0u);
  return sc;
}

// One block: x[16] (fp32) with tensor scale st and d = fp32(st * 6). Returns
// the E4M3 block scale; `codes` gets the sixteen e2m1 codes (element j of each
// half in nibble j of .x / .y).
NVFP4_DEV uint32_t quant_block16(const float (&v)[16], float st, float d, uint2& codes) {
  float ab = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) ab = fmaxf(ab, fabsf(v[e]));
  const uint32_t sc = f32_to_e4m3(__fdiv_rn(ab, d));
  codes = sc != 0 ? e2m1x16(v, __fmul_rn(e4m3_to_f32(sc), st)) : make_uint2(0u, 0u);
  return sc;
}

}  // namespace nvfp4
