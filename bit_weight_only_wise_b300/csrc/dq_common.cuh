// Device helpers shared by the W4A16 / NF4 kernels: inline-PTX wrappers and
// the exact 4-bit -> fp16 / bf16 dequantization of packed words.
//
// Dequantization contract (cloud.tencent.com/developer/article/2726413 §2.1:
// asymmetric quantization with a stored zero point):
//     w_hat = RNE_dtype((q - z) * s),   q, z in 0..15, s an fp16 scale.
// (q - z) * s is exact in fp32 (4-bit integer times an 11-bit significand), so
// the value is one rounding of the exact product.  The routines below reach
// that value with packed 16-bit arithmetic on pairs of codes:
//
//   fp16: a code is placed in the mantissa of a "magic" fp16 whose ulp is 1
//         (1024 + q: magic 0x6400 with the code in bits 0..3, or 64 + q:
//         magic 0x5400 with the code in bits 4..7).  Subtracting the same
//         magic plus z is exact and gives (q - z); one fp16 multiply by s is
//         the single IEEE rounding of the exact product.
//   bf16: the code goes into bits 0..3 of 0x4300 (128 + q); subtracting
//         128 + z gives (q - z) exactly.  s is split as s = s_hi + s_lo with
//         s_hi the first 8 significant bits of s (exact in bf16) and s_lo the
//         remaining <= 3 bits (also exact); t = (q - z) * s_lo is exact (<= 7
//         bits) and fma(q - z, s_hi, t) rounds the exact (q - z) * s once.
//   bf16 through fp32 (the decode kernel): the fp16 magic codes go through
//         one mixed-precision FMA each, which gives (q - z) * s exactly in
//         fp32, and one pair conversion rounds it (see below).
//
// A packed word holds the codes of 8 consecutive K rows of one column; pair j
// (j = 0..3) of a word holds rows (j, j + 4) in its (low, high) halves.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace w4a16 {

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t d;
  // (a & mask) | magic
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(magic));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t hsub2_f16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hsub2_bf16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hmul2_bf16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hfma2_bf16(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Two fp32 values -> packed 16-bit pair (lo in bits 0..15), one RNE each.
__device__ __forceinline__ uint32_t pack2_rn(float lo, float hi, bool bf16) {
  uint32_t d;
  if (bf16)
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float lo16_to_f32(uint32_t v, bool bf16) {
  if (bf16) return __uint_as_float(v << 16);
  return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu)));
}
__device__ __forceinline__ float hi16_to_f32(uint32_t v, bool bf16) {
  if (bf16) return __uint_as_float(v & 0xFFFF0000u);
  return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

// An act-order map entry outside [0, G) would index past the scale and zero
// arrays.  It is clamped into range (so nothing outside them is read) and
// reported as W4A16_ERR_INVALID_ARG (1) through the caller's status word.
__device__ __forceinline__ int checked_group(int gr, int G, int* dev_status) {
  if ((unsigned)gr >= (unsigned)G) {
    if (dev_status) atomicExch(dev_status, 1 /* W4A16_ERR_INVALID_ARG */);
    gr = gr < 0 ? 0 : G - 1;
  }
  return gr;
}

// ------------------------------------------------- INT4, exact differences
// The 8 codes of word w as the exact integers (q - z) in fp16, 4 pairs (row
// j, row j + 4): the 1024 + q / 64 + q forms of dq_word_f16 minus z_lo /
// z_hi (as in DqConstF16).  Every difference is an integer of at most 4
// bits, so each subtraction is exact.
__device__ __forceinline__ void dq_word_codes_f16(uint32_t w, uint32_t z_lo, uint32_t z_hi, uint32_t out[4]) {
  const uint32_t w8 = w >> 8;
  out[0] = hsub2_f16(lop3_and_or(w, 0x000F000Fu, 0x64006400u), z_lo);
  out[1] = hsub2_f16(lop3_and_or(w, 0x00F000F0u, 0x54005400u), z_hi);
  out[2] = hsub2_f16(lop3_and_or(w8, 0x000F000Fu, 0x64006400u), z_lo);
  out[3] = hsub2_f16(lop3_and_or(w8, 0x00F000F0u, 0x54005400u), z_hi);
}

// ---------------------------------------------------------------- INT4, fp16
// Per-(group, column) constants for the fp16 route; each half of a register
// may belong to a different (group, column), so act-order can mix them.
struct DqConstF16 {
  uint32_t z_lo;  // (1024 + z) in both halves: for pairs 0 and 2
  uint32_t z_hi;  // (64 + z): for pairs 1 and 3
  uint32_t s;     // fp16 scale
};

__device__ __forceinline__ DqConstF16 dq_const_f16(uint32_t z, uint32_t s_bits) {
  DqConstF16 c;
  c.z_lo = (0x6400u | z) * 0x00010001u;
  c.z_hi = (0x5400u | (z << 4)) * 0x00010001u;
  c.s = (s_bits & 0xFFFFu) * 0x00010001u;
  return c;
}

// Two (z, s) per register half: lane 0 for the low element, lane 1 for the high.
__device__ __forceinline__ DqConstF16 dq_const_f16_2(uint32_t z0, uint32_t s0, uint32_t z1, uint32_t s1) {
  DqConstF16 c;
  c.z_lo = (0x6400u | z0) | ((0x6400u | z1) << 16);
  c.z_hi = (0x5400u | (z0 << 4)) | ((0x5400u | (z1 << 4)) << 16);
  c.s = (s0 & 0xFFFFu) | (s1 << 16);
  return c;
}

// The 8 codes of word w -> 4 fp16 pairs: out[j] = (row j, row j + 4).
__device__ __forceinline__ void dq_word_f16(uint32_t w, const DqConstF16& c, uint32_t out[4]) {
  const uint32_t w8 = w >> 8;
  const uint32_t p0 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
  const uint32_t p1 = lop3_and_or(w, 0x00F000F0u, 0x54005400u);
  const uint32_t p2 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);
  const uint32_t p3 = lop3_and_or(w8, 0x00F000F0u, 0x54005400u);
  out[0] = hmul2_f16(hsub2_f16(p0, c.z_lo), c.s);
  out[1] = hmul2_f16(hsub2_f16(p1, c.z_hi), c.s);
  out[2] = hmul2_f16(hsub2_f16(p2, c.z_lo), c.s);
  out[3] = hmul2_f16(hsub2_f16(p3, c.z_hi), c.s);
}

// Same with a separate constant set per pair (act-order: every row of the word
// may sit in a different group).
__device__ __forceinline__ void dq_word_f16_rows(uint32_t w, const DqConstF16 c[4], uint32_t out[4]) {
  const uint32_t w8 = w >> 8;
  const uint32_t p0 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
  const uint32_t p1 = lop3_and_or(w, 0x00F000F0u, 0x54005400u);
  const uint32_t p2 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);
  const uint32_t p3 = lop3_and_or(w8, 0x00F000F0u, 0x54005400u);
  out[0] = hmul2_f16(hsub2_f16(p0, c[0].z_lo), c[0].s);
  out[1] = hmul2_f16(hsub2_f16(p1, c[1].z_hi), c[1].s);
  out[2] = hmul2_f16(hsub2_f16(p2, c[2].z_lo), c[2].s);
  out[3] = hmul2_f16(hsub2_f16(p3, c[3].z_hi), c[3].s);
}

// ---------------------------------------------------------------- INT4, bf16
struct DqConstBF16 {
  uint32_t z;     // (128 + z) as bf16 in both halves
  uint32_t s_hi;  // first 8 significant bits of s, bf16
  uint32_t s_lo;  // s - s_hi, exact in bf16
};

__device__ __forceinline__ void split_scale_bf16(uint32_t s_bits, uint32_t& hi16, uint32_t& lo16) {
  const float s = __half2float(__ushort_as_half((unsigned short)(s_bits & 0xFFFFu)));
  const uint32_t hb = __float_as_uint(s) & 0xFFFF0000u;
  const float lo = s - __uint_as_float(hb);  // exact: at most 3 significant bits
  hi16 = hb >> 16;
  // lo has the sign of s or is zero; giving a zero lo the sign of s keeps
  // (q - z) == 0 with a negative scale at -0, as the exact product is
  lo16 = (__float_as_uint(lo) | (__float_as_uint(s) & 0x80000000u)) >> 16;
}

__device__ __forceinline__ DqConstBF16 dq_const_bf16(uint32_t z, uint32_t s_bits) {
  DqConstBF16 c;
  uint32_t hi, lo;
  split_scale_bf16(s_bits, hi, lo);
  c.z = (0x4300u | z) * 0x00010001u;
  c.s_hi = hi * 0x00010001u;
  c.s_lo = lo * 0x00010001u;
  return c;
}

__device__ __forceinline__ DqConstBF16 dq_const_bf16_2(uint32_t z0, uint32_t s0, uint32_t z1, uint32_t s1) {
  DqConstBF16 c;
  uint32_t hi0, lo0, hi1, lo1;
  split_scale_bf16(s0, hi0, lo0);
  split_scale_bf16(s1, hi1, lo1);
  c.z = (0x4300u | z0) | ((0x4300u | z1) << 16);
  c.s_hi = hi0 | (hi1 << 16);
  c.s_lo = lo0 | (lo1 << 16);
  return c;
}

__device__ __forceinline__ uint32_t dq_pair_bf16(uint32_t p, const DqConstBF16& c) {
  const uint32_t v = hsub2_bf16(p, c.z);   // q - z, exact
  const uint32_t t = hmul2_bf16(v, c.s_lo);  // exact
  return hfma2_bf16(v, c.s_hi, t);           // one rounding of (q - z) * s
}

__device__ __forceinline__ void dq_word_bf16(uint32_t w, const DqConstBF16& c, uint32_t out[4]) {
  out[0] = dq_pair_bf16(lop3_and_or(w, 0x000F000Fu, 0x43004300u), c);
  out[1] = dq_pair_bf16(lop3_and_or(w >> 4, 0x000F000Fu, 0x43004300u), c);
  out[2] = dq_pair_bf16(lop3_and_or(w >> 8, 0x000F000Fu, 0x43004300u), c);
  out[3] = dq_pair_bf16(lop3_and_or(w >> 12, 0x000F000Fu, 0x43004300u), c);
}

__device__ __forceinline__ void dq_word_bf16_rows(uint32_t w, const DqConstBF16 c[4], uint32_t out[4]) {
  out[0] = dq_pair_bf16(lop3_and_or(w, 0x000F000Fu, 0x43004300u), c[0]);
  out[1] = dq_pair_bf16(lop3_and_or(w >> 4, 0x000F000Fu, 0x43004300u), c[1]);
  out[2] = dq_pair_bf16(lop3_and_or(w >> 8, 0x000F000Fu, 0x43004300u), c[2]);
  out[3] = dq_pair_bf16(lop3_and_or(w >> 12, 0x000F000Fu, 0x43004300u), c[3]);
}

// ------------------------------------------ INT4, bf16 through fp32 FMAs
// The same bf16 value from the fp16 route's magic codes and one
// mixed-precision FMA per weight (fp16 operands, exact product, fp32 sum):
//     fma(1024 + q, s, -(1024 + z) * s) = (q - z) * s   exactly,
// because -(1024 + z) * s has at most 22 significant bits (an exact fp32
// constant) and the result at most 15; likewise with 64 + q for the codes in
// bits 4..7.  One cvt.rn.bf16x2 then rounds each value of a pair once.  The
// FMAs issue on the fp32 pipe at full rate, leaving the packed 16-bit pipe
// idle: per pair 2 FMAs, 1 conversion and 1.25 logic operations, against 3
// packed operations and 1.75 logic operations above.  Only the sign of a
// zero weight can differ from the IEEE product (x + (-x) is +0); a product
// cannot show it, since its fp32 sums start from +0.
struct DqConstBF16Fma {
  float z_lo;  // -(1024 + z) * s: pairs 0 and 2
  float z_hi;  // -(64 + z) * s: pairs 1 and 3
  uint32_t s;  // fp16 scale in the low half
};

__device__ __forceinline__ DqConstBF16Fma dq_const_bf16_fma(uint32_t z, uint32_t s_bits) {
  const float s = __half2float(__ushort_as_half((unsigned short)(s_bits & 0xFFFFu)));
  DqConstBF16Fma c;
  c.z_lo = __fmul_rn(-(1024.f + (float)z), s);  // exact
  c.z_hi = __fmul_rn(-(64.f + (float)z), s);    // exact
  c.s = s_bits & 0xFFFFu;
  return c;
}

// fma(half H of p, low half of s, zs) with fp16 operands and an fp32 sum
template <int H>
__device__ __forceinline__ float fma_f16_f32(uint32_t p, uint32_t s, float zs) {
  float d;
  if (H == 0)
    asm("{\n\t.reg .f16 a0, a1, s0, s1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "mov.b32 {s0, s1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, s0, %3;\n\t}"
        : "=f"(d)
        : "r"(p), "r"(s), "f"(zs));
  else
    asm("{\n\t.reg .f16 a0, a1, s0, s1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "mov.b32 {s0, s1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a1, s0, %3;\n\t}"
        : "=f"(d)
        : "r"(p), "r"(s), "f"(zs));
  return d;
}

__device__ __forceinline__ uint32_t dq_pair_bf16_fma(uint32_t p, float zs, uint32_t s) {
  return pack2_rn(fma_f16_f32<0>(p, s, zs), fma_f16_f32<1>(p, s, zs), true);
}

__device__ __forceinline__ void dq_word_bf16_fma(uint32_t w, const DqConstBF16Fma& c, uint32_t out[4]) {
  const uint32_t w8 = w >> 8;
  out[0] = dq_pair_bf16_fma(lop3_and_or(w, 0x000F000Fu, 0x64006400u), c.z_lo, c.s);
  out[1] = dq_pair_bf16_fma(lop3_and_or(w, 0x00F000F0u, 0x54005400u), c.z_hi, c.s);
  out[2] = dq_pair_bf16_fma(lop3_and_or(w8, 0x000F000Fu, 0x64006400u), c.z_lo, c.s);
  out[3] = dq_pair_bf16_fma(lop3_and_or(w8, 0x00F000F0u, 0x54005400u), c.z_hi, c.s);
}

// -------------------------------------------------- natural K order pairs
// The tensor-memory A operand needs each 32-bit cell to hold two consecutive
// K rows, (2j, 2j+1).  Byte j of a word holds exactly those two codes; a byte
// permute copies it into both 16-bit halves and the magic masks pick the low
// code in the low half and the high code in the high half.
//   fp16: low half 1024 + q (code in bits 0..3), high half 64 + q (code in
//         bits 4..7 of that half), so the zero-point constant differs by half.
//   bf16: the high half takes byte j of (w >> 4), so both codes sit in bits
//         0..3 of their half under the 128 magic.
__device__ __forceinline__ uint32_t dq_zmix_f16(uint32_t z) {
  return (0x6400u | z) | ((0x5400u | (z << 4)) << 16);
}

__device__ __forceinline__ void dq_word_nat_f16(uint32_t w, uint32_t zmix, uint32_t s2, uint32_t out[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t u = prmt(w, 0u, 0x1111u * j);
    out[j] = hmul2_f16(hsub2_f16(lop3_and_or(u, 0x00F0000Fu, 0x54006400u), zmix), s2);
  }
}

// The FMA route in natural K order costs no more than in the (j, j + 4)
// order: each FMA yields its own fp32 value and the conversion pairs any two,
// so pair (2j, 2j + 1) takes its codes from two magic registers, the
// 1024 + q one (rows 0, 4 / 2, 6) and the 64 + q one (rows 1, 5 / 3, 7).
__device__ __forceinline__ void dq_word_nat_bf16_fma(uint32_t w, const DqConstBF16Fma& c, uint32_t out[4]) {
  const uint32_t w8 = w >> 8;
  const uint32_t p04 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
  const uint32_t p15 = lop3_and_or(w, 0x00F000F0u, 0x54005400u);
  const uint32_t p26 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);
  const uint32_t p37 = lop3_and_or(w8, 0x00F000F0u, 0x54005400u);
  out[0] = pack2_rn(fma_f16_f32<0>(p04, c.s, c.z_lo), fma_f16_f32<0>(p15, c.s, c.z_hi), true);
  out[1] = pack2_rn(fma_f16_f32<0>(p26, c.s, c.z_lo), fma_f16_f32<0>(p37, c.s, c.z_hi), true);
  out[2] = pack2_rn(fma_f16_f32<1>(p04, c.s, c.z_lo), fma_f16_f32<1>(p15, c.s, c.z_hi), true);
  out[3] = pack2_rn(fma_f16_f32<1>(p26, c.s, c.z_lo), fma_f16_f32<1>(p37, c.s, c.z_hi), true);
}

__device__ __forceinline__ void dq_word_nat_bf16(uint32_t w, const DqConstBF16& c, uint32_t out[4]) {
  const uint32_t w4 = w >> 4;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t sel = (uint32_t)j * 0x0011u + (uint32_t)(4 + j) * 0x1100u;
    const uint32_t u = prmt(w, w4, sel);
    out[j] = dq_pair_bf16(lop3_and_or(u, 0x000F000Fu, 0x43004300u), c);
  }
}

// (ca, cb) * absmax as two IEEE fp32 products (round to nearest, no flush),
// issued as one packed fp32x2 multiply, then one pair conversion
__device__ __forceinline__ uint32_t nf4_pair(float ca, float cb, float absmax, bool bf16) {
  uint64_t x, m, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(ca), "f"(cb));
  asm("mov.b64 %0, {%1, %1};" : "=l"(m) : "f"(absmax));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(m));
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
  return pack2_rn(lo, hi, bf16);
}

template <bool BF16>
__device__ __forceinline__ void dq_word_nat_nf4(uint32_t w, const float* cb, float absmax, uint32_t out[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    out[j] = nf4_pair(cb[(w >> (8 * j)) & 0xFu], cb[(w >> (8 * j + 4)) & 0xFu], absmax, BF16);
  }
}

// ---------------------------------------------------------------------- NF4
// w_hat = RNE_dtype(fl32(C[q] * absmax)): an fp32 product, then one rounding.
// `cb` is the 16-entry codebook (shared or register copy).
template <bool BF16>
__device__ __forceinline__ void dq_word_nf4(uint32_t w, const float* cb, float absmax, uint32_t out[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    out[j] = nf4_pair(cb[(w >> (4 * j)) & 0xFu], cb[(w >> (4 * j + 16)) & 0xFu], absmax, BF16);
  }
}

}  // namespace w4a16
