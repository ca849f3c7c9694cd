// Device pieces shared by the split-K decode kernels (gemv.cu, gemv_ws.cu):
// the stream-K split of the units over the persistent grid, the m16n8k16
// tensor-core step, and the write-out of a finished 256-column block, either
// directly or through the deterministic split-K reduction.
//
// Units: 256 weight columns x one 128-row K block, numbered column-block-major
// (u = b * KB + kb).  CTA i of P owns units [U*i/P, U*(i+1)/P).  Within a CTA,
// 8 warps own a 32-column slice each; lane (g, c) = (lane / 4, lane % 4)
// accumulates columns 4g .. 4g+3 of the slice for tokens 2c, 2c+1 (+8t) in
// the m16n8k16 accumulator layout (column = MMA row, token = MMA column).
// Slice w of block b is output column b * cpb + 32 (w % 4) + (w / 4) hi2 on
// (see GemvArgs): the plain product's 256 columns, or with the fused SiLU
// epilogue the gate (w < 4) and up (w >= 4) halves of 128 output columns,
// which the write-out pairs: act = SiLU(gate) * up.
#pragma once

#include <cstdint>

#include "dq_common.cuh"
#include "sm100.cuh"
#include "w4a16_internal.h"

namespace w4a16 {

constexpr int kSliceWarps = kGemvCols / 32;  // 8 column slices per 256-column block

struct Range {
  long long U;  // units
  int P;        // CTAs
  __device__ __forceinline__ long long start(int i) const { return U * i / P; }
  // the CTA whose range holds unit u: the largest i with start(i) <= u
  __device__ __forceinline__ int owner(long long u) const { return (int)(((u + 1) * P - 1) / U); }
};

// SiLU(g) * u in fp32, the gate_up epilogue
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g, 1.f + __expf(-g)) * u; }

// A launch's column geometry (see GemvArgs), fixed at compile time for the
// plain product -- 256-column blocks, halves 128 columns apart, Y as wide as
// N -- and read from the arguments for the fused SiLU epilogue, which is a
// kernel variant of its own: the plain kernels carry none of its code or
// registers (the 32-row-group bf16 variant's spills went from 152 to 12
// bytes).
template <bool SILU>
struct Geom {
  __device__ __forceinline__ static int cpb(const GemvArgs& a) { return SILU ? a.cpb : kGemvCols; }
  __device__ __forceinline__ static int hiofs(const GemvArgs& a) { return SILU ? a.hiofs : kGemvCols / 2; }
  __device__ __forceinline__ static int hi2(const GemvArgs& a) { return SILU ? a.hi2 : kGemvCols / 2; }
  __device__ __forceinline__ static int nout(const GemvArgs& a) { return SILU ? a.Nout : a.N; }
  __device__ __forceinline__ static int ldy(const GemvArgs& a) { return SILU ? a.ldy : a.N; }
};

// first output column of warp w's slice of block b
template <bool SILU>
__device__ __forceinline__ int slice_col(const GemvArgs& a, int b, int warp) {
  return b * Geom<SILU>::cpb(a) + 32 * (warp & 3) + (warp >> 2) * Geom<SILU>::hi2(a);
}

template <bool BF16>
__device__ __forceinline__ void mma_16816(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  if (BF16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d = A * B with a zero accumulator (the first step of a sum)
template <bool BF16>
__device__ __forceinline__ void mma_16816_zc(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  if (BF16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// The word-row of a 16-row tile that lane quarter-index c reads at step o;
// under the 128-byte swizzle the four quarters then hit distinct banks.
__device__ __forceinline__ int tile_row(int c, int o) { return 2 * c + 8 * (o & 1) + (o >> 1); }

// Activation pairs for the MMA's B operand: 8 consecutive K rows of one token
// (xv = rows 0..7, two per word) -> pairs (0,4), (1,5), (2,6), (3,7), the K
// order in which a packed word's codes come out of the dequantizer.
__device__ __forceinline__ void x_pairs(const uint4& xv, uint32_t bf[4]) {
  bf[0] = prmt(xv.x, xv.z, 0x5410u);
  bf[1] = prmt(xv.x, xv.z, 0x7632u);
  bf[2] = prmt(xv.y, xv.w, 0x5410u);
  bf[3] = prmt(xv.y, xv.w, 0x7632u);
}

// Warp `warp`'s slice of column block b is finished.  When CTA `cta` owns
// the whole block the slice is rounded and written to Y here.  Otherwise its
// fp32 partial goes to the CTA's slot for the block (slot 0 for the CTA's
// first block, 1 for its last) and the function returns true: the block's
// ticket is taken later, by finish_blocks, once the CTA has nothing else to
// do, so that no warp waits on a memory round trip in the middle of its work.
// this warp's fp32 fragment of a block into a slice slot (the split-K layout)
template <int NT>
__device__ __forceinline__ void store_slot(const GemvArgs& a, float* slot, int lane, const float (&acc)[NT][2][4]) {
  const int gl = lane >> 2, c = lane & 3;
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int tok = 8 * t + 2 * c;
      const int cl = 4 * gl + 2 * r;
      if (tok < a.M) *reinterpret_cast<float2*>(slot + tok * 32 + cl) = make_float2(acc[t][r][0], acc[t][r][2]);
      if (tok + 1 < a.M)
        *reinterpret_cast<float2*>(slot + (tok + 1) * 32 + cl) = make_float2(acc[t][r][1], acc[t][r][3]);
    }
}

// Slot of CTA cta's segment seg (0: its first block, 1: its last), slice w.
// With the fused SiLU epilogue the grid holds at most 2 CTAs per SM; the
// workspace is sized for kGemvMaxCTAsPerSM (3), so the slots of CTA indices
// kNumSMs * 2 .. kNumSMs * 3 - 1 are unused by the split-K reduction, and
// (CTA kNumSMs * 2 + i / 2, segment i % 2) carries CTA i's fully owned
// blocks' gate and up halves between its warps.
static_assert(kGemvMaxCTAsPerSM >= 3, "the SiLU exchange slots lie past two CTAs per SM");
__device__ __forceinline__ float* slice_slot(const GemvArgs& a, int cta, int seg, int warp) {
  return a.partial + ((size_t)(cta * 2 + seg) * kSliceWarps + warp) * a.M * 32;
}

// Warp `warp`'s slice of column block b is finished.  When CTA `cta` owns
// the whole block the slice is rounded and written to Y here.  Otherwise its
// fp32 partial goes to the CTA's slot for the block (slot 0 for the CTA's
// first block, 1 for its last) and the function returns true: the block's
// ticket is taken later, by finish_blocks, once the CTA has nothing else to
// do, so that no warp waits on a memory round trip in the middle of its work.
// Fused SiLU, whole block: both halves pass through the CTA's exchange slot,
// a barrier of the consumer warps (named barrier 1, all kSliceWarps warps)
// orders the writes before the gate warps read.
template <int NT, bool BF16, bool SILU>
__device__ __forceinline__ bool store_block(const GemvArgs& a, const Range& R, int cta, int first_block, int warp,
                                            int lane, int b, const float (&acc)[NT][2][4]) {
  const int gl = lane >> 2, c = lane & 3;
  using G = Geom<SILU>;
  const int col0 = slice_col<SILU>(a, b, warp) + 4 * gl;
  const int i_first = R.owner((long long)b * a.KB);
  const int i_last = R.owner((long long)(b + 1) * a.KB - 1);
  if (SILU && i_first == i_last) {
    float* xs = slice_slot(a, kNumSMs * 2 + cta / 2, cta % 2, 0);
    store_slot<NT>(a, xs + (size_t)warp * a.M * 32, lane, acc);
    asm volatile("bar.sync 1, %0;" ::"r"(kSliceWarps * 32) : "memory");
    if (warp < kSliceWarps / 2) {
      const int col = slice_col<SILU>(a, b, warp) + lane;
      const float* gp = xs + (size_t)warp * a.M * 32 + lane;
      const float* up = xs + (size_t)(warp + kSliceWarps / 2) * a.M * 32 + lane;
      if (col < G::nout(a))
        for (int t = 0; t < a.M; ++t)
          a.Y[(size_t)t * G::ldy(a) + col] =
              (uint16_t)(pack2_rn(silu_mul(gp[t * 32], up[t * 32]), 0.f, BF16) & 0xFFFFu);
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kSliceWarps * 32) : "memory");  // the slot is free again
    return false;
  }
  if (i_first == i_last) {
    if (col0 >= G::nout(a)) return false;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int tok = 8 * t + 2 * c;
        const int col = col0 + 2 * r;
        if (tok < a.M)
          *reinterpret_cast<uint32_t*>(a.Y + (size_t)tok * G::ldy(a) + col) = pack2_rn(acc[t][r][0], acc[t][r][2], BF16);
        if (tok + 1 < a.M)
          *reinterpret_cast<uint32_t*>(a.Y + (size_t)(tok + 1) * G::ldy(a) + col) =
              pack2_rn(acc[t][r][1], acc[t][r][3], BF16);
      }
    return false;
  }
  store_slot<NT>(a, slice_slot(a, cta, b == first_block ? 0 : 1, warp), lane, acc);
  return true;
}

// Sum the partials of split block b for this warp's slice, in contributor
// order (deterministic whatever order the contributors finished in), round
// once and write Y.  Contributor i wrote the block as its first block (slot 0)
// unless its range starts before the block, which only the first contributor's
// can.  Several contributors' loads are in flight at once.
template <int NT, bool BF16, bool SILU>
__device__ __forceinline__ void reduce_block(const GemvArgs& a, const Range& R, int warp, int lane, int b) {
  using G = Geom<SILU>;
  const int col = slice_col<SILU>(a, b, warp) + lane;
  if (col >= G::nout(a)) return;
  const int i_first = R.owner((long long)b * a.KB);
  const int i_last = R.owner((long long)(b + 1) * a.KB - 1);
  const int sg_first = R.start(i_first) == (long long)b * a.KB ? 0 : 1;
  const size_t stride = (size_t)a.M * 32;  // floats per slice slot
  auto slot = [&](int i) -> const float* {
    return a.partial + ((size_t)(i * 2 + (i == i_first ? sg_first : 0)) * kSliceWarps + warp) * stride + lane;
  };
  if (SILU) {  // slices warp (gate) and warp + 4 (up), both summed in contributor order
    for (int t = 0; t < a.M; ++t) {
      float g = 0.f, u = 0.f;
      for (int i = i_first; i <= i_last; ++i) {
        g += __ldcg(slot(i) + t * 32);
        u += __ldcg(slot(i) + (size_t)(kSliceWarps / 2) * stride + t * 32);
      }
      a.Y[(size_t)t * G::ldy(a) + col] = (uint16_t)(pack2_rn(silu_mul(g, u), 0.f, BF16) & 0xFFFFu);
    }
    return;
  }
  if (a.M == 1) {  // single token: sixteen contributors per round trip
    float sum = 0.f;
    for (int i0 = i_first; i0 <= i_last; i0 += 16) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = i0 + j <= i_last ? __ldcg(slot(i0 + j)) : 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) sum += v[j];
    }
    a.Y[col] = (uint16_t)(pack2_rn(sum, 0.f, BF16) & 0xFFFFu);
    return;
  }
  constexpr int kChunk = NT == 1 ? 4 : 2;
  float sum[8 * NT];
#pragma unroll
  for (int t = 0; t < 8 * NT; ++t) sum[t] = 0.f;
  for (int i0 = i_first; i0 <= i_last; i0 += kChunk) {
    float v[kChunk][8 * NT];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const int i = i0 + j;
      const float* pp = slot(i);
#pragma unroll
      for (int t = 0; t < 8 * NT; ++t) v[j][t] = (i <= i_last && t < a.M) ? __ldcg(pp + t * 32) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kChunk; ++j)
#pragma unroll
      for (int t = 0; t < 8 * NT; ++t) sum[t] += v[j][t];
  }
#pragma unroll
  for (int t = 0; t < 8 * NT; ++t)
    if (t < a.M) a.Y[(size_t)t * G::ldy(a) + col] = (uint16_t)(pack2_rn(sum[t], 0.f, BF16) & 0xFFFFu);
}

// reduce_block for two blocks at M = 1 with every contributor's load of both
// in flight at once (a warp that completes both of its blocks' counts; the
// plain product only)
template <bool BF16>
__device__ __forceinline__ void reduce_two_blocks_m1(const GemvArgs& a, const Range& R, int warp, int lane, int b0,
                                                     int b1) {
  int first[2], last[2], sgf[2], col[2];
  const int bs[2] = {b0, b1};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    first[h] = R.owner((long long)bs[h] * a.KB);
    last[h] = R.owner((long long)(bs[h] + 1) * a.KB - 1);
    sgf[h] = R.start(first[h]) == (long long)bs[h] * a.KB ? 0 : 1;
    col[h] = slice_col<false>(a, bs[h], warp) + lane;
  }
  float sum[2] = {0.f, 0.f};
  const int n = max(last[0] - first[0], last[1] - first[1]) + 1;
  for (int j0 = 0; j0 < n; j0 += 8) {
    float v[2][8];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = first[h] + j0 + j;
        const float* pp =
            a.partial + ((size_t)(i * 2 + (i == first[h] ? sgf[h] : 0)) * kSliceWarps + warp) * 32 + lane;
        v[h][j] = (i <= last[h] && col[h] < a.N) ? __ldcg(pp) : 0.f;
      }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int j = 0; j < 8; ++j) sum[h] += v[h][j];
  }
#pragma unroll
  for (int h = 0; h < 2; ++h)
    if (col[h] < a.N) a.Y[col[h]] = (uint16_t)(pack2_rn(sum[h], 0.f, BF16) & 0xFFFFu);
}

// The CTA is done: publish this warp's partials of split blocks p0 and p1
// (the CTA's first and last block; -1 for none) and take their tickets; the
// contributor that completes a block's count sums it.
template <int NT, bool BF16, bool SILU>
__device__ __forceinline__ void finish_blocks(const GemvArgs& a, const Range& R, int warp, int lane, int p0, int p1) {
  if (p0 < 0 && p1 < 0) return;
  // the warp barrier orders every lane's partial stores before lane 0's
  // fence, whose release covers them before the tickets move; the acquire
  // increments order the summing loads after the other contributors' stores
  __syncwarp();
  // Fused SiLU: the gate slice w and the up slice w + 4 of every contributor
  // count on one ticket (slice w % 4), so the warp that completes it sums
  // both halves: a wrap of 2 contributors - 1.
  int last0 = 0, last1 = 0;
  if (lane == 0) {
    __threadfence();
    const int tw = SILU ? (warp & (kSliceWarps / 2 - 1)) : warp;
    if (p0 >= 0) {
      uint32_t w = (uint32_t)(R.owner((long long)(p0 + 1) * a.KB - 1) - R.owner((long long)p0 * a.KB));
      if (SILU) w = 2 * w + 1;
      last0 = sm100::ticket_inc_acquire(a.counters + p0 * kSliceWarps + tw, w) == w;
    }
    if (p1 >= 0) {
      uint32_t w = (uint32_t)(R.owner((long long)(p1 + 1) * a.KB - 1) - R.owner((long long)p1 * a.KB));
      if (SILU) w = 2 * w + 1;
      last1 = sm100::ticket_inc_acquire(a.counters + p1 * kSliceWarps + tw, w) == w;
    }
  }
  __syncwarp();
  last0 = __shfl_sync(0xFFFFFFFFu, last0, 0);
  last1 = __shfl_sync(0xFFFFFFFFu, last1, 0);
  if (SILU) {  // the completing warp may be the gate or the up one: sum from the gate slice
    if (last0) reduce_block<NT, BF16, SILU>(a, R, warp & (kSliceWarps / 2 - 1), lane, p0);
    if (last1) reduce_block<NT, BF16, SILU>(a, R, warp & (kSliceWarps / 2 - 1), lane, p1);
    return;
  }
  if (last0 && last1 && a.M == 1) {  // both blocks: one round trip for the two
    reduce_two_blocks_m1<BF16>(a, R, warp, lane, p0, p1);
    return;
  }
  if (last0) reduce_block<NT, BF16, SILU>(a, R, warp, lane, p0);
  if (last1) reduce_block<NT, BF16, SILU>(a, R, warp, lane, p1);
}

}  // namespace w4a16
