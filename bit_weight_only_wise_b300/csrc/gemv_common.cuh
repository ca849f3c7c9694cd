// Device pieces shared by the split-K decode kernels (gemv.cu, gemv_ws.cu):
// the stream-K split of the units over the persistent grid, the m16n8k16
// tensor-core step, and the write-out of a finished 256-column block, either
// directly or through the deterministic split-K reduction.
//
// Units: 256 output columns x one 128-row K group, numbered column-block-major
// (u = b * G + g).  CTA i of P owns units [U*i/P, U*(i+1)/P).  Within a CTA,
// 8 warps own a 32-column slice each; lane (g, c) = (lane / 4, lane % 4)
// accumulates columns 4g .. 4g+3 of the slice for tokens 2c, 2c+1 (+8t) in
// the m16n8k16 accumulator layout (column = MMA row, token = MMA column).
#pragma once

#include <cstdint>

#include "dq_common.cuh"
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

// Warp `warp`'s slice of column block b is finished: write it directly when
// CTA `cta` owns the whole block, else through a partial and a ticket; the
// last contributor sums the partials in contributor order (deterministic
// whatever the arrival order), rounds once and resets the ticket.
template <int NT, bool BF16>
__device__ __forceinline__ void flush_block(const GemvArgs& a, const Range& R, int cta, int first_block, int warp,
                                            int lane, int b, const float (&acc)[NT][2][4]) {
  const int gl = lane >> 2, c = lane & 3;
  const int col0 = b * kGemvCols + warp * 32 + 4 * gl;
  const int i_first = R.owner((long long)b * a.G);
  const int i_last = R.owner((long long)(b + 1) * a.G - 1);
  if (i_first == i_last) {
    if (col0 >= a.N) return;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int tok = 8 * t + 2 * c;
        const int col = col0 + 2 * r;
        if (tok < a.M)
          *reinterpret_cast<uint32_t*>(a.Y + (size_t)tok * a.N + col) = pack2_rn(acc[t][r][0], acc[t][r][2], BF16);
        if (tok + 1 < a.M)
          *reinterpret_cast<uint32_t*>(a.Y + (size_t)(tok + 1) * a.N + col) =
              pack2_rn(acc[t][r][1], acc[t][r][3], BF16);
      }
    return;
  }
  const int seg = (b == first_block) ? 0 : 1;
  float* slot = a.partial + ((size_t)(cta * 2 + seg) * kSliceWarps + warp) * a.M * 32;
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
  __threadfence();
  __syncwarp();
  int last = 0;
  int* ticket = a.counters + b * kSliceWarps + warp;
  if (lane == 0) {
    last = atomicAdd(ticket, 1) == i_last - i_first;
    if (last) {
      *ticket = 0;  // ready for the next call
      __threadfence();
    }
  }
  last = __shfl_sync(0xFFFFFFFFu, last, 0);
  if (!last) return;
  const int col = b * kGemvCols + warp * 32 + lane;
  if (col >= a.N) return;
  // contributor i wrote this block as its first (slot 0) or last (slot 1)
  // block; the partials of kChunk contributors (all tokens) are loaded at
  // once and added in contributor order, so the sum is deterministic and a
  // block split over many CTAs costs few round trips
  constexpr int kChunk = NT == 1 ? 4 : 2;
  float sum[8 * NT];
#pragma unroll
  for (int t = 0; t < 8 * NT; ++t) sum[t] = 0.f;
  for (int i0 = i_first; i0 <= i_last; i0 += kChunk) {
    float v[kChunk][8 * NT];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const int i = i0 + j;
      const int sg = (i <= i_last && b == (int)(R.start(i) / a.G)) ? 0 : 1;
      const float* pp = a.partial + ((size_t)(i * 2 + sg) * kSliceWarps + warp) * a.M * 32 + lane;
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
    if (t < a.M) a.Y[(size_t)t * a.N + col] = (uint16_t)(pack2_rn(sum[t], 0.f, BF16) & 0xFFFFu);
}

}  // namespace w4a16
