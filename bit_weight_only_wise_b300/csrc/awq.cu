// Repack an AWQ checkpoint into this library's layout.
//
// AWQ checkpoints ("模型量化实践：GPTQ 与 AWQ 在生产环境的精度与速度权衡" §3.1:
// zero_point=True, q_group_size=128, w_bit=4, version="GEMM") are what the
// fastest rows of "LLM量化技术深度对比" §5 serve, through a kernel of their
// own layout.  The pages do not print that layout; the one taken here is AWQ's
// published GEMM layout:
//   qweight int32 [K, N/8]: word [k, c] holds row k, columns 8c .. 8c+7, with
//                           column 8c + ORDER[j] in bits 4j .. 4j+3,
//                           ORDER = (0, 2, 4, 6, 1, 3, 5, 7);
//   qzeros  int32 [G, N/8]: zero points, packed the same way;
//   scales  fp16  [G, N]:   as in this library (no conversion needed).
// This library packs codes along K (8 rows of one column per word) and zero
// points along N in natural column order, so the repack is a pure
// rearrangement of nibbles: each thread reads the 8 AWQ words of rows
// 8i .. 8i+7 for column group c (coalesced across threads), transposes the
// 8 x 8 nibble block in registers and writes the 8 words [i, 8c .. 8c+7].
#include <cstdint>

#include "w4a16_internal.h"

namespace w4a16 {

namespace {

// bit position (x 4) of natural column j within an AWQ word: ORDER^-1
__device__ __forceinline__ int awq_slot(int j) { return (j >> 1) + 4 * (j & 1); }

__global__ void __launch_bounds__(256) awq_repack_kernel(const uint32_t* __restrict__ qa, int K, int N,
                                                         uint32_t* __restrict__ qw) {
  const int C = N / 8;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;  // column group
  const int i = blockIdx.y;                             // word-row (8 rows)
  if (c >= C) return;
  uint32_t in[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) in[r] = qa[(size_t)(8 * i + r) * C + c];
  uint32_t out[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {  // natural column 8c + j
    const int sh = 4 * awq_slot(j);
    uint32_t w = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) w |= ((in[r] >> sh) & 0xFu) << (4 * r);
    out[j] = w;
  }
  uint32_t* dst = qw + (size_t)i * N + 8 * c;
  if ((N & 3) == 0 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(out[0], out[1], out[2], out[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(out[4], out[5], out[6], out[7]);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[j] = out[j];
  }
}

// zero points: the nibble of natural column j moves from slot ORDER^-1[j] to j
__global__ void __launch_bounds__(256) awq_zeros_kernel(const uint32_t* __restrict__ za, int total,
                                                        uint32_t* __restrict__ zw) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= total) return;
  const uint32_t v = za[t];
  uint32_t w = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) w |= ((v >> (4 * awq_slot(j))) & 0xFu) << (4 * j);
  zw[t] = w;
}

}  // namespace

cudaError_t launch_awq_repack(const uint32_t* qweight_awq, const uint32_t* qzeros_awq, int K, int N, int G,
                              uint32_t* qweight, uint32_t* qzeros, cudaStream_t st) {
  const int C = N / 8;
  dim3 block(256), grid((C + 255) / 256, K / 8);
  awq_repack_kernel<<<grid, block, 0, st>>>(qweight_awq, K, N, qweight);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !qzeros_awq) return e;
  const int total = G * C;
  awq_zeros_kernel<<<(total + 255) / 256, 256, 0, st>>>(qzeros_awq, total, qzeros);
  return cudaGetLastError();
}

}  // namespace w4a16
