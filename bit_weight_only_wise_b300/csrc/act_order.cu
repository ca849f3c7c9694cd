// Act-order prepack: a one-time reordering of an act-order checkpoint's rows so
// that every group's rows are contiguous, in group order.
//
// With GPTQ's act-order ("GPTQ与bitsandbytes对比：谁是2024年大模型量化的终极选择？",
// GPTQ section, --act-order; "模型量化实践：GPTQ 与 AWQ 在生产环境的精度与速度权衡"
// §3.1, desc_act) each K row k belongs to group g_idx[k], and the rows of one
// group are scattered over K, so a kernel that streams the rows in storage
// order needs a different (scale, zero) for nearly every row.  Reordering the
// rows by group turns the product into a plain grouped one:
//
//   Y = X . W_hat = X[:, perm] . W_hat[perm, :],   sorted row j = original row perm[j]
//
// where group g holds sorted rows [g*128, (g+1)*128).  The reorder is exact
// (the same products, summed in another order), needs every group to hold
// exactly 128 rows, and is done once, when the checkpoint is loaded; at run
// time only X's columns are gathered (M*K values).
//
//   act_order_perm_kernel    one CTA per group: the group's rows in their
//                            original order (a ballot prefix count per chunk
//                            of rows), and a count check;
//   act_order_repack_kernel  sorted word (i, n) = the nibbles of rows
//                            perm[8i .. 8i+7] of column n;
//   gather_columns_kernel    X_perm[m, j] = X[m, perm[j]].
//
// Every index read from a caller's buffer (g_idx, perm) is clamped into range,
// so a malformed map produces wrong numbers and a status, never an access
// outside the arrays.
#include <cstdint>

#include "sm100.cuh"
#include "w4a16_internal.h"

namespace w4a16 {

namespace {

constexpr int kPermThreads = 256;

__global__ void __launch_bounds__(kPermThreads)
    act_order_perm_kernel(const int32_t* __restrict__ g_idx, int K, int group_size, int32_t* __restrict__ perm,
                          int* dev_status) {
  const int g = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int warp_count[kPermThreads / 32];
  int base = 0;  // rows of group g found before the current chunk
  for (int k0 = 0; k0 < K; k0 += kPermThreads) {
    const int k = k0 + threadIdx.x;
    const bool hit = k < K && g_idx[k] == g;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, hit);
    if (lane == 0) warp_count[warp] = __popc(m);
    __syncthreads();
    int before = base;
    for (int w = 0; w < warp; ++w) before += warp_count[w];
    before += __popc(m & ((1u << lane) - 1u));
    if (hit && before < group_size) perm[g * group_size + before] = k;
    int total = 0;
    for (int w = 0; w < kPermThreads / 32; ++w) total += warp_count[w];
    base += total;
    __syncthreads();
  }
  // every group must hold exactly group_size rows for the sorted layout
  if (threadIdx.x == 0 && base != group_size && dev_status) atomicExch(dev_status, 2 /* W4A16_ERR_UNSUPPORTED */);
}

__global__ void __launch_bounds__(256)
    act_order_repack_kernel(const uint32_t* __restrict__ qw, const int32_t* __restrict__ perm, int K, int N,
                            uint32_t* __restrict__ out) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = blockIdx.y;  // sorted word-row
  if (n >= N) return;
  uint32_t w = 0;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    int src = perm[8 * i + r];
    src = src < 0 ? 0 : (src >= K ? K - 1 : src);
    w |= ((qw[(size_t)(src >> 3) * N + n] >> (4 * (src & 7))) & 0xFu) << (4 * r);
  }
  out[(size_t)i * N + n] = w;
}

// Launched as a programmatic dependent of the previous kernel in the stream
// and letting the next one (the product) launch at once, so that the
// product's launch overlaps this one; X, perm and the scratch it writes are
// touched only after the previous kernel has completed.
__global__ void __launch_bounds__(256)
    gather_columns_kernel(const uint16_t* __restrict__ X, const int32_t* __restrict__ perm, int M, int K,
                          uint16_t* __restrict__ out) {
  sm100::griddep_launch_dependents();
  sm100::griddep_wait();
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= K) return;
  int src = perm[j];
  src = src < 0 ? 0 : (src >= K ? K - 1 : src);
  for (int m = blockIdx.y; m < M; m += gridDim.y) out[(size_t)m * K + j] = X[(size_t)m * K + src];
}

}  // namespace

cudaError_t launch_act_order_prepack(const uint32_t* qw, const int32_t* g_idx, int K, int N, int group_size,
                                     uint32_t* qw_sorted, int32_t* perm, int* dev_status, cudaStream_t st) {
  act_order_perm_kernel<<<K / group_size, kPermThreads, 0, st>>>(g_idx, K, group_size, perm, dev_status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  act_order_repack_kernel<<<dim3((N + 255) / 256, K / 8), 256, 0, st>>>(qw, perm, K, N, qw_sorted);
  return cudaGetLastError();
}

cudaError_t launch_gather_columns(const uint16_t* X, const int32_t* perm, int M, int K, uint16_t* out,
                                  cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((K + 255) / 256, M < 65535 ? M : 65535);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_columns_kernel, X, perm, M, K, out);
}

}  // namespace w4a16
