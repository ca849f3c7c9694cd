// Allocation-free variant of the decode entry point (w4a16_gemv_noalloc).
//
// Some callers cannot allocate device memory at the moment they need a
// product: code running inside a memory pool they do not own, a runtime that
// forbids cudaMalloc on its hot path (allocation can synchronise the device
// or fail under fragmentation), or a host whose framework hands it only the
// input and output tensors.  w4a16_gemv needs a caller-provided workspace for
// its split-K partial sums; this entry point instead uses a scratch array that
// lives in the library itself, in device global memory, reserved once per GPU
// when the library's code is loaded there.
//
// The array's device address is looked up with cudaGetSymbolAddress the first
// time the entry point runs on a device (with that device current) and cached.
// Each call clears the part of the array that must start at zero (the split-K
// tickets) and then runs the ordinary decode kernel with the array as its
// workspace.  All calls share the one array, so calls that overlap on the GPU
// (different streams, no ordering between them) race on it and must not be
// issued.
#include <cstdint>
#include <mutex>

#include "w4a16.h"
#include "w4a16_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// The scratch: split-K tickets first, then fp32 partial sums (the same layout
// the caller's workspace has for w4a16_gemv).  Zero-initialised at load.
static __device__ __align__(256) unsigned char g_noalloc_scratch[W4A16_NOALLOC_SCRATCH_BYTES];

void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" w4a16_status w4a16_gemv_noalloc(const void* X, const uint32_t* qweight, const void* scales,
                                           const uint32_t* qzeros, const int32_t* g_idx, void* Y, int M, int N,
                                           int K, int group_size, w4a16_dtype dtype, int* dev_status,
                                           cudaStream_t stream) {
  // every check of w4a16_gemv, in its order, before the scratch or the stream
  // is touched: a rejected call has no side effect
  if (dtype != W4A16_F16 && dtype != W4A16_BF16) return W4A16_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K <= 0 || M > W4A16_MAX_M || N > W4A16_MAX_N || K > W4A16_MAX_K)
    return W4A16_ERR_INVALID_ARG;
  if (N % 8 || K % 8 || group_size <= 0 || K % group_size) return W4A16_ERR_INVALID_ARG;
  if (!w4a16::int4_group_supported(K, group_size)) return W4A16_ERR_UNSUPPORTED;
  if (M > W4A16_GEMV_MAX_M) return W4A16_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return W4A16_OK;
  auto ok16 = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!ok16(X) || !ok16(qweight) || !ok16(scales) || !ok16(Y)) return W4A16_ERR_INVALID_ARG;
  if (qzeros && (reinterpret_cast<uintptr_t>(qzeros) & 15u)) return W4A16_ERR_INVALID_ARG;  // NULL: symmetric
  if (g_idx && (reinterpret_cast<uintptr_t>(g_idx) & 15u)) return W4A16_ERR_INVALID_ARG;
  const size_t need = w4a16_workspace_bytes(M, N, K);
  if (need > (size_t)W4A16_NOALLOC_SCRATCH_BYTES) return W4A16_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return W4A16_ERR_CUDA;
  // tickets of the column blocks this shape uses must start at zero
  const size_t tickets = (size_t)((N + w4a16::kGemvCols - 1) / w4a16::kGemvCols) * (w4a16::kGemvCols / 32) * sizeof(int);
  if (tickets > w4a16::kCountersBytes) return W4A16_ERR_INVALID_ARG;
  if (cudaMemsetAsync(scratch, 0, tickets, stream) != cudaSuccess) return W4A16_ERR_CUDA;
  return w4a16_gemv(X, qweight, scales, qzeros, g_idx, Y, M, N, K, group_size, dtype, scratch,
                    (size_t)W4A16_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
