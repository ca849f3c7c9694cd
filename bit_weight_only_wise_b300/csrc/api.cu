// C ABI: argument validation and dispatch (see include/w4a16.h).
//
// Every entry point validates its arguments on the host and returns
// W4A16_ERR_INVALID_ARG / W4A16_ERR_UNSUPPORTED without launching anything
// when they are wrong; otherwise it enqueues its kernel(s) on the caller's
// stream and returns the launch status.
#include "w4a16.h"

#include <cstdint>

#include "w4a16_internal.h"

using namespace w4a16;

namespace {

constexpr int kNF4Block = 64;
static_assert(W4A16_MAX_K == 65535 * 8, "word-rows index a grid dimension");
static_assert(W4A16_MAX_N == kMaxColBlocks * kGemvCols, "one split-K ticket slice per column block");
// token tiles of the tensor-core kernel (up to 128 tokens with act-order)
// index a grid dimension; tiles = column tiles x token tiles then fits int
static_assert(W4A16_MAX_M == 65535 * 128, "token tiles index a grid dimension");

bool in_limits(int M, int N, int K) { return M <= W4A16_MAX_M && N <= W4A16_MAX_N && K <= W4A16_MAX_K; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }
bool ok_dtype(w4a16_dtype d) { return d == W4A16_F16 || d == W4A16_BF16; }
size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

w4a16_status from_cuda(cudaError_t e) { return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA; }

// Shape checks common to the INT4 entry points.  Returns OK, or the error.
w4a16_status check_int4_shape(int M, int N, int K, int group_size) {
  if (M < 0 || N < 0 || K <= 0 || !in_limits(M, N, K)) return W4A16_ERR_INVALID_ARG;
  if (N % 8 || K % 8) return W4A16_ERR_INVALID_ARG;
  if (group_size <= 0 || K % group_size) return W4A16_ERR_INVALID_ARG;
  if (!int4_group_supported(K, group_size)) return W4A16_ERR_UNSUPPORTED;
  return W4A16_OK;
}

w4a16_status check_nf4_shape(int M, int N, int K, int blocksize) {
  if (M < 0 || N < 0 || K <= 0 || !in_limits(M, N, K)) return W4A16_ERR_INVALID_ARG;
  if (N % 8 || K % 8) return W4A16_ERR_INVALID_ARG;
  if (blocksize <= 0 || K % blocksize) return W4A16_ERR_INVALID_ARG;
  if (blocksize != kNF4Block) return W4A16_ERR_UNSUPPORTED;
  return W4A16_OK;
}

w4a16_status check_gemm_workspace(const GemmSplit& sp, void* ws, size_t ws_bytes) {
  if (sp.workspace_bytes == 0) return W4A16_OK;
  if (!ok_ptr(ws) || ws_bytes < sp.workspace_bytes) return W4A16_ERR_INVALID_ARG;
  return W4A16_OK;
}

w4a16_status check_workspace(const GemvPlan& p, void* ws, size_t ws_bytes) {
  if (p.workspace_bytes == 0) return W4A16_OK;
  if (!ok_ptr(ws) || ws_bytes < p.workspace_bytes) return W4A16_ERR_INVALID_ARG;
  return W4A16_OK;
}

GemvArgs gemv_args(const void* X, const uint32_t* qw, void* Y, int M, int N, int K, const GemvPlan& p,
                   void* ws, int* dev_status) {
  GemvArgs a{};
  a.X = static_cast<const uint16_t*>(X);
  a.qw = qw;
  a.Y = static_cast<uint16_t*>(Y);
  a.dev_status = dev_status;
  a.M = M;
  a.N = N;
  a.K = K;
  a.KB = p.KB;
  a.blocks_n = p.blocks_n;
  // the plain product: 256-column blocks (the fused SiLU entry overrides these)
  a.cpb = kGemvCols;
  a.hiofs = a.hi2 = kGemvCols / 2;
  a.Nout = a.ldy = N;
  a.ctas = p.ctas;
  a.counters = static_cast<int*>(ws);
  a.partial = reinterpret_cast<float*>(static_cast<char*>(ws) + kCountersBytes);
  return a;
}

w4a16_status int4_gemv_impl(const void* X, const uint32_t* qweight, const void* scales, const uint32_t* qzeros,
                            const int32_t* g_idx, void* Y, int M, int N, int K, int group_size, w4a16_dtype dtype,
                            void* workspace, size_t workspace_bytes, int* dev_status, cudaStream_t stream,
                            bool silu = false) {
  const GemvPlan p = gemv_plan(M, N, K, g_idx ? kInt4Act : kInt4);
  w4a16_status st = check_workspace(p, workspace, workspace_bytes);
  if (st != W4A16_OK) return st;
  GemvArgs a = gemv_args(X, qweight, Y, M, N, K, p, workspace, dev_status);
  if (silu) {  // gate columns [0, F), up columns [F, 2F): 128 output columns per block
    a.silu = 1;
    a.cpb = kGemvCols / 2;
    a.hiofs = N / 2;
    a.hi2 = 0;
    a.Nout = a.ldy = N / 2;
  }
  a.scales = static_cast<const uint16_t*>(scales);
  a.qz = qzeros;
  a.g_idx = g_idx;
  a.gsize = group_size;
  a.NG = K / group_size;
  return from_cuda(launch_gemv_int4(a, dtype == W4A16_BF16, stream));
}

// qzeros may be NULL: symmetric weights (every zero point 8)
w4a16_status check_int4_ptrs(const void* X, const uint32_t* qweight, const void* scales, const uint32_t* qzeros,
                             const int32_t* g_idx, const void* Y) {
  if (!ok_ptr(X) || !ok_ptr(qweight) || !ok_ptr(scales) || !ok_ptr(Y)) return W4A16_ERR_INVALID_ARG;
  if ((qzeros && !aligned16(qzeros)) || (g_idx && !aligned16(g_idx))) return W4A16_ERR_INVALID_ARG;
  return W4A16_OK;
}

// w4a16_gemv's checks before anything launches; *empty: a valid call with
// nothing to compute (M or N zero)
w4a16_status gemv_check(const void* X, const uint32_t* qweight, const void* scales, const uint32_t* qzeros,
                        const int32_t* g_idx, const void* Y, int M, int N, int K, int group_size,
                        w4a16_dtype dtype, bool* empty) {
  *empty = false;
  if (!ok_dtype(dtype)) return W4A16_ERR_INVALID_ARG;
  w4a16_status st = check_int4_shape(M, N, K, group_size);
  if (st != W4A16_OK) return st;
  if (M > W4A16_GEMV_MAX_M) return W4A16_ERR_INVALID_ARG;
  if (M == 0 || N == 0) {
    *empty = true;
    return W4A16_OK;
  }
  return check_int4_ptrs(X, qweight, scales, qzeros, g_idx, Y);
}

}  // namespace

extern "C" {

w4a16_status w4a16_gemv(const void* X, const uint32_t* qweight, const void* scales, const uint32_t* qzeros,
                        const int32_t* g_idx, void* Y, int M, int N, int K, int group_size, w4a16_dtype dtype,
                        void* workspace, size_t workspace_bytes, int* dev_status, cudaStream_t stream) {
  bool empty = false;
  const w4a16_status st = gemv_check(X, qweight, scales, qzeros, g_idx, Y, M, N, K, group_size, dtype, &empty);
  if (st != W4A16_OK || empty) return st;
  return int4_gemv_impl(X, qweight, scales, qzeros, g_idx, Y, M, N, K, group_size, dtype, workspace,
                        workspace_bytes, dev_status, stream);
}

w4a16_status w4a16_gemv_batch(const w4a16_gemv_item* items, int count, void* workspace, size_t workspace_bytes,
                              int* dev_status, cudaStream_t stream) {
  if (count < 0 || (count > 0 && items == nullptr)) return W4A16_ERR_INVALID_ARG;
  // every item is checked before the first launch
  for (int i = 0; i < count; ++i) {
    const w4a16_gemv_item& it = items[i];
    bool empty = false;
    w4a16_status st = gemv_check(it.X, it.qweight, it.scales, it.qzeros, it.g_idx, it.Y, it.M, it.N, it.K,
                                 it.group_size, it.dtype, &empty);
    if (st != W4A16_OK) return st;
    if (empty) continue;
    st = check_workspace(gemv_plan(it.M, it.N, it.K, it.g_idx ? kInt4Act : kInt4), workspace, workspace_bytes);
    if (st != W4A16_OK) return st;
  }
  for (int i = 0; i < count; ++i) {
    const w4a16_gemv_item& it = items[i];
    if (it.M == 0 || it.N == 0) continue;
    const w4a16_status st = int4_gemv_impl(it.X, it.qweight, it.scales, it.qzeros, it.g_idx, it.Y, it.M, it.N, it.K,
                                           it.group_size, it.dtype, workspace, workspace_bytes, dev_status, stream);
    if (st != W4A16_OK) return st;
  }
  return W4A16_OK;
}

w4a16_status w4a16_gemm(const void* X, const uint32_t* qweight, const void* scales, const uint32_t* qzeros,
                        const int32_t* g_idx, void* Y, int M, int N, int K, int group_size, w4a16_dtype dtype,
                        void* workspace, size_t workspace_bytes, int* dev_status, cudaStream_t stream) {
  if (!ok_dtype(dtype)) return W4A16_ERR_INVALID_ARG;
  w4a16_status st = check_int4_shape(M, N, K, group_size);
  if (st != W4A16_OK) return st;
  if (M == 0 || N == 0) return W4A16_OK;
  st = check_int4_ptrs(X, qweight, scales, qzeros, g_idx, Y);
  if (st != W4A16_OK) return st;
  if (M <= W4A16_GEMV_MAX_M)
    return int4_gemv_impl(X, qweight, scales, qzeros, g_idx, Y, M, N, K, group_size, dtype, workspace,
                          workspace_bytes, dev_status, stream);
  if (g_idx && !gemm_act_order_fits(K / group_size)) return W4A16_ERR_UNSUPPORTED;
  st = check_gemm_workspace(gemm_split_plan(M, N, K, g_idx != nullptr), workspace, workspace_bytes);
  if (st != W4A16_OK) return st;
  GemmArgs a{};
  a.X = X;
  a.qw = qweight;
  a.scales = static_cast<const uint16_t*>(scales);
  a.qz = qzeros;
  a.g_idx = g_idx;
  a.Y = static_cast<uint16_t*>(Y);
  a.dev_status = dev_status;
  a.M = M;
  a.N = N;
  a.K = K;
  a.gsize = group_size;
  a.NG = K / group_size;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  return from_cuda(launch_gemm_tc(a, dtype == W4A16_BF16, false, stream));
}

}  // extern "C"

namespace {

// NF4 product with fp32 absmax (absmax_q == nullptr) or double-quantized
// absmax (absmax_q, absmax_s2); validation common to both entry points.
w4a16_status nf4_gemm_impl(const void* X, const uint32_t* qweight, const float* absmax, const uint8_t* absmax_q,
                           const float* absmax_s2, const float* codebook16, void* Y, int M, int N, int K,
                           int blocksize, w4a16_dtype dtype, void* workspace, size_t workspace_bytes,
                           int* dev_status, cudaStream_t stream) {
  if (!ok_dtype(dtype)) return W4A16_ERR_INVALID_ARG;
  w4a16_status st = check_nf4_shape(M, N, K, blocksize);
  if (st != W4A16_OK) return st;
  if (M == 0 || N == 0) return W4A16_OK;
  if (!ok_ptr(X) || !ok_ptr(qweight) || !ok_ptr(Y)) return W4A16_ERR_INVALID_ARG;
  if (absmax_q ? (!ok_ptr(absmax_q) || !ok_ptr(absmax_s2)) : !ok_ptr(absmax)) return W4A16_ERR_INVALID_ARG;
  if (codebook16 && !aligned16(codebook16)) return W4A16_ERR_INVALID_ARG;
  if (M <= W4A16_GEMV_MAX_M) {
    const GemvPlan p = gemv_plan(M, N, K, kNF4);
    st = check_workspace(p, workspace, workspace_bytes);
    if (st != W4A16_OK) return st;
    GemvArgs a = gemv_args(X, qweight, Y, M, N, K, p, workspace, dev_status);
    a.absmax = absmax;
    a.absmax_q = absmax_q;
    a.absmax_s2 = absmax_s2;
    a.codebook = codebook16;
    a.cb_builtin = nf4_builtin_codebook();
    return from_cuda(launch_gemv_nf4(a, dtype == W4A16_BF16, stream));
  }
  st = check_gemm_workspace(gemm_split_plan(M, N, K, false), workspace, workspace_bytes);
  if (st != W4A16_OK) return st;
  GemmArgs a{};
  a.X = X;
  a.qw = qweight;
  a.absmax = absmax;
  a.absmax_q = absmax_q;
  a.absmax_s2 = absmax_s2;
  a.codebook = codebook16;
  a.cb_builtin = nf4_builtin_codebook();
  a.Y = static_cast<uint16_t*>(Y);
  a.dev_status = dev_status;
  a.M = M;
  a.N = N;
  a.K = K;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  return from_cuda(launch_gemm_tc(a, dtype == W4A16_BF16, true, stream));
}

}  // namespace

extern "C" {

w4a16_status w4a16_gemm_silu_mul(const void* X, const uint32_t* qweight, const void* scales,
                                 const uint32_t* qzeros, void* A, int M, int N, int K, int group_size,
                                 w4a16_dtype dtype, void* workspace, size_t workspace_bytes, int* dev_status,
                                 cudaStream_t stream) {
  if (!ok_dtype(dtype)) return W4A16_ERR_INVALID_ARG;
  w4a16_status st = check_int4_shape(M, N, K, group_size);
  if (st != W4A16_OK) return st;
  if (N % 16) return W4A16_ERR_INVALID_ARG;  // F = N / 2 a multiple of 8
  if (M == 0 || N == 0) return W4A16_OK;
  st = check_int4_ptrs(X, qweight, scales, qzeros, nullptr, A);
  if (st != W4A16_OK) return st;
  if (M <= W4A16_GEMV_MAX_M)
    return int4_gemv_impl(X, qweight, scales, qzeros, nullptr, A, M, N, K, group_size, dtype, workspace,
                          workspace_bytes, dev_status, stream, true);
  st = check_gemm_workspace(gemm_split_plan(M, N, K, false), workspace, workspace_bytes);
  if (st != W4A16_OK) return st;
  GemmArgs a{};
  a.X = X;
  a.qw = qweight;
  a.scales = static_cast<const uint16_t*>(scales);
  a.qz = qzeros;
  a.Y = static_cast<uint16_t*>(A);
  a.dev_status = dev_status;
  a.M = M;
  a.N = N;
  a.K = K;
  a.gsize = group_size;
  a.NG = K / group_size;
  a.silu = 1;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  return from_cuda(launch_gemm_tc(a, dtype == W4A16_BF16, false, stream));
}

w4a16_status nf4_gemm(const void* X, const uint32_t* qweight, const float* absmax, const float* codebook16,
                      void* Y, int M, int N, int K, int blocksize, w4a16_dtype dtype, void* workspace,
                      size_t workspace_bytes, int* dev_status, cudaStream_t stream) {
  return nf4_gemm_impl(X, qweight, absmax, nullptr, nullptr, codebook16, Y, M, N, K, blocksize, dtype, workspace,
                       workspace_bytes, dev_status, stream);
}

w4a16_status nf4dq_gemm(const void* X, const uint32_t* qweight, const uint8_t* absmax_q, const float* absmax_s2,
                        const float* codebook16, void* Y, int M, int N, int K, int blocksize, w4a16_dtype dtype,
                        void* workspace, size_t workspace_bytes, int* dev_status, cudaStream_t stream) {
  if (!absmax_q) return W4A16_ERR_INVALID_ARG;
  return nf4_gemm_impl(X, qweight, nullptr, absmax_q, absmax_s2, codebook16, Y, M, N, K, blocksize, dtype,
                       workspace, workspace_bytes, dev_status, stream);
}

w4a16_status nf4_double_quantize(const float* absmax, int K, int N, int blocksize, uint8_t* absmax_q,
                                 float* absmax_s2, cudaStream_t stream) {
  w4a16_status st = check_nf4_shape(0, N, K, blocksize);
  if (st != W4A16_OK) return st;
  if (N == 0) return W4A16_OK;
  if (!ok_ptr(absmax) || !ok_ptr(absmax_q) || !ok_ptr(absmax_s2)) return W4A16_ERR_INVALID_ARG;
  return from_cuda(launch_double_quantize(absmax, K / blocksize, N, absmax_q, absmax_s2, stream));
}

w4a16_status nf4dq_dequant(const uint32_t* qweight, const uint8_t* absmax_q, const float* absmax_s2,
                           const float* codebook16, void* W_out, int K, int N, int blocksize, w4a16_dtype dtype,
                           cudaStream_t stream) {
  if (!ok_dtype(dtype)) return W4A16_ERR_INVALID_ARG;
  w4a16_status st = check_nf4_shape(0, N, K, blocksize);
  if (st != W4A16_OK) return st;
  if (N == 0) return W4A16_OK;
  if (!ok_ptr(qweight) || !ok_ptr(absmax_q) || !ok_ptr(absmax_s2) || !ok_ptr(W_out)) return W4A16_ERR_INVALID_ARG;
  if (codebook16 && !aligned16(codebook16)) return W4A16_ERR_INVALID_ARG;
  return from_cuda(launch_dequant_nf4dq(qweight, absmax_q, absmax_s2, codebook16, static_cast<uint16_t*>(W_out), K,
                                        N, blocksize, dtype == W4A16_BF16, stream));
}

w4a16_status w4a16_dequant(const uint32_t* qweight, const void* scales, const uint32_t* qzeros,
                           const int32_t* g_idx, void* W_out, int K, int N, int group_size, w4a16_dtype dtype,
                           cudaStream_t stream) {
  if (!ok_dtype(dtype)) return W4A16_ERR_INVALID_ARG;
  w4a16_status st = check_int4_shape(0, N, K, group_size);
  if (st != W4A16_OK) return st;
  if (N == 0) return W4A16_OK;
  if (!ok_ptr(qweight) || !ok_ptr(scales) || !ok_ptr(W_out)) return W4A16_ERR_INVALID_ARG;
  if ((qzeros && !aligned16(qzeros)) || (g_idx && !aligned16(g_idx))) return W4A16_ERR_INVALID_ARG;
  return from_cuda(launch_dequant_int4(qweight, static_cast<const uint16_t*>(scales), qzeros, g_idx,
                                       static_cast<uint16_t*>(W_out), K, N, group_size, dtype == W4A16_BF16,
                                       stream));
}

w4a16_status nf4_dequant(const uint32_t* qweight, const float* absmax, const float* codebook16, void* W_out, int K,
                         int N, int blocksize, w4a16_dtype dtype, cudaStream_t stream) {
  if (!ok_dtype(dtype)) return W4A16_ERR_INVALID_ARG;
  w4a16_status st = check_nf4_shape(0, N, K, blocksize);
  if (st != W4A16_OK) return st;
  if (N == 0) return W4A16_OK;
  if (!ok_ptr(qweight) || !ok_ptr(absmax) || !ok_ptr(W_out)) return W4A16_ERR_INVALID_ARG;
  if (codebook16 && !aligned16(codebook16)) return W4A16_ERR_INVALID_ARG;
  return from_cuda(launch_dequant_nf4(qweight, absmax, codebook16, static_cast<uint16_t*>(W_out), K, N, blocksize,
                                      dtype == W4A16_BF16, stream));
}

w4a16_status w4a16_quantize(const float* W, int K, int N, int group_size, uint32_t* qweight, void* scales,
                            uint32_t* qzeros, cudaStream_t stream) {
  w4a16_status st = check_int4_shape(0, N, K, group_size);
  if (st != W4A16_OK) return st;
  if (N == 0) return W4A16_OK;
  // qzeros NULL: symmetric quantization (no zero points stored)
  if (!ok_ptr(W) || !ok_ptr(qweight) || !ok_ptr(scales) || (qzeros && !aligned16(qzeros)))
    return W4A16_ERR_INVALID_ARG;
  return from_cuda(
      launch_quantize_rtn(W, K, N, group_size, qweight, static_cast<uint16_t*>(scales), qzeros, stream));
}

w4a16_status nf4_quantize(const float* W, int K, int N, int blocksize, const float* codebook16, uint32_t* qweight,
                          float* absmax, cudaStream_t stream) {
  w4a16_status st = check_nf4_shape(0, N, K, blocksize);
  if (st != W4A16_OK) return st;
  if (N == 0) return W4A16_OK;
  if (!ok_ptr(W) || !ok_ptr(qweight) || !ok_ptr(absmax)) return W4A16_ERR_INVALID_ARG;
  if (codebook16 && !aligned16(codebook16)) return W4A16_ERR_INVALID_ARG;
  return from_cuda(launch_quantize_nf4(W, K, N, blocksize, codebook16, qweight, absmax, stream));
}

size_t w4a16_workspace_bytes(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0 || !in_limits(M, N, K)) return 0;
  if (M <= W4A16_GEMV_MAX_M) return gemv_plan(M, N, K, kInt4).workspace_bytes;
  // the tensor-core kernel's split-K tiles; act-order uses a smaller token tile
  const size_t a = gemm_split_plan(M, N, K, false).workspace_bytes;
  const size_t b = gemm_split_plan(M, N, K, true).workspace_bytes;
  return a > b ? a : b;
}

w4a16_status w4a16_act_order_prepack(const uint32_t* qweight, const int32_t* g_idx, int K, int N, int group_size,
                                     uint32_t* qweight_sorted, int32_t* perm, int* dev_status,
                                     cudaStream_t stream) {
  w4a16_status st = check_int4_shape(0, N, K, group_size);
  if (st != W4A16_OK) return st;
  if (N == 0) return W4A16_OK;
  if (!ok_ptr(qweight) || !ok_ptr(g_idx) || !ok_ptr(qweight_sorted) || !ok_ptr(perm)) return W4A16_ERR_INVALID_ARG;
  if (qweight_sorted == qweight) return W4A16_ERR_INVALID_ARG;  // rows are gathered: no in-place reorder
  return from_cuda(launch_act_order_prepack(qweight, g_idx, K, N, group_size, qweight_sorted, perm, dev_status,
                                            stream));
}

// [plain-kernel workspace, at least the ticket area | X with its columns in
// sorted order]: the ticket area stays in front whatever M is, so a buffer
// shared with the other entry points keeps its tickets
static size_t prepacked_front_bytes(int M, int N, int K) {
  const size_t plain = w4a16_workspace_bytes(M, N, K);
  return align256(plain > kCountersBytes ? plain : kCountersBytes);
}

size_t w4a16_prepacked_workspace_bytes(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0 || !in_limits(M, N, K)) return 0;
  return prepacked_front_bytes(M, N, K) + align256((size_t)M * K * 2);
}

w4a16_status w4a16_gemm_prepacked(const void* X, const uint32_t* qweight_sorted, const void* scales,
                                  const uint32_t* qzeros, const int32_t* perm, void* Y, int M, int N, int K,
                                  int group_size, w4a16_dtype dtype, void* workspace, size_t workspace_bytes,
                                  int* dev_status, cudaStream_t stream) {
  if (!ok_dtype(dtype)) return W4A16_ERR_INVALID_ARG;
  w4a16_status st = check_int4_shape(M, N, K, group_size);
  if (st != W4A16_OK) return st;
  if (M == 0 || N == 0) return W4A16_OK;
  st = check_int4_ptrs(X, qweight_sorted, scales, qzeros, nullptr, Y);
  if (st != W4A16_OK) return st;
  if (!ok_ptr(perm) || !ok_ptr(workspace) || workspace_bytes < w4a16_prepacked_workspace_bytes(M, N, K))
    return W4A16_ERR_INVALID_ARG;
  const size_t plain = w4a16_workspace_bytes(M, N, K);
  uint16_t* Xp = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + prepacked_front_bytes(M, N, K));
  cudaError_t e = launch_gather_columns(static_cast<const uint16_t*>(X), perm, M, K, Xp, stream);
  if (e != cudaSuccess) return W4A16_ERR_CUDA;
  return w4a16_gemm(Xp, qweight_sorted, scales, qzeros, nullptr, Y, M, N, K, group_size, dtype,
                    plain ? workspace : nullptr, plain, dev_status, stream);
}

w4a16_status w4a16_repack_awq(const uint32_t* qweight_awq, const uint32_t* qzeros_awq, int K, int N, int group_size,
                              uint32_t* qweight, uint32_t* qzeros, cudaStream_t stream) {
  w4a16_status st = check_int4_shape(0, N, K, group_size);
  if (st != W4A16_OK) return st;
  if (N == 0) return W4A16_OK;
  if (!ok_ptr(qweight_awq) || !ok_ptr(qweight)) return W4A16_ERR_INVALID_ARG;
  if (!qzeros_awq != !qzeros) return W4A16_ERR_INVALID_ARG;  // both or neither (symmetric)
  if (qzeros_awq && (!aligned16(qzeros_awq) || !aligned16(qzeros))) return W4A16_ERR_INVALID_ARG;
  if (qweight == qweight_awq || (qzeros && qzeros == qzeros_awq)) return W4A16_ERR_INVALID_ARG;  // not in place
  return from_cuda(launch_awq_repack(qweight_awq, qzeros_awq, K, N, K / group_size, qweight, qzeros, stream));
}

const char* w4a16_status_string(w4a16_status status) {
  switch (status) {
    case W4A16_OK: return "ok";
    case W4A16_ERR_INVALID_ARG: return "invalid argument (shape, pointer, alignment, dtype or workspace)";
    case W4A16_ERR_UNSUPPORTED: return "not supported by this library (group or block size, or shape)";
    case W4A16_ERR_CUDA: return "CUDA runtime or launch error";
    case W4A16_ERR_TIMEOUT: return "device-side bounded wait expired";
  }
  return "unknown status";
}

}  // extern "C"
