// Internal declarations shared by the library's translation units.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime_api.h>

namespace w4a16 {

// B300: 148 SMs.  The split-K plan is a pure function of the shape so that the
// workspace size can be computed on the host without a device query.
constexpr int kNumSMs = 148;

// A 16-entry NF4 table passed to kernels by value (used when the caller gives
// no table of its own).
struct Cb16 {
  float v[16];
};
// The library's built-in NF4 table (host; built once per process).
const Cb16& nf4_builtin_codebook();

// ----------------------------------------------------------- split-K GEMV
constexpr int kGemvThreads = 256;            // 8 warps, one 32-column slice each
constexpr int kGemvCols = 256;               // columns per unit
// kInt4: grouped scales and zero points (any supported group size, symmetric
// or not); kInt4Act: the same with an act-order map; kNF4: fp32 absmax;
// kNF4DQ: NF4 with double-quantized absmax (8-bit codes and a second-level
// fp32 scale)
enum GemvFmt { kInt4 = 0, kInt4Act = 1, kNF4 = 2, kNF4DQ = 3 };
// persistent grid: CTAs resident per SM, by token tiles (M <= 8: one tile of
// 8 tokens) and format (register and shared-memory budget of each variant)
constexpr int kGemvMaxCTAsPerSM = 3;
constexpr int gemv_ctas_per_sm(int M, int fmt) { return fmt != kInt4Act ? 2 : M <= 8 ? 3 : 2; }
// The workspace starts with a fixed-size area of split-K tickets (one int per
// 32-column slice) and the fp32 partial sums follow it.  The area's size does
// not depend on the shape, so partial sums of one call never land where a
// later call with another shape keeps its tickets.
constexpr int kMaxColBlocks = 4096;          // N <= 4096 * 256
constexpr size_t kCountersBytes = (size_t)kMaxColBlocks * (kGemvCols / 32) * sizeof(int);

struct GemvPlan {
  int blocks_n;  // 256-column blocks
  int KB;        // 128-row blocks along K (units per column block)
  int ctas;      // persistent grid size
  size_t workspace_bytes;
};

GemvPlan gemv_plan(int M, int N, int K, int fmt);

struct GemvArgs {
  const uint16_t* X;
  const uint32_t* qw;
  const uint16_t* scales;   // INT4: fp16 scales [NG, N]
  const uint32_t* qz;       // INT4 packed zeros [NG, N/8], or nullptr: symmetric (every zero point 8)
  const int32_t* g_idx;     // INT4 act-order map or nullptr
  const float* absmax;      // NF4: fp32 [K/64, N]
  const uint8_t* absmax_q;  // NF4 double quantization: 8-bit codes [K/64, N]
  const float* absmax_s2;   // NF4 double quantization: fp32 [K/64, ceil(N/256)]
  const float* codebook;    // NF4 table in device memory, or nullptr: cb_builtin
  Cb16 cb_builtin;          // NF4 table used when codebook is nullptr
  uint16_t* Y;
  float* partial;
  int* counters;
  int* dev_status;
  int M, N, K;
  int KB;          // 128-row blocks along K (units per column block)
  int NG;          // scale groups along K
  int gsize;       // rows per group (INT4)
  int kbpg;        // 128-row units per group (set by the launcher)
  int nwz;         // zero words per row to copy: N / 8, or 0 for symmetric weights (launcher)
  // Output columns.  Plain product: a column block is 256 output columns, the
  // unit's second half starting 128 columns on (cpb = 256, hiofs = hi2 = 128,
  // Nout = ldy = N).  Fused SiLU(gate) * up (silu = 1): the weight holds gate
  // columns [0, F) then up columns [F, 2F); a block is 128 output columns,
  // its unit the 128 gate columns then the 128 matching up columns (cpb =
  // 128, hiofs = F, hi2 = 0, Nout = ldy = F = N / 2).
  int silu;
  int cpb, hiofs, hi2, Nout, ldy;
  uint32_t zxor;   // 0, or 0x88888888 for symmetric weights: zero points of 8 (launcher)
  int blocks_n;    // 256-column blocks
  int ctas;
  int stages;      // pipeline depth (set by the launcher)
  int tab_stride;  // act-order: bytes per group in the shared-memory table (set by the launcher)
};

cudaError_t launch_gemv_int4(const GemvArgs& a, bool bf16, cudaStream_t st);
// the warp-specialized decode kernel: grouped INT4 (any supported group
// size, symmetric or not), act-order through a shared-memory table of the
// column block's scales and zeros (when it fits: gemv_ws_act_fits), NF4
cudaError_t launch_gemv_ws_int4(const GemvArgs& a, bool bf16, cudaStream_t st);
cudaError_t launch_gemv_ws_act(const GemvArgs& a, bool bf16, cudaStream_t st);
bool gemv_ws_act_fits(int NG);
cudaError_t launch_gemv_ws_nf4(const GemvArgs& a, bool bf16, cudaStream_t st);
cudaError_t launch_gemv_nf4(const GemvArgs& a, bool bf16, cudaStream_t st);
// Group sizes the decode kernel supports: 32 and 64 (several groups per
// 128-row unit), multiples of 128, and a single group (per-channel, g = K).
inline bool int4_group_supported(int K, int g) {
  return g == 32 || g == 64 || g % 128 == 0 || g == K;
}

// ------------------------------------------------------ tensor-core GEMM
struct GemmArgs {
  const void* X;
  const uint32_t* qw;
  const uint16_t* scales;  // INT4
  const uint32_t* qz;      // INT4, or nullptr: symmetric (every zero point 8)
  const int32_t* g_idx;    // INT4 act-order map or nullptr
  int gsize;               // INT4 rows per group
  int NG;                  // INT4 groups along K
  int silu;                // fused SiLU(gate) * up: Y [M, N/2] from gate [0, N/2) and up [N/2, N)
  const float* absmax;     // NF4
  const uint8_t* absmax_q; // NF4 double quantization: 8-bit codes [K/64, N], or nullptr
  const float* absmax_s2;  // NF4 double quantization: fp32 [K/64, ceil(N/256)]
  const float* codebook;   // NF4 table in device memory, or nullptr: cb_builtin
  Cb16 cb_builtin;
  uint16_t* Y;
  int* dev_status;
  int M, N, K;
  void* workspace;  // split-K tickets and partial tiles (see gemm_split_plan)
  size_t workspace_bytes;
};

// Tokens per CTA (the MMA's N) the tensor-core kernel uses for M tokens.
int gemm_tokens_per_cta(int M, bool act_order);
// Split-K plan of the tensor-core kernel for a shape (pure function).
struct GemmSplit {
  int BT;
  int tiles;
  int dp_tiles;  // tiles run whole, in full waves; the rest are split along K
  int splits;
  int kb_per_split;
  size_t workspace_bytes;  // 0 when not split
};
GemmSplit gemm_split_plan(int M, int N, int K, bool act_order);
// Whether the act-order variant's per-CTA (scale, zero) table fits for NG groups.
bool gemm_act_order_fits(int NG);
cudaError_t launch_gemm_tc(const GemmArgs& a, bool bf16, bool nf4, cudaStream_t st);

// ------------------------------------------------- per-device kernel setup
// cudaFuncSetAttribute acts on a kernel as loaded on the current device, so a
// launcher sets its kernel's attributes once per device: `done` keeps one bit
// per device index.  Returns whether they still have to be set here; *bit is
// the bit to record afterwards (0 past device 63: those set them every call).
inline bool attrs_pending(const std::atomic<unsigned long long>& done, unsigned long long* bit) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  *bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  return *bit == 0 || (done.load(std::memory_order_acquire) & *bit) == 0;
}

// ------------------------------------------------------ act-order prepack
cudaError_t launch_act_order_prepack(const uint32_t* qw, const int32_t* g_idx, int K, int N, int group_size,
                                     uint32_t* qw_sorted, int32_t* perm, int* dev_status, cudaStream_t st);
cudaError_t launch_gather_columns(const uint16_t* X, const int32_t* perm, int M, int K, uint16_t* out,
                                  cudaStream_t st);

// ------------------------------------------------------------ AWQ layout
cudaError_t launch_awq_repack(const uint32_t* qweight_awq, const uint32_t* qzeros_awq, int K, int N, int G,
                              uint32_t* qweight, uint32_t* qzeros, cudaStream_t st);

// ------------------------------------------------------- standalone kernels
cudaError_t launch_dequant_int4(const uint32_t* qw, const uint16_t* scales, const uint32_t* qz,
                                const int32_t* g_idx, uint16_t* out, int K, int N, int group_size,
                                bool bf16, cudaStream_t st);
// codebook: a device table, or nullptr for the built-in one
cudaError_t launch_dequant_nf4(const uint32_t* qw, const float* absmax, const float* codebook, uint16_t* out,
                               int K, int N, int blocksize, bool bf16, cudaStream_t st);
cudaError_t launch_dequant_nf4dq(const uint32_t* qw, const uint8_t* absmax_q, const float* absmax_s2,
                                 const float* codebook, uint16_t* out, int K, int N, int blocksize, bool bf16,
                                 cudaStream_t st);
cudaError_t launch_double_quantize(const float* absmax, int rows, int N, uint8_t* absmax_q, float* absmax_s2,
                                   cudaStream_t st);
cudaError_t launch_quantize_rtn(const float* W, int K, int N, int group_size, uint32_t* qw, uint16_t* scales,
                                uint32_t* qz, cudaStream_t st);
cudaError_t launch_quantize_nf4(const float* W, int K, int N, int blocksize, const float* codebook, uint32_t* qw,
                                float* absmax, cudaStream_t st);

}  // namespace w4a16
