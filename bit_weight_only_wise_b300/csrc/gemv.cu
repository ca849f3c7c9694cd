// Split-K weight-streaming kernel for act-order decode shapes (1 <= M <= 16,
// g_idx as stored: every K row may belong to a different group) with more
// groups than the warp-specialized kernel's shared-memory table holds (that
// kernel, gemv_ws.cu, serves every other decode format).  Each packed word
// needs the (scale, zero) of eight different groups, gathered here from
// global memory per row.  For speed, prepack act-order checkpoints once
// (act_order.cu) and use the plain kernels.
//
// Y[M,N] = X[M,K] . W_hat[K,N] ("GPTQ与bitsandbytes对比：谁是2024年大模型量化的终极选择？",
// GPTQ section, --act-order).
//
// Work split (stream-K).  The work is cut into units of 256 output columns x
// one 128-row K group (16 KB of packed weights).  A persistent grid of
// 148 x (2 to 3) CTAs takes contiguous, equal-sized ranges of the units in
// column-block-major order, so every SM streams the same number of bytes
// whatever the shape.  Inside a CTA each of the 8 warps owns a 32-column slice
// of the unit and runs its own TMA ring: lane 0 keeps 2 2-KB tiles
// (16 word-rows x 32 columns, 128-byte swizzle) in flight into the warp's
// shared-memory stages, signalled by per-stage mbarriers.
//
// Inner product.  Lane (g = lane/4, c = lane%4) reads, per unit, four 16-byte
// vectors (columns [4g, 4g+4) of word-rows 2c, 2c+8, 2c+1, 2c+9 -- an order
// that makes the swizzled reads bank-conflict free), dequantizes them in
// registers to exact fp16/bf16 pairs and feeds them to m16n8k16 tensor-core
// MMAs as the A operand, the output columns being the MMA's M dimension and
// the (up to 16) tokens its N dimension (fp32 accumulation).
//
// Reduction: the deterministic split-K write-out of gemv_common.cuh.
#include <cuda.h>

#include "dq_common.cuh"
#include "gemv_common.cuh"
#include "sm100.cuh"
#include "tma_host.h"
#include "w4a16_internal.h"

namespace w4a16 {

using namespace sm100;

namespace {


constexpr int kWarps = kGemvThreads / 32;  // 8 column slices per CTA
constexpr int kTileBytes = 16 * 32 * 4;    // 16 word-rows x 32 columns
// the unit's activations ride in the same stage: 8 tokens per tile x 128 rows
template <int NT>
constexpr int x_tile_bytes() { return NT * 8 * 128 * 2; }
template <int NT>
constexpr int stage_bytes() { return kTileBytes + x_tile_bytes<NT>(); }
// TMA stages per warp.  Measured on B300: streaming 2-KB boxes runs at ~82%
// of the copy bandwidth with about 48 copies outstanding per SM (3 CTAs x 8
// warps x 2, or 2 x 8 x 3); twice as many outstanding copies halve the rate.
template <int NT>
constexpr int ring_depth() { return 2; }
template <int NT>
constexpr int gemv_smem() { return 1024 + kWarps * ring_depth<NT>() * stage_bytes<NT>(); }
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------- dequantizers
// fetch(): raw constants of a unit, one unit ahead; begin(): turn them into
// the current unit's constants; word(): dequantize the word of column
// col0 + c4 at step o into 4 pairs (rows (j, j+4) of that word-row).
template <int FMT, bool BF16>
struct Dq;

template <bool BF16>
struct Dq<kInt4Act, BF16> {
  uint32_t* tab;
  __device__ __forceinline__ void fetch(const GemvArgs&, int, int, int) {}
  __device__ __forceinline__ void publish(int) {}
  __device__ __forceinline__ void begin(int) {}
  // every row of the word-row sits in its own group
  __device__ __forceinline__ void word(const GemvArgs& a, int, uint32_t w, int c4, int row0, int col0, bool ok,
                                       uint32_t out[4]) {
    uint32_t z[8], s[8];
    if (ok) {
      const int4 g0 = __ldg(reinterpret_cast<const int4*>(a.g_idx + row0));
      const int4 g1 = __ldg(reinterpret_cast<const int4*>(a.g_idx + row0 + 4));
      const int gr[8] = {checked_group(g0.x, a.NG, a.dev_status), checked_group(g0.y, a.NG, a.dev_status),
                         checked_group(g0.z, a.NG, a.dev_status), checked_group(g0.w, a.NG, a.dev_status),
                         checked_group(g1.x, a.NG, a.dev_status), checked_group(g1.y, a.NG, a.dev_status),
                         checked_group(g1.z, a.NG, a.dev_status), checked_group(g1.w, a.NG, a.dev_status)};
      const int col = col0 + c4;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        s[r] = __ldg(a.scales + (size_t)gr[r] * a.N + col);
        // symmetric weights (no zero points): every zero point is 8
        z[r] = a.qz ? (__ldg(a.qz + (size_t)gr[r] * (a.N >> 3) + (col >> 3)) >> (4 * (col & 7))) & 0xFu : 8u;
      }
    } else {
#pragma unroll
      for (int r = 0; r < 8; ++r) s[r] = z[r] = 0;
    }
    if (BF16) {
      DqConstBF16 k[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) k[j] = dq_const_bf16_2(z[j], s[j], z[j + 4], s[j + 4]);
      dq_word_bf16_rows(w, k, out);
    } else {
      DqConstF16 k[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) k[j] = dq_const_f16_2(z[j], s[j], z[j + 4], s[j + 4]);
      dq_word_f16_rows(w, k, out);
    }
  }
};

template <int NT, int FMT, bool BF16>
__global__ void __launch_bounds__(kGemvThreads, gemv_ctas_per_sm(NT == 1 ? 1 : 16, FMT))
    gemv_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const GemvArgs a) {
  constexpr int kRing = ring_depth<NT>();
  constexpr int kStage = stage_bytes<NT>();
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kWarps][kRing];
  __shared__ __align__(16) uint32_t s_tab[kWarps][2 * 96];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int gl = lane >> 2, c = lane & 3;
  uint8_t* ring = smem + warp * (kRing * kStage);
  uint64_t* bar = full[warp];
  volatile int abort_flag = 0;  // per-warp pipeline: nobody else raises it

  const Range R{(long long)a.blocks_n * a.KB, (int)gridDim.x};
  const int cta = blockIdx.x;
  const long long u0 = R.start(cta);
  const int nu = (int)(R.start(cta + 1) - u0);
  const int first_block = (int)(u0 / a.KB);

  Dq<FMT, BF16> dq;
  dq.tab = s_tab[warp];
  if (lane == 0) {
    for (int s = 0; s < kRing; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // lane 0 streams this warp's slice of the CTA's units, kRing ahead: (tx, ty)
  // is the TMA coordinate of the next unit to copy, is_ its stage
  int tx = first_block * kGemvCols + warp * 32, ty = (int)(u0 % a.KB) * 16, is_ = 0;
  const int ty_end = a.KB * 16;
  auto advance = [&]() {
    is_ = (is_ + 1 == kRing) ? 0 : is_ + 1;
    ty += 16;
    if (ty == ty_end) {
      ty = 0;
      tx += kGemvCols;
    }
  };
  auto issue = [&]() {
    mbar_arrive_expect_tx(&bar[is_], kStage);
    tma_load_2d(ring + is_ * kStage, &tmW, &bar[is_], tx, ty);
    tma_load_2d(ring + is_ * kStage + kTileBytes, &tmX, &bar[is_], ty * 8, 0);
    advance();
  };
  // Nothing the caller owns is read into shared memory before griddep_wait
  // (the kernel before this one may still be writing it); until then the
  // first stages' weights are only prefetched into L2.
  const int n_first = nu < kRing ? nu : kRing;
  if (lane == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
    int px = tx, py = ty;
    for (int k = 0; k < n_first; ++k) {
      tma_prefetch_l2_2d(&tmW, px, py);
      py += 16;
      if (py == ty_end) {
        py = 0;
        px += kGemvCols;
      }
    }
  }
  griddep_wait();
  if (lane == 0)
    for (int k = 0; k < n_first; ++k) issue();
  griddep_launch_dependents();

  float acc[NT][2][4];
  auto zero_acc = [&]() {
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][r][i] = 0.f;
  };
  zero_acc();

  int p0 = -1, p1 = -1;  // split blocks whose tickets are still to be taken
  auto flush = [&](int b) {
    if (store_block<NT, BF16, false>(a, R, cta, first_block, warp, lane, b, acc)) (b == first_block ? p0 : p1) = b;
  };

  // lane-invariant parts of the shared-memory and activation addresses
  uint32_t lds_off[4];
  int xrow[4];
#pragma unroll
  for (int o = 0; o < 4; ++o) {
    const int r = tile_row(c, o);
    lds_off[o] = (uint32_t)(r * 128 + ((gl ^ (r & 7)) << 4));
    xrow[o] = 8 * r;
  }
  // this lane's activations in a stage: token 8t + gl, rows 8r .. 8r + 7
  const uint32_t x_lane = (uint32_t)(kTileBytes + gl * 256);
  const uint32_t ring_s = smem_u32(ring);

  int cur_b = -1;
  int b = first_block, g = (int)(u0 % a.KB);  // current unit
  int s = 0;
  uint32_t phase = 0;
  if (nu > 0) dq.fetch(a, g, b * kGemvCols + warp * 32, lane);
#pragma unroll 1
  for (int k = 0; k < nu; ++k) {
    if (b != cur_b) {
      if (cur_b >= 0) {
        flush(cur_b);
        zero_acc();
      }
      cur_b = b;
    }
    const int col0 = b * kGemvCols + warp * 32 + 4 * gl;
    const bool ok = col0 < a.N;
    dq.publish(lane);
    __syncwarp();
    dq.begin(gl);
    int bn = b, gn = g + 1;  // next unit
    if (gn == a.KB) {
      gn = 0;
      ++bn;
    }
    if (k + 1 < nu) dq.fetch(a, gn, bn * kGemvCols + warp * 32, lane);  // its constants, early
    if (!mbar_wait(&bar[s], phase, &abort_flag, a.dev_status, kWaitLimitNs)) {
      // let this warp's copies in flight land before its shared memory goes away
      for (int kk = k, ss = s, ph = phase; kk < k + kRing && kk < nu; ++kk) {
        (void)mbar_drain(&bar[ss], ph, kWaitLimitNs);
        if (++ss == kRing) {
          ss = 0;
          ph ^= 1;
        }
      }
      return;
    }
    const uint32_t st = ring_s + (uint32_t)(s * kStage);
    // read the whole stage first and hand it back to the TMA right away, so
    // the next copy overlaps this unit's arithmetic
    uint4 wvs[4], xvs[NT][4];
#pragma unroll
    for (int o = 0; o < 4; ++o) {
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(wvs[o].x), "=r"(wvs[o].y), "=r"(wvs[o].z), "=r"(wvs[o].w)
                   : "r"(st + lds_off[o]));
#pragma unroll
      for (int t = 0; t < NT; ++t)  // zero beyond M and K: the copy fills out-of-range elements with 0
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(xvs[t][o].x), "=r"(xvs[t][o].y), "=r"(xvs[t][o].z), "=r"(xvs[t][o].w)
                     : "r"(st + x_lane + (uint32_t)(t * 8 * 256 + 2 * xrow[o])));
    }
    __syncwarp();
    if (lane == 0 && k + kRing < nu) {
      fence_proxy_async_smem();  // the warp's reads of this stage precede the next copy into it
      issue();
    }
#pragma unroll
    for (int o = 0; o < 4; ++o) {
      const uint4 wv = wvs[o];
      const int row0 = g * 128 + xrow[o];
      uint32_t bf[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) x_pairs(xvs[t][o], bf[t]);
      const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        uint32_t pa[4], pb[4];
        dq.word(a, o, ws[2 * rr], 2 * rr, row0, col0, ok, pa);
        dq.word(a, o, ws[2 * rr + 1], 2 * rr + 1, row0, col0, ok, pb);
        const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
        const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          mma_16816<BF16>(acc[t][rr], a0, bf[t][0], bf[t][1]);
          mma_16816<BF16>(acc[t][rr], a1, bf[t][2], bf[t][3]);
        }
      }
    }
    if (++s == kRing) {
      s = 0;
      phase ^= 1;
    }
    b = bn;
    g = gn;
  }
  if (cur_b >= 0) flush(cur_b);
  finish_blocks<NT, BF16, false>(a, R, warp, lane, p0, p1);
}

template <int NT, int FMT, bool BF16>
cudaError_t launch_one(const CUtensorMap& tm, const GemvArgs& a, cudaStream_t st) {
  auto enc = tensor_map_encoder();
  CUtensorMap tx;  // X [M, K], boxes of 128 rows x 8*NT tokens
  cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
  cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
  cuuint32_t box[2] = {128, (cuuint32_t)(8 * NT)};
  cuuint32_t estr[2] = {1, 1};
  if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(a.X), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> attr_done{0};
  unsigned long long dev_bit = 0;
  if (attrs_pending(attr_done, &dev_bit)) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NT, FMT, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         gemv_smem<NT>());
    if (e != cudaSuccess) return e;
    // as much shared memory as the SM has, so that the intended number of
    // CTAs fits next to each other
    e = cudaFuncSetAttribute(gemv_kernel<NT, FMT, BF16>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(dev_bit, std::memory_order_release);
  }
  // programmatic dependent launch: this grid may start while the previous
  // kernel on the stream finishes (it waits for it before touching its data)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.ctas);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = gemv_smem<NT>();
  cfg.stream = st;
  cudaLaunchAttribute attr_pdl[1];
  attr_pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr_pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr_pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<NT, FMT, BF16>, tm, tx, a);
}

template <int FMT>
cudaError_t launch_gemv(const GemvArgs& a, bool bf16, cudaStream_t st) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tm;
  cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)(a.K / 8)};
  cuuint64_t strides[1] = {(cuuint64_t)a.N * 4};
  cuuint32_t box[2] = {32, 16};
  cuuint32_t estr[2] = {1, 1};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(a.qw), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (a.M <= 8) return bf16 ? launch_one<1, FMT, true>(tm, a, st) : launch_one<1, FMT, false>(tm, a, st);
  return bf16 ? launch_one<2, FMT, true>(tm, a, st) : launch_one<2, FMT, false>(tm, a, st);
}

}  // namespace

cudaError_t launch_gemv_int4(const GemvArgs& a, bool bf16, cudaStream_t st) {
  // grouped weights: the warp-specialized kernel (gemv_ws.cu); act-order: the
  // same kernel with its shared-memory table when every group fits, else this
  // one (global-memory lookups)
  if (!a.g_idx) return launch_gemv_ws_int4(a, bf16, st);
  return gemv_ws_act_fits(a.NG) ? launch_gemv_ws_act(a, bf16, st) : launch_gemv<kInt4Act>(a, bf16, st);
}

// NF4 runs on the warp-specialized kernel as well (gemv_ws.cu)
cudaError_t launch_gemv_nf4(const GemvArgs& a, bool bf16, cudaStream_t st) { return launch_gemv_ws_nf4(a, bf16, st); }

GemvPlan gemv_plan(int M, int N, int K, int fmt) {
  GemvPlan p{};
  p.blocks_n = (N + kGemvCols - 1) / kGemvCols;
  p.KB = (K + 127) / 128;
  const long long U = (long long)p.blocks_n * p.KB;
  // at least kMinUnits units (64 KB of weights) per CTA: below that the
  // per-CTA start-up and the split reduction cost more than the bytes
  constexpr long long kMinUnits = 4;
  long long target = kNumSMs * gemv_ctas_per_sm(M, fmt);
  const long long cap = U / kMinUnits > 0 ? U / kMinUnits : 1;
  if (target > cap) target = cap;
  p.ctas = (int)target;
  // sized for the largest grid any format may use, so one size serves all
  if (M > 0 && N > 0 && K > 0)
    p.workspace_bytes =
        kCountersBytes + (size_t)kNumSMs * kGemvMaxCTAsPerSM * 2 * kWarps * (size_t)M * 32 * sizeof(float);
  return p;
}

}  // namespace w4a16
