// Warp-specialized split-K weight-streaming kernel for INT4 decode shapes
// (1 <= M <= 16, one scale and zero point per 128-row group, no act-order).
//
// At M <= 16 the product is bound by streaming the packed weights once
// ("LLM量化技术深度对比:GPTQ vs AWQ vs bitsandbytes 2026基准全解析", key-data
// item 3: a 4-bit forward moves a quarter of the FP16 bytes; item 1: the fused
// kernel that never writes 16-bit weights is the fast one).  What keeps such
// a kernel from the bandwidth is instruction issue: exact dequantization costs
// two packed 16-bit operations per pair of weights (fp16) or two fp32 FMAs and
// a conversion (bf16), so every other instruction per weight has to go.  The
// CTA is therefore split by role:
//
//   producer warp  streams each unit (256 columns x one 128-row group) into a
//                  shared-memory stage: eight 2-KB weight boxes (16 word-rows
//                  x 32 columns, 128-byte swizzle) and the activation box by
//                  TMA, the unit's 256 scales and 32 zero words by cp.async,
//                  all completing on the stage's `full` barrier;
//   helper warp    turns the raw scales and zeros into the packed per-column
//                  dequantization constants, and the raw activations into the
//                  MMA B-operand pairs, once per stage for all consumers, then
//                  arrives on `ready`;
//   8 consumer     each own a 32-column slice of the unit: four 16-byte
//   warps          weight loads, the activation pairs and the constants from
//                  shared memory, exact dequantization in registers and
//                  m16n8k16 tensor-core MMAs (columns as the MMA's M, tokens as
//                  its N); they arrive on `empty` when done with the stage.
//
// The units are split over a persistent grid of 2 CTAs per SM as contiguous
// equal ranges in column-block-major order (stream-K); finished column blocks
// are written through the deterministic split-K reduction of gemv_common.cuh.
//
// Every wait is bounded; a wait that gives up raises the CTA's abort flag and
// the caller's status word, and the producer lets its copies in flight land
// before the CTA exits.
#include <cuda.h>

#include "dq_common.cuh"
#include "gemv_common.cuh"
#include "sm100.cuh"
#include "tma_host.h"
#include "w4a16_internal.h"

namespace w4a16 {

using namespace sm100;

namespace {

constexpr int kCW = kSliceWarps;              // consumer warps, one 32-column slice each
constexpr int kProducer = kCW, kHelper = kCW + 1;
constexpr int kWsThreads = (kCW + 2) * 32;
constexpr int kWBox = 16 * 32 * 4;            // one slice: 16 word-rows x 32 columns
constexpr int kWBytes = kCW * kWBox;          // the unit's packed weights, 16 KB
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Shared memory: a ring of STAGES weight stages (16 KB each, 1024-byte
// aligned as the 128-byte swizzle of the weight boxes requires), then a ring
// of as many side stages holding the rest of each unit (byte offsets within a
// side stage below).  The activations arrive raw ([8NT tokens][128 rows]) and
// the helper rewrites them in place as B-operand pairs ([NT][4 steps][32
// lanes] x 16 B, the same size).
template <int NT>
struct WsLayout {
  static constexpr int STAGES = NT == 1 ? 5 : 4;     // as many as two CTAs per SM can hold
  static constexpr int CT = 0;                        // INT4 constants: [kCW][3][32] words
  static constexpr int AM = 0;                        // NF4 absmax: [2 blocks][256 columns] fp32
  static constexpr int X = CT + kCW * 3 * 32 * 4;     // activations, raw then paired
  static constexpr int SR = X + NT * 8 * 128 * 2;     // raw scales: 256 x fp16
  static constexpr int ZR = SR + kGemvCols * 2;       // raw zeros: 32 words
  static constexpr int SIDE = ZR + 32 * 4;            // a multiple of 128 bytes
  static constexpr int SIDE_RING = STAGES * kWBytes;
  static constexpr int SMEM = 1024 + STAGES * (kWBytes + SIDE);
  static constexpr uint32_t TX = kWBytes + NT * 8 * 128 * 2;  // TMA bytes per stage (INT4)
  static constexpr uint32_t TX_NF4 = TX + 2 * kGemvCols * 4;    // + the unit's absmax
};
static_assert(WsLayout<1>::SIDE % 128 == 0 && WsLayout<2>::SIDE % 128 == 0, "side stages keep TMA alignment");

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0) : "memory");
}
// arrive on `bar` once this thread's cp.async copies so far have landed
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// ------------------------------------------------------------------ roles
template <int NT, int FMT>
__device__ __forceinline__ void ws_producer(const CUtensorMap* tmW, const CUtensorMap* tmX, const CUtensorMap* tmA,
                                            const GemvArgs& a, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                            volatile int* abort, int nu, int b0, int g0, int lane) {
  using L = WsLayout<NT>;
  const uint32_t side0 = smem_u32(smem) + L::SIDE_RING;
  const int nw = a.N >> 3;  // zero words per row
  // weights and their group metadata for unit (b, g) into stage s: INT4
  // scales and zeros by cp.async, NF4 absmax (the unit's two 64-row blocks)
  // by TMA
  auto issue_weights = [&](int s, int b, int g) {
    if (lane == 0) mbar_arrive_expect_tx(&full[s], FMT == kNF4 ? L::TX_NF4 : L::TX);
    __syncwarp();
    if (lane < kCW)
      tma_load_2d(smem + s * kWBytes + lane * kWBox, tmW, &full[s], b * kGemvCols + lane * 32, g * 16);
    if constexpr (FMT == kNF4) {
      if (lane == kCW) tma_load_2d(smem + L::SIDE_RING + s * L::SIDE + L::AM, tmA, &full[s], b * kGemvCols, g * 2);
    } else {
      const uint32_t side = side0 + s * L::SIDE;
      const int col = b * kGemvCols + 8 * lane;
      const bool sv = col < a.N;
      cp_async_16(side + L::SR + 16 * lane, sv ? a.scales + (size_t)g * a.N + col : a.scales, sv);
      const int zc = b * 32 + lane;
      const bool zv = zc < nw;
      cp_async_4(side + L::ZR + 4 * lane, zv ? a.qz + (size_t)g * nw + zc : a.qz, zv);
      cp_async_arrive_noinc(&full[s]);
    }
  };
  auto issue_x = [&](int s, int g) {
    if (lane == 0) tma_load_2d(smem + L::SIDE_RING + s * L::SIDE + L::X, tmX, &full[s], g * 128, 0);
  };
  if (lane == 0) {
    prefetch_tmap(tmW);
    prefetch_tmap(tmX);
    if (FMT == kNF4) prefetch_tmap(tmA);
  }
  // The packed weights and their constants do not depend on the previous
  // kernel in the stream, so the first stages start before waiting for it;
  // the activations follow after griddep_wait.
  constexpr int S = L::STAGES;
  const int n_first = nu < S ? nu : S;
  int b = b0, g = g0;
  for (int k = 0; k < n_first; ++k) {
    issue_weights(k, b, g);
    if (++g == a.G) {
      g = 0;
      ++b;
    }
  }
  griddep_wait();
  griddep_launch_dependents();
  for (int k = 0, gg = g0; k < n_first; ++k) {
    issue_x(k, gg);
    if (++gg == a.G) gg = 0;
  }
  int s = 0;
  uint32_t ph = 0;  // parity of the release of stage s to wait for
  for (int k = S; k < nu; ++k) {
    // stage s was last filled for unit k - S: wait until it is released
    if (!mbar_wait(&empty[s], ph, abort, a.dev_status, kWaitLimitNs)) {
      // let this CTA's copies in flight land before its shared memory goes away
      cp_async_wait_all();
      for (int kk = k - S; kk < k; ++kk) (void)mbar_drain(&full[kk % S], (uint32_t)(kk / S) & 1u, kWaitLimitNs);
      return;
    }
    issue_weights(s, b, g);
    issue_x(s, g);
    if (++g == a.G) {
      g = 0;
      ++b;
    }
    if (++s == S) {
      s = 0;
      ph ^= 1;
    }
  }
  cp_async_wait_all();
}

template <int NT, int FMT, bool BF16>
__device__ __forceinline__ void ws_helper(const GemvArgs& a, uint8_t* smem, uint64_t* full, uint64_t* ready,
                                          volatile int* abort, int nu, int lane) {
  using L = WsLayout<NT>;
  const int gl = lane >> 2, c = lane & 3;
  int s = 0;
  uint32_t ph = 0;
  for (int k = 0; k < nu; ++k) {
    if (!mbar_wait(&full[s], ph, abort, a.dev_status, kWaitLimitNs)) return;
    uint8_t* st = smem + L::SIDE_RING + s * L::SIDE;
    if constexpr (FMT == kInt4) {
      // constants of columns 8*lane .. 8*lane+7 of the unit: consumer warp
      // lane/4, slice columns 8*(lane%4) ..
      const uint4 sv = *reinterpret_cast<const uint4*>(st + L::SR + 16 * lane);
      const uint32_t zw = *reinterpret_cast<const uint32_t*>(st + L::ZR + 4 * lane);
      const uint32_t sb[8] = {sv.x, sv.x >> 16, sv.y, sv.y >> 16, sv.z, sv.z >> 16, sv.w, sv.w >> 16};
      uint32_t k0[8], k1[8], k2[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t z = (zw >> (4 * j)) & 0xFu;
        if (BF16) {
          const DqConstBF16Fma q = dq_const_bf16_fma(z, sb[j] & 0xFFFFu);
          k0[j] = __float_as_uint(q.z_lo);
          k1[j] = __float_as_uint(q.z_hi);
          k2[j] = q.s;
        } else {
          const DqConstF16 q = dq_const_f16(z, sb[j] & 0xFFFFu);
          k0[j] = q.z_lo;
          k1[j] = q.z_hi;
          k2[j] = q.s;
        }
      }
      uint4* ct = reinterpret_cast<uint4*>(st + L::CT) + (lane >> 2) * 24 + (lane & 3) * 2;
      ct[0] = make_uint4(k0[0], k0[1], k0[2], k0[3]);
      ct[1] = make_uint4(k0[4], k0[5], k0[6], k0[7]);
      ct[8] = make_uint4(k1[0], k1[1], k1[2], k1[3]);
      ct[9] = make_uint4(k1[4], k1[5], k1[6], k1[7]);
      ct[16] = make_uint4(k2[0], k2[1], k2[2], k2[3]);
      ct[17] = make_uint4(k2[4], k2[5], k2[6], k2[7]);
    }
    // activation pairs: lane (gl, c) of every consumer reads, at step o, the
    // pairs of token 8t + gl for word-row tile_row(c, o).  The 32 lanes'
    // loads cover the raw tile exactly once, so it is rewritten in place.
    uint4 xv[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int o = 0; o < 4; ++o)
        xv[t][o] = *reinterpret_cast<const uint4*>(st + L::X + ((8 * t + gl) * 128 + 8 * tile_row(c, o)) * 2);
    __syncwarp();
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int o = 0; o < 4; ++o) {
        uint32_t bf[4];
        x_pairs(xv[t][o], bf);
        *reinterpret_cast<uint4*>(st + L::X + ((t * 4 + o) * 32 + lane) * 16) = make_uint4(bf[0], bf[1], bf[2], bf[3]);
      }
    // the next copy into this stage comes from the TMA unit
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive(&ready[s]);
    if (++s == L::STAGES) {
      s = 0;
      ph ^= 1;
    }
  }
}

template <int NT, int FMT, bool BF16>
__device__ __forceinline__ void ws_consumer(const GemvArgs& a, const Range& R, uint8_t* smem, const float* cbk,
                                            uint64_t* ready, uint64_t* empty, volatile int* abort, int nu, int b0,
                                            int g0, int warp, int lane) {
  using L = WsLayout<NT>;
  const int gl = lane >> 2, c = lane & 3;
  const uint32_t wbase = smem_u32(smem);
  const uint32_t sbase = wbase + L::SIDE_RING;
  uint32_t w_off[4];
#pragma unroll
  for (int o = 0; o < 4; ++o) {
    const int r = tile_row(c, o);
    w_off[o] = (uint32_t)(warp * kWBox + r * 128 + ((gl ^ (r & 7)) << 4));
  }
  const uint32_t x_off = (uint32_t)(L::X + lane * 16);
  const uint32_t c_off = (uint32_t)(L::CT + warp * 384 + gl * 16);
  const uint32_t am_off = (uint32_t)(L::AM + (warp * 32 + 4 * gl) * 4);  // NF4: this lane's 4 columns

  // Y, the partial sums and the tickets may still be in use by the previous
  // kernel in the stream
  griddep_wait();
  griddep_launch_dependents();

  // two accumulators per (token tile, column pair): even and odd steps o, so
  // that consecutive MMAs do not wait on each other
  float acc[NT][2][2][4];
  int s = 0;
  uint32_t ph = 0;
  int p0 = -1, p1 = -1;  // split blocks whose tickets are still to be taken
  for (int b = b0, g = g0, left = nu; left > 0; ++b, g = 0) {
    const int n = a.G - g < left ? a.G - g : left;  // units of column block b
    left -= n;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[t][r][h][i] = 0.f;
#pragma unroll 1
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait(&ready[s], ph, abort, a.dev_status, kWaitLimitNs)) return;
      const uint32_t ws_ = wbase + (uint32_t)(s * kWBytes);
      const uint32_t ss = sbase + (uint32_t)(s * L::SIDE);
      uint4 wv[4], xv[NT][4];
#pragma unroll
      for (int o = 0; o < 4; ++o) wv[o] = lds128(ws_ + w_off[o]);
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int o = 0; o < 4; ++o) xv[t][o] = lds128(ss + x_off + (uint32_t)((t * 4 + o) * 512));
      // INT4: the columns' packed constants; NF4: their two blocks' absmax
      const uint4 c0 = lds128(ss + (FMT == kNF4 ? am_off : c_off));
      const uint4 c1 = lds128(ss + (FMT == kNF4 ? am_off + kGemvCols * 4 : c_off + 128));
      const uint4 c2 = FMT == kNF4 ? c1 : lds128(ss + c_off + 256);
      // One token tile: release the stage as soon as it has been read (the
      // arrive orders the loads above before the producer's next copy into
      // the stage).  Two tiles: the loaded values and the accumulators do not
      // all fit in registers at once, so the loads stay interleaved with the
      // arithmetic and the stage is released after it.
      if (NT == 1) mbar_arrive(&empty[s]);
      const uint32_t k0[4] = {c0.x, c0.y, c0.z, c0.w}, k1[4] = {c1.x, c1.y, c1.z, c1.w},
                     k2[4] = {c2.x, c2.y, c2.z, c2.w};
#pragma unroll
      for (int o = 0; o < 4; ++o) {
        const uint32_t wd[4] = {wv[o].x, wv[o].y, wv[o].z, wv[o].w};
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          uint32_t pa[4], pb[4];
          if constexpr (FMT == kNF4) {
            // word-row tile_row(c, o) lies in the unit's 64-row block o & 1
            const uint32_t* am = (o & 1) ? k1 : k0;
            dq_word_nf4<BF16>(wd[2 * rr], cbk, __uint_as_float(am[2 * rr]), pa);
            dq_word_nf4<BF16>(wd[2 * rr + 1], cbk, __uint_as_float(am[2 * rr + 1]), pb);
          } else if (BF16) {
            dq_word_bf16_fma(wd[2 * rr], DqConstBF16Fma{__uint_as_float(k0[2 * rr]), __uint_as_float(k1[2 * rr]), k2[2 * rr]},
                             pa);
            dq_word_bf16_fma(wd[2 * rr + 1],
                             DqConstBF16Fma{__uint_as_float(k0[2 * rr + 1]), __uint_as_float(k1[2 * rr + 1]), k2[2 * rr + 1]},
                             pb);
          } else {
            dq_word_f16(wd[2 * rr], DqConstF16{k0[2 * rr], k1[2 * rr], k2[2 * rr]}, pa);
            dq_word_f16(wd[2 * rr + 1], DqConstF16{k0[2 * rr + 1], k1[2 * rr + 1], k2[2 * rr + 1]}, pb);
          }
          const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
          const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            mma_16816<BF16>(acc[t][rr][o & 1], a0, xv[t][o].x, xv[t][o].y);
            mma_16816<BF16>(acc[t][rr][o & 1], a1, xv[t][o].z, xv[t][o].w);
          }
        }
      }
      if (NT != 1) mbar_arrive(&empty[s]);
      if (++s == L::STAGES) {
        s = 0;
        ph ^= 1;
      }
    }
    float out[NT][2][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i) out[t][r][i] = acc[t][r][0][i] + acc[t][r][1][i];
    if (store_block<NT, BF16>(a, R, (int)blockIdx.x, b0, warp, lane, b, out)) (b == b0 ? p0 : p1) = b;
  }
  finish_blocks<NT, BF16>(a, R, warp, lane, p0, p1);
}

template <int NT, int FMT, bool BF16>
__global__ void __launch_bounds__(kWsThreads, 2)
    gemv_ws_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmA, const GemvArgs a) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int S = WsLayout<NT>::STAGES;
  __shared__ uint64_t full[S], ready[S], empty[S];
  __shared__ int abort_flag;
  __shared__ float s_cb[16];  // NF4 codebook
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  const Range R{(long long)a.blocks_n * a.G, (int)gridDim.x};
  const long long u0 = R.start(blockIdx.x);
  const int nu = (int)(R.start(blockIdx.x + 1) - u0);
  const int b0 = (int)(u0 / a.G), g0 = (int)(u0 % a.G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // the producer's expect-tx arrival (+ INT4: its 32 lanes' cp.async arrivals)
      mbar_init(&full[s], FMT == kNF4 ? 1 : 1 + 32);
      mbar_init(&ready[s], 32);
      mbar_init(&empty[s], kCW * 32);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (FMT == kNF4 && threadIdx.x < 16) s_cb[threadIdx.x] = a.codebook ? a.codebook[threadIdx.x] : a.cb_builtin.v[threadIdx.x];
  __syncthreads();
  volatile int* abort = &abort_flag;
  if (warp == kProducer)
    ws_producer<NT, FMT>(&tmW, &tmX, &tmA, a, smem, full, empty, abort, nu, b0, g0, lane);
  else if (warp == kHelper)
    ws_helper<NT, FMT, BF16>(a, smem, full, ready, abort, nu, lane);
  else
    ws_consumer<NT, FMT, BF16>(a, R, smem, s_cb, ready, empty, abort, nu, b0, g0, warp, lane);
}

template <int NT, int FMT, bool BF16>
cudaError_t launch_ws(const CUtensorMap& tmW, const CUtensorMap& tmA, const GemvArgs& a, cudaStream_t st) {
  using L = WsLayout<NT>;
  CUtensorMap tmX;  // X [M, K], boxes of 128 rows x 8*NT tokens
  if (!encode_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.X, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.K * 2, 128,
                 (uint32_t)(8 * NT), CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> attr_done{0};
  unsigned long long dev_bit = 0;
  if (attrs_pending(attr_done, &dev_bit)) {
    cudaError_t e = cudaFuncSetAttribute(gemv_ws_kernel<NT, FMT, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemv_ws_kernel<NT, FMT, BF16>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(dev_bit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.ctas);
  cfg.blockDim = dim3(kWsThreads);
  cfg.dynamicSmemBytes = L::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr_pdl[1];
  attr_pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr_pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr_pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_ws_kernel<NT, FMT, BF16>, tmW, tmX, tmA, a);
}

}  // namespace

template <int FMT>
cudaError_t launch_gemv_ws(const GemvArgs& a, bool bf16, cudaStream_t st) {
  CUtensorMap tmW;  // packed weights [K/8, N] words, boxes of 16 word-rows x 32 columns
  if (!encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.qw, (uint64_t)a.N, (uint64_t)(a.K / 8), (uint64_t)a.N * 4, 32,
                 16, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  CUtensorMap tmA = tmW;  // NF4 absmax [K/64, N] fp32, boxes of 2 blocks x 256 columns
  if (FMT == kNF4 && !encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.absmax, (uint64_t)a.N, (uint64_t)(a.K / 64),
                                (uint64_t)a.N * 4, kGemvCols, 2, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (a.M <= 8) return bf16 ? launch_ws<1, FMT, true>(tmW, tmA, a, st) : launch_ws<1, FMT, false>(tmW, tmA, a, st);
  return bf16 ? launch_ws<2, FMT, true>(tmW, tmA, a, st) : launch_ws<2, FMT, false>(tmW, tmA, a, st);
}

cudaError_t launch_gemv_ws_int4(const GemvArgs& a, bool bf16, cudaStream_t st) {
  return launch_gemv_ws<kInt4>(a, bf16, st);
}

cudaError_t launch_gemv_ws_nf4(const GemvArgs& a, bool bf16, cudaStream_t st) {
  return launch_gemv_ws<kNF4>(a, bf16, st);
}

}  // namespace w4a16
