// Warp-specialized split-K weight-streaming kernel for decode shapes
// (1 <= M <= 16): INT4 with grouped scales and zero points (groups of 32, 64,
// any multiple of 128, or one group per column; symmetric or asymmetric),
// INT4 act-order with the map as stored, and NF4 (fp32 absmax, or
// double-quantized absmax).
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
//   producer warp  streams each unit (256 columns x 128 rows along K) into a
//                  shared-memory stage: eight 2-KB weight boxes (16 word-rows
//                  x 32 columns, 128-byte swizzle) and the activation box by
//                  TMA, and the unit's metadata (NF4: the absmax of its two
//                  64-row blocks by TMA, or their 8-bit codes and
//                  second-level scales by cp.async; act-order: the 128 rows'
//                  group indices by cp.async), all completing on the stage's
//                  `full` barrier;
//   helper warp    copies grouped INT4 metadata (the scales and zero words of
//                  a unit's 1, 2 or 4 groups, by cp.async onto the same
//                  barrier, S units ahead), turns the raw metadata into what
//                  the consumers read (packed per-column dequantization
//                  constants; fp32 absmax; table offsets), and the raw
//                  activations into the MMA B-operand pairs, once per stage
//                  for all consumers, then arrives on `ready`;
//   8 consumer     each own a 32-column slice of the unit: four 16-byte
//   warps          weight loads, the activation pairs and the constants from
//                  shared memory, exact dequantization in registers and
//                  m16n8k16 tensor-core MMAs (columns as the MMA's M, tokens as
//                  its N); they arrive on `empty` when done with the stage.
//
// Act-order ("GPTQ与bitsandbytes对比" GPTQ section, --act-order): every K row
// may sit in its own group, so the dequantization constants change from row
// to row.  The consumers keep the scales and zero words of every group for
// the current 256 columns in shared memory (a copy of that slice of the
// caller's arrays, reloaded when the CTA moves to the next column block), and
// each weight looks up its row's entry there.
//
// The units are split over a persistent grid of 1 or 2 CTAs per SM as
// contiguous equal ranges in column-block-major order (stream-K); finished
// column blocks are written through the deterministic split-K reduction of
// gemv_common.cuh.
//
// Every wait is bounded; a wait that gives up raises the CTA's abort flag and
// the caller's status word, and the producer and helper let their copies in
// flight land before the CTA exits.
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
constexpr int kCtBytes = kCW * 3 * 32 * 4;    // one group's packed constants for 256 columns
constexpr int kMaxStages = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// Shared memory a CTA may use with two CTAs per SM (228 KB per SM, 1 KB
// reserved per CTA, a little static shared memory), and with one.
constexpr int kTwoCtaSmem = 113 * 1024;
constexpr int kOneCtaSmem = 226 * 1024;
// Act-order table: per group, 256 fp16 scales then 32 zero words, padded so
// that consecutive groups start in different banks.
constexpr int kTabStride = 256 * 2 + 32 * 4 + 16;

// Shared memory: a ring of `stages` weight stages (16 KB each, 1024-byte
// aligned as the 128-byte swizzle of the weight boxes requires), then a ring
// of as many side stages holding the rest of each unit (byte offsets within a
// side stage below), then (act-order) the table.  The activations arrive raw
// ([8NT tokens][128 rows]) and the helper rewrites them in place as B-operand
// pairs ([NT][4 steps][32 lanes] x 16 B, the same size).
template <int NT, int FMT, int GPU>
struct WsLayout {
  static constexpr bool NF = FMT == kNF4 || FMT == kNF4DQ;
  static constexpr int NGRP = FMT == kInt4 && GPU > 1 ? GPU : 1;  // groups per unit
  // INT4: NGRP x [kCW][3][32] words of constants; NF4: [2 blocks][256] fp32 absmax
  static constexpr int CT = 0;
  static constexpr int CT_BYTES = FMT == kInt4 ? NGRP * kCtBytes : NF ? 2 * kGemvCols * 4 : 0;
  static constexpr int X = CT + CT_BYTES;               // activations, raw then paired
  static constexpr int RAW = X + NT * 8 * 128 * 2;      // raw metadata
  // INT4: NGRP x 256 fp16 scales, then NGRP x 32 zero words; NF4DQ: 2 x 256
  // absmax codes, then the 2 second-level scales; act-order: the 128 rows'
  // group indices (turned into table offsets in place)
  static constexpr int RAW_BYTES = FMT == kInt4      ? NGRP * (kGemvCols * 2 + 32 * 4)
                                   : FMT == kNF4DQ   ? 2 * kGemvCols + 16
                                   : FMT == kInt4Act ? 128 * 4
                                                     : 0;
  static constexpr int SIDE = (RAW + RAW_BYTES + 127) / 128 * 128;
  static constexpr int STAGE = kWBytes + SIDE;
  // bytes the TMA delivers per stage
  static constexpr uint32_t TX = kWBytes + NT * 8 * 128 * 2 + (FMT == kNF4 ? 2 * kGemvCols * 4 : 0);
  // stages that leave room for two CTAs per SM (at most 5: more in flight
  // measured no faster)
  static constexpr int TWO_CTA_FIT = (kTwoCtaSmem - 1024 - 512) / STAGE;
  static constexpr int TWO_CTA_STAGES = TWO_CTA_FIT < 5 ? TWO_CTA_FIT : 5;
};

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
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
// Pipeline depth: fixed per variant, except act-order, whose table takes a
// share of shared memory that depends on the number of groups.
template <int NT, int FMT, int GPU>
__device__ __forceinline__ int stages_of(const GemvArgs& a) {
  return FMT == kInt4Act ? a.stages : WsLayout<NT, FMT, GPU>::TWO_CTA_STAGES;
}

// the consumer warps only (named barrier 1)
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory"); }

// The producer's walk over its units: column block b, 128-row block kb, and
// (grouped INT4) the group of the unit's first row.  The producer warp is on
// the critical path -- every instruction it spends per unit shows in the
// kernel's time -- so the group index is a compile-time function of kb where
// it can be: GPU = 4 or 2 groups of 32 or 64 rows per unit (kb * GPU + j),
// 1 for groups of exactly 128 rows (kb), and 0 for groups spanning a.kbpg
// whole units, or all of K (then tracked incrementally).
template <int GPU>
struct UnitWalk {
  int b, kb, gi, kq;  // kq: units of the current group already passed (GPU = 0)
  __device__ __forceinline__ UnitWalk(const GemvArgs& a, int b0, int k0) : b(b0), kb(k0), gi(0), kq(0) {
    if (GPU == 0) {
      gi = k0 / a.kbpg;
      kq = k0 % a.kbpg;
    }
  }
  __device__ __forceinline__ void next(const GemvArgs& a) {
    if (++kb == a.KB) {
      kb = 0;
      ++b;
      if (GPU == 0) gi = kq = 0;
    } else if (GPU == 0 && ++kq == a.kbpg) {
      kq = 0;
      ++gi;
    }
  }
  __device__ __forceinline__ int group(int j) const { return GPU == 0 ? gi : GPU == 1 ? kb : kb * GPU + j; }
};

// The scale-after-sum route: fp16 INT4 whose groups do not split a 16-row
// MMA step between two scales (every group size but 32).  The weights enter
// the MMAs as the exact integers q - z and each group's scale multiplies its
// fp32 partial sum, so a product is sum_g s_g * sum_k x_k (q_k - z): the
// exact dequantized weight (q - z) * s times x, where the dequantize-then-
// multiply form uses RNE_fp16((q - z) * s).  The two differ by at most one
// fp16 rounding of each weight (relative 2^-11), well inside the product
// tolerance; a one-hot row still gives RNE((q - z) * s) bit for bit (one
// exact fp32 product, rounded once).  bf16 keeps the dequantize-then-
// multiply form: there one rounding of each weight (relative 2^-8) is
// already close to the tolerance on its own.
template <int FMT, int GPU, bool BF16>
__host__ __device__ constexpr bool fact_route() {
  return FMT == kInt4 && GPU <= 2 && !BF16;
}

// ------------------------------------------------------- act-order pairs
// One dequantized pair (row j of the word in the low half, row j + 4 in the
// high half) from the code pair `code` and the zero-point pair `zm`, both in
// the same magic form (1024 + v for a value in bits 0..3 of each half, or
// 64 + v for one in bits 4..7): their fp16 difference is q - z exactly; one
// mixed-precision FMA per weight gives (q - z) * s exactly in fp32 (4 x 11
// significant bits; the addend -0 keeps the product's sign), and one pair
// conversion rounds each value once.  sa / sb hold the two rows' fp16 scales,
// the one used being half H of each.
template <bool BF16, int H>
__device__ __forceinline__ uint32_t dq_pair_rows(uint32_t code, uint32_t zm, uint32_t sa, uint32_t sb) {
  const uint32_t v = hsub2_f16(code, zm);
  float lo, hi;
  if (H == 0)
    asm("{\n\t.reg .f16 v0, v1, a0, a1, b0, b1;\n\t"
        "mov.b32 {v0, v1}, %2;\n\tmov.b32 {a0, a1}, %3;\n\tmov.b32 {b0, b1}, %4;\n\t"
        "fma.rn.f32.f16 %0, v0, a0, 0f80000000;\n\t"
        "fma.rn.f32.f16 %1, v1, b0, 0f80000000;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(v), "r"(sa), "r"(sb));
  else
    asm("{\n\t.reg .f16 v0, v1, a0, a1, b0, b1;\n\t"
        "mov.b32 {v0, v1}, %2;\n\tmov.b32 {a0, a1}, %3;\n\tmov.b32 {b0, b1}, %4;\n\t"
        "fma.rn.f32.f16 %0, v0, a1, 0f80000000;\n\t"
        "fma.rn.f32.f16 %1, v1, b1, 0f80000000;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(v), "r"(sa), "r"(sb));
  return pack2_rn(lo, hi, BF16);
}

// INT4: unit u's scales and zero words into the raw area of a side stage
// (side: its shared address), one cp.async arrival on `bar` per lane.  The
// helper warp issues these, S units ahead of the unit it converts: the
// producer warp is on the critical path (every instruction it spends per unit
// shows in the kernel's time) and the helper has time to spare; moving them
// measured 1-6% faster across the decode shapes.  Symmetric weights: a.nwz =
// 0, so the zero words are zero-filled (the helper turns them into 8s).
template <int NT, int FMT, int GPU, bool SILU>
__device__ __forceinline__ void int4_meta_copy(const GemvArgs& a, uint32_t side, const UnitWalk<GPU>& u, int lane,
                                               uint64_t* bar) {
  using L = WsLayout<NT, FMT, GPU>;
  using G = Geom<SILU>;
  const int cpb = G::cpb(a);
  const int scol_l = 8 * (lane & 15) + (lane >> 4) * G::hiofs(a);
  const int ocol_l = 8 * (lane & 15) + (lane >> 4) * G::hi2(a);
  const int zw_l = (lane >> 4) * (G::hiofs(a) >> 3) + (lane & 15);
  const int nw = a.N >> 3;
  const int b = u.b;
#pragma unroll
  for (int j = 0; j < L::NGRP; ++j) {
    const int gi = u.group(j);
    const bool gv = GPU <= 1 || gi < a.NG;  // only 32/64-row groups can run past K
    const int col = b * cpb + scol_l;
    const bool sv = gv && b * cpb + ocol_l < G::nout(a);
    cp_async_16(side + L::RAW + j * (kGemvCols * 2) + 16 * lane, sv ? a.scales + (size_t)gi * a.N + col : a.scales,
                sv);
    const int zc = b * (cpb >> 3) + zw_l;
    const bool zv = sv && zc < a.nwz;
    cp_async_4(side + L::RAW + L::NGRP * (kGemvCols * 2) + j * 128 + 4 * lane, zv ? a.qz + (size_t)gi * nw + zc : a.qw,
               zv);
  }
  cp_async_arrive_noinc(bar);
}

// ------------------------------------------------------------------ roles
template <int NT, int FMT, int GPU, bool SILU>
__device__ __forceinline__ void ws_producer(const CUtensorMap* tmW, const CUtensorMap* tmX, const CUtensorMap* tmA,
                                            const GemvArgs& a, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                            volatile int* abort, int nu, int b0, int k0, int lane) {
  using L = WsLayout<NT, FMT, GPU>;
  const int S = stages_of<NT, FMT, GPU>(a);
  const uint32_t side0 = smem_u32(smem) + S * kWBytes;
  const int nw = a.N >> 3;  // zero words per row
  const int nb64 = a.K / 64;
  const int nc2 = (a.N + kGemvCols - 1) / kGemvCols;
  // this lane's constant column offsets within a block (see GemvArgs: the
  // unit's second half starts a.hiofs weight columns and a.hi2 output
  // columns after its first): its weight box (lanes < 8), its 8 scales, their
  // output column, and their zero word
  using G = Geom<SILU>;
  // every weight byte is read once per call: stream them evict-first, so
  // that they do not push the activations, partial sums and tickets, or the
  // next launch's data, out of L2 (1.9% on the decode stack)
  const uint64_t wpol = l2_evict_first_policy();
  const int cpb = G::cpb(a);
  const int wcol_l = 32 * (lane & 3) + (lane >> 2) * G::hiofs(a);
  const int scol_l = 8 * (lane & 15) + (lane >> 4) * G::hiofs(a);
  const int ocol_l = 8 * (lane & 15) + (lane >> 4) * G::hi2(a);
  const int zw_l = (lane >> 4) * (G::hiofs(a) >> 3) + (lane & 15);
  // the unit's metadata into stage s: by cp.async (NF4's absmax by TMA;
  // INT4's scales and zeros by the helper warp)
  auto issue_meta = [&](int s, const UnitWalk<GPU>& u) {
    const uint32_t side = side0 + s * L::SIDE;
    const int b = u.b, kb = u.kb;
    if constexpr (FMT == kInt4) {
      // INT4 metadata: copied by the helper warp (int4_meta_copy)
    } else if constexpr (FMT == kNF4) {
      if (lane == kCW) tma_load_2d(smem + S * kWBytes + s * L::SIDE + L::CT, tmA, &full[s], b * kGemvCols, kb * 2);
    } else if constexpr (FMT == kNF4DQ) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int idx = lane * 4 + q;  // 128 four-byte pieces: [2 blocks][64]
        const int r = idx >> 6, cb = (idx & 63) * 4;
        const int row = kb * 2 + r, col = b * kGemvCols + cb;
        const bool v = row < nb64 && col < a.N;
        cp_async_4(side + L::RAW + r * kGemvCols + cb, v ? a.absmax_q + (size_t)row * a.N + col : a.absmax_q, v);
      }
      if (lane < 2) {
        const int row = kb * 2 + lane;
        const bool v = row < nb64;
        cp_async_4(side + L::RAW + 2 * kGemvCols + 4 * lane, v ? a.absmax_s2 + (size_t)row * nc2 + b : a.absmax_s2,
                   v);
      }
      cp_async_arrive_noinc(&full[s]);
    } else {  // act-order: the rows' group indices
      const int row = kb * 128 + 4 * lane;
      const bool v = row < a.K;
      cp_async_16(side + L::RAW + 16 * lane, v ? a.g_idx + row : a.g_idx, v);
      cp_async_arrive_noinc(&full[s]);
    }
  };
  auto issue_unit = [&](int s, const UnitWalk<GPU>& u) {
    if (lane == 0) mbar_arrive_expect_tx(&full[s], L::TX);
    __syncwarp();
    if (lane < kCW)
      tma_load_2d_hint(smem + s * kWBytes + lane * kWBox, tmW, &full[s], u.b * cpb + wcol_l, u.kb * 16, wpol);
    if (lane == 0) tma_load_2d(smem + S * kWBytes + s * L::SIDE + L::X, tmX, &full[s], u.kb * 128, 0);
    issue_meta(s, u);
  };
  if (lane == 0) {
    prefetch_tmap(tmW);
    prefetch_tmap(tmX);
    if (FMT == kNF4) prefetch_tmap(tmA);
  }
  // Nothing the caller owns is read into shared memory before griddep_wait
  // (the kernel before this one may still be writing it); until then the
  // first stages' weights and metadata are only prefetched into L2, so that
  // the copies issued after the wait find them there.
  const int n_first = nu < S ? nu : S;
  {
    UnitWalk<GPU> u(a, b0, k0);
    for (int k = 0; k < n_first; ++k) {
      if (lane < kCW) tma_prefetch_l2_2d(tmW, u.b * cpb + wcol_l, u.kb * 16);
      if constexpr (FMT == kInt4) {
        const int col = u.b * cpb + scol_l;
#pragma unroll
        for (int j = 0; j < L::NGRP; ++j) {
          const int gi = u.group(j);
          if (gi < a.NG && u.b * cpb + ocol_l < G::nout(a)) prefetch_l2(a.scales + (size_t)gi * a.N + col);
          if (gi < a.NG && a.nwz && (lane & 15) == 0) prefetch_l2(a.qz + (size_t)gi * nw + u.b * (cpb >> 3) + zw_l);
        }
      } else if constexpr (FMT == kNF4) {
        if (lane == kCW) tma_prefetch_l2_2d(tmA, u.b * kGemvCols, u.kb * 2);
      }
      u.next(a);
    }
  }
  griddep_wait();
  griddep_launch_dependents();
  UnitWalk<GPU> u(a, b0, k0);
  for (int k = 0; k < n_first; ++k) {
    issue_unit(k, u);
    u.next(a);
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
    issue_unit(s, u);
    u.next(a);
    if (++s == S) {
      s = 0;
      ph ^= 1;
    }
  }
  cp_async_wait_all();
}

template <int NT, int FMT, bool BF16, int GPU, bool SILU>
__device__ __forceinline__ void ws_helper(const GemvArgs& a, uint8_t* smem, uint64_t* full, uint64_t* ready,
                                          volatile int* abort, int nu, int b0, int k0, int lane) {
  using L = WsLayout<NT, FMT, GPU>;
  const int S = stages_of<NT, FMT, GPU>(a);
  const int gl = lane >> 2, c = lane & 3;
  const uint32_t side0 = smem_u32(smem) + S * kWBytes;
  // INT4: this warp copies each unit's metadata, S units ahead: a stage's raw
  // area is free once this warp has converted it
  UnitWalk<GPU> um(a, b0, k0);
  if constexpr (FMT == kInt4) {
    griddep_wait();  // the scales and zeros may be written by the previous kernel
    const int n_first = nu < S ? nu : S;
    for (int k = 0; k < n_first; ++k) {
      int4_meta_copy<NT, FMT, GPU, SILU>(a, side0 + k * L::SIDE, um, lane, &full[k]);
      um.next(a);
    }
  }
  int s = 0;
  uint32_t ph = 0;
  for (int k = 0; k < nu; ++k) {
    if (!mbar_wait(&full[s], ph, abort, a.dev_status, kWaitLimitNs)) {
      cp_async_wait_all();
      return;
    }
    uint8_t* st = smem + S * kWBytes + s * L::SIDE;
    if constexpr (FMT == kInt4) {
      // constants of columns 8*lane .. 8*lane+7 of the unit: consumer warp
      // lane/4, slice columns 8*(lane%4) ..; one set per group of the unit
#pragma unroll
      for (int j = 0; j < L::NGRP; ++j) {
        const uint4 sv = *reinterpret_cast<const uint4*>(st + L::RAW + j * (kGemvCols * 2) + 16 * lane);
        // symmetric weights (no zero points, zero-filled words): a.zxor
        // turns them into zero points of 8
        const uint32_t zw = *reinterpret_cast<const uint32_t*>(st + L::RAW + L::NGRP * (kGemvCols * 2) + j * 128 +
                                                                4 * lane) ^
                            a.zxor;
        const uint32_t sb[8] = {sv.x, sv.x >> 16, sv.y, sv.y >> 16, sv.z, sv.z >> 16, sv.w, sv.w >> 16};
        uint32_t k0[8], k1[8], k2[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const uint32_t z = (zw >> (4 * jj)) & 0xFu;
          if (fact_route<FMT, GPU, BF16>()) {
            // scale after the sum: the zero point's code forms and the
            // scale as fp32
            k0[jj] = (0x6400u | z) * 0x00010001u;
            k1[jj] = (0x5400u | (z << 4)) * 0x00010001u;
            k2[jj] = __float_as_uint(__half2float(__ushort_as_half((unsigned short)(sb[jj] & 0xFFFFu))));
          } else if (BF16) {
            const DqConstBF16Fma q = dq_const_bf16_fma(z, sb[jj] & 0xFFFFu);
            k0[jj] = __float_as_uint(q.z_lo);
            k1[jj] = __float_as_uint(q.z_hi);
            k2[jj] = q.s;
          } else {
            const DqConstF16 q = dq_const_f16(z, sb[jj] & 0xFFFFu);
            k0[jj] = q.z_lo;
            k1[jj] = q.z_hi;
            k2[jj] = q.s;
          }
        }
        uint4* ct = reinterpret_cast<uint4*>(st + L::CT + j * kCtBytes) + (lane >> 2) * 24 + (lane & 3) * 2;
        ct[0] = make_uint4(k0[0], k0[1], k0[2], k0[3]);
        ct[1] = make_uint4(k0[4], k0[5], k0[6], k0[7]);
        ct[8] = make_uint4(k1[0], k1[1], k1[2], k1[3]);
        ct[9] = make_uint4(k1[4], k1[5], k1[6], k1[7]);
        ct[16] = make_uint4(k2[0], k2[1], k2[2], k2[3]);
        ct[17] = make_uint4(k2[4], k2[5], k2[6], k2[7]);
      }
      if (k + S < nu) {
        int4_meta_copy<NT, FMT, GPU, SILU>(a, side0 + s * L::SIDE, um, lane, &full[s]);
        um.next(a);
      }
    } else if constexpr (FMT == kNF4DQ) {
      // absmax_hat = fl32(code * s2) for [2 blocks][256 columns]: lane takes
      // columns 8*lane .. 8*lane+7 of both blocks
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float s2 = *reinterpret_cast<const float*>(st + L::RAW + 2 * kGemvCols + 4 * r);
        const uint2 cw = *reinterpret_cast<const uint2*>(st + L::RAW + r * kGemvCols + 8 * lane);
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = __fmul_rn((float)(((q < 4 ? cw.x : cw.y) >> (8 * (q & 3))) & 0xFFu), s2);
        float4* am = reinterpret_cast<float4*>(st + L::CT + (r * kGemvCols + 8 * lane) * 4);
        am[0] = make_float4(v[0], v[1], v[2], v[3]);
        am[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    } else if constexpr (FMT == kInt4Act) {
      // rows' group indices -> byte offsets of their groups in the table (an
      // index outside [0, NG) is clamped and reported)
      uint4* gp = reinterpret_cast<uint4*>(st + L::RAW) + lane;
      const uint4 g = *gp;
      *gp = make_uint4((uint32_t)(checked_group((int)g.x, a.NG, a.dev_status) * a.tab_stride),
                       (uint32_t)(checked_group((int)g.y, a.NG, a.dev_status) * a.tab_stride),
                       (uint32_t)(checked_group((int)g.z, a.NG, a.dev_status) * a.tab_stride),
                       (uint32_t)(checked_group((int)g.w, a.NG, a.dev_status) * a.tab_stride));
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
    if (++s == S) {
      s = 0;
      ph ^= 1;
    }
  }
}

// Act-order: copy the scales and zero words of every group for column block
// b into the table (consumer warps only; symmetric weights: zero words of 8).
__device__ __forceinline__ void act_table_load(const GemvArgs& a, uint32_t tab, int b, int warp, int lane) {
  const int t = warp * 32 + lane;
  const int nw = a.N >> 3;
  for (int i = t; i < a.NG * 32; i += kCW * 32) {
    const int g = i >> 5, ch = i & 31;
    const int col = b * kGemvCols + 8 * ch;
    const bool v = col < a.N;
    cp_async_16(tab + g * a.tab_stride + 16 * ch, v ? a.scales + (size_t)g * a.N + col : a.scales, v);
    const uint32_t zd = tab + g * a.tab_stride + kGemvCols * 2 + 4 * ch;
    if (a.qz) {
      const int zc = b * 32 + ch;
      const bool zv = zc < nw;
      cp_async_4(zd, zv ? a.qz + (size_t)g * nw + zc : a.qz, zv);
    } else {
      asm volatile("st.shared.u32 [%0], %1;" ::"r"(zd), "r"(0x88888888u) : "memory");
    }
  }
  cp_async_wait_all();
  consumers_sync();
}

template <int NT, int FMT, bool BF16, int GPU, bool SILU>
__device__ __forceinline__ void ws_consumer(const GemvArgs& a, const Range& R, uint8_t* smem, const float* cbk,
                                            uint64_t* ready, uint64_t* empty, volatile int* abort, int nu, int b0,
                                            int k0, int warp, int lane) {
  using L = WsLayout<NT, FMT, GPU>;
  constexpr bool FACT = fact_route<FMT, GPU, BF16>();
  const int S = stages_of<NT, FMT, GPU>(a);
  const int gl = lane >> 2, c = lane & 3;
  const uint32_t wbase = smem_u32(smem);
  const uint32_t sbase = wbase + S * kWBytes;
  const uint32_t tab = sbase + S * L::SIDE;  // act-order table
  uint32_t w_off[4];
#pragma unroll
  for (int o = 0; o < 4; ++o) {
    const int r = tile_row(c, o);
    w_off[o] = (uint32_t)(warp * kWBox + r * 128 + ((gl ^ (r & 7)) << 4));
  }
  const uint32_t x_off = (uint32_t)(L::X + lane * 16);
  // INT4: this lane's constant sets.  With 4 groups per unit (g = 32) the
  // group of word-row tile_row(c, o) is 2 (o & 1) + c / 2; with 2 (g = 64) it
  // is o & 1; with one it is the unit's.
  const int set0 = GPU == 4 ? (c >> 1) : 0;
  const int set1 = GPU == 4 ? 2 + (c >> 1) : GPU == 2 ? 1 : 0;  // (used when GPU > 1)
  const uint32_t c_off0 = (uint32_t)(L::CT + set0 * kCtBytes + warp * 384 + gl * 16);
  const uint32_t c_off1 = (uint32_t)(L::CT + set1 * kCtBytes + warp * 384 + gl * 16);
  const uint32_t am_off = (uint32_t)(L::CT + (warp * 32 + 4 * gl) * 4);  // NF4: this lane's 4 columns
  // act-order: this lane's 4 columns in a table row, and the byte of a zero
  // word holding columns (4gl + 2h, 4gl + 2h + 1), h = 0, 1
  const uint32_t tcol_s = (uint32_t)((warp * 32 + 4 * gl) * 2);
  const uint32_t tcol_z = (uint32_t)(kGemvCols * 2 + ((warp * 32 + 4 * gl) >> 3) * 4);
  const uint32_t zb = 2u * (uint32_t)(gl & 1);
  const uint32_t zsel0 = zb | ((4u + zb) << 8), zsel1 = (zb + 1) | ((5u + zb) << 8);

  // Y, the partial sums, the tickets and every caller buffer may still be in
  // use by the previous kernel in the stream
  griddep_wait();
  griddep_launch_dependents();

  // two accumulators per (token tile, column pair): even and odd steps o, so
  // that consecutive MMAs do not wait on each other -- except for two token
  // tiles on the scale-after-sum route with one group per unit, where the
  // registers are short and the tiles' MMAs already interleave
  constexpr int NPAR = FACT && GPU <= 1 && NT == 2 ? 1 : 2;
  float acc[NT][2][NPAR][4];
  // FACT: the block's sums so far, each unit's scaled sums added in order
  float tot[NT][2][4];
  int s = 0;
  uint32_t ph = 0;
  int p0 = -1, p1 = -1;  // split blocks whose tickets are still to be taken
  for (int b = b0, kb0 = k0, left = nu; left > 0; ++b, kb0 = 0) {
    const int n = a.KB - kb0 < left ? a.KB - kb0 : left;  // units of column block b
    left -= n;
    if constexpr (FMT == kInt4Act) {
      if (b != b0) consumers_sync();  // every consumer is done with the previous block's table
      act_table_load(a, tab, b, warp, lane);
    }
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int h = 0; h < NPAR; ++h)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[t][r][h][i] = 0.f;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i) tot[t][r][i] = 0.f;
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
      // INT4: the columns' packed constants (one or two sets); NF4: their two
      // blocks' absmax; act-order: the table offsets of this lane's rows
      uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0, c2 = c0, d0 = c0, d1 = c0, d2 = c0;
      uint4 ro[4][2];
      if constexpr (FMT == kInt4Act) {
#pragma unroll
        for (int o = 0; o < 4; ++o) {
          const uint32_t rb = ss + L::RAW + (uint32_t)(32 * tile_row(c, o));
          ro[o][0] = lds128(rb);
          ro[o][1] = lds128(rb + 16);
        }
      } else if constexpr (L::NF) {
        c0 = lds128(ss + am_off);
        c1 = lds128(ss + am_off + kGemvCols * 4);
      } else {
        c0 = lds128(ss + c_off0);
        c1 = lds128(ss + c_off0 + 128);
        c2 = lds128(ss + c_off0 + 256);
        if (GPU > 1) {
          d0 = lds128(ss + c_off1);
          d1 = lds128(ss + c_off1 + 128);
          d2 = lds128(ss + c_off1 + 256);
        }
      }
      // One token tile: release the stage as soon as it has been read (the
      // arrive orders the loads above before the producer's next copy into
      // the stage).  Two tiles: the loaded values and the accumulators do not
      // all fit in registers at once, so the loads stay interleaved with the
      // arithmetic and the stage is released after it.
      if (NT == 1) mbar_arrive(&empty[s]);
#pragma unroll
      for (int o = 0; o < 4; ++o) {
        const uint32_t wd[4] = {wv[o].x, wv[o].y, wv[o].z, wv[o].w};
        if constexpr (FMT == kInt4Act) {
          uint32_t pq[4][4];  // [column i][pair j]: rows (j, j + 4) of the word of column 4gl + i
          const uint32_t off[8] = {ro[o][0].x, ro[o][0].y, ro[o][0].z, ro[o][0].w,
                                   ro[o][1].x, ro[o][1].y, ro[o][1].z, ro[o][1].w};
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint2 sa = lds64(tab + off[jj] + tcol_s), sb = lds64(tab + off[jj + 4] + tcol_s);
            const uint32_t za = lds32(tab + off[jj] + tcol_z), zz = lds32(tab + off[jj + 4] + tcol_z);
            const uint32_t zp0 = prmt(za, zz, zsel0), zp1 = prmt(za, zz, zsel1);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t zp = (i >> 1) ? zp1 : zp0;
              const uint32_t sra = (i >> 1) ? sa.y : sa.x, srb = (i >> 1) ? sb.y : sb.x;
              if ((i & 1) == 0) {  // zero point in bits 0..3 of its byte: the 1024 + v form
                const uint32_t zm = lop3_and_or(zp, 0x000F000Fu, 0x64006400u);
                const uint32_t cd = lop3_and_or(wd[i] >> (4 * jj), 0x000F000Fu, 0x64006400u);
                pq[i][jj] = dq_pair_rows<BF16, 0>(cd, zm, sra, srb);
              } else {  // bits 4..7: the 64 + v form
                const uint32_t zm = lop3_and_or(zp, 0x00F000F0u, 0x54005400u);
                const uint32_t wsh = jj == 0 ? wd[i] << 4 : wd[i] >> (4 * jj - 4);
                const uint32_t cd = lop3_and_or(wsh, 0x00F000F0u, 0x54005400u);
                pq[i][jj] = dq_pair_rows<BF16, 1>(cd, zm, sra, srb);
              }
            }
          }
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const uint32_t* pa = pq[2 * rr];
            const uint32_t* pb = pq[2 * rr + 1];
            const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
            const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              mma_16816<BF16>(acc[t][rr][(o & 1) % NPAR], a0, xv[t][o].x, xv[t][o].y);
              mma_16816<BF16>(acc[t][rr][(o & 1) % NPAR], a1, xv[t][o].z, xv[t][o].w);
            }
          }
        } else {
          // a column pair at a time: its two words' dequantization, then its
          // MMAs, so that the arithmetic of one pair overlaps the other's MMAs
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            uint32_t pa[4], pb[4];
            if constexpr (L::NF) {
              // word-row tile_row(c, o) lies in the unit's 64-row block o & 1
              const uint4 am = (o & 1) ? c1 : c0;
              const uint32_t amv[4] = {am.x, am.y, am.z, am.w};
              dq_word_nf4<BF16>(wd[2 * rr], cbk, __uint_as_float(amv[2 * rr]), pa);
              dq_word_nf4<BF16>(wd[2 * rr + 1], cbk, __uint_as_float(amv[2 * rr + 1]), pb);
            } else if constexpr (FACT) {
              const bool second = GPU > 1 && (o & 1);
              const uint4 e0 = second ? d0 : c0, e1 = second ? d1 : c1;
              const uint32_t k0v[4] = {e0.x, e0.y, e0.z, e0.w}, k1v[4] = {e1.x, e1.y, e1.z, e1.w};
              dq_word_codes_f16(wd[2 * rr], k0v[2 * rr], k1v[2 * rr], pa);
              dq_word_codes_f16(wd[2 * rr + 1], k0v[2 * rr + 1], k1v[2 * rr + 1], pb);
            } else {
              const bool second = GPU > 1 && (o & 1);
              const uint4 e0 = second ? d0 : c0, e1 = second ? d1 : c1, e2 = second ? d2 : c2;
              const uint32_t k0v[4] = {e0.x, e0.y, e0.z, e0.w}, k1v[4] = {e1.x, e1.y, e1.z, e1.w},
                             k2v[4] = {e2.x, e2.y, e2.z, e2.w};
              if (BF16) {
                dq_word_bf16_fma(
                    wd[2 * rr],
                    DqConstBF16Fma{__uint_as_float(k0v[2 * rr]), __uint_as_float(k1v[2 * rr]), k2v[2 * rr]}, pa);
                dq_word_bf16_fma(wd[2 * rr + 1],
                                 DqConstBF16Fma{__uint_as_float(k0v[2 * rr + 1]), __uint_as_float(k1v[2 * rr + 1]),
                                                k2v[2 * rr + 1]},
                                 pb);
              } else {
                dq_word_f16(wd[2 * rr], DqConstF16{k0v[2 * rr], k1v[2 * rr], k2v[2 * rr]}, pa);
                dq_word_f16(wd[2 * rr + 1], DqConstF16{k0v[2 * rr + 1], k1v[2 * rr + 1], k2v[2 * rr + 1]}, pb);
              }
            }
            const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
            const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              // FACT: each unit's sums start from zero (its scales differ
              // from the previous unit's)
              float* d = acc[t][rr][(o & 1) % NPAR];
              if (FACT && o < NPAR)
                mma_16816_zc<BF16>(d, a0, xv[t][o].x, xv[t][o].y);
              else
                mma_16816<BF16>(d, a0, xv[t][o].x, xv[t][o].y);
              mma_16816<BF16>(d, a1, xv[t][o].z, xv[t][o].w);
            }
          }
        }
      }
      if constexpr (FACT) {
        // the unit's sums times their columns' scales (fp32, exact fp16
        // values); with two groups per unit, even steps o hold the first
        // group's rows and odd steps the second's
        const uint4 sa = c2, sb = GPU == 2 ? d2 : c2;
        const float s0[4] = {__uint_as_float(sa.x), __uint_as_float(sa.y), __uint_as_float(sa.z),
                             __uint_as_float(sa.w)};
        const float s1[4] = {__uint_as_float(sb.x), __uint_as_float(sb.y), __uint_as_float(sb.z),
                             __uint_as_float(sb.w)};
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int col = 2 * r + (i >> 1);  // this value's column: 4gl + col
              if (GPU == 2) {
                tot[t][r][i] = fmaf(s0[col], acc[t][r][0][i], tot[t][r][i]);
                tot[t][r][i] = fmaf(s1[col], acc[t][r][NPAR - 1][i], tot[t][r][i]);
              } else {
                const float v = NPAR == 2 ? acc[t][r][0][i] + acc[t][r][NPAR - 1][i] : acc[t][r][0][i];
                tot[t][r][i] = fmaf(s0[col], v, tot[t][r][i]);
              }
            }
      }
      if (NT != 1) mbar_arrive(&empty[s]);
      if (++s == S) {
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
        for (int i = 0; i < 4; ++i) out[t][r][i] = FACT ? tot[t][r][i] : acc[t][r][0][i] + acc[t][r][NPAR - 1][i];
    if (store_block<NT, BF16, SILU>(a, R, (int)blockIdx.x, b0, warp, lane, b, out)) (b == b0 ? p0 : p1) = b;
  }
  finish_blocks<NT, BF16, SILU>(a, R, warp, lane, p0, p1);
}

template <int NT, int FMT, bool BF16, int GPU, bool SILU>
__global__ void __launch_bounds__(kWsThreads, FMT == kInt4Act ? 1 : 2)
    gemv_ws_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmA, const GemvArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kMaxStages], ready[kMaxStages], empty[kMaxStages];
  __shared__ int abort_flag;
  __shared__ float s_cb[16];  // NF4 codebook
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  const Range R{(long long)a.blocks_n * a.KB, (int)gridDim.x};
  const long long u0 = R.start(blockIdx.x);
  const int nu = (int)(R.start(blockIdx.x + 1) - u0);
  const int b0 = (int)(u0 / a.KB), k0 = (int)(u0 % a.KB);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages_of<NT, FMT, GPU>(a); ++s) {
      // the producer's expect-tx arrival (+ its 32 lanes' cp.async arrivals,
      // for every format whose metadata comes by cp.async)
      mbar_init(&full[s], FMT == kNF4 ? 1 : 1 + 32);
      mbar_init(&ready[s], 32);
      mbar_init(&empty[s], kCW * 32);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if ((FMT == kNF4 || FMT == kNF4DQ) && threadIdx.x < 16)
    s_cb[threadIdx.x] = a.codebook ? a.codebook[threadIdx.x] : a.cb_builtin.v[threadIdx.x];
  __syncthreads();
  volatile int* abort = &abort_flag;
  if (warp == kProducer)
    ws_producer<NT, FMT, GPU, SILU>(&tmW, &tmX, &tmA, a, smem, full, empty, abort, nu, b0, k0, lane);
  else if (warp == kHelper)
    ws_helper<NT, FMT, BF16, GPU, SILU>(a, smem, full, ready, abort, nu, b0, k0, lane);
  else
    ws_consumer<NT, FMT, BF16, GPU, SILU>(a, R, smem, s_cb, ready, empty, abort, nu, b0, k0, warp, lane);
}

// Pipeline depth and CTAs per SM of a launch.  Act-order: its consumers hold
// more registers (137-168 a thread) than two CTAs per SM leave, so one CTA
// per SM, with the table of all groups and then as many stages as fit (up to
// kMaxStages).  Returns false if fewer than 2 stages fit beside the table.
template <int NT, int FMT, int GPU>
bool ws_shape(int NG, int* stages, int* ctas_per_sm, int* smem) {
  using L = WsLayout<NT, FMT, GPU>;
  if (FMT != kInt4Act) {
    *stages = L::TWO_CTA_STAGES;
    *ctas_per_sm = 2;
    *smem = 1024 + L::TWO_CTA_STAGES * L::STAGE;
    return true;
  }
  const long long table = (long long)NG * kTabStride;
  const long long one = (kOneCtaSmem - 1024 - 512 - table) / L::STAGE;
  if (one < 2) return false;
  *stages = one < kMaxStages ? (int)one : kMaxStages;
  *ctas_per_sm = 1;
  *smem = (int)(1024 + (long long)*stages * L::STAGE + table);
  return true;
}

template <int NT, int FMT, bool BF16, int GPU, bool SILU>
cudaError_t launch_ws(const CUtensorMap& tmW, const CUtensorMap& tmA, const GemvArgs& a0, cudaStream_t st) {
  GemvArgs a = a0;
  int stages = 0, cps = 0, smem = 0;
  if (!ws_shape<NT, FMT, GPU>(a.NG, &stages, &cps, &smem)) return cudaErrorInvalidValue;
  a.stages = stages;
  a.tab_stride = kTabStride;
  // 128-row units per group (groups of a multiple of 128 rows, or one group)
  a.kbpg = a.gsize >= 128 && a.gsize % 128 == 0 ? a.gsize / 128 : a.KB;
  // symmetric weights: no zero words to copy; the helper makes them 8s
  a.nwz = a.qz ? a.N / 8 : 0;
  a.zxor = a.qz ? 0u : 0x88888888u;
  // the persistent grid: at most cps CTAs per SM, at least 4 units (64 KB of
  // weights) per CTA, and no more CTAs than the workspace has partial slots
  // for (the plan's grid)
  const long long U = (long long)a.blocks_n * a.KB;
  long long ctas = (long long)kNumSMs * cps;
  const long long cap = U / 4 > 0 ? U / 4 : 1;
  if (ctas > cap) ctas = cap;
  if (ctas > a.ctas) ctas = a.ctas;
  CUtensorMap tmX;  // X [M, K], boxes of 128 rows x 8*NT tokens
  if (!encode_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.X, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.K * 2, 128,
                 (uint32_t)(8 * NT), CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> attr_done{0};
  unsigned long long dev_bit = 0;
  if (attrs_pending(attr_done, &dev_bit)) {
    cudaError_t e = cudaFuncSetAttribute(gemv_ws_kernel<NT, FMT, BF16, GPU, SILU>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kOneCtaSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemv_ws_kernel<NT, FMT, BF16, GPU, SILU>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(dev_bit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kWsThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr_pdl[1];
  attr_pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr_pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr_pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_ws_kernel<NT, FMT, BF16, GPU, SILU>, tmW, tmX, tmA, a);
}

template <int FMT, int GPU, bool SILU>
cudaError_t launch_fmt_s(const CUtensorMap& tmW, const CUtensorMap& tmA, const GemvArgs& a, bool bf16,
                         cudaStream_t st) {
  if (a.M <= 8)
    return bf16 ? launch_ws<1, FMT, true, GPU, SILU>(tmW, tmA, a, st)
                : launch_ws<1, FMT, false, GPU, SILU>(tmW, tmA, a, st);
  return bf16 ? launch_ws<2, FMT, true, GPU, SILU>(tmW, tmA, a, st)
              : launch_ws<2, FMT, false, GPU, SILU>(tmW, tmA, a, st);
}

// the fused SiLU epilogue exists for plain INT4 groups only
template <int FMT, int GPU>
cudaError_t launch_fmt(const CUtensorMap& tmW, const CUtensorMap& tmA, const GemvArgs& a, bool bf16,
                       cudaStream_t st) {
  if constexpr (FMT == kInt4) {
    if (a.silu) return launch_fmt_s<FMT, GPU, true>(tmW, tmA, a, bf16, st);
  } else {
    if (a.silu) return cudaErrorInvalidValue;
  }
  return launch_fmt_s<FMT, GPU, false>(tmW, tmA, a, bf16, st);
}

bool encode_weights(CUtensorMap* tmW, const GemvArgs& a) {
  // packed weights [K/8, N] words, boxes of 16 word-rows x 32 columns
  return encode_2d(tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.qw, (uint64_t)a.N, (uint64_t)(a.K / 8), (uint64_t)a.N * 4,
                   32, 16, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

cudaError_t launch_gemv_ws_int4(const GemvArgs& a, bool bf16, cudaStream_t st) {
  CUtensorMap tmW;
  if (!encode_weights(&tmW, a)) return cudaErrorInvalidValue;
  if (a.NG > 1 && a.gsize == 32) return launch_fmt<kInt4, 4>(tmW, tmW, a, bf16, st);
  if (a.NG > 1 && a.gsize == 64) return launch_fmt<kInt4, 2>(tmW, tmW, a, bf16, st);
  if (a.gsize == 128) return launch_fmt<kInt4, 1>(tmW, tmW, a, bf16, st);
  return launch_fmt<kInt4, 0>(tmW, tmW, a, bf16, st);  // groups spanning several units, or one group
}

bool gemv_ws_act_fits(int NG) {
  int stages, cps, smem;
  return ws_shape<2, kInt4Act, 1>(NG, &stages, &cps, &smem) && ws_shape<1, kInt4Act, 1>(NG, &stages, &cps, &smem);
}

cudaError_t launch_gemv_ws_act(const GemvArgs& a, bool bf16, cudaStream_t st) {
  CUtensorMap tmW;
  if (!encode_weights(&tmW, a)) return cudaErrorInvalidValue;
  return launch_fmt<kInt4Act, 1>(tmW, tmW, a, bf16, st);
}

cudaError_t launch_gemv_ws_nf4(const GemvArgs& a, bool bf16, cudaStream_t st) {
  CUtensorMap tmW;
  if (!encode_weights(&tmW, a)) return cudaErrorInvalidValue;
  if (a.absmax_q) return launch_fmt<kNF4DQ, 1>(tmW, tmW, a, bf16, st);
  CUtensorMap tmA;  // NF4 absmax [K/64, N] fp32, boxes of 2 blocks x 256 columns
  if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.absmax, (uint64_t)a.N, (uint64_t)(a.K / 64),
                 (uint64_t)a.N * 4, kGemvCols, 2, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  return launch_fmt<kNF4, 1>(tmW, tmA, a, bf16, st);
}

}  // namespace w4a16
