// Split-K weight-streaming kernel for decode shapes (1 <= M <= 16).
//
// Y[M,N] = X[M,K] . W_hat[K,N].  At M <= 16 the product moves 0.5 byte of
// packed weight per multiply-add pair per token, so the kernel is bound by
// HBM bandwidth: decode time is the time to stream the weights once
// ("LLM量化技术深度对比:GPTQ vs AWQ vs bitsandbytes 2026基准全解析", key-data
// item 3: 16 GB of 4-bit weights vs 64 GB at FP16 per forward; item 1: the
// fused kernel that never writes 16-bit weights is the fast one).
//
// Work split.  A CTA (8 warps) owns 256 consecutive output columns and a
// contiguous range of K groups (128 rows each); a warp owns 32 columns.  Per
// group, lane (g = lane/4, c = lane%4) loads the 16-byte vectors holding
// columns [4g, 4g+4) of the packed word-rows c, c+4, c+8, c+12 of the group
// (128-bit coalesced loads, 512 contiguous bytes per warp and word-row),
// dequantizes them in registers to exact fp16/bf16 pairs, and feeds them to
// the tensor cores as the A operand of m16n8k16 MMAs, with the weights' output
// columns as the MMA's M dimension and the (up to 16) tokens as its N
// dimension (fp32 accumulation).  The MMA needs matching K orderings for A
// and B, not the natural one: each lane's pair j = rows (j, j+4) of its word
// is paired with the activations of the same two rows.
//
// Split-K reduction.  With more than one split, each CTA writes its fp32
// partial tile to the workspace, and the last CTA to arrive for a column block
// (an atomic ticket) sums the splits in index order -- so the result does not
// depend on arrival order -- rounds once to the output dtype and resets the
// ticket to zero for the next call.
#include "dq_common.cuh"
#include "w4a16_internal.h"

namespace w4a16 {

enum GemvFmt { kInt4 = 0, kInt4Act = 1, kNF4 = 2 };

__device__ __forceinline__ uint4 ldg_stream_v4(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
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

// Dequantize the 4 words (4 columns) of one word-row into pr[column][pair].
template <int FMT, bool BF16>
struct Dequantizer;

template <bool BF16>
struct Dequantizer<kInt4, BF16> {
  // constants of the 4 columns for the current group
  DqConstF16 cf[4];
  DqConstBF16 cb[4];
  __device__ __forceinline__ void load_group(const GemvArgs& a, int gi, int col0, bool ok) {
    uint2 sv = make_uint2(0, 0);
    uint32_t zw = 0;
    if (ok) {
      sv = __ldg(reinterpret_cast<const uint2*>(a.scales + (size_t)gi * a.N + col0));
      zw = __ldg(a.qz + (size_t)gi * (a.N >> 3) + (col0 >> 3)) >> (4 * (col0 & 7));
    }
    const uint32_t sb[4] = {sv.x & 0xFFFFu, sv.x >> 16, sv.y & 0xFFFFu, sv.y >> 16};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t z = (zw >> (4 * c)) & 0xFu;
      if (BF16) cb[c] = dq_const_bf16(z, sb[c]);
      else cf[c] = dq_const_f16(z, sb[c]);
    }
  }
  __device__ __forceinline__ void word_row(const GemvArgs&, const uint4& w, int, int, bool, uint32_t pr[4][4]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (BF16) dq_word_bf16(ws[c], cb[c], pr[c]);
      else dq_word_f16(ws[c], cf[c], pr[c]);
    }
  }
};

template <bool BF16>
struct Dequantizer<kInt4Act, BF16> {
  __device__ __forceinline__ void load_group(const GemvArgs&, int, int, bool) {}
  // row0: first K row of the word-row; every row has its own group
  __device__ __forceinline__ void word_row(const GemvArgs& a, const uint4& w, int row0, int col0, bool ok,
                                           uint32_t pr[4][4]) {
    uint32_t sv[8][2], zw[8];
    if (ok) {
      const int4 g0 = __ldg(reinterpret_cast<const int4*>(a.g_idx + row0));
      const int4 g1 = __ldg(reinterpret_cast<const int4*>(a.g_idx + row0 + 4));
      const int gr[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const uint2 s2 = __ldg(reinterpret_cast<const uint2*>(a.scales + (size_t)gr[r] * a.N + col0));
        sv[r][0] = s2.x;
        sv[r][1] = s2.y;
        zw[r] = __ldg(a.qz + (size_t)gr[r] * (a.N >> 3) + (col0 >> 3)) >> (4 * (col0 & 7));
      }
    } else {
#pragma unroll
      for (int r = 0; r < 8; ++r) sv[r][0] = sv[r][1] = zw[r] = 0;
    }
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t z[8], s[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        z[r] = (zw[r] >> (4 * c)) & 0xFu;
        s[r] = (sv[r][c >> 1] >> (16 * (c & 1))) & 0xFFFFu;
      }
      if (BF16) {
        DqConstBF16 k[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) k[j] = dq_const_bf16_2(z[j], s[j], z[j + 4], s[j + 4]);
        dq_word_bf16_rows(ws[c], k, pr[c]);
      } else {
        DqConstF16 k[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) k[j] = dq_const_f16_2(z[j], s[j], z[j + 4], s[j + 4]);
        dq_word_f16_rows(ws[c], k, pr[c]);
      }
    }
  }
};

template <bool BF16>
struct Dequantizer<kNF4, BF16> {
  const float* cbk;  // shared-memory codebook
  __device__ __forceinline__ void load_group(const GemvArgs&, int, int, bool) {}
  __device__ __forceinline__ void word_row(const GemvArgs& a, const uint4& w, int row0, int col0, bool ok,
                                           uint32_t pr[4][4]) {
    float4 am = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ok && row0 < a.K) am = __ldg(reinterpret_cast<const float4*>(a.absmax + (size_t)(row0 >> 6) * a.N + col0));
    dq_word_nf4<BF16>(w.x, cbk, am.x, pr[0]);
    dq_word_nf4<BF16>(w.y, cbk, am.y, pr[1]);
    dq_word_nf4<BF16>(w.z, cbk, am.z, pr[2]);
    dq_word_nf4<BF16>(w.w, cbk, am.w, pr[3]);
  }
};

template <int NT, int FMT, bool BF16>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const GemvArgs a) {
  __shared__ float s_cb[16];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int col_blk = blockIdx.x * kGemvCols;
  const int col0 = col_blk + warp * 32 + 4 * g;
  const bool col_ok = col0 < a.N;
  const int split = blockIdx.y;
  const int g_begin = split * a.groups_per_split;
  const int g_end = min(a.G, g_begin + a.groups_per_split);
  const size_t N = (size_t)a.N;

  Dequantizer<FMT, BF16> dq;
  if constexpr (FMT == kNF4) {
    if (threadIdx.x < 16) s_cb[threadIdx.x] = a.codebook[threadIdx.x];
    __syncthreads();
    dq.cbk = s_cb;
  }

  float acc[NT][2][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[t][r][i] = 0.f;

  // weights of the next group are loaded while the current one is consumed
  uint4 wq[4], wn[4];
  auto load_w = [&](int gi, uint4 (&dst)[4]) {
#pragma unroll
    for (int o = 0; o < 4; ++o) {
      const int wrow = gi * 16 + c + 4 * o;
      if (col_ok && 8 * wrow < a.K) dst[o] = ldg_stream_v4(a.qw + (size_t)wrow * N + col0);
      else dst[o] = make_uint4(0, 0, 0, 0);
    }
  };
  if (g_begin < g_end) load_w(g_begin, wq);

#pragma unroll 1
  for (int gi = g_begin; gi < g_end; ++gi) {
    if (gi + 1 < g_end) load_w(gi + 1, wn);
    dq.load_group(a, gi, col0, col_ok);
#pragma unroll
    for (int o = 0; o < 4; ++o) {
      const int row0 = gi * 128 + 8 * (c + 4 * o);  // first K row of this lane's word-row
      // activations of the same 8 rows, for this lane's token(s)
      uint32_t b[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int tok = 8 * t + g;
        uint4 xv = make_uint4(0, 0, 0, 0);
        if (tok < a.M && row0 < a.K) xv = __ldg(reinterpret_cast<const uint4*>(a.X + (size_t)tok * a.K + row0));
        b[t][0] = prmt(xv.x, xv.z, 0x5410u);  // rows (0, 4)
        b[t][1] = prmt(xv.x, xv.z, 0x7632u);  // rows (1, 5)
        b[t][2] = prmt(xv.y, xv.w, 0x5410u);  // rows (2, 6)
        b[t][3] = prmt(xv.y, xv.w, 0x7632u);  // rows (3, 7)
      }
      uint32_t pr[4][4];
      dq.word_row(a, wq[o], row0, col0, col_ok, pr);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint32_t a0[4] = {pr[2 * r][0], pr[2 * r + 1][0], pr[2 * r][1], pr[2 * r + 1][1]};
        const uint32_t a1[4] = {pr[2 * r][2], pr[2 * r + 1][2], pr[2 * r][3], pr[2 * r + 1][3]};
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          mma_16816<BF16>(acc[t][r], a0, b[t][0], b[t][1]);
          mma_16816<BF16>(acc[t][r], a1, b[t][2], b[t][3]);
        }
      }
    }
#pragma unroll
    for (int o = 0; o < 4; ++o) wq[o] = wn[o];
  }

  // D fragment: acc[t][r] = {(tok 2c, colA), (tok 2c+1, colA), (tok 2c, colB), (tok 2c+1, colB)}
  // with colA = col0 + 2r, colB = colA + 1, tok relative to 8t.
  if (a.splits == 1) {
    if (!col_ok) return;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int tok = 8 * t + 2 * c;
        const int col = col0 + 2 * r;
        if (tok < a.M) *reinterpret_cast<uint32_t*>(a.Y + (size_t)tok * N + col) = pack2_rn(acc[t][r][0], acc[t][r][2], BF16);
        if (tok + 1 < a.M) *reinterpret_cast<uint32_t*>(a.Y + (size_t)(tok + 1) * N + col) = pack2_rn(acc[t][r][1], acc[t][r][3], BF16);
      }
    return;
  }

  if (col_ok) {
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int tok = 8 * t + 2 * c;
        const int col = col0 + 2 * r;
        if (tok < a.M)
          *reinterpret_cast<float2*>(a.partial + ((size_t)split * a.M + tok) * N + col) = make_float2(acc[t][r][0], acc[t][r][2]);
        if (tok + 1 < a.M)
          *reinterpret_cast<float2*>(a.partial + ((size_t)split * a.M + tok + 1) * N + col) = make_float2(acc[t][r][1], acc[t][r][3]);
      }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(a.counters + blockIdx.x, 1);
    s_last = (prev == a.splits - 1);
    if (s_last) {
      a.counters[blockIdx.x] = 0;  // ready for the next call
      __threadfence();
    }
  }
  __syncthreads();
  if (!s_last) return;
  const int col = col_blk + threadIdx.x;
  if (col >= a.N) return;
  for (int tok = 0; tok < a.M; ++tok) {
    float s = 0.f;
    for (int sp = 0; sp < a.splits; ++sp) s += __ldcg(a.partial + ((size_t)sp * a.M + tok) * N + col);
    const uint32_t v = pack2_rn(s, 0.f, BF16);
    a.Y[(size_t)tok * N + col] = (uint16_t)(v & 0xFFFFu);
  }
}

template <int FMT>
static cudaError_t launch_gemv(const GemvArgs& a, bool bf16, cudaStream_t st) {
  dim3 grid(a.N > 0 ? (a.N + kGemvCols - 1) / kGemvCols : 0, a.splits), block(kGemvThreads);
  if (a.M <= 8) {
    if (bf16) gemv_kernel<1, FMT, true><<<grid, block, 0, st>>>(a);
    else gemv_kernel<1, FMT, false><<<grid, block, 0, st>>>(a);
  } else {
    if (bf16) gemv_kernel<2, FMT, true><<<grid, block, 0, st>>>(a);
    else gemv_kernel<2, FMT, false><<<grid, block, 0, st>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_gemv_int4(const GemvArgs& a, bool bf16, cudaStream_t st) {
  return a.g_idx ? launch_gemv<kInt4Act>(a, bf16, st) : launch_gemv<kInt4>(a, bf16, st);
}

cudaError_t launch_gemv_nf4(const GemvArgs& a, bool bf16, cudaStream_t st) {
  return launch_gemv<kNF4>(a, bf16, st);
}

GemvPlan gemv_plan(int M, int N, int K, int rows_per_group) {
  GemvPlan p{};
  p.blocks_n = (N + kGemvCols - 1) / kGemvCols;
  const int G = (K + 127) / 128;  // chunks of 128 rows
  (void)rows_per_group;
  int s = p.blocks_n > 0 ? (kGemvTargetCTAs + p.blocks_n / 2) / p.blocks_n : 1;
  s = s < 1 ? 1 : (s > G ? G : s);
  p.groups_per_split = G > 0 ? (G + s - 1) / s : 1;
  p.splits = G > 0 ? (G + p.groups_per_split - 1) / p.groups_per_split : 1;
  if (p.splits > 1 && M > 0) {
    p.workspace_bytes = kCountersBytes + (size_t)p.splits * M * N * sizeof(float);
  }
  return p;
}

}  // namespace w4a16
