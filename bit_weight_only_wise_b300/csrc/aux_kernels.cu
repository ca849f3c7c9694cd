// Standalone dequantization (the bit-exact check target) and the on-device
// quantizers (round-to-nearest INT4, blockwise NF4) that build checkpoints.
//
// Dequantization: cloud.tencent.com/developer/article/2726413 §2.1-2.2
// (asymmetric, group-wise); "GPTQ、AWQ与Bitsandbytes：大模型量化三大技术路径
// 深度对比" §2.3 (block-wise NF4).  Quantization: "GPTQ与bitsandbytes对比"
// GPTQ section (round-to-nearest is the plain baseline quantizer).
#include "dq_common.cuh"
#include "w4a16_internal.h"

namespace w4a16 {

// ------------------------------------------------------------ dequant INT4
// One thread: one packed word-row i (8 K rows) x 4 columns [n, n+4).
template <bool BF16, bool ACT>
__global__ void __launch_bounds__(256) dequant_int4_kernel(const uint32_t* __restrict__ qw,
                                                           const uint16_t* __restrict__ scales,
                                                           const uint32_t* __restrict__ qz,
                                                           const int32_t* __restrict__ g_idx,
                                                           uint16_t* __restrict__ out, int K, int N,
                                                           int group_size) {
  const int n4 = blockIdx.x * blockDim.x + threadIdx.x;  // column quad
  const int i = blockIdx.y;                               // word-row
  const int n = 4 * n4;
  if (n >= N) return;
  const uint4 w = *reinterpret_cast<const uint4*>(qw + (size_t)i * N + n);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  uint32_t pr[4][4];  // [column][pair]
  if (!ACT) {
    const int g = (8 * i) / group_size;
    const uint2 sv = *reinterpret_cast<const uint2*>(scales + (size_t)g * N + n);
    // symmetric weights (no zero points): every zero point is 8
    const uint32_t zw = qz ? qz[(size_t)g * (N / 8) + n / 8] >> (4 * (n & 7)) : 0x8888u;
    const uint32_t sb[4] = {sv.x & 0xFFFFu, sv.x >> 16, sv.y & 0xFFFFu, sv.y >> 16};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t z = (zw >> (4 * c)) & 0xFu;
      if (BF16) {
        DqConstBF16 k = dq_const_bf16(z, sb[c]);
        dq_word_bf16(ws[c], k, pr[c]);
      } else {
        DqConstF16 k = dq_const_f16(z, sb[c]);
        dq_word_f16(ws[c], k, pr[c]);
      }
    }
  } else {
    int gr[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) gr[r] = checked_group(g_idx[8 * i + r], K / group_size, nullptr);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t z[8], s[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        s[r] = scales[(size_t)gr[r] * N + n + c];
        z[r] = qz ? (qz[(size_t)gr[r] * (N / 8) + (n + c) / 8] >> (4 * ((n + c) & 7))) & 0xFu : 8u;
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
  // pair j of column c holds rows (j, j+4): transpose to rows x 4 columns
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint2 lo, hi;
    lo.x = prmt(pr[0][j], pr[1][j], 0x5410u);
    lo.y = prmt(pr[2][j], pr[3][j], 0x5410u);
    hi.x = prmt(pr[0][j], pr[1][j], 0x7632u);
    hi.y = prmt(pr[2][j], pr[3][j], 0x7632u);
    *reinterpret_cast<uint2*>(out + (size_t)(8 * i + j) * N + n) = lo;
    *reinterpret_cast<uint2*>(out + (size_t)(8 * i + j + 4) * N + n) = hi;
  }
}

// ------------------------------------------------------------- dequant NF4
template <bool BF16>
__global__ void __launch_bounds__(256) dequant_nf4_kernel(const uint32_t* __restrict__ qw,
                                                          const float* __restrict__ absmax,
                                                          const float* __restrict__ codebook, const Cb16 cb_builtin,
                                                          uint16_t* __restrict__ out, int K, int N,
                                                          int blocksize) {
  __shared__ float cb[16];
  if (threadIdx.x < 16) cb[threadIdx.x] = codebook ? codebook[threadIdx.x] : cb_builtin.v[threadIdx.x];
  __syncthreads();
  const int n4 = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = blockIdx.y;
  const int n = 4 * n4;
  if (n >= N) return;
  const uint4 w = *reinterpret_cast<const uint4*>(qw + (size_t)i * N + n);
  const float4 am = *reinterpret_cast<const float4*>(absmax + (size_t)((8 * i) / blocksize) * N + n);
  uint32_t pr[4][4];
  dq_word_nf4<BF16>(w.x, cb, am.x, pr[0]);
  dq_word_nf4<BF16>(w.y, cb, am.y, pr[1]);
  dq_word_nf4<BF16>(w.z, cb, am.z, pr[2]);
  dq_word_nf4<BF16>(w.w, cb, am.w, pr[3]);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint2 lo, hi;
    lo.x = prmt(pr[0][j], pr[1][j], 0x5410u);
    lo.y = prmt(pr[2][j], pr[3][j], 0x5410u);
    hi.x = prmt(pr[0][j], pr[1][j], 0x7632u);
    hi.y = prmt(pr[2][j], pr[3][j], 0x7632u);
    *reinterpret_cast<uint2*>(out + (size_t)(8 * i + j) * N + n) = lo;
    *reinterpret_cast<uint2*>(out + (size_t)(8 * i + j + 4) * N + n) = hi;
  }
}

// ------------------------------------------- dequant NF4, double-quantized absmax
// As dequant_nf4_kernel with absmax_hat = fl32(code * s2) ("GPTQ、AWQ与
// Bitsandbytes" §3.3 use_double_quant; §4.3: a scale of the scale): codes
// [K/bs, N] bytes, s2 [K/bs, ceil(N/256)] fp32, one per 256 columns of a row.
template <bool BF16>
__global__ void __launch_bounds__(256) dequant_nf4dq_kernel(const uint32_t* __restrict__ qw,
                                                            const uint8_t* __restrict__ absmax_q,
                                                            const float* __restrict__ absmax_s2,
                                                            const float* __restrict__ codebook, const Cb16 cb_builtin,
                                                            uint16_t* __restrict__ out, int K, int N, int blocksize) {
  __shared__ float cb[16];
  if (threadIdx.x < 16) cb[threadIdx.x] = codebook ? codebook[threadIdx.x] : cb_builtin.v[threadIdx.x];
  __syncthreads();
  const int n4 = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = blockIdx.y;
  const int n = 4 * n4;
  if (n >= N) return;
  const int blk = (8 * i) / blocksize;
  const uint4 w = *reinterpret_cast<const uint4*>(qw + (size_t)i * N + n);
  const uint32_t codes = *reinterpret_cast<const uint32_t*>(absmax_q + (size_t)blk * N + n);
  const float s2 = absmax_s2[(size_t)blk * ((N + 255) / 256) + n / 256];  // the 4 columns share a 256-block
  float am[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) am[c] = __fmul_rn((float)((codes >> (8 * c)) & 0xFFu), s2);
  uint32_t pr[4][4];
  dq_word_nf4<BF16>(w.x, cb, am[0], pr[0]);
  dq_word_nf4<BF16>(w.y, cb, am[1], pr[1]);
  dq_word_nf4<BF16>(w.z, cb, am[2], pr[2]);
  dq_word_nf4<BF16>(w.w, cb, am[3], pr[3]);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint2 lo, hi;
    lo.x = prmt(pr[0][j], pr[1][j], 0x5410u);
    lo.y = prmt(pr[2][j], pr[3][j], 0x5410u);
    hi.x = prmt(pr[0][j], pr[1][j], 0x7632u);
    hi.y = prmt(pr[2][j], pr[3][j], 0x7632u);
    *reinterpret_cast<uint2*>(out + (size_t)(8 * i + j) * N + n) = lo;
    *reinterpret_cast<uint2*>(out + (size_t)(8 * i + j + 4) * N + n) = hi;
  }
}

// ------------------------------------------------- NF4 double quantization
// One CTA per (absmax row r, 256-column block c): s2 = fl32(max / 255) (the
// fp64 quotient rounded to fp32; a zero scale becomes 1), code =
// clamp(rint(absmax / s2), 0, 255) with the division in fp64.
__global__ void __launch_bounds__(256) double_quantize_kernel(const float* __restrict__ absmax, int N,
                                                              uint8_t* __restrict__ absmax_q,
                                                              float* __restrict__ absmax_s2) {
  __shared__ float red[8];
  const int r = blockIdx.y, c = blockIdx.x, t = threadIdx.x;
  const int n = c * 256 + t;
  const float v = n < N ? absmax[(size_t)r * N + n] : 0.f;
  float m = v;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((t & 31) == 0) red[t >> 5] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
  float s2 = __double2float_rn(__ddiv_rn((double)m, 255.0));
  if (s2 == 0.f) s2 = 1.f;
  const int nc = (N + 255) / 256;
  if (t == 0) absmax_s2[(size_t)r * nc + c] = s2;
  if (n < N) {
    const double q = fmin(fmax(rint(__ddiv_rn((double)v, (double)s2)), 0.0), 255.0);
    absmax_q[(size_t)r * N + n] = (uint8_t)q;
  }
}

// ------------------------------------------------------------ quantize RTN
__device__ __forceinline__ uint16_t f64_to_f16_rn(double x) {
  unsigned short h;
  asm("cvt.rn.f16.f64 %0, %1;" : "=h"(h) : "d"(x));
  return h;
}

// One thread: one group g of `group_size` rows x one column n.  The whole
// warp must be present for the zero-point shuffle, so out-of-range columns
// compute on dummy data and skip their stores.
//   asymmetric (qz given): range [min(w, 0), max(w, 0)], s = fp16((mx - mn) / 15),
//     z = clamp(rint(-mn / s), 0, 15), q = clamp(rint(w / s) + z, 0, 15);
//   symmetric (qz == nullptr; cloud.tencent.com/developer/article/2726413 §2.1,
//     zero point fixed at 0): s = fp16(max |w| / 7), q = clamp(rint(w / s), -8, 7)
//     + 8, so the implied zero point is 8.
// A zero scale becomes 1; divisions in fp64, rint half to even.
__global__ void __launch_bounds__(256) quantize_rtn_kernel(const float* __restrict__ W, int K, int N,
                                                           int group_size, uint32_t* __restrict__ qw,
                                                           uint16_t* __restrict__ scales,
                                                           uint32_t* __restrict__ qz) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int g = blockIdx.y;
  const bool ok = n < N;
  const int nn = ok ? n : 0;
  const bool sym = qz == nullptr;
  const float* col = W + (size_t)g * group_size * N + nn;
  float mn = 0.f, mx = 0.f;  // zero is always inside the range
  for (int r = 0; r < group_size; ++r) {
    const float v = col[(size_t)r * N];
    mn = fminf(mn, v);
    mx = fmaxf(mx, v);
  }
  const double span = sym ? fmax(-(double)mn, (double)mx) : __dsub_rn((double)mx, (double)mn);
  uint16_t sh = f64_to_f16_rn(__ddiv_rn(span, sym ? 7.0 : 15.0));
  if ((sh & 0x7FFFu) == 0) sh = 0x3C00u;  // a zero scale becomes 1
  const double s = (double)__half2float(__ushort_as_half(sh));
  double zd = sym ? 8.0 : rint(__ddiv_rn(-(double)mn, s));
  zd = fmin(fmax(zd, 0.0), 15.0);
  if (!sym) {
    // zero points: 8 consecutive columns per word
    uint32_t zp = (uint32_t)zd << (4 * (n & 7));
    zp |= __shfl_xor_sync(0xFFFFFFFFu, zp, 1);
    zp |= __shfl_xor_sync(0xFFFFFFFFu, zp, 2);
    zp |= __shfl_xor_sync(0xFFFFFFFFu, zp, 4);
    if (ok && (n & 7) == 0) qz[(size_t)g * (N / 8) + n / 8] = zp;
  }
  if (!ok) return;
  scales[(size_t)g * N + n] = sh;
  for (int i = 0; i < group_size / 8; ++i) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const double v = (double)col[(size_t)(8 * i + j) * N];
      double q = rint(__ddiv_rn(v, s)) + zd;
      q = fmin(fmax(q, 0.0), 15.0);  // symmetric: rint(w/s) in [-8, 7], stored + 8
      word |= (uint32_t)q << (4 * j);
    }
    qw[(size_t)(g * (group_size / 8) + i) * N + n] = word;
  }
}

// ------------------------------------------------------------ quantize NF4
__global__ void __launch_bounds__(256) quantize_nf4_kernel(const float* __restrict__ W, int K, int N,
                                                           int blocksize, const float* __restrict__ codebook,
                                                           const Cb16 cb_builtin, uint32_t* __restrict__ qw,
                                                           float* __restrict__ absmax) {
  __shared__ double cb[16];
  if (threadIdx.x < 16) cb[threadIdx.x] = (double)(codebook ? codebook[threadIdx.x] : cb_builtin.v[threadIdx.x]);
  __syncthreads();
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int b = blockIdx.y;
  if (n >= N) return;
  const float* col = W + (size_t)b * blocksize * N + n;
  float am = 0.f;
  for (int r = 0; r < blocksize; ++r) am = fmaxf(am, fabsf(col[(size_t)r * N]));
  absmax[(size_t)b * N + n] = am;
  for (int i = 0; i < blocksize / 8; ++i) {
    uint32_t word = 0;
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
      uint32_t code = 7;
      if (am != 0.f) {
        const double v = (double)__fdiv_rn(col[(size_t)(8 * i + j) * N], am);
        double best = fabs(cb[0] - v);
        code = 0;
#pragma unroll
        for (int c = 1; c < 16; ++c) {
          const double d = fabs(cb[c] - v);  // exact: both operands are fp32 values
          if (d < best) {
            best = d;
            code = c;
          }
        }
      }
      word |= code << (4 * j);
    }
    qw[(size_t)(b * (blocksize / 8) + i) * N + n] = word;
  }
}

// ------------------------------------------------------------- launchers
cudaError_t launch_dequant_int4(const uint32_t* qw, const uint16_t* scales, const uint32_t* qz,
                                const int32_t* g_idx, uint16_t* out, int K, int N, int group_size,
                                bool bf16, cudaStream_t st) {
  dim3 block(256), grid((N / 4 + 255) / 256, K / 8);
  if (bf16) {
    if (g_idx) dequant_int4_kernel<true, true><<<grid, block, 0, st>>>(qw, scales, qz, g_idx, out, K, N, group_size);
    else dequant_int4_kernel<true, false><<<grid, block, 0, st>>>(qw, scales, qz, g_idx, out, K, N, group_size);
  } else {
    if (g_idx) dequant_int4_kernel<false, true><<<grid, block, 0, st>>>(qw, scales, qz, g_idx, out, K, N, group_size);
    else dequant_int4_kernel<false, false><<<grid, block, 0, st>>>(qw, scales, qz, g_idx, out, K, N, group_size);
  }
  return cudaGetLastError();
}

cudaError_t launch_dequant_nf4(const uint32_t* qw, const float* absmax, const float* codebook, uint16_t* out,
                               int K, int N, int blocksize, bool bf16, cudaStream_t st) {
  dim3 block(256), grid((N / 4 + 255) / 256, K / 8);
  const Cb16& cb = nf4_builtin_codebook();
  if (bf16) dequant_nf4_kernel<true><<<grid, block, 0, st>>>(qw, absmax, codebook, cb, out, K, N, blocksize);
  else dequant_nf4_kernel<false><<<grid, block, 0, st>>>(qw, absmax, codebook, cb, out, K, N, blocksize);
  return cudaGetLastError();
}

cudaError_t launch_dequant_nf4dq(const uint32_t* qw, const uint8_t* absmax_q, const float* absmax_s2,
                                 const float* codebook, uint16_t* out, int K, int N, int blocksize, bool bf16,
                                 cudaStream_t st) {
  dim3 block(256), grid((N / 4 + 255) / 256, K / 8);
  const Cb16& cb = nf4_builtin_codebook();
  if (bf16)
    dequant_nf4dq_kernel<true><<<grid, block, 0, st>>>(qw, absmax_q, absmax_s2, codebook, cb, out, K, N, blocksize);
  else
    dequant_nf4dq_kernel<false><<<grid, block, 0, st>>>(qw, absmax_q, absmax_s2, codebook, cb, out, K, N, blocksize);
  return cudaGetLastError();
}

cudaError_t launch_double_quantize(const float* absmax, int rows, int N, uint8_t* absmax_q, float* absmax_s2,
                                   cudaStream_t st) {
  dim3 block(256), grid((N + 255) / 256, rows);
  double_quantize_kernel<<<grid, block, 0, st>>>(absmax, N, absmax_q, absmax_s2);
  return cudaGetLastError();
}

cudaError_t launch_quantize_rtn(const float* W, int K, int N, int group_size, uint32_t* qw, uint16_t* scales,
                                uint32_t* qz, cudaStream_t st) {
  dim3 block(256), grid((N + 255) / 256, K / group_size);
  quantize_rtn_kernel<<<grid, block, 0, st>>>(W, K, N, group_size, qw, scales, qz);
  return cudaGetLastError();
}

cudaError_t launch_quantize_nf4(const float* W, int K, int N, int blocksize, const float* codebook, uint32_t* qw,
                                float* absmax, cudaStream_t st) {
  dim3 block(256), grid((N + 255) / 256, K / blocksize);
  quantize_nf4_kernel<<<grid, block, 0, st>>>(W, K, N, blocksize, codebook, nf4_builtin_codebook(), qw, absmax);
  return cudaGetLastError();
}

}  // namespace w4a16
