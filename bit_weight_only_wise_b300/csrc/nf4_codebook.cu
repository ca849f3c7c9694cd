// The library's built-in NF4 table (host code).
//
// NF4 puts its 16 values where normally distributed weights are dense, near 0
// ("LLM量化技术深度对比:GPTQ vs AWQ vs bitsandbytes 2026基准全解析", key-data
// item 2; "GPTQ、AWQ与Bitsandbytes：大模型量化三大技术路径深度对比" §2.3: the
// type is built from a normal-distribution prior).  The table:
//   C[7] = 0,
//   C[8 + i] =  Phi^-1(d - (d - 1/2) i / 8) / Phi^-1(d),  i = 0..7  (8 positives)
//   C[6 - i] = -Phi^-1(d - (d - 1/2) i / 7) / Phi^-1(d),  i = 0..6  (7 negatives)
// with d = 1 - (1/30 + 1/32) / 2, so that C[0] = -1 and C[15] = +1; each
// quotient is formed in double and rounded once to float.
//
// Phi^-1 is computed here by Newton's method on Phi(x) = erfc(-x / sqrt 2) / 2
// (libm's erfc), kept inside a bisection bracket, to double precision.  The
// table is built once per process, on first use.
#include <cmath>
#include <mutex>

#include "w4a16.h"
#include "w4a16_internal.h"

namespace w4a16 {

namespace {

double normal_cdf(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); }

// Standard-normal quantile for p in (0, 1).
double normal_quantile(double p) {
  const double inv_sqrt_2pi = 0.39894228040143267794;
  double lo = -40.0, hi = 40.0, x = 0.0;
  for (int it = 0; it < 200; ++it) {
    const double f = normal_cdf(x) - p;
    if (f == 0.0) return x;
    if (f < 0.0) lo = x;
    else hi = x;
    const double dens = inv_sqrt_2pi * std::exp(-0.5 * x * x);
    double nx = x - f / dens;
    if (!(nx > lo && nx < hi)) nx = 0.5 * (lo + hi);  // Newton left the bracket: bisect
    if (nx == x || hi - lo <= 0.0) break;
    x = nx;
  }
  return x;
}

Cb16 build_table() {
  const double d = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0);
  const double top = normal_quantile(d);
  Cb16 t{};
  t.v[7] = 0.0f;
  for (int i = 0; i < 8; ++i) t.v[15 - i] = (float)(normal_quantile(d - (d - 0.5) * i / 8.0) / top);
  for (int i = 0; i < 7; ++i) t.v[i] = (float)(-normal_quantile(d - (d - 0.5) * i / 7.0) / top);
  return t;
}

}  // namespace

const Cb16& nf4_builtin_codebook() {
  static Cb16 table;
  static std::once_flag once;
  std::call_once(once, [] { table = build_table(); });
  return table;
}

}  // namespace w4a16

extern "C" w4a16_status nf4_default_codebook(float* out16) {
  if (!out16) return W4A16_ERR_INVALID_ARG;
  const w4a16::Cb16& t = w4a16::nf4_builtin_codebook();
  for (int i = 0; i < 16; ++i) out16[i] = t.v[i];
  return W4A16_OK;
}
