/*
 * The library used through include/w4a16.h from a plain C program, with no
 * GPU: every entry point the header declares is referenced (so the link
 * checks that each has C linkage), and the calls made are the pure host
 * functions and calls that fail validation before anything is launched.
 * Prints "ok" and exits 0 when every check holds; otherwise prints the first
 * failing check and exits 1.  Built and run by tests/test_c_abi_host.py.
 */
#include <limits.h>
#include <stdint.h>
#include <stdio.h>
#include <stddef.h>
#include <string.h>

#include "w4a16.h"

#define CHECK(c)                                          \
  do {                                                    \
    if (!(c)) {                                           \
      printf("failed: %s (line %d)\n", #c, __LINE__);     \
      return 1;                                           \
    }                                                     \
  } while (0)

/* stand-ins for device pointers: 16-byte aligned, never dereferenced,
   because every call below is rejected (or is an empty problem) first */
#define P(a) ((void*)(uintptr_t)(a))
#define PU(a) ((uint32_t*)(uintptr_t)(a))
#define PF(a) ((float*)(uintptr_t)(a))
#define PI(a) ((int32_t*)(uintptr_t)(a))
#define PU8(a) ((uint8_t*)(uintptr_t)(a))

static int defined_host_status(w4a16_status s) {
  return s == W4A16_OK || s == W4A16_ERR_INVALID_ARG || s == W4A16_ERR_UNSUPPORTED;
}

/* Every entry point over extreme and boundary sizes, block sizes and both
 * dtypes.  Each call passes NULL as its first pointer, which every entry
 * point checks after the sizes and before anything else, so no call can
 * launch; what runs is the size and shape arithmetic, which a sanitizer
 * build checks for undefined behaviour. */
static int fuzz_sizes(void) {
  const int sizes[] = {INT_MIN, -8, -1, 0, 1, 8, 16, 17, 128, 256, 4096, 524160,
                       W4A16_MAX_M, W4A16_MAX_M + 1, W4A16_MAX_N, W4A16_MAX_N + 8, W4A16_MAX_K,
                       W4A16_MAX_K + 8, INT_MAX - 7, INT_MAX};
  const int blocks[] = {INT_MIN, -1, 0, 64, 128, INT_MAX};
  const w4a16_dtype dts[] = {W4A16_F16, W4A16_BF16};
  const size_t ns = sizeof(sizes) / sizeof(sizes[0]), nb = sizeof(blocks) / sizeof(blocks[0]);
  for (size_t a = 0; a < ns; ++a)
    for (size_t b = 0; b < ns; ++b)
      for (size_t c = 0; c < ns; ++c) {
        const int M = sizes[a], N = sizes[b], K = sizes[c];
        (void)w4a16_workspace_bytes(M, N, K);
        (void)w4a16_prepacked_workspace_bytes(M, N, K);
        for (size_t g = 0; g < nb; ++g)
          for (int d = 0; d < 2; ++d) {
            const int G = blocks[g];
            const w4a16_dtype dt = dts[d];
            w4a16_status s1, s2;
            CHECK(defined_host_status(
                w4a16_gemm(NULL, PU(16), P(16), PU(16), NULL, P(16), M, N, K, G, dt, NULL, 0, NULL, NULL)));
            s1 = w4a16_gemv(NULL, PU(16), P(16), PU(16), NULL, P(16), M, N, K, G, dt, NULL, 0, NULL, NULL);
            s2 = w4a16_gemv_noalloc(NULL, PU(16), P(16), PU(16), NULL, P(16), M, N, K, G, dt, NULL, NULL);
            CHECK(defined_host_status(s1) && s1 == s2);
            {  /* a one-item batch answers as w4a16_gemv */
              const w4a16_gemv_item it = {NULL, PU(16), P(16), PU(16), NULL, P(16), M, N, K, G, dt};
              CHECK(w4a16_gemv_batch(&it, 1, NULL, 0, NULL, NULL) == s1);
            }
            CHECK(defined_host_status(w4a16_gemm_prepacked(NULL, PU(16), P(16), PU(16), PI(16), P(16), M, N, K, G,
                                                           dt, P(16), 1u << 20, NULL, NULL)));
            CHECK(defined_host_status(
                nf4_gemm(NULL, PU(16), PF(16), PF(16), P(16), M, N, K, G, dt, NULL, 0, NULL, NULL)));
            CHECK(defined_host_status(w4a16_gemm_silu_mul(NULL, PU(16), P(16), PU(16), P(16), M, N, K, G, dt, NULL, 0,
                                                          NULL, NULL)));
            CHECK(defined_host_status(
                nf4dq_gemm(NULL, PU(16), PU8(16), PF(16), PF(16), P(16), M, N, K, G, dt, NULL, 0, NULL, NULL)));
            if (a == 0) { /* the weight-only entry points take no M */
              CHECK(defined_host_status(w4a16_dequant(NULL, P(16), PU(16), NULL, P(16), K, N, G, dt, NULL)));
              CHECK(defined_host_status(nf4_dequant(NULL, PF(16), PF(16), P(16), K, N, G, dt, NULL)));
              CHECK(defined_host_status(nf4dq_dequant(NULL, PU8(16), PF(16), PF(16), P(16), K, N, G, dt, NULL)));
              CHECK(defined_host_status(nf4_double_quantize(NULL, K, N, G, PU8(16), PF(16), NULL)));
              CHECK(defined_host_status(w4a16_repack_awq(NULL, PU(16), K, N, G, PU(32), PU(48), NULL)));
              if (d == 0) {
                CHECK(defined_host_status(w4a16_quantize(NULL, K, N, G, PU(16), P(16), PU(16), NULL)));
                CHECK(defined_host_status(nf4_quantize(NULL, K, N, G, PF(16), PU(16), PF(16), NULL)));
                CHECK(defined_host_status(w4a16_act_order_prepack(NULL, PI(16), K, N, G, PU(32), PI(48), NULL,
                                                                  NULL)));
              }
            }
          }
      }
  return 0;
}

int main(void) {
  typedef void (*fn_t)(void);
  const fn_t fns[] = {
      (fn_t)w4a16_gemm,          (fn_t)w4a16_gemv,
      (fn_t)nf4_gemm,            (fn_t)w4a16_dequant,
      (fn_t)nf4_dequant,         (fn_t)w4a16_quantize,
      (fn_t)nf4_quantize,        (fn_t)w4a16_gemv_noalloc,
      (fn_t)w4a16_workspace_bytes, (fn_t)w4a16_act_order_prepack,
      (fn_t)w4a16_gemm_prepacked, (fn_t)w4a16_prepacked_workspace_bytes,
      (fn_t)w4a16_selftest_wait_timeout, (fn_t)w4a16_status_string,
      (fn_t)nf4_default_codebook, (fn_t)nf4dq_gemm,
      (fn_t)nf4dq_dequant,       (fn_t)nf4_double_quantize,
      (fn_t)w4a16_repack_awq,    (fn_t)w4a16_gemm_silu_mul,
      (fn_t)w4a16_gemv_batch,
  };
  for (size_t i = 0; i < sizeof(fns) / sizeof(fns[0]); ++i) CHECK(fns[i] != NULL);

  for (int s = W4A16_OK; s <= W4A16_ERR_TIMEOUT; ++s) {
    const char* msg = w4a16_status_string((w4a16_status)s);
    CHECK(msg != NULL && strlen(msg) >= 2);
  }

  /* pure host functions */
  CHECK(w4a16_workspace_bytes(0, 4096, 4096) == 0);
  CHECK(w4a16_workspace_bytes(1, 4096, 4096) == w4a16_workspace_bytes(1, 4096, 4096));
  CHECK(w4a16_prepacked_workspace_bytes(4, 64, 256) >= (size_t)4 * 256 * 2);

  /* the built-in NF4 table: -1 .. 1, zero at index 7, ascending */
  {
    float cb[16];
    CHECK(nf4_default_codebook(cb) == W4A16_OK);
    CHECK(cb[0] == -1.0f && cb[7] == 0.0f && cb[15] == 1.0f);
    for (int i = 1; i < 16; ++i) CHECK(cb[i] > cb[i - 1]);
    CHECK(nf4_default_codebook(NULL) == W4A16_ERR_INVALID_ARG);
  }

  /* validation: rejected before any launch */
  CHECK(w4a16_gemm(P(16), PU(16), P(16), PU(16), NULL, P(16), 4, 64, 256, 128, (w4a16_dtype)7, NULL, 0, NULL,
                   NULL) == W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemm(P(16), PU(16), P(16), PU(16), NULL, P(16), 4, 60, 256, 128, W4A16_BF16, NULL, 0, NULL, NULL) ==
        W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemm(P(16), PU(16), P(16), PU(16), NULL, P(16), 4, 64, 384, 48, W4A16_BF16, NULL, 0, NULL, NULL) ==
        W4A16_ERR_UNSUPPORTED);
  CHECK(w4a16_gemm(NULL, PU(16), P(16), PU(16), NULL, P(16), 4, 64, 256, 128, W4A16_F16, NULL, 0, NULL, NULL) ==
        W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemv(P(16), PU(16), P(16), PU(16), NULL, P(16), 17, 64, 256, 128, W4A16_BF16, NULL, 0, NULL, NULL) ==
        W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemv_noalloc(P(16), PU(16), P(16), PU(16), NULL, P(16), 17, 64, 256, 128, W4A16_BF16, NULL, NULL) ==
        W4A16_ERR_INVALID_ARG);
  CHECK(nf4_gemm(P(16), PU(16), PF(16), PF(16), P(16), 4, 64, 256, 32, W4A16_BF16, NULL, 0, NULL, NULL) ==
        W4A16_ERR_UNSUPPORTED);
  CHECK(w4a16_selftest_wait_timeout(NULL, 1000, NULL) == W4A16_ERR_INVALID_ARG);

  /* the batch entry: its item layout (the Python binding mirrors it), the
   * empty batch, and an invalid item anywhere in the list rejected before
   * any launch */
  CHECK(sizeof(w4a16_gemv_item) == 72 && offsetof(w4a16_gemv_item, M) == 48 &&
        offsetof(w4a16_gemv_item, dtype) == 64);
  CHECK(w4a16_gemv_batch(NULL, 0, NULL, 0, NULL, NULL) == W4A16_OK);
  CHECK(w4a16_gemv_batch(NULL, -1, NULL, 0, NULL, NULL) == W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemv_batch(NULL, 1, NULL, 0, NULL, NULL) == W4A16_ERR_INVALID_ARG);
  {
    const w4a16_gemv_item two[2] = {
        {P(16), PU(16), P(16), PU(16), NULL, P(16), 1, 64, 256, 128, W4A16_BF16},   /* valid */
        {P(16), PU(16), P(16), PU(16), NULL, P(16), 17, 64, 256, 128, W4A16_BF16},  /* M > 16 */
    };
    CHECK(w4a16_gemv_batch(two, 2, NULL, 0, NULL, NULL) == W4A16_ERR_INVALID_ARG);
  }

  /* size limits */
  CHECK(w4a16_gemm(P(16), PU(16), P(16), PU(16), NULL, P(16), W4A16_MAX_M + 1, 64, 256, 128, W4A16_BF16, NULL, 0,
                   NULL, NULL) == W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemm(P(16), PU(16), P(16), PU(16), NULL, P(16), 4, W4A16_MAX_N + 8, 256, 128, W4A16_BF16, NULL, 0,
                   NULL, NULL) == W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_workspace_bytes(W4A16_MAX_M + 1, 64, 256) == 0);
  CHECK(w4a16_prepacked_workspace_bytes(4, W4A16_MAX_N + 8, 256) == 0);

  /* empty problems: valid no-ops that launch nothing and touch no pointer */
  CHECK(w4a16_gemm(NULL, PU(16), P(16), PU(16), NULL, NULL, 0, 64, 256, 128, W4A16_BF16, NULL, 0, NULL, NULL) ==
        W4A16_OK);
  CHECK(w4a16_gemv_noalloc(NULL, PU(16), P(16), PU(16), NULL, NULL, 0, 64, 256, 128, W4A16_BF16, NULL, NULL) ==
        W4A16_OK);

  if (fuzz_sizes()) return 1;

  printf("ok\n");
  return 0;
}
