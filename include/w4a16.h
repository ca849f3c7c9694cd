/*
 * w4a16.h -- C ABI of the B300 (sm_103a) library for 4-bit weight-only
 * quantized linear layers: Y[M,N] = X[M,K] . W_hat[K,N], with W_hat
 * dequantized on the fly from packed 4-bit codes.
 *
 * Two weight formats:
 *
 *  INT4 (GPTQ / AWQ checkpoints).  Round-to-nearest quantization with one
 *    fp16 scale and one 4-bit zero point per group of group_size rows along K
 *    (cloud.tencent.com/developer/article/2726413 §2.1 asymmetric
 *    quantization stores a zero point; §2.2 group-wise granularity, e.g. 128
 *    elements per scale, or one per channel; "模型量化实践：GPTQ 与 AWQ 在生产
 *    环境的精度与速度权衡" §3.1 bits=4, group_size=128, zero_point=True;
 *    "GPTQ、AWQ与Bitsandbytes" §3.1 node 3: groups of 128, 64 or 32).
 *    group_size: 32, 64, any multiple of 128, or K (one group per column).
 *    Symmetric weights (same §2.1: zero point fixed at 0) are passed with
 *    qzeros == NULL: their signed codes are stored as code + 8, i.e. every
 *    zero point is 8.  An optional act-order map g_idx assigns every K row to
 *    its group ("GPTQ与bitsandbytes对比" GPTQ section, --act-order; "模型量化
 *    实践" §3.1, desc_act=True).
 *      W_hat[k,n] = RNE_dtype((q[k,n] - z[g,n]) * s[g,n]),
 *      g = g_idx[k] or k / group_size,  z = 8 when qzeros is NULL
 *
 *  NF4 (bitsandbytes).  Codes index a 16-entry normal-float codebook, scaled
 *    per block of 64 consecutive K rows by an fp32 absmax ("LLM量化技术深度对比:
 *    GPTQ vs AWQ vs bitsandbytes 2026基准全解析" key-data item 2; "GPTQ、AWQ与
 *    Bitsandbytes：大模型量化三大技术路径深度对比" §2.3 block-wise NF4).
 *      W_hat[k,n] = RNE_dtype(fl32(C[q[k,n]] * absmax[k/64, n]))
 *    With double quantization ("GPTQ、AWQ与Bitsandbytes" §3.3
 *    use_double_quant; §4.3: a scale of the scale is stored) absmax is held
 *    as 8-bit codes with one fp32 second-level scale per 256 consecutive
 *    columns of an absmax row:  absmax = fl32(code * s2)  (nf4dq_* calls).
 *
 * Fusing the dequantization into the product -- never writing 16-bit weights
 * to memory -- is what makes the format fast ("LLM量化技术深度对比" key-data
 * item 1: the same AWQ weights run 10.9x faster with a fused kernel); the
 * product is the plain one.
 *
 * Tensor layouts (all row-major, contiguous, little-endian):
 *   X       [M, K]     fp16 or bf16 (the compute dtype)
 *   Y       [M, N]     same dtype as X
 *   qweight uint32 [K/8, N]: code of row 8i+j, column n in bits 4j..4j+3 of
 *                      word [i, n] (8 codes per word, packed along K)
 *   scales  fp16 [G, N], G = K / group_size  (INT4)
 *   qzeros  uint32 [G, N/8]: zero point of column 8c+j in bits 4j.. of
 *                      word [g, c] (packed along N; the stored value is z);
 *                      NULL: symmetric weights (every zero point 8)
 *   g_idx   int32 [K]  row -> group, each value in [0, G); NULL means k/group_size
 *   absmax  fp32 [K/64, N]                  (NF4)
 *   absmax_q  uint8 [K/64, N], absmax_s2 fp32 [K/64, ceil(N/256)]
 *                      (NF4 with double-quantized absmax)
 *   codebook16 fp32 [16], ascending         (NF4; NULL = the built-in table,
 *                      see nf4_default_codebook)
 *
 * Conventions shared by every entry point:
 *  - Every pointer is a device pointer owned by the caller.  The library
 *    allocates and frees nothing and never synchronises; each call is
 *    enqueued on `stream` and returns as soon as it is enqueued.
 *  - The return value reports host-side errors only: argument validation
 *    (nothing is launched) and launch errors.  Faults inside a kernel surface
 *    at the caller's next synchronisation, as for any CUDA call.
 *  - Pointers must be 16-byte aligned.  N and K must be multiples of 8;
 *    K a multiple of the group / block size.
 *  - Sizes: 0 <= M <= W4A16_MAX_M, 0 <= N <= W4A16_MAX_N and
 *    0 < K <= W4A16_MAX_K; outside them W4A16_ERR_INVALID_ARG, nothing
 *    launched.
 *  - M == 0 or N == 0 is a valid empty problem: W4A16_OK, nothing launched.
 *  - The decode and tensor-core product kernels are launched as programmatic
 *    dependents of the kernel before them on `stream`, so their start
 *    overlaps its end.  Until that kernel has completed they only set up
 *    their own barriers and tensor memory and (decode) prefetch weight lines
 *    into L2 (the device's point of coherence, so a prefetch cannot return
 *    stale data); every read or write of a caller's buffer happens after it.
 *    Callers need no ordering beyond the stream's.
 *  - The dtype of X and Y is `dtype`; scales are always fp16, absmax fp32.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  W4A16_OK = 0,
  W4A16_ERR_INVALID_ARG = 1, /* bad shape, null or misaligned pointer, bad dtype */
  W4A16_ERR_UNSUPPORTED = 2, /* valid request the library does not implement */
  W4A16_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  W4A16_ERR_TIMEOUT = 4      /* a device-side bounded wait expired (written to dev_status) */
} w4a16_status;

typedef enum { W4A16_F16 = 0, W4A16_BF16 = 1 } w4a16_dtype;

/* Largest token count the split-K decode kernel (w4a16_gemv) accepts. */
#define W4A16_GEMV_MAX_M 16

/* Size limits of every entry point.  M: 65535 token tiles of 128 (a grid
 * dimension); N: 4096 column blocks of 256 (the split-K ticket area); K:
 * 65535 packed word-rows of 8 (a grid dimension), so the largest K that is a
 * multiple of 128 is 524160. */
#define W4A16_MAX_M 8388480
#define W4A16_MAX_N 1048576
#define W4A16_MAX_K 524280

/*
 * Y = X . W_hat for the INT4 format, any M >= 0.  Dispatches on M: M <= 16
 * runs the split-K decode kernel (as w4a16_gemv), larger M the tcgen05
 * tensor-core kernel: output tiles of 128 columns x up to 256 tokens run
 * whole in full waves of the SMs, and the tiles left over for a ragged last
 * wave (all tiles, when they do not fill one wave) are split along K (fp32
 * partial tiles summed in a fixed order: deterministic).
 *   group_size: 32, 64, a multiple of 128, or K; others W4A16_ERR_UNSUPPORTED.
 *   qzeros: NULL for symmetric weights.
 *   g_idx with M > 16: the tensor-core kernel keeps every group's (scale,
 *     zero) of its 128 columns in shared memory, which holds at most 290
 *     groups (K <= 37120 at group_size 128); beyond that the call returns
 *     W4A16_ERR_UNSUPPORTED -- prepack such checkpoints
 *     (w4a16_act_order_prepack).
 *   workspace: device scratch of at least w4a16_workspace_bytes(M, N, K)
 *     bytes, zero-filled by the caller before its first use.  Its first part
 *     holds the split-K tickets, which every call that completes leaves at
 *     zero again; the rest is scratch for fp32 partial sums.  After a call
 *     whose status word reports W4A16_ERR_TIMEOUT, zero-fill it again.  May
 *     be NULL when that size is 0.  Calls that run at the same time must not
 *     share a workspace.
 *   dev_status: NULL, or a device int the caller zeroes; a kernel whose
 *     bounded wait expires writes W4A16_ERR_TIMEOUT there and stops early
 *     (its Y is then undefined); a g_idx entry outside [0, K/128) writes
 *     W4A16_ERR_INVALID_ARG there (the entry is clamped into range, so no
 *     memory outside the scale and zero arrays is read; Y is meaningless).
 */
w4a16_status w4a16_gemm(const void* X, const uint32_t* qweight, const void* scales,
                        const uint32_t* qzeros, const int32_t* g_idx, void* Y,
                        int M, int N, int K, int group_size, w4a16_dtype dtype,
                        void* workspace, size_t workspace_bytes, int* dev_status,
                        cudaStream_t stream);

/* Y = X . W_hat for the INT4 format and 0 <= M <= W4A16_GEMV_MAX_M: the
 * weight-streaming decode kernel (split along K, fp32 partial sums reduced
 * in a fixed order, so results are deterministic).  Arguments as w4a16_gemm. */
w4a16_status w4a16_gemv(const void* X, const uint32_t* qweight, const void* scales,
                        const uint32_t* qzeros, const int32_t* g_idx, void* Y,
                        int M, int N, int K, int group_size, w4a16_dtype dtype,
                        void* workspace, size_t workspace_bytes, int* dev_status,
                        cudaStream_t stream);

/*
 * A list of decode products launched by one call: items[i] holds the
 * arguments of one w4a16_gemv call (same meaning, layouts and limits), and
 * the products run in the order given on `stream`, each computing exactly
 * what w4a16_gemv computes for its item.  They use `workspace` in turn, so
 * it must hold at least the largest w4a16_workspace_bytes(M, N, K) of the
 * items.  The call spares a caller that runs many small products per step
 * (a decoder's linears for one token) a library call per product.
 *   items: host memory, read during the call only (count 0: nothing to do).
 *   Errors: every item is checked before anything is launched; an invalid
 *   item returns its status (W4A16_ERR_INVALID_ARG or _UNSUPPORTED) with
 *   nothing launched.  A launch error returns W4A16_ERR_CUDA after the items
 *   before it were launched.
 */
typedef struct w4a16_gemv_item {
  const void* X;
  const uint32_t* qweight;
  const void* scales;
  const uint32_t* qzeros; /* NULL: symmetric */
  const int32_t* g_idx;   /* NULL: groups in order */
  void* Y;
  int M, N, K, group_size;
  w4a16_dtype dtype;
} w4a16_gemv_item;

w4a16_status w4a16_gemv_batch(const w4a16_gemv_item* items, int count, void* workspace, size_t workspace_bytes,
                              int* dev_status, cudaStream_t stream);

/*
 * Fused decoder-MLP activation: A[M, F] = SiLU(X . W_hat[:, :F]) * (X . W_hat[:, F:])
 * for a gate_up weight of N = 2F columns (gate in columns [0, F), up in
 * [F, 2F)), SiLU(t) = t / (1 + e^-t), both products and the activation in
 * fp32 and one rounding of A to dtype.  The 2F-wide product never goes to
 * memory: per-token latency follows the bytes moved per forward
 * ("LLM量化技术深度对比" key-data items 1 and 3), and the activation is the
 * gate_up product's epilogue.  The pages do not spell the layer out; the
 * gate-then-up column order is this library's reading.
 *   A: [M, N/2] in dtype; N a multiple of 16.  No act-order map (prepack such
 *   checkpoints).  Other arguments, workspace and limits as w4a16_gemm.
 */
w4a16_status w4a16_gemm_silu_mul(const void* X, const uint32_t* qweight, const void* scales,
                                 const uint32_t* qzeros, void* A, int M, int N, int K, int group_size,
                                 w4a16_dtype dtype, void* workspace, size_t workspace_bytes, int* dev_status,
                                 cudaStream_t stream);

/* Y = X . W_hat for the NF4 format, any M >= 0.  blocksize: 64.
 * codebook16: a device table of 16 fp32 values, or NULL for the library's
 * built-in table (nf4_default_codebook).  Other arguments as w4a16_gemm. */
w4a16_status nf4_gemm(const void* X, const uint32_t* qweight, const float* absmax,
                      const float* codebook16, void* Y, int M, int N, int K, int blocksize,
                      w4a16_dtype dtype, void* workspace, size_t workspace_bytes,
                      int* dev_status, cudaStream_t stream);

/* W_out[K, N] (dtype) = W_hat, the INT4 dequantization written out; bit-exact
 * with the definition above.  g_idx may be NULL; qzeros NULL: symmetric. */
w4a16_status w4a16_dequant(const uint32_t* qweight, const void* scales, const uint32_t* qzeros,
                           const int32_t* g_idx, void* W_out, int K, int N, int group_size,
                           w4a16_dtype dtype, cudaStream_t stream);

/* W_out[K, N] (dtype) = W_hat for NF4; bit-exact with the definition above.
 * codebook16: as nf4_gemm (NULL = built-in table). */
w4a16_status nf4_dequant(const uint32_t* qweight, const float* absmax, const float* codebook16,
                         void* W_out, int K, int N, int blocksize, w4a16_dtype dtype,
                         cudaStream_t stream);

/*
 * Round-to-nearest INT4 quantization of fp32 W[K, N] with contiguous groups
 * ("GPTQ与bitsandbytes对比" GPTQ section: RTN is the plain baseline quantizer;
 * cloud.tencent.com/developer/article/2726413 §2.1-2.2).  Per group g and
 * column n, in fp64:
 *   asymmetric (qzeros given):
 *     mn = min(min_k w, 0), mx = max(max_k w, 0), s = RNE_fp16((mx - mn) / 15)
 *     (s = 1 if that is 0), z = clamp(rint(-mn / s), 0, 15),
 *     q = clamp(rint(w / s) + z, 0, 15)      (rint: half to even)
 *   symmetric (qzeros == NULL): s = RNE_fp16(max_k |w| / 7) (1 if 0),
 *     q = clamp(rint(w / s), -8, 7) + 8
 * Outputs qweight [K/8, N], scales fp16 [G, N], qzeros [G, N/8].
 */
w4a16_status w4a16_quantize(const float* W, int K, int N, int group_size, uint32_t* qweight,
                            void* scales, uint32_t* qzeros, cudaStream_t stream);

/*
 * NF4 quantization of fp32 W[K, N] ("GPTQ、AWQ与Bitsandbytes" §2.3: block-wise,
 * calibration-free).  absmax = max |w| over each block of 64 rows of a
 * column; v = fl32(w / absmax); q = the index of the codebook entry nearest
 * to v (exact comparison, ties to the lower index; code 7 for an all-zero
 * block).  Outputs qweight [K/8, N] and absmax fp32 [K/64, N].
 * codebook16: as nf4_gemm (NULL = built-in table).
 */
w4a16_status nf4_quantize(const float* W, int K, int N, int blocksize, const float* codebook16,
                          uint32_t* qweight, float* absmax, cudaStream_t stream);

/*
 * Allocation-free decode: the same product as w4a16_gemv (INT4, 0 <= M <= 16,
 * same arguments and results) for callers that cannot allocate a workspace --
 * e.g. code that runs inside someone else's memory pool, or on a path where
 * cudaMalloc (which may synchronise the device or fail when memory is
 * fragmented) is not allowed.  The pages have no counterpart; this is a
 * library convenience.
 *
 * The scratch it needs lives in the library: one static device array of
 * W4A16_NOALLOC_SCRATCH_BYTES per GPU, held from the time the library is
 * loaded on that GPU until the process exits.  Calls that would need more
 * scratch than that return W4A16_ERR_UNSUPPORTED (with the current split-K
 * plan every M <= 16 fits).  The function allocates and frees nothing.
 *  - The first call on each device looks up the array's address
 *    (cudaGetSymbolAddress, with that device current) and keeps it.  A
 *    cudaDeviceReset makes the kept address stale: do not call this function
 *    on a device after resetting it in the same process.
 *  - Each call clears the scratch area that must start at zero, on `stream`.
 *  - All calls share the one array and it keeps the last call's contents:
 *    calls that may run at the same time on the GPU (different streams with
 *    no ordering between them) race and must not be issued.
 */
#define W4A16_NOALLOC_SCRATCH_BYTES (16u << 20)
w4a16_status w4a16_gemv_noalloc(const void* X, const uint32_t* qweight, const void* scales,
                                const uint32_t* qzeros, const int32_t* g_idx, void* Y, int M, int N, int K,
                                int group_size, w4a16_dtype dtype, int* dev_status, cudaStream_t stream);

/*
 * NF4 with double-quantized absmax: the same product as nf4_gemm with
 * absmax = fl32(absmax_q * s2), s2 = absmax_s2[k/64, n/256] (see the format
 * notes above; the 4-bit codes are those of the first level, computed with
 * the original absmax).  absmax_q uint8 [K/64, N], absmax_s2 fp32
 * [K/64, ceil(N/256)].  Other arguments as nf4_gemm.
 */
w4a16_status nf4dq_gemm(const void* X, const uint32_t* qweight, const uint8_t* absmax_q,
                        const float* absmax_s2, const float* codebook16, void* Y, int M, int N, int K,
                        int blocksize, w4a16_dtype dtype, void* workspace, size_t workspace_bytes,
                        int* dev_status, cudaStream_t stream);

/* W_out[K, N] (dtype) = W_hat for NF4 with double-quantized absmax;
 * bit-exact with the definition above. */
w4a16_status nf4dq_dequant(const uint32_t* qweight, const uint8_t* absmax_q, const float* absmax_s2,
                           const float* codebook16, void* W_out, int K, int N, int blocksize,
                           w4a16_dtype dtype, cudaStream_t stream);

/*
 * Second-level quantization of an NF4 absmax array [K/blocksize, N] (fp32):
 * per row and block of 256 consecutive columns, s2 = fl32(max / 255) (the
 * fp64 quotient rounded once to fp32; 1 if the block is all zero) and
 * code = clamp(rint(absmax / s2), 0, 255) with the division in fp64.
 * Outputs absmax_q uint8 [K/blocksize, N] and absmax_s2 fp32
 * [K/blocksize, ceil(N/256)].  The pages do not describe bitsandbytes' own
 * second level; this is the plain reading of "a scale of the scale".
 */
w4a16_status nf4_double_quantize(const float* absmax, int K, int N, int blocksize, uint8_t* absmax_q,
                                 float* absmax_s2, cudaStream_t stream);

/* Bytes of workspace w4a16_gemm / w4a16_gemv / nf4_gemm need for this
 * shape (0 when none is needed, and for shapes outside the size limits,
 * which those calls reject).  Pure host function.  For M > 16: the ticket
 * area (128 KiB) plus one fp32 partial tile (128 columns x BT tokens) per
 * K part of each leftover tile, where BT = min(round_up(M, 32), 256) (128
 * with g_idx), rest = tiles mod 148, parts = min(148 / rest, (K / 64) / 8)
 * rounded to group-aligned ranges; 0 when no tile is split. */
size_t w4a16_workspace_bytes(int M, int N, int K);

/*
 * Act-order prepack, run once when a checkpoint is loaded.  With act-order
 * ("GPTQ与bitsandbytes对比" GPTQ section, --act-order; "模型量化实践" §3.1,
 * desc_act) the rows of one group are scattered over K.  This reorders them
 * so that group g occupies rows [g*128, (g+1)*128), each group's rows keeping
 * their original order:
 *   perm[j]            = the original row of sorted row j
 *   qweight_sorted row j = qweight row perm[j]          (same nibble packing)
 * after which  Y = X . W_hat = X[:, perm] . W_hat_sorted  with plain groups
 * (scales and qzeros are unchanged).  Every group must hold exactly
 * group_size rows (GPTQ's layout); otherwise *dev_status (when not NULL)
 * receives W4A16_ERR_UNSUPPORTED and the outputs are unspecified -- use the
 * g_idx entry points for such maps.  Entries of g_idx outside [0, K/128) are
 * never matched, so they show up the same way.
 *   qweight_sorted: uint32 [K/8, N], not aliasing qweight; perm: int32 [K].
 *   Both caller-owned device buffers, written asynchronously on `stream`.
 */
w4a16_status w4a16_act_order_prepack(const uint32_t* qweight, const int32_t* g_idx, int K, int N,
                                     int group_size, uint32_t* qweight_sorted, int32_t* perm,
                                     int* dev_status, cudaStream_t stream);

/*
 * Y = X . W_hat for act-order weights prepacked by w4a16_act_order_prepack:
 * X's columns are gathered by perm into the workspace, then the plain-group
 * kernels run (the decode kernel for M <= 16, the tensor-core kernel above),
 * so act-order costs one gather of M*K values per call.  Arguments as
 * w4a16_gemm, with perm in place of g_idx; workspace: at least
 * w4a16_prepacked_workspace_bytes(M, N, K) bytes, zero-filled before its first
 * use.  Its first part is laid out as w4a16_gemm's workspace (always at least
 * the split-K ticket area, whatever M is, so one buffer can serve every entry
 * point); the rest is scratch for the gathered X.  perm values outside
 * [0, K) are clamped (no access outside X).
 */
w4a16_status w4a16_gemm_prepacked(const void* X, const uint32_t* qweight_sorted, const void* scales,
                                  const uint32_t* qzeros, const int32_t* perm, void* Y, int M, int N,
                                  int K, int group_size, w4a16_dtype dtype, void* workspace,
                                  size_t workspace_bytes, int* dev_status, cudaStream_t stream);

/* Bytes of workspace w4a16_gemm_prepacked needs (0 for shapes outside the
 * size limits).  Pure host function. */
size_t w4a16_prepacked_workspace_bytes(int M, int N, int K);

/*
 * Repack an AWQ checkpoint ("模型量化实践" §3.1: zero_point=True,
 * q_group_size, w_bit=4, version="GEMM"; served by a faster kernel's layout
 * in "LLM量化技术深度对比" §5) into this library's layout, once at load.
 * The pages do not print AWQ's packing; the layout read here is AWQ's
 * published GEMM layout (equality with files written by AWQ's own tools is
 * not verified here):
 *   qweight_awq int32 [K, N/8]: word [k, c] = row k, columns 8c .. 8c+7, with
 *                               column 8c + ORDER[j] in bits 4j .. 4j+3,
 *                               ORDER = (0, 2, 4, 6, 1, 3, 5, 7)
 *   qzeros_awq  int32 [G, N/8]: zero points packed the same way (NULL for
 *                               symmetric weights, with qzeros NULL too)
 * Outputs qweight [K/8, N] and qzeros [G, N/8] in this library's layout
 * (caller-owned device buffers, not aliasing the inputs); the fp16 scales
 * [G, N] are already in this library's layout.  G = K / group_size.
 */
w4a16_status w4a16_repack_awq(const uint32_t* qweight_awq, const uint32_t* qzeros_awq, int K, int N,
                              int group_size, uint32_t* qweight, uint32_t* qzeros, cudaStream_t stream);

/*
 * Self-test of the bounded device-side wait that every pipeline wait in this
 * library uses (no counterpart in the pages: a library diagnostic).  One warp
 * waits on a barrier that nothing completes; after limit_ns (1 ns .. 10 s) of
 * wall-clock time the wait gives up, writes W4A16_ERR_TIMEOUT to *dev_status
 * and the kernel returns, so the caller can check that a stuck pipeline ends
 * with a status rather than a hang and that the context stays usable.
 * dev_status must not be NULL.
 */
w4a16_status w4a16_selftest_wait_timeout(int* dev_status, unsigned long long limit_ns, cudaStream_t stream);

/*
 * The library's built-in NF4 table, written to out16[0..15] (host memory):
 * the table NULL stands for in nf4_gemm, nf4_dequant and nf4_quantize.  NF4
 * places its 16 values where normally distributed weights are dense
 * ("LLM量化技术深度对比" key-data item 2; "GPTQ、AWQ与Bitsandbytes" §2.3:
 * built from a normal-distribution prior).  With d = 1 - (1/30 + 1/32) / 2
 * and Phi the standard-normal CDF:
 *   C[7] = 0,
 *   C[8 + i] =  Phi^-1(d - (d - 1/2) i / 8) / Phi^-1(d),   i = 0..7,
 *   C[6 - i] = -Phi^-1(d - (d - 1/2) i / 7) / Phi^-1(d),   i = 0..6,
 * each quotient formed in double and rounded once to fp32 (C[0] = -1,
 * C[15] = 1, ascending).  The pages print no table; equality with any other
 * library's shipped table is not claimed.  Pure host function;
 * W4A16_ERR_INVALID_ARG if out16 is NULL.
 */
w4a16_status nf4_default_codebook(float* out16);

/* Static, human-readable text for a status code.  Pure host function. */
const char* w4a16_status_string(w4a16_status status);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
