/*
 * dg.h — C ABI of the GB300 (sm_103a) FP8 fine-grained-scaled GEMM library.
 *
 * The operation is DeepGEMM-style FP8 matrix multiplication,
 *     D[M,N] = A[M,K] . B[N,K]^T,
 * with E4M3 operands, one fp32 scale per 1x128 K-group of A (per token) and
 * one per 128x128 block of B, the tensor-core partial sum of every 128-wide K
 * block promoted to fp32 on the CUDA cores and scaled there
 *     acc = fmaf(P_kb[m,n], sfa[m,kb] * sfb[n/128,kb], acc),  kb ascending,
 * and a bf16 (round-to-nearest-even) output.  Sources, by page title and
 * section:
 *   "DeepGEMM：一款支持FP8通用矩阵乘法(GEMM)的开源库": 功能特色 (高性能, 支持多种数据
 *     排列方式, 细粒度缩放功能) and 技术细节 (两级累加技术, 非标准块大小支持,
 *     线程专业化技术, 统一的计算任务调度系统);
 *   the 2kiu.com DeepGEMM tutorial: 4.1-4.4 (tiling, pipelining, edges,
 *     precision control) and 5.3 (no hidden temporary allocations).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller, except
 *     where marked "host".  The library never allocates, frees or copies the
 *     caller's memory, never synchronises `stream` (except
 *     dg_read_device_status) and never prints.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All work is enqueued asynchronously on it.
 *   - Arguments are checked before anything is enqueued; a failed check
 *     returns an error code and enqueues nothing.  Launch failures return
 *     DG_ERR_CUDA.  Nothing is ever thrown across the ABI.
 *   - Device pointers must be 16-byte aligned (DG_ERR_MISALIGNED otherwise).
 *   - K must be a positive multiple of 128 and N a positive multiple of 8
 *     (16-byte output rows); DG_ERR_UNSUPPORTED_SHAPE otherwise.  M and N need
 *     not be multiples of the tile: edge tiles read zeros and store clipped.
 *   - E4M3: bias 7, max 448, NaN 0x7F/0xFF, no infinities.
 *   - Layouts (all row-major, no padding between rows):
 *       A    uint8 E4M3 [M][K]                (K-major)
 *       B    uint8 E4M3 [N][K]                (K-major, i.e. the "NT" form)
 *       SFA  fp32 [K/128][ldsfa], ldsfa = round_up(M, 4): sfa[kb*ldsfa + m]
 *       SFB  fp32 [ceil(N/128)][K/128]:                   sfb[nb*(K/128) + kb]
 *       D    bf16 bits (uint16) [M][N]
 *   - The device status word (dg_read_device_status) collects problems that
 *     only the GPU can see: bad MoE metadata and pipeline timeouts.
 *   - Thread safety: entry points may be called concurrently from several
 *     host threads; per-device setup happens once behind a lock.
 *   - Stream order: the kernels let the next kernel of the stream start its
 *     set-up early (programmatic dependent launch) and wait for the previous
 *     kernel to complete before reading its outputs, with one exception: a
 *     dense GEMM copies the first K blocks of B before that wait.  B (the
 *     weights) must therefore not be written by the kernel immediately before
 *     the call in the same stream if that kernel signals its dependents early
 *     (the activation quantiser and the GEMMs of this library do; kernels that
 *     do not use programmatic launch never let the GEMM start early).
 */
#ifndef DG_H_
#define DG_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DG_OK = 0,
    DG_ERR_INVALID_ARG = 1,       /* null pointer, non-positive size, bad enum */
    DG_ERR_UNSUPPORTED_SHAPE = 2, /* K % 128 != 0, N % 8 != 0, size limits */
    DG_ERR_MISALIGNED = 3,        /* a device pointer is not 16-byte aligned */
    DG_ERR_UNSUPPORTED_DEVICE = 4,/* current device is not compute capability 10.3 */
    DG_ERR_CUDA = 5,              /* a CUDA runtime/driver call or launch failed */
    DG_ERR_DEVICE_TIMEOUT = 6     /* dg_read_device_status saw a pipeline timeout */
} dg_status_t;

typedef enum { DG_DTYPE_F32 = 0, DG_DTYPE_BF16 = 1 } dg_dtype_t;

typedef enum { DG_LAYOUT_DENSE = 0, DG_LAYOUT_CONTIGUOUS = 1, DG_LAYOUT_MASKED = 2 } dg_layout_t;

/* Bits of the device status word. */
#define DG_DEVFLAG_MASKED_M_CLAMPED 0x1 /* some masked_m[g] < 0 or > max_m (clamped) */
#define DG_DEVFLAG_BAD_EXPERT 0x2       /* an m_indices entry >= G (block or row skipped) */
#define DG_DEVFLAG_MIXED_BLOCK 0x4      /* a 128-row block held rows of two experts */
#define DG_DEVFLAG_TIMEOUT 0x8          /* a pipeline wait gave up; outputs are incomplete */

/* Tile plan chosen for a problem (host-only query, see dg_query_plan). */
typedef struct {
    int block_m;   /* rows of D per tile */
    int block_n;   /* columns of D per tile */
    int stages;    /* depth of the shared-memory operand ring */
    int num_tiles; /* tiles in the problem (masked layout: upper bound, G*ceil(max_m/BM)*n-blocks) */
    int grid;      /* persistent CTAs launched */
    int smem_bytes;/* dynamic shared memory per CTA */
} dg_plan_t;

/* Per-token 1x128 activation quantiser ("DeepGEMM：一款支持FP8通用矩阵乘法(GEMM)的开源库",
 * 功能特色/细粒度缩放功能; 2kiu.com tutorial 4.4: scales from data statistics,
 * saturation of out-of-range values).
 * For each row m and K-group kb (128 values):
 *     amax = max |x|;  s = max(amax, 1e-4f) / 448.0f  (IEEE fp32 division);
 *     q    = E4M3 round-to-nearest-even, saturating, of fp32(x / s);
 *     sfa[kb*ldsfa + m] = s,  ldsfa = round_up(M, 4).
 *   x       [M][K] fp32 (x_dtype = DG_DTYPE_F32) or bf16 bits (DG_DTYPE_BF16)
 *   q       out, uint8 E4M3 [M][K]
 *   sfa     out, fp32 [K/128][round_up(M,4)]; columns m >= M are not written
 * Bit-exact: the same inputs give the same bytes and scales on every run. */
dg_status_t dg_quant_act_1x128(const void *x, int x_dtype, uint8_t *q, float *sfa, int M, int K,
                               void *stream);

/* Per-block 128x128 weight quantiser (same rule per block; weights are
 * quantised once, offline).  G independent [N][K] matrices back to back.
 *   w    fp32 [G][N][K];  q out uint8 [G][N][K];
 *   sfb  out fp32 [G][ceil(N/128)][K/128] */
dg_status_t dg_quant_weight_128x128(const float *w, uint8_t *q, float *sfb, int G, int N, int K,
                                    void *stream);

/* Dense NT GEMM ("DeepGEMM：一款支持FP8通用矩阵乘法(GEMM)的开源库",
 * 功能特色/支持多种数据排列方式: the normal layout; 技术细节/两级累加技术).
 *   a [M][K], sfa [K/128][round_up(M,4)], b [N][K], sfb [ceil(N/128)][K/128],
 *   d out bf16 [M][N] (every element written). */
dg_status_t dg_fp8_gemm_nt(const uint8_t *a, const float *sfa, const uint8_t *b, const float *sfb,
                           uint16_t *d, int M, int N, int K, void *stream);

/* MoE grouped GEMM, contiguous layout (same page, 支持多种数据排列方式 and
 * 应用场景/混合专家模型).  The experts' rows are concatenated in A; m_indices[m]
 * is the expert of row m, or -1 for a padding row.  Every expert's segment
 * starts at a multiple of 128 rows (pad with -1 rows), so each 128-row block
 * belongs to one expert, read from its first row on the device (no host sync).
 *   a [sum_M][K], sfa [K/128][sum_M], b [G][N][K], sfb [G][ceil(N/128)][K/128],
 *   m_indices int32 [sum_M] (device), d out bf16 [sum_M][N].
 * Rows whose index is -1 are not written.  sum_M must be a multiple of 128.
 * A block whose first index is >= G, or a row whose index disagrees with its
 * block's, is skipped and flagged in the device status word. */
dg_status_t dg_fp8_grouped_contiguous(const uint8_t *a, const float *sfa, const uint8_t *b,
                                      const float *sfb, uint16_t *d, const int32_t *m_indices,
                                      int sum_M, int N, int K, int G, void *stream);

/* MoE grouped GEMM, masked layout (same page, 支持多种数据排列方式).  Expert g
 * owns rows [g*max_m, (g+1)*max_m) of A and D of which the first masked_m[g]
 * are valid; masked_m lives on the device and is read by the kernel, so the
 * call enqueues the same work whatever its contents and can be captured in a
 * CUDA graph and replayed after masked_m changes.
 *   a [G][max_m][K], sfa [G][K/128][round_up(max_m,4)], b [G][N][K],
 *   sfb [G][ceil(N/128)][K/128], masked_m int32 [G] (device),
 *   d out bf16 [G][max_m][N]: rows >= masked_m[g] are never written.
 * masked_m[g] outside [0, max_m] is clamped and flagged.  expected_m is a
 * host hint of the typical masked_m (0 = unknown: every buffer full) used
 * only to pick the tile width (the m-blocks an expert is expected to fill
 * decide how many tiles a wave has); it never changes results and the launch
 * stays the same whatever masked_m holds. */
dg_status_t dg_fp8_grouped_masked(const uint8_t *a, const float *sfa, const uint8_t *b,
                                  const float *sfb, uint16_t *d, const int32_t *masked_m, int G,
                                  int max_m, int N, int K, int expected_m, void *stream);

/* The three GEMMs above with the output re-quantised in the epilogue as the
 * next GEMM's activation operand (2kiu.com tutorial 7: fuse the operations
 * around a GEMM so that its result makes no extra round trip; DeepGEMM page
 * 应用场景/混合专家模型: the expert GEMMs run back to back).  Instead of bf16 D the
 * call writes, for every row it would have written:
 *   q   out uint8 E4M3 codes, D's layout ([M][N], [sum_M][N], [G][max_m][N]);
 *   sfo out fp32 one scale per 1x128 group of the row, M-major like sfa:
 *       dense [N/128][round_up(M,4)], contiguous [N/128][sum_M],
 *       masked [G][N/128][round_up(max_m,4)].
 * Per row and 128-column group: D rounded to bf16 (round to nearest even),
 * then the dg_quant_act_1x128 rule on those values, so that the result equals
 * dg_fp8_gemm_nt (or the grouped call) followed by dg_quant_act_1x128 on D,
 * bit for bit.  Rows not written by the bf16 call (padding, masked tails)
 * keep their q bytes and sfo entries.  N must be a multiple of 128
 * (DG_ERR_UNSUPPORTED_SHAPE); q and sfo 16-byte aligned (DG_ERR_MISALIGNED).
 * Dense and contiguous problems take the bf16 call's CTA-pair tiles where its
 * plan has them (256 x 256; DG_FORCE_BN=128 or 256 pins the choice), every
 * other problem 128 x 128 tiles on one SM.  The masked call's expected_m is
 * accepted so that its arguments match dg_fp8_grouped_masked; its tiles are
 * always 128 x 128, so the hint does not change its plan. */
dg_status_t dg_fp8_gemm_nt_q(const uint8_t *a, const float *sfa, const uint8_t *b, const float *sfb,
                             uint8_t *q, float *sfo, int M, int N, int K, void *stream);
dg_status_t dg_fp8_grouped_contiguous_q(const uint8_t *a, const float *sfa, const uint8_t *b,
                                        const float *sfb, uint8_t *q, float *sfo,
                                        const int32_t *m_indices, int sum_M, int N, int K, int G,
                                        void *stream);
dg_status_t dg_fp8_grouped_masked_q(const uint8_t *a, const float *sfa, const uint8_t *b,
                                    const float *sfb, uint8_t *q, float *sfo, const int32_t *masked_m,
                                    int G, int max_m, int N, int K, int expected_m, void *stream);

/* ------------------------------------------------------------------------
 * Beyond per-group-scaled FP8: the two formats the 2kiu.com DeepGEMM tutorial
 * names beside it.  Both keep the accumulator in tensor memory across all of
 * K (no promotion on the CUDA cores): 256 x 256 tiles on pairs of SMs when
 * there are at least half the SMs' worth of them, 128 x 256 tiles on one SM
 * otherwise (the environment variable DG_FORCE_ACC_PAIR=1 or 0 overrides the
 * choice).  The result does not depend on the choice beyond the tensor
 * core's summation order.
 * ------------------------------------------------------------------------ */

/* BF16 GEMM (2kiu.com tutorial 1 and 2.2: BF16 beside FP8 as a
 * low-precision format):
 *     D[m][n] = bf16_rn(sum_k A[m][k] * B[n][k])
 * with bf16 operands and an fp32 accumulator (the tensor core's summation of
 * the exact products; on integer-valued inputs whose sums stay exact in
 * fp32 the result is unique).
 *   a bf16 bits [M][K] (K-major), b bf16 bits [N][K] (K-major),
 *   d out bf16 [M][N].
 * K must be a multiple of 64 and N of 8 (DG_ERR_UNSUPPORTED_SHAPE). */
dg_status_t dg_bf16_gemm_nt(const uint16_t *a, const uint16_t *b, uint16_t *d, int M, int N, int K,
                            void *stream);

/* MX (micro-scaling) quantiser (2kiu.com tutorial 7: MX formats with finer
 * scale granularity; the format as the OCP Microscaling Formats (MX) v1.0
 * specification defines it, with E4M3 elements): per row and 32-wide block
 * of K values, e = floor(log2 amax) - 8 clamped to [-127, 127] (an all-zero
 * block takes -127), scale code e + 127 (E8M0), codes E4M3 round-to-nearest-
 * even with saturation of x * 2^-e (the block maximum lands in [256, 448]).
 *   x fp32 [R][K]; q out E4M3 [R][K];
 *   sx out E8M0, chunk-major: [K/128][R] 32-bit words, the word of row r and
 *   128-wide chunk g holding in byte j (little-endian) the scale code of the
 *   row's 32-wide block 4 g + j.  (The row-major [R][K/32] codes, permuted so
 *   that the GEMM reads one chunk's scales of consecutive rows as one
 *   contiguous run, the order in which the tensor core takes them: four
 *   scales per row per 128 K values.)
 * K must be a multiple of 128.  Bit-exact and deterministic. */
dg_status_t dg_quant_mx_1x32(const float *x, uint8_t *q, uint8_t *sx, int R, int K, void *stream);

/* MX GEMM (same sources): E4M3 operands with one E8M0 scale per 32
 * consecutive K values of each row, applied per block by the tensor core
 * (tcgen05.mma kind::mxf8f6f4, block scaling):
 *     D[m][n] = bf16_rn(sum_kb 2^(sa[m][kb]-127) 2^(sb[n][kb]-127)
 *                              sum_{k in block kb} dec(A[m][k]) dec(B[n][k]))
 * with an fp32 accumulator.
 *   a E4M3 [M][K], b E4M3 [N][K]; sa, sb E8M0 scales in the chunk-major
 *   layout dg_quant_mx_1x32 writes ([K/128][M] and [K/128][N] 32-bit words,
 *   byte j of a word = block 4 g + j of chunk g); d out bf16 [M][N].
 * K must be a multiple of 128 and N of 8 (DG_ERR_UNSUPPORTED_SHAPE). */
dg_status_t dg_mx_gemm_nt(const uint8_t *a, const uint8_t *sa, const uint8_t *b, const uint8_t *sb,
                          uint16_t *d, int M, int N, int K, void *stream);

/* Host-only: the tile plan the bf16-output GEMM entry points would launch for
 * this problem on a GPU with `num_sms` SMs (num_sms <= 0: the current
 * device's).  Makes no CUDA call when num_sms > 0.  For DG_LAYOUT_DENSE, M is
 * the row count; CONTIGUOUS: M = sum_M; MASKED: M = max_m, and expected_m the
 * masked call's hint (0 = none; ignored by the other layouts; < 0 invalid).
 * Dense and contiguous problems with at least 16 K blocks that fill a wave of
 * CTA pairs take 256 x 256 tiles on pairs of SMs (block_m = 256; contiguous:
 * at most 1024 blocks of 128 rows); otherwise tiles are 128 x 192 when the
 * problem has at least one full wave of them, else 128 x 128 or 128 x 96,
 * whichever leaves the busiest CTA the fewest operand bytes.  The
 * environment variable DG_FORCE_BN=96|128|192|256 (read at every call) pins
 * the width (256: the CTA-pair tiles, dense and contiguous only).  Results do
 * not depend on the plan. */
dg_status_t dg_query_plan(int layout, int M, int N, int K, int G, int expected_m, int num_sms,
                          dg_plan_t *out);

/* Human-readable name of a status code (static string, never NULL). */
const char *dg_status_string(dg_status_t status);

/* Synchronises `stream`, copies the current device's status word into
 * *flags (host) and clears it.  Returns DG_ERR_DEVICE_TIMEOUT if the timeout
 * bit was set, DG_OK otherwise (other bits are reported through *flags). */
dg_status_t dg_read_device_status(int *flags, void *stream);

/* Diagnostic of the failure-detection path: every pipeline wait of the GEMM
 * kernels is bounded.  Enqueues one small kernel whose single thread
 * waits, with the same bounded wait the GEMM pipelines use, on an mbarrier
 * that nothing ever arrives on.  The wait gives up after `limit_cycles` SM
 * cycles (1000 <= limit_cycles <= 4e9, about 2 s; DG_ERR_INVALID_ARG
 * otherwise), sets DG_DEVFLAG_TIMEOUT in the device status word and the
 * kernel returns: the context stays usable, and the next
 * dg_read_device_status on the stream returns DG_ERR_DEVICE_TIMEOUT.  No copy,
 * MMA or tensor memory is involved. */
dg_status_t dg_selftest_wait_timeout(long long limit_cycles, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DG_H_ */
