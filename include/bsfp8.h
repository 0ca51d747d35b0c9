/*
 * bsfp8.h -- C ABI of libbsfp8: block-scaled E4M3 GEMM with bf16 output on one
 * GB300 (sm_103a).
 *
 * Operation (FP8 GEMM library article, hncyxsy.com/news/241433, section 2.2
 * "scale granularity" and section 2.3 "where the scales live": one fp32 scale
 * per 32x32 block of each operand, taking part in the accumulation, no separate
 * dequantisation pass; section 6 gives the operand shapes A [M,K], B [N,K],
 * scale_a [M/32,K/32], scale_b [N/32,K/32]):
 *
 *   C[m,n] = bf16( sum_kb sA[m/32][kb] * sB[n/32][kb] * sum_{k in kb} A[m,k]*B[n,k] )
 *
 * kb runs over the K/32 blocks of 32 consecutive k in ascending order.  The
 * K-reduction order is the same for every M: no split-K, no shape-dependent
 * tile configuration ("AI Infra 进阶：如何让大模型输出确定的结果",
 * aif.amtbbs.org post 29992, section 1: a row's result changes with the batch
 * only through the reduction split).  Hence every output row is bit-identical
 * whatever M (and whatever other rows) it is computed with, given the same
 * path; FP8_PATH_* below says when AUTO's choice of path can itself depend on
 * other rows, and FP8_PATH_PROMOTE is batch-invariant for any scales.
 *
 * Layouts (all device memory, all row-major, caller-owned):
 *   A   [M, K]           E4M3 codes, one byte each (row stride K bytes)
 *   B   [N, K]           E4M3 codes, K contiguous ("K-major" weights)
 *   sA  [ceil(M/32), K/32] fp32 (the last row block may be partial)
 *   sB  [N/32, K/32]     fp32
 *   C   [M, N]           bf16, fully overwritten (no beta*C term)
 *
 * Constraints: M >= 0; N and K multiples of 32 (N, K >= 0); M, N, K < 2^31.
 * A, B and C 16-byte aligned; sA and sB 4-byte aligned.  E4M3 NaN codes
 * (0x7F, 0xFF) and NaN/inf scales give undefined values (never a fault).
 *
 * Execution: every call is asynchronous on `stream` (0 = legacy default
 * stream), allocates no per-call device memory and never synchronises the
 * host.  The first call on a device does a one-time set-up for that device
 * (kernel attributes, a 256-byte device status word); make it outside any
 * stream capture.  Calls are thread-safe.
 *
 * Errors: functions return FP8_OK (0) or a negative FP8_ERR_* code; argument
 * errors are detected on the host before anything is enqueued.  Conditions
 * found on the device (a bounded wait that ran out, a forced native path with
 * non-power-of-two scales) are recorded in a sticky per-device status word
 * read by fp8_status_query().
 */
#ifndef BSFP8_H
#define BSFP8_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BSFP8_VERSION 10000 /* 1.0.0 */

enum {
    FP8_OK = 0,
    FP8_ERR_NULL = -1,       /* a required pointer is NULL */
    FP8_ERR_SHAPE = -2,      /* negative size, N or K not a multiple of 32, size >= 2^31, G out of range */
    FP8_ERR_ALIGN = -3,      /* A/B/C not 16-byte aligned or sA/sB not 4-byte aligned */
    FP8_ERR_ARCH = -4,       /* current device is not sm_103 */
    FP8_ERR_CUDA = -5,       /* a CUDA runtime/driver call failed (launch, attribute, ...) */
    FP8_ERR_MODE = -6,       /* unknown path mode or debug key */
    FP8_ERR_SCALE = -7,      /* device status: FP8_PATH_NATIVE with a scale that is not 2^e */
    FP8_ERR_TIMEOUT = -8,    /* device status: a bounded wait inside a kernel ran out */
    FP8_ERR_RECORD = -9      /* device status: a device-resident group record was rejected */
};

/* Path selection.
 * FP8_PATH_AUTO: per output tile (256 rows x 256 columns), the native path is
 *   taken when every scale the tile reads (its row blocks of sA and column
 *   blocks of sB, all of K) is a positive normal power of two; otherwise the
 *   promotion path.  A row's bits therefore depend only on the scales of the
 *   rows in its own 256-row tile (rows 256*floor(m/256) ...), and only when
 *   sA's 32-row blocks mix kinds: AUTO is batch-invariant (a row gets the same
 *   bits for every M) whenever every row block of sA is of one kind -- all of
 *   its K/32 scales powers of two in every block, or at least one scale that
 *   is not in every block -- whatever sB holds (every launch reads the same
 *   sB).  Where sA's row blocks do mix, a row computed with fewer rows (M
 *   ending inside its tile) may take the native path while the full batch
 *   promotes the tile; its bits are then those of one of the two pinned paths
 *   below.  Callers that need batch invariance for any scales pin
 *   FP8_PATH_PROMOTE.
 * FP8_PATH_NATIVE: block-scaled tensor-core path (kind::mxf8f6f4 with UE8M0
 *   scales, exact for power-of-two scales).  A tile that finds another scale
 *   is computed by the promotion path and FP8_ERR_SCALE is recorded.
 * FP8_PATH_PROMOTE: per-K-block fp32 promotion for arbitrary fp32 scales:
 *   unscaled 32-deep tensor-core partials, scaled and accumulated in fp32.
 *   Every tile takes this path whatever the scales, so each row's bits are
 *   the same for every M (batch-invariant unconditionally); each element
 *   equals, bit for bit, what AUTO computes for it on a promoted tile. */
enum { FP8_PATH_AUTO = 0, FP8_PATH_NATIVE = 1, FP8_PATH_PROMOTE = 2 };

/* Block-scaled GEMM, AUTO path.  Returns FP8_OK or FP8_ERR_*.
 * M == 0, N == 0: nothing is enqueued.  K == 0: C is zero-filled. */
int fp8_gemm_blockscaled(const void *A, const float *sA, const void *B, const float *sB,
                         void *C, int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* Same with an explicit path (FP8_PATH_*). */
int fp8_gemm_blockscaled_ex(const void *A, const float *sA, const void *B, const float *sB,
                            void *C, int64_t M, int64_t N, int64_t K, int mode,
                            cudaStream_t stream);

/* Block-scaled GEMM with a residual added in the epilogue (FP8 GEMM library
 * article, hncyxsy.com/news/241433, section 2.3 and the pitfalls of section 5:
 * element-wise work fused into the GEMM's tail instead of another pass over
 * the output):
 *   C[m,n] = bf16( sum_kb sA*sB*sum_k A*B  +  R[m,n] )
 * The accumulator and R (bf16, exact in fp32) are added in fp32 and rounded
 * once to bf16 (nearest even).  R: bf16 [M, N] row-major, 16-byte aligned,
 * read only; it may be the same buffer as C (in place).  Everything else as
 * fp8_gemm_blockscaled (AUTO path); K = 0 gives C = R.
 * Returns FP8_OK or FP8_ERR_SHAPE / FP8_ERR_NULL / FP8_ERR_ALIGN / FP8_ERR_CUDA. */
int fp8_gemm_blockscaled_residual(const void *A, const float *sA, const void *B, const float *sB,
                                  const void *R, void *C, int64_t M, int64_t N, int64_t K,
                                  cudaStream_t stream);

/* Block-scaled GEMM whose output is quantized in the epilogue to the operand
 * format of the next GEMM (FP8 GEMM library article, hncyxsy.com/news/241433,
 * sections 2.1-2.2: E4M3 with one fp32 scale per 32x32 block; section 2.3:
 * element-wise work fused into the GEMM's tail instead of another pass over
 * the output):
 *   (Cq, sC) = fp8_quantize_blocks( fp8_gemm_blockscaled(A, sA, B, sB) )
 * bit for bit: the bf16 output of the AUTO-path GEMM is never written; each
 * 32x32 block of it gets s = amax/448 (1 for an all-zero block) and codes
 * E4M3(x/s) with the quantizer's arithmetic.  A 32-row block's scale depends
 * on all its rows, so results are batch-invariant per 32-row block.
 * Cq: E4M3 codes [M, N] row-major (16-byte aligned), fully overwritten.
 * sC: fp32 [ceil(M/32), N/32] row-major (4-byte aligned), fully overwritten.
 * Everything else as fp8_gemm_blockscaled; K = 0 gives codes 0 and scales 1.
 * Returns FP8_OK or FP8_ERR_SHAPE / FP8_ERR_NULL / FP8_ERR_ALIGN / FP8_ERR_CUDA. */
int fp8_gemm_blockscaled_quant(const void *A, const float *sA, const void *B, const float *sB,
                               void *Cq, float *sC, int64_t M, int64_t N, int64_t K,
                               cudaStream_t stream);

/* GEMM with scales that do not vary along K (FP8 GEMM library article,
 * hncyxsy.com/news/241433, section 2.2: per-tensor, per-channel and per-token
 * scale granularities; section 2.3: such scales are applied in the GEMM's
 * epilogue):
 *   C[m,n] = bf16( sA[m] * sB[n] * sum_k A[m,k] * B[n,k] )
 * A, B, C, M, N, K: as fp8_gemm_blockscaled.  sA: fp32 [M] (per token / row
 * of A), sB: fp32 [N] (per output channel / row of B), 4-byte aligned, read
 * only; a per-tensor scale is a constant vector.  The MMAs run with unit
 * scales and accumulate over all of K in fp32; the epilogue multiplies by
 * sA[m] * sB[n] (one fp32 product) and rounds to bf16 (nearest even).  Same
 * tiles and K order as the block-scaled call, so rows are batch-invariant.
 * Returns FP8_OK or FP8_ERR_SHAPE / FP8_ERR_NULL / FP8_ERR_ALIGN / FP8_ERR_CUDA. */
int fp8_gemm_rowcol(const void *A, const float *sA, const void *B, const float *sB, void *C,
                    int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* Block-scaled GEMM with per-token scales for A (FP8 GEMM library article,
 * hncyxsy.com/news/241433, section 2.2: per-token scales for activations, a
 * finer granularity than 32x32 blocks): one fp32 scale per row of A per
 * 32-K block, B keeping its 32x32 blocks:
 *   C[m,n] = bf16( sum_kb sA[m][kb] * sB[n/32][kb] * sum_{k in kb} A[m,k]*B[n,k] )
 * sA: fp32 [M, K/32] row-major (4-byte aligned); everything else as
 * fp8_gemm_blockscaled.  Any finite scales: every tile takes the per-K-block
 * fp32 promotion (unscaled 32-deep tensor-core partials, acc += (sA*sB) *
 * partial in fp32, K ascending), so each row's bits are the same for every M.
 * With scales equal within each 32-row block the result equals
 * fp8_gemm_blockscaled_ex(..., FP8_PATH_PROMOTE) on the block scales, bit for
 * bit.  Returns FP8_OK or FP8_ERR_SHAPE / FP8_ERR_NULL / FP8_ERR_ALIGN /
 * FP8_ERR_CUDA. */
int fp8_gemm_pertoken(const void *A, const float *sA, const void *B, const float *sB, void *C,
                      int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* Same with an explicit path.  FP8_PATH_AUTO and FP8_PATH_PROMOTE: the
 * promotion path above.  FP8_PATH_NATIVE: the block-scaled tensor-core path
 * (kind::mxf8f6f4, UE8M0 scales) on CTA pairs with 256 x 256 tiles, each row
 * of A carrying its own scale per 32-K block (1 x 32 scale vectors along K,
 * the scale layout of MX formats), B its 32 x 32 blocks; every sA and sB
 * value must be a positive normal power of two.  The scales are not scanned
 * before the launch: a value that is not is reported as FP8_ERR_SCALE by
 * fp8_status_query and the result is undefined.  Tiles and K order depend on
 * N and K only, so each row's bits are the same for every M; the bits differ
 * from the promotion path's (a different accumulation), both within the
 * acceptance bound.  Returns as fp8_gemm_pertoken, or FP8_ERR_MODE. */
int fp8_gemm_pertoken_ex(const void *A, const float *sA, const void *B, const float *sB, void *C,
                         int64_t M, int64_t N, int64_t K, int mode, cudaStream_t stream);

/* Per-token A scales given as UE8M0 bytes, the exponent-only 8-bit scale
 * format of the block-scaled MMA (FP8 GEMM library article,
 * hncyxsy.com/news/241433, section 2.2, per-token granularity):
 *   C[m,n] = bf16( sum_kb 2^(sA[m][kb] - 127) * sB[n/32][kb] * sum_k A*B )
 * sA: uint8 [M, K/32] row-major, any alignment (rows that start on 8 bytes
 * with K a multiple of 256 are read 8 bytes at a time); a byte 0xFF (not a
 * number in UE8M0) is reported as FP8_ERR_SCALE through fp8_status_query.
 * sB: fp32 [N/32, K/32] powers of two (else FP8_ERR_SCALE, as NATIVE mode).
 * Always the native path (CTA pairs, the bytes copied into per-row scale
 * lines without conversion); its results equal fp8_gemm_pertoken_ex with
 * FP8_PATH_NATIVE and the same scales given as fp32 powers of two, bit for
 * bit, for bytes 1-254 (the byte 0, 2^-127, has no fp32 normal counterpart).
 * Scale products below the fp32 normal range (2^-126) may be flushed.
 * Everything else as fp8_gemm_pertoken.  Returns FP8_OK or FP8_ERR_SHAPE /
 * FP8_ERR_NULL / FP8_ERR_ALIGN / FP8_ERR_CUDA. */
int fp8_gemm_pertoken_e8m0(const void *A, const void *sA, const void *B, const float *sB, void *C,
                           int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* Block quantization of activations to the operand format above (FP8 GEMM
 * library article, hncyxsy.com/news/241433, section 2.1: E4M3, largest value
 * 448; section 2.2: one scale per 32x32 block).  For each 32x32 block of x:
 *   s = amax / 448 (fp32 division; s = 1 when the block is all zero),
 *   q = E4M3(x / s) (fp32 division, round to nearest even, saturating at +-448).
 * x: bf16 [M, K] row-major (16-byte aligned), read only.
 * q: E4M3 codes [M, K] row-major (16-byte aligned), fully overwritten.
 * s: fp32 [ceil(M/32), K/32] row-major (4-byte aligned), fully overwritten;
 *    the last row block may be partial (rows past M do not exist).
 * q and s are the A and sA operands of fp8_gemm_blockscaled.  K must be a
 * multiple of 32; M = 0 or K = 0 is a no-op.  NaN or infinite inputs give
 * undefined codes.  Asynchronous on `stream`; all buffers caller-owned device
 * memory.  Returns FP8_OK or FP8_ERR_SHAPE / FP8_ERR_NULL / FP8_ERR_ALIGN /
 * FP8_ERR_CUDA (launch failure). */
int fp8_quantize_blocks(const void *x, void *q, float *s, int64_t M, int64_t K, cudaStream_t stream);

/* Allocation-free variant of fp8_gemm_blockscaled (AUTO path, same layouts
 * and constraints).  It runs one CTA per 128 x 256 tile instead of CTA pairs
 * on 256 x 256 tiles, with the same per-element arithmetic: its output equals
 * fp8_gemm_blockscaled's bit for bit whenever both choose the same path for
 * every element, which holds when sA's row blocks are all of one kind (see
 * FP8_PATH_AUTO).  Where sA's row blocks mix kinds, AUTO's 128-row and
 * 256-row tiles can choose differently; both results are then within the
 * same tolerance of the exact value.  The pages have no counterpart: this entry point
 * exists for callers that cannot allocate device memory: an inference server
 * whose caching allocator owns the whole device (a stray cudaMalloc there can
 * fail, fragment the pool or stall the device while it synchronises), or a
 * deployment whose memory budget is fixed at start-up and must not grow per
 * call.  The only extra device memory the kernel needs (its status
 * word) lives in a static array inside the library: FP8_NOALLOC_SCRATCH_BYTES
 * on every GPU that loads the library, held until the process exits.  Its
 * size does not depend on M, N or K, so no problem size exceeds it.
 * The call never invokes cudaMalloc, cudaFree or any allocating routine.
 * The first call on each device performs a one-time set-up for that device
 * (looks up the array's device address and clears it); make that first call
 * before any stream capture.  All calls share the array: calls that overlap
 * on the GPU race on it (only their status bits mix; results are not
 * affected).  Device-side conditions of these calls (a wait that ran out)
 * are recorded in word 0 of that array; fp8_status_query reads and clears it
 * together with the regular status word, and allocates nothing either. */
#define FP8_NOALLOC_SCRATCH_BYTES 256
int fp8_gemm_blockscaled_noalloc(const void *A, const float *sA, const void *B, const float *sB,
                                 void *C, int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* One group of a grouped launch: device pointers with the layouts above,
 * sized by that group's M_g (sA_g has ceil(M_g/32) group-local row blocks). */
typedef struct fp8_group_desc {
    const void *A;    /* [M_g, K] E4M3 */
    const float *sA;  /* [ceil(M_g/32), K/32] fp32 */
    const void *B;    /* [N, K] E4M3 */
    const float *sB;  /* [N/32, K/32] fp32 */
    void *C;          /* [M_g, N] bf16 */
} fp8_group_desc;

#define FP8_MAX_GROUPS_PER_LAUNCH 64

/* Grouped GEMM for ragged decode batches (FP8 GEMM library article, section
 * 4.1-4.2: many small GEMMs of different shapes merged into one launch, each
 * block finding its problem from a parameter table; section 4.3: shapes kept
 * in device memory so a captured CUDA graph stays valid when they change).
 *
 * groups: HOST array of G descriptors (copied into the launch; the caller may
 *         reuse it as soon as the call returns).
 * Ms:     DEVICE int32[G], the row count of each group, read only by the
 *         kernel (so it may change between graph replays).  M_g < 0 is
 *         treated as 0.
 * N, K:   shared by all groups (multiples of 32).
 * Groups are independent GEMMs: group g's result is bit-identical to
 * fp8_gemm_blockscaled on that group alone with the same path.
 * G <= FP8_MAX_GROUPS_PER_LAUNCH runs as one launch; larger G is split into
 * consecutive launches of at most that many groups on the same stream.
 * K = 0 returns FP8_ERR_SHAPE (the row counts live on the device, so the
 * host cannot zero-fill the outputs); G = 0 or N = 0 enqueues nothing. */
int fp8_gemm_grouped(const fp8_group_desc *groups, const int32_t *Ms, int64_t N, int64_t K,
                     int32_t G, cudaStream_t stream);

int fp8_gemm_grouped_ex(const fp8_group_desc *groups, const int32_t *Ms, int64_t N,
                        int64_t K, int32_t G, int mode, cudaStream_t stream);

/* Grouped GEMM with the group records in DEVICE memory (FP8 GEMM library
 * article, hncyxsy.com/news/241433, section 4.2: the grouped kernel finds its
 * problems in a parameter table; section 4.3: what a captured CUDA graph reads
 * must live in device memory so that the graph stays valid as requests
 * change).  Everything the launch depends on is in device memory: the
 * records, the row counts and the tensor maps, which a first small kernel
 * builds from the records on the device; a graph captured once therefore
 * computes whatever groups the table and Ms hold at each replay.
 *
 * groups:    DEVICE array of G fp8_group_desc (8-byte aligned), read by the
 *            launch's kernels; the pointers follow fp8_group_desc's layouts.
 * Ms:        DEVICE int32[G] row counts (M_g < 0 counts as 0).
 * N, K:      shared by all groups, multiples of 32; K = 0 gives FP8_ERR_SHAPE.
 * workspace: DEVICE memory of at least fp8_grouped_workspace_bytes(G) bytes,
 *            128-byte aligned, caller-owned, holding the per-group tensor
 *            maps between the two kernels; launches that overlap on the GPU
 *            need separate workspaces.
 * A record with a null pointer, or A, B or C not 16-byte aligned, or sA or
 * sB not 4-byte aligned, is rejected on the device: its group is skipped
 * (its C is not written) and FP8_ERR_RECORD is recorded for
 * fp8_status_query.  Results equal fp8_gemm_grouped's for the same records,
 * bit for bit.  AUTO path.  G > FP8_MAX_GROUPS_PER_LAUNCH is split into
 * consecutive launch pairs.  Returns FP8_OK or FP8_ERR_SHAPE / FP8_ERR_NULL /
 * FP8_ERR_ALIGN (groups, Ms or workspace) / FP8_ERR_CUDA. */
int fp8_gemm_grouped_device(const fp8_group_desc *groups, const int32_t *Ms, int64_t N, int64_t K,
                            int32_t G, void *workspace, int64_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes fp8_gemm_grouped_device needs for G groups (0 for G < 0). */
int64_t fp8_grouped_workspace_bytes(int32_t G);

/* Synchronises `stream`, then reads and clears the current device's status
 * words: the one the regular entry points write (including FP8_ERR_RECORD
 * from fp8_gemm_grouped_device) and word 0 of the
 * allocation-free entry point's static array (each only once its entry point
 * has run on this device).  Allocates nothing.  *status = FP8_OK, or the
 * FP8_ERR_* code of a condition recorded since the last query
 * (FP8_ERR_TIMEOUT takes precedence, then FP8_ERR_RECORD, then FP8_ERR_SCALE).  The status comes
 * back through the out-pointer so that the return value stays the call's own
 * FP8_OK / FP8_ERR_CUDA / FP8_ERR_NULL. */
int fp8_status_query(cudaStream_t stream, int *status);

/* Human-readable name of an FP8_* code (static storage). */
const char *fp8_strerror(int code);

/* BSFP8_VERSION of the loaded library. */
int fp8_version(void);

/* Debug/test controls (process-wide, affect launches enqueued afterwards).
 * FP8_DEBUG_WAIT_LIMIT_CYCLES: SM clock cycles a device-side wait may spin
 *   before the kernel records FP8_ERR_TIMEOUT and returns cleanly (default
 *   2^31, about one second; the environment variable BSFP8_WAIT_LIMIT_CYCLES
 *   sets the initial value).  value <= 0 restores the default.
 * FP8_DEBUG_WITHHOLD_STAGE: when >= 0, the producer of CTA 0 never loads
 *   that pipeline stage (counted from 0 over the CTA's whole K loop), so the
 *   waits behind it run out; the output is then incomplete.  -1 (default)
 *   disables it.  Used by the bounded-wait test.
 * FP8_DEBUG_TRACE_BUFFER: device address (0 = off) of a buffer of
 *   2 x 24 x 1024 uint64 words; CTAs 0 and 1 of later launches write the SM
 *   clock of their pipeline events there (CTA b, event e, index i at word
 *   (b*24 + e)*1024 + i).  A profiling aid; the event numbering is listed
 *   with the kernel.
 * Returns FP8_OK or FP8_ERR_MODE for an unknown key. */
enum { FP8_DEBUG_WAIT_LIMIT_CYCLES = 1, FP8_DEBUG_WITHHOLD_STAGE = 2, FP8_DEBUG_TRACE_BUFFER = 3 };
int fp8_debug_set(int key, int64_t value);

/* Frees the per-device status words and empties the host cache of TMA
 * descriptors (each is a pure function of a call's pointers and sizes, so the
 * cache never holds a stale one).  Later calls set both up again.  The
 * allocation-free entry point's static array is part of the loaded library
 * and stays; its per-device set-up (the array's device address, kernel
 * attributes) is forgotten and runs again on that entry point's next call,
 * which must then again come before any stream capture. */
void fp8_lib_shutdown(void);

#ifdef __cplusplus
}
#endif
#endif /* BSFP8_H */
