/*
 * sgemm.h — C ABI of the GB300 (sm_103a) single-precision GEMM library.
 *
 * The operation (one call computes it for one problem):
 *
 *     C[i*ldc + j] = sum_{k=0}^{K-1} A[i*lda + k] * B[k*ldb + j]
 *                    for 0 <= i < M, 0 <= j < N
 *
 * Definition: "Перемножение матриц: наивное и тайловое" (Matrix
 * multiplication: naive and tiled), section 1 — element C_row,col is the dot
 * product of row `row` of A and column `col` of B; matrices are stored row by
 * row, element (row, col) at offset row * n + col. The leading dimensions
 * lda, ldb, ldc generalise that row length n. Work: Chapter 9, Optimised
 * Matrix Multiplication, section 9.1 — M*N*K multiply-adds, 2*M*N*K FLOPs.
 *
 * Conventions fixed by this library where the pages are silent:
 *   - C is overwritten and never read (no alpha/beta scaling): every listing
 *     on the pages ends with a plain assignment of the sum to C.
 *   - Entries of a C row between column N and ldc are never touched.
 *   - K == 0 writes zeros to C (the empty sum); M == 0 or N == 0 is a no-op.
 *   - Arithmetic is IEEE FP32 with round-to-nearest fused multiply-adds,
 *     denormals kept, NaN/Inf propagated; the order of the K-sum is not
 *     specified (results are not bit-identical across kernel configs on
 *     general float inputs; they are on integer-valued inputs whose partial
 *     sums stay below 2^24 in magnitude).
 *
 * Layout: all matrices are row-major FP32 in device memory (HBM).
 * Ownership: every pointer is caller-owned device memory; the library never
 * frees, retains or reads host memory through it. Scratch space the library
 * needs (a packed copy of an operand whose rows are not 16-byte aligned, the
 * transposed K x M copy of A that the k-major configurations read, the
 * partial sums and arrival counters of a stream-K tail, the hi/lo operand
 * planes of the 3xTF32 configurations) is taken from a library-owned,
 * stream-ordered
 * memory pool on `stream` and returned on `stream`; it is never exposed.
 * Asynchrony: calls return after enqueueing work on `stream`; results are
 * ready when the stream's work completes. An FFMA call enqueues at most
 * three kernels: one layout pass for the operands that need it, which also
 * zeroes the arrival counters of the stream-K tail and of the last-rows
 * kernel (with no operand to lay out but counters to zero it runs as one
 * block); the product, which for K a multiple of its slab depth may start
 * while that pass finishes (programmatic dependent launch; its threads wait
 * for the pass before they touch memory); and the kernel of the last rows
 * that sgemm_plan_row_tail() describes. A 3xTF32 call enqueues two split
 * passes and the product per batch entry (and a memset of its stream-K
 * counters). No call synchronises the host.
 * Graph capture: sgemm(), sgemm_ex(), sgemm_general() and sgemm_general_ex()
 * may be captured into a CUDA graph once one call has run on the device
 * (the first call sets the device up); a replay computes the product of
 * whatever the operand buffers hold at replay time.
 * Thread safety: calls on different host threads/streams are safe.
 */
#ifndef DENSE_FP32_MATRIX_07_GB300_SGEMM_H
#define DENSE_FP32_MATRIX_07_GB300_SGEMM_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. A nonzero code returned by a call means that C is untouched:
 * argument errors return before anything is enqueued; a failing launch may
 * follow scratch-only work (an operand pack, a TF32 split) already enqueued
 * on the stream. Two exceptions: in a batched call on a 3xTF32
 * configuration, which launches entry after entry, a launch that fails at
 * entry b leaves entries 0 .. b-1 computed; and when the launch of the
 * last-rows kernel (sgemm_plan_row_tail()) fails, the product of the other
 * rows has been enqueued. */
enum {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_VALUE = 1, /* negative size, short leading dimension,
                                    NULL pointer with a non-empty extent,
                                    C overlapping A or B, unknown config */
    SGEMM_ERR_OVERFLOW = 2,      /* an index or byte offset would overflow,
                                    or a size exceeds the kernels' 2^31-1
                                    coordinate range */
    SGEMM_ERR_ALLOC = 3,         /* scratch allocation failed */
    SGEMM_ERR_LAUNCH = 4,        /* a kernel launch failed (cudaGetLastError), or, from
                                    sgemm_check_status(), a kernel found its launch shape
                                    wrong (a cluster kernel without its cluster) and did
                                    nothing */
    SGEMM_ERR_TIMEOUT = 5,       /* a device-side wait hit its bounded spin
                                    limit; reported by sgemm_check_status() */
    SGEMM_ERR_CUDA = 6,          /* another CUDA runtime failure (no device,
                                    device query, sticky context error) */
    SGEMM_ERR_UNSUPPORTED = 7,   /* the forced config cannot run this problem */
    SGEMM_ERR_SCRATCH_LIMIT = 8  /* sgemm_noalloc(): the packed operands would
                                    not fit its fixed scratch array */
};

/*
 * sgemm — C = A . B (see the top of this file for the exact semantics).
 *
 *   M, N, K   problem sizes, >= 0.
 *   A         device pointer, M rows of K floats, row i at A + i*lda;
 *             lda >= max(1, K). May be NULL when M == 0, N == 0 or K == 0.
 *   B         device pointer, K rows of N floats, row k at B + k*ldb;
 *             ldb >= max(1, N). May be NULL when M == 0, N == 0 or K == 0.
 *   C         device pointer, M rows of N floats, row i at C + i*ldc;
 *             ldc >= max(1, N). Must not overlap A or B. May be NULL only
 *             when M == 0 or N == 0.
 *   stream    CUDA stream to enqueue on (0 = the legacy default stream).
 *
 * Any alignment of A, B, C and any leading dimension is accepted. Operands
 * whose base address is 16-byte aligned and whose leading dimension is a
 * multiple of 4 floats are read in place by the tensor-memory-accelerator
 * (TMA) path; others are first packed into aligned scratch. For products of
 * 128x256 or 128x128 tiles with N >= 2048 and M*N*K >= 6e9 the automatic
 * choice is a k-major configuration ("ffma2_128x256_k32_s4_ka",
 * "ffma2_128x128_k32_s4_ka"), whose kernel reads A as a K x M matrix: A is
 * first transposed into scratch (K * round_up(M, 32) floats, about 8*M*K
 * bytes of traffic and a fixed few microseconds), which its faster inner
 * loop repays at those sizes. C is written with 16-byte vector stores when
 * it is aligned the same way, else with scalar stores.
 *
 * Returns SGEMM_OK or one of the codes above. A device-side timeout cannot
 * be known when the call returns; see sgemm_check_status().
 */
int sgemm(int64_t M, int64_t N, int64_t K,
          const float *A, int64_t lda,
          const float *B, int64_t ldb,
          float *C, int64_t ldc,
          cudaStream_t stream);

/*
 * sgemm_ex — sgemm() with an explicit kernel configuration.
 *
 *   config    -1 picks the configuration automatically (exactly sgemm());
 *             0 .. sgemm_num_configs()-1 forces that configuration.
 *
 * Returns SGEMM_ERR_INVALID_VALUE for an unknown config and
 * SGEMM_ERR_UNSUPPORTED when the forced config cannot run the problem.
 * Intended for tests and tuning sweeps.
 */
int sgemm_ex(int64_t M, int64_t N, int64_t K,
             const float *A, int64_t lda,
             const float *B, int64_t ldb,
             float *C, int64_t ldc,
             int config, cudaStream_t stream);

/*
 * sgemm_general — the BLAS-style general form, over a strided batch:
 *
 *     C_b = alpha * op(A_b) . op(B_b) + beta * C_b      for 0 <= b < batch
 *
 * An extension for users of this library; the pages define only C = A . B
 * (the definition at the top of this file, which this reduces to with
 * op_a = op_b = 0, alpha = 1, beta = 0, batch = 1).
 *
 *   op_a      0: A_b is stored M x K (row i at A + b*stride_a + i*lda,
 *             lda >= K); 1: A_b is stored transposed, K x M (lda >= M).
 *   op_b      0: B_b stored K x N (ldb >= N); 1: stored N x K (ldb >= K).
 *   alpha     scales the product. alpha == 0 (or K == 0) reads neither A
 *             nor B: C_b = beta * C_b.
 *   beta      scales the old C. beta == 0: C is written without being read
 *             (it may hold NaN); beta == 1 with alpha == 0 is a no-op.
 *   stride_a, stride_b, stride_c
 *             batch strides in elements (>= 0; ignored when batch == 1). A
 *             stride of 0 shares one A (or B) across the batch; C entries
 *             must not overlap (stride_c >= (M-1)*ldc + N when batch > 1).
 *   batch     number of products (0 is a no-op).
 *
 * Pointers are device pointers; C must not overlap A or B (over the whole
 * batch). Transposed operands and rows or batch strides that are not 16-byte
 * multiples are packed into pool scratch first, except that the k-major
 * configurations read a transposed A (stored K x M, aligned) in place and
 * transpose a plain one; the automatic choice takes a k-major configuration
 * for a transposed A wherever it would take its row-major twin. Alpha and
 * beta are applied in the kernels' epilogues; on the FFMA configurations
 * batch entries share one
 * persistent launch (their tiles are one schedule), on the 3xTF32 ones each
 * entry is split and multiplied in turn. Status codes as sgemm();
 * SGEMM_ERR_UNSUPPORTED if
 * a forced configuration cannot run the general form (the simple, the
 * kernel-ladder and the small-product configurations run only the plain
 * form; the automatic choice gives the general form TMA tiles instead).
 */
int sgemm_general(int op_a, int op_b, int64_t M, int64_t N, int64_t K, float alpha,
                  const float *A, int64_t lda, int64_t stride_a,
                  const float *B, int64_t ldb, int64_t stride_b,
                  float beta, float *C, int64_t ldc, int64_t stride_c,
                  int64_t batch, cudaStream_t stream);

/* sgemm_general() with a forced kernel configuration (-1 = automatic). */
int sgemm_general_ex(int op_a, int op_b, int64_t M, int64_t N, int64_t K, float alpha,
                     const float *A, int64_t lda, int64_t stride_a,
                     const float *B, int64_t ldb, int64_t stride_b,
                     float beta, float *C, int64_t ldc, int64_t stride_c,
                     int64_t batch, int config, cudaStream_t stream);

/*
 * sgemm_general_plan — host-only view of the choice sgemm_general_ex() makes
 * (the pages have no counterpart); needs no GPU.
 *
 *   op_a ... batch           as sgemm_general_ex(), with the operands given
 *                            by address (only their alignment matters; 0
 *                            means aligned; null and overlap are not checked).
 *   num_sms                  streaming multiprocessors of the target device.
 *   config                   -1 (automatic) or a forced configuration.
 *   out_config               (nullable) receives the configuration of the
 *                            product, or -1 when the call runs none (no
 *                            output entries, or K == 0 or alpha == 0, which
 *                            only scale C).
 *   out_pack_a, out_pack_b   (nullable) receive 1 if that operand goes
 *                            through scratch first (packed, transposed or,
 *                            for A under a k-major configuration, transposed
 *                            to K x M), else 0.
 *
 * Returns SGEMM_OK, or the code sgemm_general_ex() would return for these
 * sizes, strides and configuration.
 */
int sgemm_general_plan(int op_a, int op_b, int64_t M, int64_t N, int64_t K, float alpha,
                       int64_t lda, int64_t stride_a, int64_t ldb, int64_t stride_b,
                       float beta, int64_t ldc, int64_t stride_c, int64_t batch,
                       uint64_t a_addr, uint64_t b_addr, uint64_t c_addr,
                       int num_sms, int config,
                       int *out_config, int *out_pack_a, int *out_pack_b);

/*
 * sgemm_general_plan_launches — host only: how many of this library's
 * kernels sgemm_general_ex() enqueues for these arguments (sgemm_ex() is the
 * plain form: op 0, alpha 1, beta 0, batch 1). An FFMA configuration runs
 * the product, the layout pass when an operand goes through scratch or
 * arrival counters must be zeroed (stream-K tail, split last-rows kernel),
 * and the last-rows kernel (sgemm_plan_row_tail()); a 3xTF32 configuration
 * two split passes and the product per batch entry; K == 0 or alpha == 0 one
 * scaling kernel unless beta == 1. Memory copies and memsets are not
 * counted.
 *
 * Arguments as sgemm_general_plan(); out_launches (not NULL) receives the
 * count (0 when the call enqueues nothing). Returns SGEMM_OK, or the code
 * sgemm_general_ex() would return, or SGEMM_ERR_INVALID_VALUE for a NULL
 * out_launches or num_sms <= 0.
 */
int sgemm_general_plan_launches(int op_a, int op_b, int64_t M, int64_t N, int64_t K, float alpha,
                                int64_t lda, int64_t stride_a, int64_t ldb, int64_t stride_b,
                                float beta, int64_t ldc, int64_t stride_c, int64_t batch,
                                uint64_t a_addr, uint64_t b_addr, uint64_t c_addr,
                                int num_sms, int config, int *out_launches);

/*
 * sgemm_check_status — waits for `stream`, then reads and clears the current
 * device's error word. Returns SGEMM_ERR_TIMEOUT if any kernel of this
 * library on the device gave up a bounded wait since the last check (its
 * output is then incomplete), SGEMM_ERR_LAUNCH if a kernel found itself
 * launched in a shape it cannot run in (a cluster kernel without its
 * cluster; it then wrote nothing), SGEMM_ERR_CUDA if the stream reports a
 * CUDA error, else SGEMM_OK. The error word is per device, not per stream.
 */
int sgemm_check_status(cudaStream_t stream);

/* Static, NUL-terminated description of a status code (never NULL). */
const char *sgemm_error_string(int code);

/* Number of kernel configurations that sgemm_ex() accepts. */
int sgemm_num_configs(void);

/* Static name of configuration `config` ("?" when out of range). */
const char *sgemm_config_name(int config);

/*
 * sgemm_plan — host-only view of the choice sgemm() makes; needs no GPU.
 *
 *   a_addr, b_addr, c_addr   the operand addresses (only their alignment
 *                            matters; 0 means aligned).
 *   num_sms                  streaming multiprocessors of the target device.
 *   out_config               (nullable) receives the chosen configuration.
 *   out_pack_a, out_pack_b   (nullable) receive 1 if that operand would be
 *                            packed into scratch first (for A under a
 *                            k-major configuration: always, transposed),
 *                            else 0.
 *
 * Returns SGEMM_OK, or the code sgemm() would return for invalid sizes.
 */
int sgemm_plan(int64_t M, int64_t N, int64_t K,
               int64_t lda, int64_t ldb, int64_t ldc,
               uint64_t a_addr, uint64_t b_addr, uint64_t c_addr,
               int num_sms,
               int *out_config, int *out_pack_a, int *out_pack_b);

/*
 * sgemm_plan_row_tail — host-only, needs no GPU: how many of the last rows
 * of C a call computes apart from its tiled product.
 *
 * The TMA configurations tile C in 128-row block rows. When M = 128 q + r
 * with 1 <= r <= 8 (M > 128) and the block row those r rows would pad is
 * large (round_up(N, tile width) * K >= 2^21), the call runs the tiled
 * product on the first M - r rows and a small kernel on the last r: each of
 * those rows is the dot product of a row of A with every column of B, as
 * the course page "Перемножение матриц: наивное и тайловое", section 1,
 * defines C, computed by CTAs that split K, the last of each column block
 * adding the parts in a fixed order. Arguments: `config`, the configuration the call runs
 * (from sgemm_plan() or sgemm_general_plan(), or a forced one); M, N, K and
 * `batch` of the call. *out_rows receives r, or 0 when the call has no such
 * kernel (which adds one launch when it runs). Returns SGEMM_OK, or
 * SGEMM_ERR_INVALID_VALUE for an unknown config, a negative size or a NULL
 * out_rows.
 */
int sgemm_plan_row_tail(int config, int64_t M, int64_t N, int64_t K, int64_t batch,
                        int64_t *out_rows);

/*
 * sgemm_test_withhold_copy — test hook for the device-side wait limit.
 *
 * Failure detection ("Перемножение матриц: наивное и тайловое", section 2:
 * a tile may be used only once it is fully loaded; here that wait is
 * bounded). Runs the product on the 128x256 TMA configuration
 * ("ffma2_128x256_k32_s4") with whole-tile scheduling, whatever the size,
 * except that the producer
 * of the first CTA never issues the copy of its `slab`-th K slab, so the
 * consumers' wait for it can never be satisfied. Every device-side wait gives
 * up after about a second; the kernel then sets the device error word and
 * exits without faulting, the context stays usable, and sgemm_check_status()
 * returns SGEMM_ERR_TIMEOUT. C is left incomplete. The call takes about one
 * to two seconds on the GPU. slab < 0 computes the product normally.
 * Arguments otherwise as sgemm(); aligned operands make the kernel read A and
 * B in place (no packing) so the withheld copy is the product's own.
 */
int sgemm_test_withhold_copy(int64_t M, int64_t N, int64_t K,
                             const float *A, int64_t lda,
                             const float *B, int64_t ldb,
                             float *C, int64_t ldc,
                             int slab, cudaStream_t stream);

/*
 * sgemm_test_fail_next_allocs — test hook for the allocation-failure paths
 * (the pages have no counterpart).
 *
 * The next n scratch allocations of sgemm(), sgemm_ex(), sgemm_general()
 * and sgemm_general_ex() (in any thread) are treated as failed without
 * asking the pool. An automatic k-major choice then falls back to its
 * row-major twin, which reads an aligned A as stored; any other call whose
 * allocation fails returns SGEMM_ERR_ALLOC with nothing enqueued. n = 0
 * clears a pending count. Returns SGEMM_OK, or SGEMM_ERR_INVALID_VALUE for
 * n < 0. Host only; needs no GPU.
 */
int sgemm_test_fail_next_allocs(int n);

/*
 * sgemm_test_schedule — test hook (host only, no GPU): the work schedule the
 * persistent kernels follow, enumerated.
 *
 * Plans the schedule of an M x N x K product (times `batch`) in bm x bn
 * tiles of bk-deep slabs on `slots` CTAs under `policy` (0 automatic, 1 whole
 * tiles, 2 stream-K everywhere, 3 tail split), with the stream-K workspace
 * available, and walks every CTA's work items in the order the kernels do.
 * Item n holds: CTA, tile, first slab, end slab, batch
 * entry, tile row, tile column, and, for a part of a tile split among
 * several CTAs, the first and the last of those CTAs and the partial-sum
 * slot this part writes when it does not reduce the tile (else -1, -1, -1).
 * Items take 10 entries each: items[10n .. 10n+9]. info[0..6] receive the
 * grid, tiles, whole tiles, stream-K CTAs, slabs per tile, tile rows and
 * tile columns.
 * *count receives the number of items; SGEMM_ERR_INVALID_VALUE if it exceeds
 * `capacity` (items then holds the first `capacity`) or an argument is out
 * of range.
 */
int sgemm_test_schedule(int64_t M, int64_t N, int64_t K, int bm, int bn, int bk,
                        int64_t slots, int policy, int64_t batch,
                        int64_t *items, int64_t capacity, int64_t *count, int64_t *info);

/*
 * sgemm_noalloc — sgemm() for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for users of
 * this library. Some callers cannot call cudaMalloc (or any allocating
 * routine, torch's caching allocator included) where they need a product:
 * code whose device memory is fully handed to another allocator or to a
 * fixed-size arena, and latency-critical loops that must not take the
 * driver's allocation path (which can block and synchronise). sgemm() takes
 * pool scratch when an operand needs packing (a base address that is not
 * 16-byte aligned, or a leading dimension that is not a multiple of 4
 * floats) and for the partial sums of a stream-K tail; this entry point packs
 * such operands into a fixed scratch array compiled into the library instead,
 * keeps the stream-K partial sums and arrival counters in a second fixed
 * array (48 MiB; a schedule needing more, on GPUs of over 190 SMs, runs
 * whole tiles), and
 * allocates nothing. Where sgemm() would take a k-major configuration, this
 * entry point makes its transposed copy of A in the fixed array when that
 * fits (K * round_up(M, 32) floats, beside a packed B), and otherwise runs
 * the configuration's twin that reads A as stored.
 *
 * Arguments, semantics, ownership and status codes: as sgemm().
 *
 * Limit: the packed operands must fit the 64 MiB array (16 Mi floats):
 * M * round_up(K, 32) floats for a packed A plus K * round_up(N, 32) floats
 * for a packed B. Larger requests return SGEMM_ERR_SCRATCH_LIMIT with nothing
 * enqueued. Aligned operands are not packed and have no size limit.
 *
 * Memory: every GPU that loads the library's device code holds the two
 * arrays (64 MiB + 48 MiB) until the process exits.
 * Set-up: the first call on a device (with that device current) looks up the
 * arrays' device addresses and caches them with the device's other
 * constants; make that first call before any stream capture begins.
 * Sharing: all calls on a device share the arrays, which keep the last call's
 * packed data and partial sums; calls whose work overlaps on the GPU (other
 * streams, other host threads) race on them, so the caller must order them.
 */
int sgemm_noalloc(int64_t M, int64_t N, int64_t K,
                  const float *A, int64_t lda,
                  const float *B, int64_t ldb,
                  float *C, int64_t ldc,
                  cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_FP32_MATRIX_07_GB300_SGEMM_H */
