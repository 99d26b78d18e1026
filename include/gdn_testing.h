/*
 * gdn_testing.h -- test hooks of the GB300 Gated DeltaNet library.
 *
 * Not part of the recurrence: these entry points exist so that the test
 * suite can pin the tensor-core building blocks (tcgen05 MMA, shared-memory
 * matrix descriptors, 128-byte swizzled operand images, TMA tensor copies,
 * TMEM read-back) against a plain matmul before any kernel of the library
 * relies on them.  Conventions as in gdn.h (device pointers, async on stream).
 */
#ifndef GDN_GB300_TESTING_H
#define GDN_GB300_TESTING_H

#include <stdint.h>

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gdn_testing_tgemm -- the backward's batched tensor-core GEMM (kind::tf32,
 * the chunk gradients' contractions with bf16 I/O) on caller arrays: for
 * each unit b < batch,
 *   C[m][n] = alpha * col[n] * sum_k A'[m][k] B'[k][n] + beta * Cin[m][n]
 * for m < 64, n < N, then zeroed where mask asks (1: n > m, 2: n >= m).
 * A' is A stored [64][lda] (tA = 0) or [K][lda] (tA = 1); B' is B stored
 * [K][ldb] (tB = 0) or [N][ldb] (tB = 1); C and Cin are [64][ldc]; unit b's
 * arrays start sA, sB, sC, sCol floats after unit 0's.  Cin and col may be
 * null.  N in {64, 256}, K in {64, 256}, lda and ldb multiples of 4, A, B,
 * sA and sB 16-byte aligned; with tA = 1, lda, sA and A 32-byte aligned (8
 * floats), and with tB = 0 (not tiled) ldb, sB and B likewise:
 * GDN_ERR_UNSUPPORTED (shapes, leading dimensions) / GDN_ERR_ALIGNMENT
 * (addresses, unit strides) otherwise.
 * b_tiled = R > 0: each unit's B is an R x 256 matrix M in the backward's
 * tiled state layout (element (r, c) at ((c / 4) R + r) 4 + c % 4) and B' = M
 * (tB = 0, R = K, N = 256) or M transposed (tB = 1, R = N, K = 256); ldb is
 * then unused.  b_bf16 = 1 (tiled B only): M's elements are bf16 (B points at
 * them, sB counts bf16 elements), widened exactly to fp32 -- the backward's
 * chunk-start states at bf16 I/O.  Operands round to tf32 (10 explicit
 * mantissa bits); fp32 accumulation.
 */
int gdn_testing_tgemm(const float* A, int64_t sA, int32_t lda, int32_t tA, const float* B,
                      int64_t sB, int32_t ldb, int32_t tB, const float* Cin, float beta, float* C,
                      int64_t sC, int32_t ldc, const float* col, int64_t sCol, int32_t N,
                      int32_t K, float alpha, int32_t mask, int64_t batch, int32_t b_tiled,
                      int32_t b_bf16, gdn_stream_t stream);

/*
 * gdn_testing_umma_gemm -- D[128][N] (fp32) = A[128][K] * B[N][K]^T with
 * bf16 row-major inputs, on one CTA through tcgen05.mma (M = 128).
 *   a_mn / b_mn : stage the operand MN-major (1) or K-major (0) in a
 *                 128-byte-swizzled shared-memory image; an MN-major image
 *                 keeps 64 MN elements per 128-byte row, 8-row K groups 1024
 *                 bytes apart and 64-element MN blocks K*128 bytes apart; a
 *                 K-major image keeps 64 K elements per row and K blocks
 *                 R*128 bytes apart (R = 128 for A, N for B).
 *   a_lbo, a_sbo, b_lbo, b_sbo : leading / stride byte offsets written into the matrix
 *                 descriptors (so a test can check the convention).
 *   a_via_tma   : 0: threads stage A in shared memory; 1: a 2-D TMA tensor
 *                 copy loads A (K-major only); 2: A is stored into TMEM
 *                 (row m in lane m, two K elements per 32-bit column, the
 *                 lower half holding the even one) and the MMA reads it there.
 * 16 <= N <= 256 (N a multiple of 16 and a power of two, or 192);
 * K in {64, 128, 192, 256}.  Returns GDN_ERR_INVALID_ARG when a descriptor
 * could reach outside the kernel's shared-memory allocation.
 */
int gdn_testing_umma_gemm(const void* A, const void* B, float* D, int32_t N, int32_t K,
                          int32_t a_mn, int32_t b_mn, uint32_t a_lbo, uint32_t a_sbo,
                          uint32_t b_lbo, uint32_t b_sbo, int32_t a_via_tma,
                          gdn_stream_t stream);

/*
 * gdn_testing_umma_timing -- cycles of `reps` back-to-back chains of K/16
 * tcgen05.mma (M=128, N, bf16, fp32 accumulate) issued by one thread: A from
 * shared memory (K-major) or TMEM, B K-major or MN-major.  cycles (device,
 * 2 x uint64): [0] SM cycles spent issuing, [1] issue plus completion.
 * Operand values are arbitrary: this measures time only.
 */
int gdn_testing_umma_timing(int32_t N, int32_t K, int32_t a_from_tmem, int32_t b_mn,
                            int32_t reps, unsigned long long* cycles, gdn_stream_t stream);

/*
 * gdn_testing_prefill_prep -- run only the first (per-chunk, fully parallel)
 * kernel of the bf16 tensor-core prefill and leave its per-(chunk, head)
 * operand images in `images` (device, image_bytes >= max_chunks * heads *
 * gdn_testing_prefill_image_stride(), where max_chunks = batch * ceil(T/64)
 * for a dense batch and (T_total + 63 * N) / 64 for a packed one).  Chunk
 * ci (global index over all sequences), head h lives at byte offset
 * (ci * heads + h) * stride and holds, for the chunked WY form:
 *   +0       W and Q^ (64 x 256 each), 128-byte rows, row c = W[0..63][c]
 *            or Q^[0..63][c] (Q^ = gamma Q / sqrt(dk)), in blocks of 64 rows
 *            interleaved W_0 Q^_0 W_1 Q^_1 W_2 Q^_2 W_3 Q^_3: block b of W
 *            (rows 64b .. 64b+63) at +16384 b, of Q^ at +16384 b + 8192
 *   +65536   P^     (64 x 64) : 64 rows of 128 B (lower(Gam Q K^T) / sqrt(dk))
 *   +73728   U~^T rows 0-127   : row i = U~[0..63][i]
 *   +90112   decay block       : fp32 d[64] (d_r = gamma_L / gamma_r for r < L,
 *                               else 0), then fp32 G[64] (cumulative log decay)
 *   +90624   U~^T rows 128-255, then a copy of the decay block at +107008
 * Every 128-byte row r stores its 16-byte chunk j at position j XOR (r % 8).
 * Other arguments as for gdn_prefill with io_dtype = GDN_BF16.
 */
int gdn_testing_prefill_prep(const void* q, const void* k, const void* v, const float* alpha,
                             const float* beta, const int32_t* cu_seqlens, int32_t batch,
                             int64_t seqlen, int32_t heads, void* images, size_t image_bytes,
                             gdn_stream_t stream);

/* Byte stride between consecutive (chunk, head) images of gdn_testing_prefill_prep. */
size_t gdn_testing_prefill_image_stride(void);

/*
 * gdn_testing_set_trace -- phase timeline of the bf16 state pass.  While set,
 * every later gdn_prefill with bf16 I/O makes thread 0 of the state unit
 * (sequence 0, head 0, first row half) write its SM cycle counter (clock64)
 * at 12 points of each of its first max_chunks (at most 256) chunks into
 * device_buf (uint64 [max_chunks][12]): loop top, MMA-1 issued, U epilogue
 * done, after the following barrier, MMA-2 issued, MMA-2 complete, state
 * epilogue done, after the closing barrier, then (8) U accumulator loaded,
 * (9) state accumulator folded into the master state, (10) bf16 state
 * operand stored, (11) output accumulator loaded.  Thread 0 of the first
 * per-chunk worker stamps 9 points of its fifth (chunk, head) item at
 * device_buf[4096 + 0..8] (start, prologue done, Q^ in registers, Gram MMA
 * done, Q^ staged and A and P^ written, T solved, T_w / T_u ready, W / U~
 * MMAs done, images staged and their stores issued), and the worker's
 * bulk-copy thread 8 points around its copy issues at device_buf[4105 +
 * 0..7] (fused form: before and after publishing the previous item, after
 * issuing the next K / Q tiles; both forms: before and after issuing the
 * Q^ stores; fused: before and after waiting for those stores to read shared
 * memory; after issuing the W / U~ stores and the next V tile).  On the GPU global
 * timer (ns) the call also leaves: for state unit u = (sequence * heads +
 * head) * 2 + half < 128, its start, the top of its first chunk and its end
 * at device_buf[3072 + 3u + 0..2]; for per-chunk worker w < 200 (CTA w of
 * the split form's per-chunk kernel, or of the fused form's workers) its
 * start and end at device_buf[3456 + 2w + 0..1]; the start of each of the
 * first 240 items of worker 0 at device_buf[3856 + i].  So device_buf must
 * hold at least 4113 entries, zeroed.  Pass NULL to switch it off.
 * Not thread-safe; for profiling only.
 */
void gdn_testing_set_trace(uint64_t* device_buf, int32_t max_chunks);

/*
 * gdn_testing_last_prefill_form -- how the last bf16 prefill of this process
 * (gdn_prefill or gdn_prefill_noalloc) was launched: 1 fused (one cooperative launch in which per-chunk
 * workers publish each chunk's operands to the state pass through ready
 * flags), 0 split (per-chunk kernel, then state-pass kernel), -1 none yet.
 */
int32_t gdn_testing_last_prefill_form(void);

/*
 * gdn_testing_bounded_wait -- fault test of the library's bounded waits.
 * One thread waits on something that never completes: which = 0, an
 * mbarrier that expects one arrival and gets none (the try-wait every
 * tensor-core kernel uses for its copies and MMAs); which = 1, a ready flag in
 * global memory that nothing sets (the relaxed-load poll the fused prefill's
 * state pass uses for the per-chunk workers' results).  After limit_ns
 * nanoseconds of GPU global time (0 .. 2e9) the wait gives up, records
 * GDN_ERR_TIMEOUT in the device status word (read back with
 * gdn_get_device_status) and the kernel returns; nothing traps or hangs.
 * Returns GDN_ERR_INVALID_ARG for other arguments.
 */
int gdn_testing_bounded_wait(int32_t which, int64_t limit_ns, gdn_stream_t stream);

/*
 * gdn_testing_scratch_reserved -- bytes the library's scratch pool on the
 * current device holds mapped right now (cudaMemPoolAttrReservedMemCurrent;
 * 0 when no call has created the pool).  GDN_ERR_INVALID_ARG for a null
 * pointer, GDN_ERR_CUDA when the attribute cannot be read.
 */
int gdn_testing_scratch_reserved(uint64_t* bytes);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_TESTING_H */
