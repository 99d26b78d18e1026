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
 * gdn_testing_umma_gemm -- D[128][N] (fp32) = A[128][K] * B[N][K]^T with
 * bf16 row-major inputs, on one CTA through tcgen05.mma (M = 128).
 *   a_mn / b_mn : stage the operand MN-major (1) or K-major (0) in a
 *                 128-byte-swizzled shared-memory image; an MN-major image
 *                 keeps 64 MN elements per 128-byte row, 8-row K groups 1024
 *                 bytes apart and 64-element MN blocks K*128 bytes apart; a
 *                 K-major image keeps 64 K elements per row and K blocks
 *                 R*128 bytes apart (R = 128 for A, N for B).
 *   *_lbo/*_sbo : leading / stride byte offsets written into the matrix
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
 * gdn_testing_prefill_prep -- run only the first (per-chunk, fully parallel)
 * kernel of the bf16 tensor-core prefill and leave its per-(chunk, head)
 * operand images in `images` (device, image_bytes >= max_chunks * heads *
 * gdn_testing_prefill_image_stride(), where max_chunks = batch * ceil(T/64)
 * for a dense batch and (T_total + 63 * N) / 64 for a packed one).  Chunk
 * ci (global index over all sequences), head h lives at byte offset
 * (ci * heads + h) * stride and holds, for the chunked WY form:
 *   +0       W      (64 x 256): 256 rows of 128 B; row c = W[0..63][c]
 *   +32768   Q^     (64 x 256): 4 blocks of 64 rows x 128 B; block b, row r
 *                               = Q^[r][64b .. 64b+63]  (Q^ = gamma Q / sqrt(dk))
 *   +65536   K^     (64 x 256): same block layout; K^ = diag(gamma_L / gamma) K
 *   +98304   P^     (64 x 64) : 64 rows of 128 B (lower(Gam Q K^T) / sqrt(dk))
 *   +106496  U~^T  (256 x 64) : row i = U~[0..63][i]
 *   +139264  G      (64 fp32) : cumulative log decay within the chunk
 * Every 128-byte row r stores its 16-byte chunk j at position j XOR (r % 8).
 * Other arguments as for gdn_prefill with io_dtype = GDN_BF16.
 */
int gdn_testing_prefill_prep(const void* q, const void* k, const void* v, const float* alpha,
                             const float* beta, const int32_t* cu_seqlens, int32_t batch,
                             int64_t seqlen, int32_t heads, void* images, size_t image_bytes,
                             gdn_stream_t stream);

/* Byte stride between consecutive (chunk, head) images of gdn_testing_prefill_prep. */
size_t gdn_testing_prefill_image_stride(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_TESTING_H */
