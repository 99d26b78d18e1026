// Launcher of the chunked backward pass (backward.cu).  Arguments and layouts
// are those of gdn_prefill_backward in include/gdn.h.
#pragma once

#include "gdn_internal.cuh"

namespace gdn {

// Device scratch the backward of a call with this many chunks needs (T_total
// is unused).  With bf16 I/O it includes the tensor-core forward's scratch:
// that forward re-run stores every chunk's start state and leaves the
// per-chunk operand images the reverse pass reads.
size_t prefill_backward_scratch_bytes(int64_t max_chunks, int32_t H, int32_t dv, int64_t T_total,
                                      int io_dtype);

// a: the forward's arguments (q, k, v, alpha, beta, S0, map, H, dv,
// max_chunks, scratch of prefill_backward_scratch_bytes); out and S_final unused.
cudaError_t launch_prefill_backward(const PrefillLaunch& a, const void* dout,
                                    const float* dS_final, void* dq, void* dk, void* dv,
                                    float* dalpha, float* dbeta, float* dS0, int io_dtype,
                                    cudaStream_t stream);

// The batched 64-row GEMM of the chunk gradients on the tensor cores
// (kind::tf32; tgemm.cu): per unit b, C = alpha * (A' B') diag(col) + beta *
// Cin, masked (1: keep n <= m, 2: n < m), m < 64.  A' = A [64][K] or (tA)
// stored [K][64]; B' = B [K][N] or (tB) stored [N][K], or (b_tiled = R > 0)
// the tiled_states layout of an R x 256 matrix, fp32 or (b_bf16) bf16.  N, K
// in {64, 256}.
bool tgemm_shape_ok(int N, int K, int lda, int ldb, int ldc, bool tA, bool tB, int b_tiled);
cudaError_t launch_tgemm(const float* A, size_t sA, int lda, const float* B, size_t sB, int ldb,
                         const float* Cin, float* C, size_t sC, int ldc, const float* col,
                         size_t sCol, int N, int K, float alpha, float beta, int mask,
                         int64_t batch, bool tA, bool tB, int b_tiled, int b_bf16,
                         unsigned* status, cudaStream_t st);

}  // namespace gdn
