// Self-test GEMM for the tcgen05 building blocks: D[128 x N] = A[128 x K] *
// B[N x K]^T with bf16 operands staged in 128-byte-swizzled shared-memory
// images (K-major or MN-major, by threads or by a TMA tensor copy), fp32
// accumulation in TMEM, read back with tcgen05.ld.  The tests compare it with
// a plain matmul, which pins the descriptor and image conventions every
// tensor-core kernel of the library relies on.
#include <cuda.h>

#include <cstring>

#include "../../include/gdn_testing.h"
#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kSmemBytes = 220 * 1024;

struct UmmaArgs {
  const __nv_bfloat16* A;
  const __nv_bfloat16* B;
  float* D;
  int N, K;
  int a_mn, b_mn;
  uint32_t a_lbo, a_sbo, b_lbo, b_sbo;
  uint32_t b_offset;     // byte offset of the B image in shared memory
  int a_via_tma;
  unsigned* status;
};

// image byte offset of logical element (mn, k) of an operand with MN extent R
__device__ __forceinline__ uint32_t image_offset(int mn_major, int R, int K, int mn, int k) {
  if (!mn_major) return (uint32_t)(k / 64) * (uint32_t)(R * 128) + sw128_offset(mn, k % 64);
  return (uint32_t)(mn / 64) * (uint32_t)(K * 128) + sw128_offset(k, mn % 64);
}

__global__ void __launch_bounds__(128) umma_gemm_kernel(UmmaArgs a,
                                                         const __grid_constant__ CUtensorMap tmA) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  __shared__ uint64_t bar_mma, bar_tma;
  __shared__ uint32_t tmem_base;
  uint8_t* imgA = smem;
  uint8_t* imgB = smem + a.b_offset;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_tma, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t a_tmem = tmem + 256;   // A operand columns when staged in TMEM (mode 2)

  // stage B (and A unless TMA) by threads
  for (int e = tid; e < a.N * a.K; e += blockDim.x) {
    const int n = e / a.K, k = e % a.K;
    *(__nv_bfloat16*)(imgB + image_offset(a.b_mn, a.N, a.K, n, k)) = a.B[e];
  }
  if (a.a_via_tma == 2) {   // row m -> TMEM lane m, K pairs packed per column
    for (int c0 = 0; c0 < a.K / 2; c0 += 32) {
      uint32_t r[32];
      const __nv_bfloat16* row = a.A + (size_t)tid * a.K + 2 * c0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t lo = __bfloat16_as_ushort(row[2 * j]);
        const uint32_t hi = __bfloat16_as_ushort(row[2 * j + 1]);
        r[j] = lo | (hi << 16);
      }
      tmem_st32(a_tmem + ((uint32_t)(warp * 32) << 16) + c0, r);
    }
    tmem_st_wait();
  } else if (!a.a_via_tma) {
    for (int e = tid; e < 128 * a.K; e += blockDim.x) {
      const int m = e / a.K, k = e % a.K;
      *(__nv_bfloat16*)(imgA + image_offset(a.a_mn, 128, a.K, m, k)) = a.A[e];
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();

  bool ok = true;
  if (tid == 0) {
    if (a.a_via_tma == 1) {
      mbar_arrive_expect_tx(&bar_tma, 128 * a.K * 2);
      for (int b = 0; b < a.K / 64; ++b) tma_load_2d(imgA + b * 128 * 128, &tmA, b * 64, 0, &bar_tma);
      ok = mbar_wait(&bar_tma, 0);
    }
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, a.N, a.a_mn, a.b_mn);
      const uint32_t sa = smem_u32(imgA), sb = smem_u32(imgB);
      for (int s = 0; s < a.K / 16; ++s) {
        const uint32_t oa = a.a_mn ? s * 2048u : (s / 4) * (128u * 128u) + (s % 4) * 32u;
        const uint32_t ob = a.b_mn ? s * 2048u : (s / 4) * (uint32_t)(a.N * 128) + (s % 4) * 32u;
        if (a.a_via_tma == 2)
          mma_bf16_ts(tmem, a_tmem + 8 * s, smem_desc(sb + ob, a.b_lbo, a.b_sbo, kSwizzle128B),
                      idesc, s > 0);
        else
          mma_bf16(tmem, smem_desc(sa + oa, a.a_lbo, a.a_sbo, kSwizzle128B),
                   smem_desc(sb + ob, a.b_lbo, a.b_sbo, kSwizzle128B), idesc, s > 0);
      }
      mma_commit(&bar_mma);
    }
  }
  __syncthreads();
  __shared__ int okflag;
  if (tid == 0) okflag = ok;
  __syncthreads();
  if (okflag && mbar_wait(&bar_mma, 0)) {
    tc_fence_after();
    for (int c0 = 0; c0 < a.N; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, r);
      tmem_ld_wait();
      float* drow = a.D + (size_t)(warp * 32 + lane) * a.N + c0;
#pragma unroll
      for (int j = 0; j < 32; ++j) drow[j] = __uint_as_float(r[j]);
    }
  } else if (tid == 0) {
    flag_status(a.status, GDN_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// Issue `reps` back-to-back chains of K/16 MMAs (M=128, N, bf16) from one
// thread and count SM cycles from the first issue to the commit's arrival.
// Operand contents are whatever the shared memory / TMEM holds: only time.
__global__ void __launch_bounds__(128) umma_timing_kernel(int N, int K, int a_tmem_mode,
                                                           int b_mn, int reps,
                                                           unsigned long long* cycles,
                                                           unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  for (int e = tid; e < 48 * 1024; e += blockDim.x) reinterpret_cast<uint32_t*>(smem)[e] = 0x3c003c00u;
  fence_proxy_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16(128, N, 0, b_mn);
    const uint32_t sa = smem_u32(smem), sb = smem_u32(smem + 65536);
    const unsigned long long t0 = clock64();
    for (int r = 0; r < reps; ++r) {
      for (int s = 0; s < K / 16; ++s) {
        const uint64_t bd = b_mn ? smem_desc(sb + s * 2048, N * 128 > 8192 ? 8192 : 8192, 1024, kSwizzle128B)
                                 : smem_desc(sb + (s / 4) * (N * 128) + (s % 4) * 32, 16, 1024, kSwizzle128B);
        if (a_tmem_mode)
          mma_bf16_ts(tmem, tmem + 256 + 8 * (s % 16), bd, idesc, (r | s) != 0);
        else
          mma_bf16(tmem, smem_desc(sa + (s / 4) * 16384 + (s % 4) * 32, 16, 1024, kSwizzle128B), bd,
                   idesc, (r | s) != 0);
      }
    }
    const unsigned long long t1 = clock64();
    mma_commit(&bar);
    if (!mbar_wait(&bar, 0)) flag_status(status, GDN_ERR_TIMEOUT);
    const unsigned long long t2 = clock64();
    cycles[0] = t1 - t0;   // issue
    cycles[1] = t2 - t0;   // issue + completion
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// furthest byte (exclusive) an MMA of this operand can read from its start
uint32_t reach(int mn_major, int R, int K, uint32_t lbo, uint32_t sbo) {
  if (!mn_major) {   // per instruction: R/8 groups at SBO, last step at K-block K/64-1
    return (uint32_t)(K / 64 - 1) * R * 128 + 96 + (R / 8 - 1) * sbo + 1024;
  }
  return (uint32_t)(K / 16 - 1) * 2048 + (uint32_t)(R / 64 - 1) * lbo + sbo + 1024;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" int gdn_testing_umma_timing(int32_t N, int32_t K, int32_t a_from_tmem, int32_t b_mn,
                                       int32_t reps, unsigned long long* cycles,
                                       gdn_stream_t stream) {
  // operands stay inside 64 KB (A) + 128 KB (B) of the allocation
  if (!cycles || N < 16 || N > 256 || N % 16 || K < 16 || K > 256 || K % 64 || reps < 1 ||
      reps > 4096)
    return GDN_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(umma_timing_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes + 1024) != cudaSuccess)
    return GDN_ERR_CUDA;
  unsigned* st = status_ptr();
  if (!st) return GDN_ERR_CUDA;
  umma_timing_kernel<<<1, 128, kSmemBytes + 1024, (cudaStream_t)stream>>>(N, K, a_from_tmem, b_mn,
                                                                          reps, cycles, st);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" int gdn_testing_umma_gemm(const void* A, const void* B, float* D, int32_t N,
                                     int32_t K, int32_t a_mn, int32_t b_mn, uint32_t a_lbo,
                                     uint32_t a_sbo, uint32_t b_lbo, uint32_t b_sbo,
                                     int32_t a_via_tma, gdn_stream_t stream) {
  if (!A || !B || !D) return GDN_ERR_INVALID_ARG;
  if (N < 16 || N > 256 || N % 16 || K < 64 || K > 256 || K % 64) return GDN_ERR_UNSUPPORTED;
  if ((N & (N - 1)) && N != 192) return GDN_ERR_UNSUPPORTED;   // TMEM allocation size
  if (a_via_tma < 0 || a_via_tma > 2 || (a_via_tma && a_mn)) return GDN_ERR_UNSUPPORTED;
  const uint32_t a_bytes = 128u * K * 2, b_bytes = (uint32_t)N * K * 2;
  const uint32_t b_off = (a_bytes + 1023u) / 1024u * 1024u;
  // every descriptor must stay inside the shared-memory allocation
  if (reach(a_mn, 128, K, a_lbo, a_sbo) > (uint32_t)kSmemBytes ||
      b_off + reach(b_mn, N, K, b_lbo, b_sbo) > (uint32_t)kSmemBytes ||
      b_off + b_bytes > (uint32_t)kSmemBytes)
    return GDN_ERR_INVALID_ARG;
  CUtensorMap tm;
  memset(&tm, 0, sizeof tm);
  if (a_via_tma == 1) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess || !fn)
      return GDN_ERR_CUDA;
    auto encode = (CUresult(*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                               const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                               const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill))fn;
    cuuint64_t dims[2] = {(cuuint64_t)K, 128};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)A, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return GDN_ERR_CUDA;
  }
  UmmaArgs a{(const __nv_bfloat16*)A, (const __nv_bfloat16*)B, D, N, K, a_mn, b_mn, a_lbo,
             a_sbo, b_lbo, b_sbo, b_off, a_via_tma, nullptr};
  a.status = status_ptr();
  if (!a.status) return GDN_ERR_CUDA;
  if (cudaFuncSetAttribute(umma_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes + 1024) != cudaSuccess)
    return GDN_ERR_CUDA;
  umma_gemm_kernel<<<1, 128, kSmemBytes + 1024, (cudaStream_t)stream>>>(a, tm);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
