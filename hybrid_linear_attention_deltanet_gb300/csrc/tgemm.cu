// Batched 64-row GEMMs of the backward's chunk gradients on the tensor cores
// (tcgen05, kind::tf32: the fp32 operands enter as tf32, products accumulate
// in fp32 in TMEM).  Used by the backward with bf16 I/O, whose tolerance the
// tf32 rounding (2^-11 relative per operand) leaves ample room; fp32 I/O keeps
// the CUDA-core GEMM.
//
// Per unit b (a chunk and head):
//   C[m][n] = alpha * col[n] * sum_k A'[m][k] B'[k][n] + beta * Cin[m][n],
//   m < 64, n < N (64 or 256), K = 64 or 256,
// A' = A stored [64][K] or (kTA) [K][64]; B' = B stored [K][N] or (kTB)
// [N][K]; mask 1 keeps n <= m, 2 keeps n < m.  B may instead be a unit in
// the 4-column tiled layout of the backward's states (b_tiled = its row count
// R: element (r, c) of the R x 256 matrix at ((c / 4) R + r) 4 + c % 4), with
// B' = that matrix (kTB: B' = its transpose, R = N; otherwise R = K).
//
// The MMA computes the transpose D = C^T: its M rows are the n (blocks of 128;
// N = 64 runs one block whose upper 64 rows are unused), its 64 columns the m,
// so that each epilogue thread owns one n and its stores of C run along n.
// Both operands are K-major images with the 128-byte swizzle (a row holds 32
// fp32 of K), staged by all threads through registers in slabs of 32 K: rows
// whose K elements are contiguous in memory are copied as 16-byte pieces;
// the others are read 4 rows of the source at a time (lane = k) and written
// transposed.  Two stages: the loads of slab s + 1 are in flight while the
// MMAs of slab s run.
#include "../../include/gdn_testing.h"
#include "backward.cuh"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kTgThreads = 256;
constexpr int kTgSlab = 32;   // K per stage: one swizzle block of fp32

struct TgArgs {
  const float* A; size_t sA; int lda;
  const float* B; size_t sB; int ldb;
  const float* Cin; float* C; size_t sC; int ldc;
  const float* col; size_t sCol;
  int N, K;
  float alpha, beta;
  int mask;
  int64_t batch;
  unsigned* status;
  int b_tiled;   // 0: B as ldb says; R > 0: the tiled layout with R rows
  int b_bf16;    // (tiled B only) its elements are bf16, widened while staging
};

template <int kNB>
struct TgLayout {
  static constexpr uint32_t X = kNB * 16384;        // per stage: X image (kNB x 128 rows of n)
  static constexpr uint32_t Y = 8192;               //            Y image (64 rows of m)
  static constexpr uint32_t STAGE = X + Y;
  static constexpr uint32_t BYTES = 2 * STAGE + 1024;
};

// byte offset of 16-byte piece q (K elements 4q .. 4q+3 of the slab) of row r
__device__ __forceinline__ uint32_t piece(uint32_t r, uint32_t q) {
  return (r >> 7) * 16384u + (r & 127u) * 128u + ((q ^ (r & 7u)) << 4);
}

// four bf16 (8 bytes, read-only path) widened exactly to fp32
__device__ __forceinline__ float4 ld4_bf16(const __nv_bfloat16* p) {
  const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}

// 32 bytes from global memory (read-only path) as two float4; p 32-byte
// aligned.  The operands are never written while the kernel runs, so the load
// may be scheduled freely (not volatile).
__device__ __forceinline__ void ld32_nc(const float* p, float4& lo, float4& hi) {
  asm("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(lo.x), "=f"(lo.y), "=f"(lo.z), "=f"(lo.w), "=f"(hi.x), "=f"(hi.y),
                 "=f"(hi.z), "=f"(hi.w)
               : "l"(p));
}

template <bool kTA, bool kTB, int kNB>
__global__ void __launch_bounds__(kTgThreads, 2) tgemm_kernel(TgArgs g) {
  using Lay = TgLayout<kNB>;
  constexpr int kN = 128 * kNB;                          // rows of the X image staged: N
  constexpr int kNr = kNB == 1 ? 64 : 256;               // the GEMM's N
  constexpr int kXL = kNr * kTgSlab / 4 / kTgThreads;    // float4 loads of X a thread (2 or 8)
  constexpr int kYL = 64 * kTgSlab / 4 / kTgThreads;     // ... of Y (2)
  static_assert(kN >= kNr && kXL >= 1 && kYL == 2, "tile shape");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align_smem_1024(smem_raw);
  __shared__ uint64_t bar_buf[2], bar_done;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bar_buf[0], 1);
    mbar_init(&bar_buf[1], 1);
    mbar_init(&bar_done, 1);
    fence_barrier_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(&tmem_base, 64 * kNB);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const int nslab = g.K / kTgSlab;

  float4 rx[kXL], ry[kYL];
  // The transposed operands are read a row of K a lane: each lane takes two
  // adjacent 16-byte pieces of its row (all of a 32-byte sector), load j
  // covering columns ym0(j) / xn0(j) .. + 3.
  // (one 256-bit load for each pair, on 32-byte aligned rows: launch_tgemm
  // checks the alignment)
  auto ym0 = [&](int j) { return 8 * warp + 4 * j; };
  auto xn0 = [&](int j) { return 8 * (warp + 8 * (j >> 1)) + 4 * (j & 1); };
  // slab s of unit b into registers
  auto load = [&](int64_t b, int s) {
    const float* A = g.A + b * g.sA;
    const float* B = g.B + b * g.sB;
    const int k0 = s * kTgSlab;
#pragma unroll
    for (int j = 0; j < kYL; ++j) {
      if (!kTA) {   // row m of A, 16-byte piece q
        const int e = tid + j * kTgThreads, m = e >> 3, q = e & 7;
        ry[j] = __ldg(reinterpret_cast<const float4*>(A + (size_t)m * g.lda + k0 + 4 * q));
      } else if ((j & 1) == 0) {   // row k0 + lane of A, m = m0 .. m0 + 7: one 32-byte load
        ld32_nc(A + (size_t)(k0 + lane) * g.lda + ym0(j), ry[j], ry[j + 1]);
      }
    }
    const __nv_bfloat16* Bh = reinterpret_cast<const __nv_bfloat16*>(g.B) + b * g.sB;
    if (kTB && g.b_bf16) {
#pragma unroll
      for (int j = 0; j < kXL; ++j) {   // tiled bf16: row n, 4 columns of piece q (256 B a warp)
        const int e = tid + j * kTgThreads, n = e % kNr, q = e / kNr;
        rx[j] = ld4_bf16(Bh + ((size_t)(k0 / 4 + q) * g.b_tiled + n) * 4);
      }
    } else if (kTB) {
#pragma unroll
      for (int j = 0; j < kXL; ++j) {   // row n of B, 16-byte piece q (tiled: n fastest, 512 B a warp)
        const int e = tid + j * kTgThreads;
        const int n = g.b_tiled ? e % kNr : e >> 3, q = g.b_tiled ? e / kNr : e & 7;
        const size_t o = g.b_tiled ? ((size_t)(k0 / 4 + q) * g.b_tiled + n) * 4
                                   : (size_t)n * g.ldb + k0 + 4 * q;
        rx[j] = __ldg(reinterpret_cast<const float4*>(B + o));
      }
    } else if (g.b_tiled && g.b_bf16) {
#pragma unroll
      for (int j = 0; j < kXL; ++j)   // tile n0 / 4, row k0 + lane (8 bytes, 256 B a warp)
        rx[j] = ld4_bf16(Bh + ((size_t)(xn0(j) / 4) * g.b_tiled + k0 + lane) * 4);
    } else if (g.b_tiled) {
#pragma unroll
      for (int j = 0; j < kXL; ++j)   // tile n0 / 4, row k0 + lane (16 bytes, 512 B a warp)
        rx[j] = __ldg(reinterpret_cast<const float4*>(
            B + ((size_t)(xn0(j) / 4) * g.b_tiled + k0 + lane) * 4));
    } else {
#pragma unroll
      for (int j = 0; j < kXL; j += 2)   // row k0 + lane of B, n = n0 .. n0 + 7: one 32-byte load
        ld32_nc(B + (size_t)(k0 + lane) * g.ldb + xn0(j), rx[j], rx[j + 1]);
    }
  };
  auto stage = [&](int bf) {
    uint8_t* X = sm + bf * Lay::STAGE;
    uint8_t* Y = X + Lay::X;
#pragma unroll
    for (int j = 0; j < kYL; ++j) {
      if (!kTA) {
        const int e = tid + j * kTgThreads, m = e >> 3, q = e & 7;
        *reinterpret_cast<float4*>(Y + piece(m, q)) = ry[j];
      } else {
        const int m0 = ym0(j);
        const float v[4] = {ry[j].x, ry[j].y, ry[j].z, ry[j].w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<float*>(Y + piece(m0 + c, lane >> 2) + 4 * (lane & 3)) = v[c];
      }
    }
#pragma unroll
    for (int j = 0; j < kXL; ++j) {
      if (kTB) {
        const int e = tid + j * kTgThreads;
        const int n = g.b_tiled ? e % kNr : e >> 3, q = g.b_tiled ? e / kNr : e & 7;
        *reinterpret_cast<float4*>(X + piece(n, q)) = rx[j];
      } else {
        const int n0 = xn0(j);
        const float v[4] = {rx[j].x, rx[j].y, rx[j].z, rx[j].w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<float*>(X + piece(n0 + c, lane >> 2) + 4 * (lane & 3)) = v[c];
      }
    }
  };

  uint32_t cnt[2] = {0, 0};   // commits on each stage's barrier
  uint32_t done_ph = 0;
  int st = 0;                 // stages used so far (alternating buffers)
  int64_t b = blockIdx.x;
  if (b < g.batch) load(b, 0);
  for (; b < g.batch; b += gridDim.x) {
    for (int s = 0; s < nslab; ++s, ++st) {
      const int bf = st & 1;
      // the MMAs that last read this stage have finished
      if (cnt[bf] && !mbar_wait(&bar_buf[bf], (cnt[bf] - 1) & 1)) s_abort = 1;
      stage(bf);
      if (s + 1 < nslab) load(b, s + 1);
      else if (b + gridDim.x < g.batch) load(b + gridDim.x, 0);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (s_abort) break;
      if (tid == 0) {
        tc_fence_after();
        const uint32_t xa = smem_u32(sm + bf * Lay::STAGE), ya = xa + Lay::X;
        const uint32_t idesc = idesc_tf32(128, 64);
#pragma unroll
        for (int nb = 0; nb < kNB; ++nb)
#pragma unroll
          for (int ks = 0; ks < kTgSlab / 8; ++ks)
            mma_tf32(tmem + 64 * nb, smem_desc(xa + nb * 16384 + ks * 32, 16, 1024, kSwizzle128B),
                     smem_desc(ya + ks * 32, 16, 1024, kSwizzle128B), idesc, (s | ks) != 0);
        mma_commit(&bar_buf[bf]);
        if (s + 1 == nslab) mma_commit(&bar_done);
      }
      ++cnt[bf];
    }
    if (s_abort) break;
    if (!mbar_wait(&bar_done, done_ph)) s_abort = 1;
    done_ph ^= 1;
    tc_fence_after();
    // epilogue: this thread's n, all (kNB = 2) or half (kNB = 1) of the m
    const int qd = warp & 3, half = warp >> 2;
    const bool mine = kNB == 2 || qd < 2;
    if (!s_abort && mine) {
      const int n = kNB == 2 ? 128 * half + 32 * qd + lane : 32 * qd + lane;
      const float cs = g.col ? g.col[b * g.sCol + n] : 1.f;
      const float* cin = g.Cin ? g.Cin + b * g.sC + n : nullptr;
      float* cout = g.C + b * g.sC + n;
#pragma unroll
      for (int part = 0; part < (kNB == 2 ? 2 : 1); ++part) {
        const int m0 = kNB == 2 ? 32 * part : 32 * half;
        const uint32_t col0 = kNB == 2 ? 64 * half + m0 : m0;
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(32 * qd) << 16) + col0, r);
        tmem_ld_wait();
        // 16 rows at a time: Cin (which may be C itself) is read for all of
        // them before any is written, so the loads are in flight together
        // instead of each waiting behind the previous row's store
#pragma unroll
        for (int i0 = 0; i0 < 32; i0 += 16) {
          float cv[16];
          if (cin) {
#pragma unroll
            for (int i = 0; i < 16; ++i) cv[i] = cin[(size_t)(m0 + i0 + i) * g.ldc];
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int m = m0 + i0 + i;
            float v = g.alpha * cs * __uint_as_float(r[i0 + i]);
            if (cin) v = fmaf(g.beta, cv[i], v);
            if ((g.mask == 1 && n > m) || (g.mask == 2 && n >= m)) v = 0.f;
            cout[(size_t)m * g.ldc] = v;
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();   // TMEM read before the next unit's first MMA overwrites it
    if (s_abort) break;
  }
  if (s_abort && tid == 0) {   // let MMAs in flight finish before the TMEM goes
    flag_status(g.status, GDN_ERR_TIMEOUT);
    for (int bf = 0; bf < 2; ++bf)
      if (cnt[bf]) mbar_wait(&bar_buf[bf], (cnt[bf] - 1) & 1, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64 * kNB);
}

template <int kNB>
cudaError_t launch_nb(const TgArgs& g, bool tA, bool tB, cudaStream_t st) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cudaErrorUnknown;
  }
  const int64_t slots = 2 * (int64_t)sms;
  const unsigned grid = (unsigned)(g.batch < slots ? g.batch : slots);
  constexpr uint32_t smem = TgLayout<kNB>::BYTES;
  auto run = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kTgThreads, smem, st>>>(g);
    return cudaGetLastError();
  };
  if (!tA && !tB) return run(tgemm_kernel<false, false, kNB>);
  if (!tA && tB) return run(tgemm_kernel<false, true, kNB>);
  if (tA && !tB) return run(tgemm_kernel<true, false, kNB>);
  return run(tgemm_kernel<true, true, kNB>);
}

}  // namespace

bool tgemm_shape_ok(int N, int K, int lda, int ldb, int ldc, bool tA, bool tB, int b_tiled) {
  // 16-byte loads: leading dimensions and K multiples of 4; 32-byte loads of
  // the transposed A and of a row-major B stored [K][N]: multiples of 8
  if ((N != 64 && N != 256) || (K != 64 && K != 256)) return false;
  if (lda % 4 || ldc < N) return false;
  if (tA && lda % 8) return false;
  if (!tA ? lda < K : lda < 64) return false;
  if (b_tiled) {   // an R x 256 tiled matrix: 256 columns, R = N (kTB) or K
    return b_tiled == (tB ? N : K) && (tB ? K : N) == 256;
  }
  if (ldb % 4 || (!tB && ldb % 8)) return false;
  if (!tB ? ldb < N : ldb < K) return false;
  return true;
}

// base addresses and unit strides the loads need: 16 bytes throughout, 32
// for the operands read with 32-byte loads
bool tgemm_aligned(const float* A, size_t sA, const float* B, size_t sB, bool tA, bool tB,
                   int b_tiled) {
  const bool a32 = tA, b32 = !tB && !b_tiled;
  if ((((uintptr_t)A | (uintptr_t)B) & 15) || sA % 4 || sB % 4) return false;
  if (a32 && (((uintptr_t)A & 31) || sA % 8)) return false;
  if (b32 && (((uintptr_t)B & 31) || sB % 8)) return false;
  return true;
}

cudaError_t launch_tgemm(const float* A, size_t sA, int lda, const float* B, size_t sB, int ldb,
                         const float* Cin, float* C, size_t sC, int ldc, const float* col,
                         size_t sCol, int N, int K, float alpha, float beta, int mask,
                         int64_t batch, bool tA, bool tB, int b_tiled, int b_bf16,
                         unsigned* status, cudaStream_t st) {
  if (batch <= 0) return cudaSuccess;
  if (!tgemm_shape_ok(N, K, lda, ldb, ldc, tA, tB, b_tiled)) return cudaErrorInvalidValue;
  if (b_bf16 && !b_tiled) return cudaErrorInvalidValue;
  if (!tgemm_aligned(A, sA, B, sB, tA, tB, b_tiled)) return cudaErrorMisalignedAddress;
  TgArgs g{A, sA, lda, B, sB, ldb, Cin, C, sC, ldc, col, sCol, N, K, alpha, beta, mask, batch,
           status, b_tiled, b_bf16 ? 1 : 0};
  const cudaError_t e = N == 256 ? launch_nb<2>(g, tA, tB, st) : launch_nb<1>(g, tA, tB, st);
  count_launches(1);
  return e;
}

}  // namespace gdn

using namespace gdn;

extern "C" int gdn_testing_tgemm(const float* A, int64_t sA, int32_t lda, int32_t tA,
                                 const float* B, int64_t sB, int32_t ldb, int32_t tB,
                                 const float* Cin, float beta, float* C, int64_t sC, int32_t ldc,
                                 const float* col, int64_t sCol, int32_t N, int32_t K,
                                 float alpha, int32_t mask, int64_t batch, int32_t b_tiled,
                                 int32_t b_bf16, gdn_stream_t stream) {
  if (!A || !B || !C || batch < 0 || sA < 0 || sB < 0 || sC < 0 || sCol < 0 || mask < 0 ||
      mask > 2)
    return GDN_ERR_INVALID_ARG;
  if (b_tiled < 0 || !tgemm_shape_ok(N, K, lda, ldb, ldc, tA != 0, tB != 0, b_tiled))
    return GDN_ERR_UNSUPPORTED;
  if (b_bf16 < 0 || b_bf16 > 1 || (b_bf16 && !b_tiled)) return GDN_ERR_UNSUPPORTED;
  if (!tgemm_aligned(A, (size_t)sA, B, (size_t)sB, tA != 0, tB != 0, b_tiled))
    return GDN_ERR_ALIGNMENT;
  unsigned* status = status_ptr();
  if (!status) return GDN_ERR_CUDA;
  return launch_tgemm(A, (size_t)sA, lda, B, (size_t)sB, ldb, Cin, C, (size_t)sC, ldc, col,
                      (size_t)sCol, N, K, alpha, beta, mask, batch, tA != 0, tB != 0, b_tiled,
                      b_bf16, status, (cudaStream_t)stream) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}
