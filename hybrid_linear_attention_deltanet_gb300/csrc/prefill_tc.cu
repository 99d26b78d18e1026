// Chunkwise prefill on the 5th-generation tensor cores (tcgen05, bf16
// operands, fp32 accumulation in TMEM, fp32 master state).  Used for bf16 I/O.
//
// Chunked form of the gated delta rule (Appendix A.3 of "Long-Context Aware
// Upcycling": chunks of C = 64 tokens, intra-chunk delta corrections batched
// through the WY representation, state carried across chunks sequentially).
// For a chunk with start state S (dv x dk), rows r, j < L, G = cumsum(log
// alpha), gamma = exp(G), Gam_rj = exp(G_r - G_j), d_r = gamma_L / gamma_r:
//   A  = strict_lower(beta_r Gam_rj k_r.k_j),   T = (I + A)^{-1}
//   W  = T diag(beta gamma) K,  U~ = T diag(beta) V,  P^ = lower(Gam Q K^T)/sqrt(dk)
//   Q^ = diag(gamma) Q / sqrt(dk)
//   U  = U~ - W S^T,  O = Q^ S^T + P^ U,  S' = gamma_L S + U^T diag(d) K
//
// Kernel 1, tc_prep (one CTA per (chunk, head), fully parallel):
//   [K;Q] K^T on tcgen05 (M=128, N=64, K=256) -> A and P^ in fp32;
//   T by a blocked (16 x 16) fp32 forward substitution on the CUDA cores;
//   W^T = K^T T_w^T and U~^T = V^T T_u^T on tcgen05 (M=128 x 2 halves);
//   writes W, Q^, P^, U~^T and G to scratch as ready-to-load swizzled
//   operand images (the state pass copies them with 1-D TMA bulk copies).
// Kernel 2, tc_state (one CTA per (sequence, head, 128-row half of S)):
//   rows of S are independent, so each CTA owns 128 rows (the MMA M) and
//   walks the sequence's chunks: D_U = S W^T, D_O = S Q^^T (M=128, N=64,
//   K=256); U = U~ - D_U -> bf16; D_S = U^T (d K) (N=256, K=64) and
//   D_O += U^T P^^T; S = gamma_L S + D_S in fp32 registers; O -> out.
//
// Shared-memory operand images use the 128-byte swizzle: rows of 64 bf16,
// 16-byte chunk index XOR (row % 8), 8-row groups 1024 bytes apart.
//   K-major image of an R x K operand: K blocks of 64 columns, R*128 bytes apart.
//   MN-major image: one 128-byte row per K index holding 64 MN elements;
//   64-element MN blocks LBO bytes apart.
#include <cuda.h>

#include <cstring>

#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

using namespace sm100;

// ---- scratch image per (chunk, head)
constexpr size_t kImgW = 0;           // W   : MN-major B image, 256 K-rows (c) x 64 (r)
constexpr size_t kImgQ = 32768;       // Q^  : K-major B image, 4 K-blocks x (64 rows x 128 B)
constexpr size_t kImgP = 65536;       // P^  : K-major B image, 64 rows x 64
constexpr size_t kImgU = 73728;       // U~^T: 256 rows (i) x 64 (r), 128-byte swizzled rows
constexpr size_t kImgG = 106496;      // G   : 64 fp32
constexpr size_t kImgStride = 107520;

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&t);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// byte offset of 16-byte chunk `ch` (0..7) of row `row` in a 128-byte-swizzled image
__device__ __forceinline__ uint32_t sw_chunk(uint32_t row, uint32_t ch) {
  return row * 128u + ((ch ^ (row & 7u)) << 4);
}

// ============================================================ prep kernel
constexpr int kPrepThreads = 128;
// shared memory layout (offsets from the 1024-aligned base)
constexpr uint32_t kP_KQ = 0;          // 64 KB: K-block b at b*16K: rows 0-63 K, 64-127 Q
constexpr uint32_t kP_V = 65536;       // 32 KB: column block b at b*8K (64 rows x 128 B)
constexpr uint32_t kP_TW = 98304;      // 8 KB : T diag(beta gamma), K-major 64 x 64
constexpr uint32_t kP_TU = 106496;     // 8 KB : T diag(beta)
constexpr uint32_t kP_A = 114688;      // fp32 [64][65]
constexpr uint32_t kP_T = kP_A + 64 * 65 * 4;
constexpr uint32_t kP_X = kP_T + 64 * 65 * 4;   // fp32 [3][256] block temporaries
constexpr uint32_t kP_G = kP_X + 3 * 256 * 4;   // fp32 [64]
constexpr uint32_t kP_B = kP_G + 256;           // fp32 [64]
constexpr uint32_t kP_END = kP_B + 256;
constexpr uint32_t kPrepSmem = kP_END + 1024;

__global__ void __launch_bounds__(kPrepThreads, 1)
tc_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const float* __restrict__ alpha,
               const float* __restrict__ beta, SeqMap map, int32_t H,
               uint8_t* __restrict__ scratch, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align_smem_1024(smem_raw);
  float* sA = (float*)(sm + kP_A);
  float* sT = (float*)(sm + kP_T);
  float* sX = (float*)(sm + kP_X);
  float* sG = (float*)(sm + kP_G);
  float* sB = (float*)(sm + kP_B);
  __shared__ uint64_t bar_kq, bar_v, bar_a, bar_bc;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;

  const int64_t ci = blockIdx.x;
  const int h = blockIdx.y;
  int n, L;
  int64_t t0;
  if (!map.locate(ci, n, t0, L)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* img = scratch + (size_t)(ci * H + h) * kImgStride;

  if (tid == 0) {
    mbar_init(&bar_kq, 1);
    mbar_init(&bar_v, 1);
    mbar_init(&bar_a, 1);
    mbar_init(&bar_bc, 1);
    fence_barrier_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(&tmem_base, 256);
  if (tid < kC) {
    const bool ok = tid < L;
    sG[tid] = ok ? logf(alpha[(t0 + tid) * H + h]) : 0.f;
    sB[tid] = ok ? beta[(t0 + tid) * H + h] : 0.f;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar_kq, 65536);
    for (int b = 0; b < 4; ++b) {
      tma_load_3d(sm + kP_KQ + b * 16384, &tm_k, b * 64, h, (int32_t)t0, &bar_kq);
      tma_load_3d(sm + kP_KQ + b * 16384 + 8192, &tm_q, b * 64, h, (int32_t)t0, &bar_kq);
    }
    mbar_arrive_expect_tx(&bar_v, 32768);
    for (int b = 0; b < 4; ++b)
      tma_load_3d(sm + kP_V + b * 8192, &tm_v, b * 64, h, (int32_t)t0, &bar_v);
    float acc = 0.f;   // decay prefix G_r = sum_{s <= r} log alpha_s
    for (int r = 0; r < kC; ++r) { acc += sG[r]; sG[r] = acc; }
  }
  __syncthreads();

  // ---- [K; Q] K^T  ->  TMEM columns [0, 64): lanes 0-63 K K^T, 64-127 Q K^T
  if (tid == 0) {
    if (!mbar_wait(&bar_kq, 0)) {
      s_abort = 1;
    } else {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, 64, 0, 0);
      const uint32_t base = smem_u32(sm + kP_KQ);
      for (int s = 0; s < 16; ++s) {
        const uint32_t off = (s >> 2) * 16384u + (s & 3) * 32u;
        const uint64_t d = smem_desc(base + off, 16, 1024, kSwizzle128B);
        mma_bf16(tmem, d, d, idesc, s > 0);
      }
      mma_commit(&bar_a);
    }
  }
  __syncthreads();
  if (s_abort) goto teardown;
  if (!mbar_wait(&bar_a, 0)) { flag_status(status, GDN_ERR_TIMEOUT); s_abort = 1; }
  __syncthreads();
  if (s_abort) goto teardown;
  tc_fence_after();
  {
    uint32_t g0[32], g1[32];
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16), g0);
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + 32, g1);
    tmem_ld_wait();
    const int row = tid;
    if (row < kC) {   // A = strict_lower(beta_r Gam_rj k_r.k_j)
      const float Gr = sG[row], br = sB[row];
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const float kk = __uint_as_float(j < 32 ? g0[j] : g1[j - 32]);
        sA[row * 65 + j] = j < row ? br * __expf(Gr - sG[j]) * kk : 0.f;
      }
    } else {          // P^ = lower(Gam_rj q_r.k_j) / sqrt(dk), bf16 K-major image
      const int r = row - kC;
      const float Gr = sG[r];
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j0 = ch * 8 + 2 * e, j1 = j0 + 1;
          const float q0 = __uint_as_float(j0 < 32 ? g0[j0] : g1[j0 - 32]);
          const float q1 = __uint_as_float(j1 < 32 ? g0[j1] : g1[j1 - 32]);
          const float p0 = (j0 <= r && r < L) ? kScale * __expf(Gr - sG[j0]) * q0 : 0.f;
          const float p1 = (j1 <= r && r < L) ? kScale * __expf(Gr - sG[j1]) * q1 : 0.f;
          w[e] = pack_bf16(p0, p1);
        }
        *reinterpret_cast<uint4*>(img + kImgP + sw_chunk(r, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    // Q^ = gamma_r Q / sqrt(dk): same swizzled rows as the Q half of the [K; Q] image
    for (int e = tid; e < 4 * 64 * 8; e += kPrepThreads) {
      const int b = e >> 9, r = (e >> 3) & 63, p = e & 7;
      const float sc = r < L ? kScale * __expf(sG[r]) : 0.f;
      uint4 v = *reinterpret_cast<const uint4*>(sm + kP_KQ + b * 16384 + 8192 + r * 128 + p * 16);
      v.x = pack_bf16(bf16_lo(v.x) * sc, bf16_hi(v.x) * sc);
      v.y = pack_bf16(bf16_lo(v.y) * sc, bf16_hi(v.y) * sc);
      v.z = pack_bf16(bf16_lo(v.z) * sc, bf16_hi(v.z) * sc);
      v.w = pack_bf16(bf16_lo(v.w) * sc, bf16_hi(v.w) * sc);
      *reinterpret_cast<uint4*>(img + kImgQ + b * 8192 + r * 128 + p * 16) = v;
    }
  }
  tc_fence_before();
  __syncthreads();

  // ---- T = (I + A)^{-1}, blocked 4 x 4 over 16 x 16 blocks, fp32
  if (tid < 64) {   // diagonal blocks: thread -> (block b, column c)
    const int b = tid >> 4, c = tid & 15, o = 16 * b;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) x[r] = r == c ? 1.f : 0.f;
#pragma unroll
    for (int r = 1; r < 16; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < r; ++j) acc = fmaf(sA[(o + r) * 65 + o + j], x[j], acc);
      if (r > c) x[r] = -acc;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) sT[(o + r) * 65 + o + c] = x[r];
  }
  __syncthreads();
  for (int bi = 1; bi < 4; ++bi) {
    // X_bj = sum_{k=j}^{bi-1} A_{bi,k} T_{k,j}   for j < bi
    for (int e = tid; e < bi * 256; e += kPrepThreads) {
      const int bj = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
      float acc = 0.f;
      for (int m = 16 * bj; m < 16 * bi; ++m)
        acc = fmaf(sA[(16 * bi + rr) * 65 + m], sT[m * 65 + 16 * bj + cc], acc);
      sX[e] = acc;
    }
    __syncthreads();
    // T_{bi,j} = -T_{bi,bi} X_bj
    for (int e = tid; e < bi * 256; e += kPrepThreads) {
      const int bj = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        acc = fmaf(sT[(16 * bi + rr) * 65 + 16 * bi + m], sX[bj * 256 + m * 16 + cc], acc);
      sT[(16 * bi + rr) * 65 + 16 * bj + cc] = -acc;
    }
    __syncthreads();
  }
  // T_w = T diag(beta gamma), T_u = T diag(beta): K-major bf16 images (row r, col j)
  {
    const int r = tid >> 1, jh = tid & 1;
#pragma unroll
    for (int cq = 0; cq < 4; ++cq) {
      const int ch = jh * 4 + cq;
      uint32_t ww[4], uu[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j0 = ch * 8 + 2 * e, j1 = j0 + 1;
        const float t0v = j0 <= r ? sT[r * 65 + j0] : 0.f;
        const float t1v = j1 <= r ? sT[r * 65 + j1] : 0.f;
        const float b0 = sB[j0], b1 = sB[j1];
        ww[e] = pack_bf16(t0v * b0 * __expf(sG[j0]), t1v * b1 * __expf(sG[j1]));
        uu[e] = pack_bf16(t0v * b0, t1v * b1);
      }
      *reinterpret_cast<uint4*>(sm + kP_TW + sw_chunk(r, ch)) = make_uint4(ww[0], ww[1], ww[2], ww[3]);
      *reinterpret_cast<uint4*>(sm + kP_TU + sw_chunk(r, ch)) = make_uint4(uu[0], uu[1], uu[2], uu[3]);
    }
  }
  fence_proxy_async_smem();
  __syncthreads();

  // ---- W^T = K^T T_w^T and U~^T = V^T T_u^T, two 128-row halves each
  if (tid == 0) {
    if (!mbar_wait(&bar_v, 0)) {
      s_abort = 1;
    } else {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, 64, 1, 0);
      const uint32_t kq = smem_u32(sm + kP_KQ), v = smem_u32(sm + kP_V);
      const uint32_t tw = smem_u32(sm + kP_TW), tu = smem_u32(sm + kP_TU);
      for (int hh = 0; hh < 2; ++hh) {
        for (int s = 0; s < 4; ++s)
          mma_bf16(tmem + hh * 64, smem_desc(kq + hh * 32768 + s * 2048, 16384, 1024, kSwizzle128B),
                   smem_desc(tw + s * 32, 16, 1024, kSwizzle128B), idesc, s > 0);
        for (int s = 0; s < 4; ++s)
          mma_bf16(tmem + 128 + hh * 64,
                   smem_desc(v + hh * 16384 + s * 2048, 8192, 1024, kSwizzle128B),
                   smem_desc(tu + s * 32, 16, 1024, kSwizzle128B), idesc, s > 0);
      }
      mma_commit(&bar_bc);
    }
  }
  __syncthreads();
  if (s_abort) goto teardown;
  if (!mbar_wait(&bar_bc, 0)) { flag_status(status, GDN_ERR_TIMEOUT); s_abort = 1; }
  __syncthreads();
  if (s_abort) goto teardown;
  tc_fence_after();
  for (int hh = 0; hh < 2; ++hh) {
    const uint32_t c = 128 * hh + 32 * warp + lane;   // d_k row of W^T / d_v row of U~^T
    for (int part = 0; part < 2; ++part) {        // 0: W, 1: U~^T
      uint32_t g0[32], g1[32];
      const uint32_t col = part * 128 + hh * 64;
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + col, g0);
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + col + 32, g1);
      tmem_ld_wait();
      uint8_t* dst = img + (part == 0 ? kImgW : kImgU);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j0 = ch * 8 + 2 * e;
          const float a0 = __uint_as_float(j0 < 32 ? g0[j0] : g1[j0 - 32]);
          const float a1 = __uint_as_float(j0 + 1 < 32 ? g0[j0 + 1] : g1[j0 + 1 - 32]);
          w[e] = pack_bf16(a0, a1);
        }
        *reinterpret_cast<uint4*>(dst + sw_chunk(c, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  if (tid < kC) reinterpret_cast<float*>(img + kImgG)[tid] = sG[tid];

teardown:
  if (s_abort && tid == 0) {
    flag_status(status, GDN_ERR_TIMEOUT);
    mbar_wait(&bar_kq, 0, 100000000ull);   // let copies still in flight land
    mbar_wait(&bar_v, 0, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// =========================================================== state kernel
constexpr int kStateThreads = 256;
constexpr uint32_t kS_S = 0;          // 64 KB: S bf16, K-major A image, 128 rows x 256
constexpr uint32_t kS_W = 65536;      // 32 KB
constexpr uint32_t kS_Q = 98304;      // 32 KB
constexpr uint32_t kS_K = 131072;     // 32 KB: K, MN-major B image (4 column blocks of 8 KB)
constexpr uint32_t kS_P = 163840;     // 8 KB
constexpr uint32_t kS_AU = 172032;    // 16 KB: U^T bf16, K-major A image, 128 rows x 64
constexpr uint32_t kS_UT = 188416;    // 16 KB: U~^T rows of this half
constexpr uint32_t kS_O = 204800;     // 16 KB: output staging [64][128] bf16
constexpr uint32_t kS_END = 221184;
constexpr uint32_t kStateSmem = kS_END + 1024;
// TMEM columns
constexpr uint32_t kT_U = 0, kT_O = 64, kT_S = 256;

__global__ void __launch_bounds__(kStateThreads, 1)
tc_state_kernel(const __grid_constant__ CUtensorMap tm_k, const float* __restrict__ S0,
                __nv_bfloat16* __restrict__ out, float* __restrict__ S_final, SeqMap map,
                int32_t H, const uint8_t* __restrict__ scratch, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align_smem_1024(smem_raw);
  __shared__ uint64_t bar_wq, bar_k, bar_u, bar_m1, bar_m2;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  __shared__ float s_d[64];
  __shared__ float s_gC;

  const int n = blockIdx.x, h = blockIdx.y, half = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, colhalf = warp >> 2;
  const uint32_t iloc = 32 * quarter + lane;            // TMEM lane = local row of S
  const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
  const int64_t cb = map.chunk_begin(n), ce = map.chunk_end(n);
  const int64_t s_begin = map.seq_begin(n), s_end = map.seq_end(n);

  if (tid == 0) {
    mbar_init(&bar_wq, 1);
    mbar_init(&bar_k, 1);
    mbar_init(&bar_u, 1);
    mbar_init(&bar_m1, 1);
    mbar_init(&bar_m2, 1);
    fence_barrier_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);

  // master state rows (fp32, registers): this thread's 128 columns of row iloc
  float S[128];
  const size_t srow = (((size_t)n * H + h) * kDV + 128 * half + iloc) * kDK + 128 * colhalf;
  if (S0) {
    const float4* p = reinterpret_cast<const float4*>(S0 + srow);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float4 t = p[j];
      S[4 * j] = t.x; S[4 * j + 1] = t.y; S[4 * j + 2] = t.z; S[4 * j + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 128; ++j) S[j] = 0.f;
  }
  auto write_S_image = [&]() {
#pragma unroll
    for (int q8 = 0; q8 < 16; ++q8) {   // 16 chunks of 8 columns
      const int kb = 2 * colhalf + (q8 >> 3), ch = q8 & 7;
      uint4 v = make_uint4(pack_bf16(S[8 * q8], S[8 * q8 + 1]), pack_bf16(S[8 * q8 + 2], S[8 * q8 + 3]),
                           pack_bf16(S[8 * q8 + 4], S[8 * q8 + 5]), pack_bf16(S[8 * q8 + 6], S[8 * q8 + 7]));
      *reinterpret_cast<uint4*>(sm + kS_S + kb * 16384 + sw_chunk(iloc, ch)) = v;
    }
  };
  write_S_image();
  fence_proxy_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  auto issue_wqu = [&](int64_t ci) {
    const uint8_t* src = scratch + (size_t)(ci * H + h) * kImgStride;
    mbar_arrive_expect_tx(&bar_wq, 65536);
    tma_load_1d(sm + kS_W, src + kImgW, 32768, &bar_wq);
    tma_load_1d(sm + kS_Q, src + kImgQ, 32768, &bar_wq);
    mbar_arrive_expect_tx(&bar_u, 16384);
    tma_load_1d(sm + kS_UT, src + kImgU + half * 16384, 16384, &bar_u);
  };
  auto issue_kp = [&](int64_t ci) {
    const uint8_t* src = scratch + (size_t)(ci * H + h) * kImgStride;
    const int32_t t0 = (int32_t)(s_begin + (ci - cb) * kC);
    mbar_arrive_expect_tx(&bar_k, 32768 + 8192);
    for (int b = 0; b < 4; ++b) tma_load_3d(sm + kS_K + b * 8192, &tm_k, b * 64, h, t0, &bar_k);
    tma_load_1d(sm + kS_P, src + kImgP, 8192, &bar_k);
  };
  // outstanding-load bookkeeping (thread 0), for a clean exit after a timeout
  int pend_wq = 0, pend_k = 0, pend_u = 0;
  if (tid == 0 && cb < ce) {
    issue_wqu(cb);
    issue_kp(cb);
    pend_wq = pend_k = pend_u = 1;
  }

  for (int64_t ci = cb; ci < ce; ++ci) {
    const uint32_t par = (uint32_t)((ci - cb) & 1);
    const int64_t t0 = s_begin + (ci - cb) * kC;
    const int L = (int)min((int64_t)kC, s_end - t0);
    const float* Gg = reinterpret_cast<const float*>(scratch + (size_t)(ci * H + h) * kImgStride + kImgG);

    // 1. D_U = S W^T, D_O = S Q^^T
    if (tid == 0) {
      if (!mbar_wait(&bar_wq, par)) {
        s_abort = 1;
      } else {
        pend_wq = 0;
        tc_fence_after();
        const uint32_t idW = idesc_bf16(128, 64, 0, 1), idQ = idesc_bf16(128, 64, 0, 0);
        const uint32_t sS = smem_u32(sm + kS_S), sW = smem_u32(sm + kS_W), sQ = smem_u32(sm + kS_Q);
        for (int s = 0; s < 16; ++s) {
          const uint64_t a = smem_desc(sS + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024, kSwizzle128B);
          mma_bf16(tmem + kT_U, a, smem_desc(sW + s * 2048, 32768, 1024, kSwizzle128B), idW, s > 0);
          mma_bf16(tmem + kT_O, a,
                   smem_desc(sQ + (s >> 2) * 8192 + (s & 3) * 32, 16, 1024, kSwizzle128B), idQ,
                   s > 0);
        }
        mma_commit(&bar_m1);
      }
    }
    // 2. decay factors for this chunk
    if (tid < kC) {
      const float GL = Gg[L - 1];
      s_d[tid] = tid < L ? __expf(GL - Gg[tid]) : 0.f;
      if (tid == 0) s_gC = __expf(GL);
    }
    __syncthreads();
    if (s_abort) break;
    // K <- diag(d) K in place (rows r: 8 lanes cover one 128-byte row)
    if (!mbar_wait(&bar_k, par)) { flag_status(status, GDN_ERR_TIMEOUT); s_abort = 1; }
    if (tid == 0) pend_k = 0;
    {
      const int p = tid & 7, r0 = tid >> 3;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int r = r0 + 32 * rr;
        const float d = s_d[r];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint4* ptr = reinterpret_cast<uint4*>(sm + kS_K + b * 8192 + r * 128 + p * 16);
          uint4 v = *ptr;
          v.x = pack_bf16(bf16_lo(v.x) * d, bf16_hi(v.x) * d);
          v.y = pack_bf16(bf16_lo(v.y) * d, bf16_hi(v.y) * d);
          v.z = pack_bf16(bf16_lo(v.z) * d, bf16_hi(v.z) * d);
          v.w = pack_bf16(bf16_lo(v.w) * d, bf16_hi(v.w) * d);
          *ptr = v;
        }
      }
    }
    // 3. U = U~ - D_U  ->  bf16 K-major A image (row iloc, columns r)
    if (!mbar_wait(&bar_m1, par) || !mbar_wait(&bar_u, par)) {
      flag_status(status, GDN_ERR_TIMEOUT);
      s_abort = 1;
    } else {
      if (tid == 0) pend_u = 0;
      tc_fence_after();
      uint32_t g[32];
      tmem_ld32(tmem + lane_off + kT_U + 32 * colhalf, g);
      tmem_ld_wait();
#pragma unroll
      for (int cq = 0; cq < 4; ++cq) {
        const int ch = 4 * colhalf + cq;
        const uint4 ut = *reinterpret_cast<const uint4*>(sm + kS_UT + sw_chunk(iloc, ch));
        const uint32_t uw[4] = {ut.x, ut.y, ut.z, ut.w};
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float u0 = bf16_lo(uw[e]) - __uint_as_float(g[8 * cq + 2 * e]);
          const float u1 = bf16_hi(uw[e]) - __uint_as_float(g[8 * cq + 2 * e + 1]);
          w[e] = pack_bf16(u0, u1);
        }
        *reinterpret_cast<uint4*>(sm + kS_AU + sw_chunk(iloc, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (s_abort) break;

    // 4. D_S = U^T (d K) ; D_O += U^T P^^T ; prefetch the next chunk's W, Q^, U~^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id2 = idesc_bf16(128, 256, 0, 1), idO = idesc_bf16(128, 64, 0, 0);
      const uint32_t sAU = smem_u32(sm + kS_AU), sK = smem_u32(sm + kS_K), sP = smem_u32(sm + kS_P);
      for (int s = 0; s < 4; ++s) {
        const uint64_t a = smem_desc(sAU + s * 32, 16, 1024, kSwizzle128B);
        mma_bf16(tmem + kT_S, a, smem_desc(sK + s * 2048, 8192, 1024, kSwizzle128B), id2, s > 0);
        mma_bf16(tmem + kT_O, a, smem_desc(sP + s * 32, 16, 1024, kSwizzle128B), idO, 1);
      }
      mma_commit(&bar_m2);
      if (ci + 1 < ce) {
        issue_wqu(ci + 1);
        pend_wq = pend_u = 1;
      }
    }

    // 5. S = gamma_L S + D_S (fp32) -> bf16 image; O -> staging
    if (!mbar_wait(&bar_m2, par)) {
      flag_status(status, GDN_ERR_TIMEOUT);
      s_abort = 1;
    } else {
      tc_fence_after();
      const float gC = s_gC;
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) {
        uint32_t g[32];
        tmem_ld32(tmem + lane_off + kT_S + 128 * colhalf + 32 * g4, g);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) S[32 * g4 + j] = fmaf(gC, S[32 * g4 + j], __uint_as_float(g[j]));
      }
      write_S_image();
      uint32_t g[32];
      tmem_ld32(tmem + lane_off + kT_O + 32 * colhalf, g);
      tmem_ld_wait();
      __nv_bfloat16* so = reinterpret_cast<__nv_bfloat16*>(sm + kS_O);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        so[(32 * colhalf + j) * 128 + iloc] = __float2bfloat16_rn(__uint_as_float(g[j]));
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (s_abort) break;

    // 6. prefetch the next chunk's K and P^; write this chunk's rows of out
    if (tid == 0 && ci + 1 < ce) {
      issue_kp(ci + 1);
      pend_k = 1;
    }
    {
      const int r = tid >> 2, seg = tid & 3;
      if (r < L) {
        const uint4* src = reinterpret_cast<const uint4*>(sm + kS_O + r * 256 + seg * 64);
        uint4* dst = reinterpret_cast<uint4*>(out + ((t0 + r) * H + h) * kDV + 128 * half + 32 * seg);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = src[q];
      }
    }
  }

  if (!s_abort && S_final) {
    float4* p = reinterpret_cast<float4*>(S_final + srow);
#pragma unroll
    for (int j = 0; j < 32; ++j) p[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
  }
  if (tid == 0 && s_abort) {   // let copies still in flight land before the CTA exits
    flag_status(status, GDN_ERR_TIMEOUT);
    if (pend_wq) mbar_wait(&bar_wq, 0, 100000000ull), mbar_wait(&bar_wq, 1, 100000000ull);
    if (pend_k) mbar_wait(&bar_k, 0, 100000000ull), mbar_wait(&bar_k, 1, 100000000ull);
    if (pend_u) mbar_wait(&bar_u, 0, 100000000ull), mbar_wait(&bar_u, 1, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------- host side
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = (EncodeFn)p;
  }
  return fn;
}

// [T_total][H][256] bf16 viewed as (feature, head, token); box 64 x 1 x 64,
// 128-byte swizzle; token rows past the end of the tensor read as zero.
bool make_token_map(CUtensorMap* m, const void* base, int64_t T_total, int32_t H) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  memset(m, 0, sizeof *m);
  cuuint64_t dims[3] = {(cuuint64_t)kDK, (cuuint64_t)H, (cuuint64_t)(T_total > 0 ? T_total : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)kDK * 2, (cuuint64_t)H * kDK * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t prefill_tc_scratch_bytes(int64_t max_chunks, int32_t H) {
  return (size_t)max_chunks * H * kImgStride;
}

size_t prefill_tc_image_stride() { return kImgStride; }

cudaError_t launch_prefill_tc(const PrefillLaunch& a, cudaStream_t stream, bool prep_only) {
  static_assert(kDK == 256 && kDV == 256, "image layouts assume 256 x 256 heads");
  const int64_t T_total = a.map.cu_seqlens ? a.map.T : (int64_t)a.map.N * a.map.T;
  CUtensorMap tq, tk, tv;
  if (!make_token_map(&tq, a.q, T_total, a.H) || !make_token_map(&tk, a.k, T_total, a.H) ||
      !make_token_map(&tv, a.v, T_total, a.H))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(tc_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kPrepSmem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(tc_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kStateSmem)) != cudaSuccess)
    return e;
  uint8_t* scr = (uint8_t*)a.scratch;
  if (a.max_chunks > 0) {
    tc_prep_kernel<<<dim3((unsigned)a.max_chunks, (unsigned)a.H), kPrepThreads, kPrepSmem,
                     stream>>>(tq, tk, tv, a.alpha, a.beta, a.map, a.H, scr, a.status);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (prep_only) return cudaSuccess;
  tc_state_kernel<<<dim3((unsigned)a.map.N, (unsigned)a.H, 2), kStateThreads, kStateSmem,
                    stream>>>(tk, a.S0, (__nv_bfloat16*)a.out, a.S_final, a.map, a.H, scr,
                              a.status);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace gdn
