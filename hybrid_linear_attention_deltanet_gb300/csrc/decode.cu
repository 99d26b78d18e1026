// Fused single-token decode step of the gated delta rule.
//
// "Long-Context Aware Upcycling", Appendix A.3, Eq. 16-19, at T = 1 against a
// cached state (the fixed-size recurrent state the serving stack keeps per
// linear layer, Section 4.4).  With the state stored as S (dv x dk), row i
// of the update is
//     r_k = s_i . k,  r_q = s_i . q,  delta_i = beta (v_i - alpha r_k)
//     s_i <- alpha s_i + delta_i k^T
//     o_i  = (alpha r_q + delta_i (k . q)) / sqrt(dk)
// i.e. Eq. 16-18 for one column of the paper's S, and Eq. 19 read from the
// updated row without a second pass over it.
//
// Roofline: HBM.  Per (sequence, head) the dv x 256 fp32 state is read once
// and written once (512 KiB at dv = 256), against ~3 KiB of q, k, v, out,
// alpha, beta.
// Each warp streams whole 1 KiB rows with two 16-byte loads per lane (a fully
// coalesced 512 B per instruction), keeps kBatch = 4 rows (8 such loads) in
// flight, and reduces
// the two dot products with warp shuffles; the state never touches shared
// memory.  Loads and stores carry the streaming cache hint because a step's
// state (hundreds of MB) does not fit in L2.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRowsPerCta = 64;                 // a quarter of one head's state at dv = 256
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = kRowsPerCta / kWarps;  // 8
constexpr int kBatch = 4;                       // rows in flight per warp

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T>
__device__ __forceinline__ void load8(const T* p, int lane, float (&r)[8]) {
  // columns 4*lane .. 4*lane+3 and 128+4*lane .. 128+4*lane+3
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    r[j] = ld_in(p + 4 * lane + j);
    r[4 + j] = ld_in(p + 128 + 4 * lane + j);
  }
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
decode_step_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const float* __restrict__ alpha, const float* __restrict__ beta,
                   float* __restrict__ S, T* __restrict__ out, int32_t dv) {
  static_assert(kDK == 256, "row layout assumes rows of 256 fp32");
  const int blocks_per_unit = dv / kRowsPerCta;
  const int64_t unit = blockIdx.x / blocks_per_unit;    // n * H + h
  const int quarter = (int)(blockIdx.x % blocks_per_unit);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  float kr[8], qr[8];
  load8(k + unit * kDK, lane, kr);
  load8(q + unit * kDK, lane, qr);
  float kq = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) kq = fmaf(kr[j], qr[j], kq);
  kq = warp_sum(kq);
  const float a = alpha[unit], b = beta[unit];

  const int row0 = quarter * kRowsPerCta + warp * kRowsPerWarp;
  float* Srow0 = S + (unit * dv + row0) * kDK;
  const float vj = lane < kRowsPerWarp ? ld_in(v + unit * dv + row0 + lane) : 0.f;
  float o_mine = 0.f;

#pragma unroll
  for (int rb = 0; rb < kRowsPerWarp; rb += kBatch) {
    float4 s[kBatch][2];
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
      const float4* rowp = reinterpret_cast<const float4*>(Srow0 + (rb + r) * kDK);
      s[r][0] = __ldcs(rowp + lane);
      s[r][1] = __ldcs(rowp + 32 + lane);
    }
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
      const float x[8] = {s[r][0].x, s[r][0].y, s[r][0].z, s[r][0].w,
                          s[r][1].x, s[r][1].y, s[r][1].z, s[r][1].w};
      float rk = 0.f, rq = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        rk = fmaf(x[j], kr[j], rk);
        rq = fmaf(x[j], qr[j], rq);
      }
      rk = warp_sum(rk);
      rq = warp_sum(rq);
      const float vi = __shfl_sync(0xffffffffu, vj, rb + r);
      const float delta = b * (vi - a * rk);
      float y[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) y[j] = fmaf(a, x[j], delta * kr[j]);
      float4* roww = reinterpret_cast<float4*>(Srow0 + (rb + r) * kDK);
      __stcs(roww + lane, make_float4(y[0], y[1], y[2], y[3]));
      __stcs(roww + 32 + lane, make_float4(y[4], y[5], y[6], y[7]));
      const float o = (a * rq + delta * kq) * kScale;
      if (lane == rb + r) o_mine = o;
    }
  }
  if (lane < kRowsPerWarp) st_out(out + unit * dv + row0 + lane, o_mine);
}

}  // namespace

cudaError_t launch_decode_step(const void* q, const void* k, const void* v, const float* alpha,
                               const float* beta, float* S, void* out, int32_t N, int32_t H,
                               int32_t dv, int io_dtype, cudaStream_t stream) {
  if (!supported_dv(dv)) return cudaErrorInvalidValue;
  const int64_t units = (int64_t)N * H;
  const int64_t blocks = units * (dv / kRowsPerCta);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (blocks == 0) return cudaSuccess;
  if (io_dtype == GDN_BF16) {
    decode_step_kernel<__nv_bfloat16><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(
        (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, alpha, beta,
        S, (__nv_bfloat16*)out, dv);
  } else {
    decode_step_kernel<float><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(
        (const float*)q, (const float*)k, (const float*)v, alpha, beta, S, (float*)out, dv);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace gdn
