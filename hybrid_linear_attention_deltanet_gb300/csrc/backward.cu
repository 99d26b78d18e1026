// Backward pass of the chunked gated delta rule: fp32 I/O on the CUDA cores,
// bf16 I/O on the tensor cores (see "bf16 I/O" below).
//
// The training kernel of "Long-Context Aware Upcycling" (Appendix A.3, last
// paragraph) splits sequences into chunks of C = 64 tokens, batches the delta
// corrections of a chunk through the WY representation and carries the state
// across chunks sequentially.  This file differentiates that chunked form.
// Per chunk (rows r, j), with start state S (dv x dk), G = cumsum(log alpha),
// gamma = e^G, Gam_rj = e^{G_r - G_j}, d_r = e^{G_L - G_r}, s = 1/sqrt(dk):
//   A = strict_lower(beta_r Gam KK^T), T = (I + A)^-1,
//   W = T diag(beta gamma) K, U~ = T diag(beta) V, U = U~ - W S^T,
//   Qh = s diag(gamma) Q, Ph = s lower(Gam QK^T),
//   O = Qh S^T + Ph U,  S' = gamma_L S + U^T diag(d) K.
// Given dO and the gradient dS' of the chunk's end state:
//   dU  = Ph^T dO + diag(d) K dS'^T
//   dS  = gamma_L dS' + dO^T Qh - dU^T W             (carried to the chunk before)
//   dQh = dO S, dPh = lower(dO U^T), dW = -dU S, dK += diag(d) U dS',
//   dd_r = u_r . (dS' k_r), dgamma_L = <dS', S>,
// then through W and U~ (dT = dW Bw^T + dU Bu^T with Bw = diag(beta gamma) K,
// Bu = diag(beta) V), T (dA = -T^T dT T^T, strictly lower), A, Ph, Qh and the
// decays down to log alpha (a reverse cumulative sum inside the chunk).
//
// Structure (every intermediate per (chunk, head) unit in scratch):
//   gather      q, k, v, dO of each chunk -> zero-padded 64-row fp32 tiles;
//               G (padding rows add log alpha = 0), beta (0 on padding) and
//               beta gamma.  Padding rows then contribute nothing anywhere.
//   prep        KK^T, QK^T (batched GEMM), T by forward substitution, Ph,
//               W and U~ (batched GEMM).
//   fwd_states  per (sequence, head, 16-row slice of S): the forward state
//               pass, storing every chunk's start state.
//   rev_states  per (sequence, head, 16-row slice): the reverse pass over
//               chunks for dS; stores dS' and dU per chunk, dS0 at the end.
//               Rows of dS are independent exactly as rows of S are.
//   then batched 64-row GEMMs and three per-chunk elementwise kernels for the
//   local gradients, and a final scatter into the token layout.
// bf16 I/O: the tensor-core forward of gdn_prefill re-runs (split form, no
// outputs), storing every chunk's start state as bf16 tiles and leaving
// KK^T, QK^T, Ph and T in fp32 from its per-chunk kernel; the tensor-core
// reverse pass stores dS' (bf16 tiles) and dU; the GEMMs run as tf32
// tcgen05 products (tgemm.cu); the re-run and the reverse pass go to an
// internal high-priority stream while the caller's stream runs the gather,
// W and U~ and the products that need no reverse output.
#include <mutex>

#include <functional>

#include "backward.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kNS = 16;              // rows of S (or dS) per state-pass CTA
constexpr int kRG = 256 / kNS;       // row groups of the C x kNS products (256 threads)
constexpr int kRPT = kC / kRG;       // rows a thread owns in them
constexpr int kCC = kC * kC;
constexpr int kSlabF = 32;           // rows of a 64 x 256 operand staged at a time (forward)
constexpr int kSlabR = 8;            // ... (reverse, which stages two operands)

// ------------------------------------------------------------------ scratch
struct Bwd {
  int64_t units;   // max_chunks * H
  int32_t dv;
  float *Q, *K, *V, *dO;          // [64][256] [64][256] [64][dv] [64][dv]
  float *G, *B, *BG;              // [64]: cumsum log alpha, beta, beta*gamma
  float *KK, *QK, *Tm, *TmB, *TmU, *Ph;   // [64][64]
  float *W, *Ut;                  // [64][256] [64][dv]
  float *Sst, *dSp;               // [dv][256]; bf16 in the tiled layout with bf16 I/O at
                                  // dv = 256 (the forward re-run's and the reverse pass's
                                  // stores), else fp32
  float *dU, *U, *TdU;            // [64][dv]
  float *dQh, *dW, *dK1, *TdW, *dKa, *dQa;   // [64][256]
  float *dPh, *dTm, *X, *dA, *Ms, *FG;       // [64][64]
  float *dGc, *dBc;               // [64]
  float *dgLp;                    // [dv / 32]
  __host__ __device__ size_t sD() const { return (size_t)kC * kDK; }
  __host__ __device__ size_t sV() const { return (size_t)kC * dv; }
  __host__ __device__ size_t sS() const { return (size_t)dv * kDK; }
};

size_t bwd_bytes_per_unit(int32_t dv) {
  const size_t D = (size_t)kC * kDK, V = (size_t)kC * dv, S = (size_t)dv * kDK;
  return 4 * (2 * D + 2 * V + 3 * kC + 6 * kCC + D + V + 2 * S + 3 * V + 6 * D + 6 * kCC +
              2 * kC + dv / kNS);
}

Bwd carve(void* base, int64_t units, int32_t dv) {
  Bwd s{};
  s.units = units;
  s.dv = dv;
  char* p = (char*)base;
  auto take = [&](size_t per_unit) {
    float* r = (float*)p;
    p += align_up((size_t)units * per_unit * 4, 256);
    return r;
  };
  const size_t D = (size_t)kC * kDK, V = (size_t)kC * dv, S = (size_t)dv * kDK;
  s.Q = take(D); s.K = take(D); s.V = take(V); s.dO = take(V);
  s.G = take(kC); s.B = take(kC); s.BG = take(kC);
  s.KK = take(kCC); s.QK = take(kCC); s.Tm = take(kCC); s.TmB = take(kCC); s.TmU = take(kCC);
  s.Ph = take(kCC);
  s.W = take(D); s.Ut = take(V);
  s.Sst = take(S); s.dSp = take(S);
  s.dU = take(V); s.U = take(V); s.TdU = take(V);
  s.dQh = take(D); s.dW = take(D); s.dK1 = take(D); s.TdW = take(D); s.dKa = take(D);
  s.dQa = take(D);
  s.dPh = take(kCC); s.dTm = take(kCC); s.X = take(kCC); s.dA = take(kCC); s.Ms = take(kCC);
  s.FG = take(kCC);
  s.dGc = take(kC); s.dBc = take(kC);
  s.dgLp = take(dv / kNS);
  return s;
}

size_t bwd_scratch_bytes(int64_t units, int32_t dv) {
  // every array is padded to 256 B: bound by the per-unit sum plus 40 paddings
  return (size_t)units * bwd_bytes_per_unit(dv) + 40 * 256;
}

// ------------------------------------------------------------------ gather
// four consecutive input elements (8- or 16-byte aligned) as fp32
__device__ __forceinline__ float4 ld4_in(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float4 ld4_in(const __nv_bfloat16* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
gather_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
              const T* __restrict__ dout, const float* __restrict__ alpha,
              const float* __restrict__ beta, SeqMap map, int32_t H, Bwd s) {
  const int64_t ci = blockIdx.x;
  const int h = blockIdx.y, tid = threadIdx.x;
  const int64_t u = ci * H + h;
  int n = 0, L = 0;
  int64_t t0 = 0;
  if (!map.locate(ci, n, t0, L)) L = 0;   // units past the last chunk stay all-zero
  const int dv = s.dv;
  // four consecutive elements a thread (16-byte fp32 stores)
  for (int e = 4 * tid; e < kC * kDK; e += 4 * kThreads) {
    const int r = e / kDK, c = e % kDK;
    const int64_t g = ((t0 + r) * H + h) * kDK + c;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(s.Q + u * s.sD() + e) = r < L ? ld4_in(q + g) : z;
    *reinterpret_cast<float4*>(s.K + u * s.sD() + e) = r < L ? ld4_in(k + g) : z;
  }
  for (int e = 4 * tid; e < kC * dv; e += 4 * kThreads) {
    const int r = e / dv, c = e % dv;
    const int64_t g = ((t0 + r) * H + h) * dv + c;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(s.V + u * s.sV() + e) = r < L ? ld4_in(v + g) : z;
    *reinterpret_cast<float4*>(s.dO + u * s.sV() + e) = r < L ? ld4_in(dout + g) : z;
  }
  if (tid < 32) {   // G = cumsum(log alpha) by warp scan over two halves
    float carry = 0.f;
    for (int half = 0; half < 2; ++half) {
      const int r = half * 32 + tid;
      float x = r < L ? logf(alpha[(t0 + r) * H + h]) : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (tid >= o) x += y;
      }
      x += carry;
      const float b = r < L ? beta[(t0 + r) * H + h] : 0.f;
      s.G[u * kC + r] = x;
      s.B[u * kC + r] = b;
      s.BG[u * kC + r] = b * expf(x);   // beta_r gamma_r
      carry = __shfl_sync(0xffffffffu, x, 31);
    }
  }
}

// ------------------------------------------------------------------ batched GEMM
// C = alpha * colscale[n] * (A' B')[m][n] + beta * Cin[m][n], m < 64, per unit b;
// K a multiple of 32, N of 64.
// A' = A [64][K] (row stride lda) or, kTA, A stored [K][64];
// B' = B [K][N] or, kTB, B stored [N][K].  mask 1: keep n <= m; 2: keep n < m.
struct BG {
  const float* A; size_t sA; int lda;
  const float* B; size_t sB; int ldb;
  const float* Cin; float* C; size_t sC; int ldc;
  const float* col; size_t sCol;
  int N, K;
  float alpha, beta;
  int mask;
  int64_t batch;
};

// 64 x TN output tiles (TN = 128: 8 x 4 outputs a thread; TN = 64: 4 x 4), K
// in slabs of 32 staged through shared memory, the next slab's global loads
// (16-byte vectors along the contiguous axis) in registers while the current
// slab computes.
template <bool kTA, bool kTB, int TN>
__global__ void __launch_bounds__(kThreads) bgemm_kernel(BG g) {
  constexpr int KS = 32;
  constexpr int RM = TN == 128 ? 8 : 4;              // rows a thread
  constexpr int TNG = TN / 4;                         // column groups of 4
  constexpr int NA = KS * kC / 4 / kThreads;          // float4 loads of A a thread (2)
  constexpr int NB = KS * TN / 4 / kThreads;          // ... of B (4 or 2)
  __shared__ __align__(16) float As[KS][kC + 4];
  __shared__ __align__(16) float Bs[KS][TN + 4];
  const int tid = threadIdx.x, tm = tid / TNG, tn = tid % TNG;
  const int n0 = blockIdx.x * TN;
  for (int64_t b = blockIdx.y; b < g.batch; b += gridDim.y) {
    const float* A = g.A + b * g.sA;
    const float* B = g.B + b * g.sB;
    float4 ra[NA], rb[NB];
    auto load = [&](int k0) {
#pragma unroll
      for (int j = 0; j < NA; ++j) {
        const int idx = tid + j * kThreads;
        ra[j] = !kTA ? *reinterpret_cast<const float4*>(A + (size_t)(idx >> 3) * g.lda + k0 + 4 * (idx & 7))
                     : *reinterpret_cast<const float4*>(A + (size_t)(k0 + (idx >> 4)) * g.lda + 4 * (idx & 15));
      }
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const int idx = tid + j * kThreads;
        rb[j] = !kTB ? *reinterpret_cast<const float4*>(B + (size_t)(k0 + idx / TNG) * g.ldb + n0 + 4 * (idx % TNG))
                     : *reinterpret_cast<const float4*>(B + (size_t)(n0 + (idx >> 3)) * g.ldb + k0 + 4 * (idx & 7));
      }
    };
    auto stage = [&]() {
#pragma unroll
      for (int j = 0; j < NA; ++j) {
        const int idx = tid + j * kThreads;
        if (!kTA) {
          const int m = idx >> 3, q = idx & 7;
          As[4 * q][m] = ra[j].x; As[4 * q + 1][m] = ra[j].y;
          As[4 * q + 2][m] = ra[j].z; As[4 * q + 3][m] = ra[j].w;
        } else {
          *reinterpret_cast<float4*>(&As[idx >> 4][4 * (idx & 15)]) = ra[j];
        }
      }
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const int idx = tid + j * kThreads;
        if (!kTB) {
          *reinterpret_cast<float4*>(&Bs[idx / TNG][4 * (idx % TNG)]) = rb[j];
        } else {
          const int nn = idx >> 3, q = idx & 7;
          Bs[4 * q][nn] = rb[j].x; Bs[4 * q + 1][nn] = rb[j].y;
          Bs[4 * q + 2][nn] = rb[j].z; Bs[4 * q + 3][nn] = rb[j].w;
        }
      }
    };
    float acc[RM][4];
#pragma unroll
    for (int i = 0; i < RM; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    __syncthreads();                     // the previous unit's last slab is consumed
    load(0);
    stage();
    __syncthreads();
    for (int k0 = 0; k0 < g.K; k0 += KS) {
      const bool more = k0 + KS < g.K;
      if (more) load(k0 + KS);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        float av[RM];
#pragma unroll
        for (int i = 0; i < RM; i += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(&As[kk][tm * RM + i]);
          av[i] = a4.x; av[i + 1] = a4.y; av[i + 2] = a4.z; av[i + 3] = a4.w;
        }
        const float4 b4 = *reinterpret_cast<const float4*>(&Bs[kk][tn * 4]);
        const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int i = 0; i < RM; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      if (more) {
        __syncthreads();
        stage();
        __syncthreads();
      }
    }
#pragma unroll
    for (int i = 0; i < RM; ++i) {
      const int m = tm * RM + i;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int nn = n0 + tn * 4 + j;
        float val = g.alpha * acc[i][j];
        if (g.col) val *= g.col[b * g.sCol + nn];
        if (g.Cin) val = fmaf(g.beta, g.Cin[b * g.sC + (size_t)m * g.ldc + nn], val);
        if ((g.mask == 1 && nn > m) || (g.mask == 2 && nn >= m)) val = 0.f;
        g.C[b * g.sC + (size_t)m * g.ldc + nn] = val;
      }
    }
  }
}

// ------------------------------------------------------------------ prep: T, Ph
__global__ void __launch_bounds__(kThreads) tprep_kernel(Bwd s) {
  __shared__ __align__(16) float As[kC][kC + 4];   // 16-byte rows: read 4 at a time
  __shared__ float Ts[kC][kC + 1];
  __shared__ float Gs[kC], Bs[kC], BGs[kC];
  const int64_t u = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid < kC) {
    Gs[tid] = s.G[u * kC + tid];
    Bs[tid] = s.B[u * kC + tid];
    BGs[tid] = Bs[tid] * expf(Gs[tid]);   // beta_j gamma_j
  }
  __syncthreads();
  for (int e = tid; e < kCC; e += kThreads) {
    const int r = e >> 6, j = e & 63;
    const float gam = j <= r ? expf(Gs[r] - Gs[j]) : 0.f;
    As[r][j] = j < r ? Bs[r] * gam * s.KK[u * kCC + e] : 0.f;
    s.Ph[u * kCC + e] = j <= r ? kScale * gam * s.QK[u * kCC + e] : 0.f;
  }
  __syncthreads();
  if (tid < kC) {   // (I + A)^-1 by forward substitution, one column per thread
    // column c in registers; row r's sum over j < r in four partial sums
    // (A is strictly lower, so the terms j >= r a float4 rounds up to are 0)
    const int c = tid;
    float x[kC];
#pragma unroll
    for (int r = 0; r < kC; ++r) x[r] = r == c ? 1.f : 0.f;
#pragma unroll
    for (int r = 1; r < kC; ++r) {
      float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
      for (int j4 = 0; j4 < r; j4 += 4) {
        const float4 a = *reinterpret_cast<const float4*>(&As[r][j4]);
        p0 = fmaf(a.x, x[j4], p0);
        p1 = fmaf(a.y, x[j4 + 1], p1);
        p2 = fmaf(a.z, x[j4 + 2], p2);
        p3 = fmaf(a.w, x[j4 + 3], p3);
      }
      if (r > c) x[r] = -((p0 + p1) + (p2 + p3));
    }
#pragma unroll
    for (int r = 0; r < kC; ++r) Ts[r][c] = x[r];
    s.BG[u * kC + c] = BGs[c];
  }
  __syncthreads();
  for (int e = tid; e < kCC; e += kThreads) {
    const int r = e >> 6, j = e & 63;
    const float t = Ts[r][j];
    s.Tm[u * kCC + e] = t;
    s.TmB[u * kCC + e] = t * BGs[j];
    s.TmU[u * kCC + e] = t * Bs[j];
  }
}

// ------------------------------------------------------------------ forward states
// Shared-memory rows are 16-byte multiples so that the inner products read
// four values a load: ~5 loads per 16 FMAs.
constexpr int kSP = kDK + 4;         // row stride of the S / dS slice
constexpr int kWS = 68;              // row stride of a 64-column W slab (forward)
constexpr int kKS = 32;              // dk columns of a K slab (reverse)
constexpr int kKSP = kKS + 4;        // its row stride
constexpr int kUP = kNS + 4;         // row stride of the C x kNS tiles
constexpr int kPP = kC + 4;          // row stride of the staged Ph

__global__ void __launch_bounds__(kThreads)
fwd_states_kernel(const float* __restrict__ S0, SeqMap map, int32_t H, Bwd s) {
  extern __shared__ __align__(16) float sm[];
  float* Ss = sm;                   // [kNS][kSP]
  float* Wt = Ss + kNS * kSP;       // [C][kWS]  64 columns of W
  float* Us = Wt + kC * kWS;        // [C][kUP]
  float* Ks = Us + kC * kUP;        // [kSlabF][256]
  float* dec = Ks + kSlabF * kDK;   // [C]
  const int n = blockIdx.x, h = blockIdx.y, slice = blockIdx.z;
  const int tid = threadIdx.x, i = tid % kNS, r4 = (tid / kNS) * kRPT;
  const int dv = s.dv;
  const int64_t sbase = ((int64_t)n * H + h) * dv * kDK + (int64_t)slice * kNS * kDK;
  for (int e = tid; e < kNS * kDK; e += kThreads)
    Ss[(e / kDK) * kSP + e % kDK] = S0 ? S0[sbase + e] : 0.f;
  const int64_t cb = map.chunk_begin(n), ce = map.chunk_end(n);
  for (int64_t ci = cb; ci < ce; ++ci) {
    const int64_t u = ci * H + h;
    __syncthreads();
    float* dst = s.Sst + u * s.sS() + (size_t)slice * kNS * kDK;
    for (int e = tid; e < kNS * kDK; e += kThreads) dst[e] = Ss[(e / kDK) * kSP + e % kDK];
    const float* G = s.G + u * kC;
    const float GL = G[kC - 1];
    if (tid < kC) dec[tid] = expf(GL - G[tid]);
    const float gL = expf(GL);
    // U = U~ - W S^T: rows r4 .. r4+3, column i; 4 columns of dk a step
    float acc[kRPT];
#pragma unroll
    for (int m = 0; m < kRPT; ++m) acc[m] = 0.f;
    const float* Wg = s.W + u * s.sD();
    // the next 64 columns of W are in flight (registers) while a slab computes
    constexpr int kWL = kC * 16 / kThreads;          // float4 loads a thread a slab
    float4 wpre[kWL];
    auto load_w = [&](int c0) {
#pragma unroll
      for (int j = 0; j < kWL; ++j) {
        const int e = tid + j * kThreads;
        wpre[j] = *reinterpret_cast<const float4*>(Wg + (e >> 4) * kDK + c0 + 4 * (e & 15));
      }
    };
    load_w(0);
    for (int c0 = 0; c0 < kDK; c0 += 64) {
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kWL; ++j) {
        const int e = tid + j * kThreads;
        *reinterpret_cast<float4*>(&Wt[(e >> 4) * kWS + 4 * (e & 15)]) = wpre[j];
      }
      __syncthreads();
      if (c0 + 64 < kDK) load_w(c0 + 64);
#pragma unroll 4
      for (int cc = 0; cc < 64; cc += 4) {
        const float4 sv = *reinterpret_cast<const float4*>(&Ss[i * kSP + c0 + cc]);
#pragma unroll
        for (int m = 0; m < kRPT; ++m) {
          const float4 w = *reinterpret_cast<const float4*>(&Wt[(r4 + m) * kWS + cc]);
          acc[m] = fmaf(w.x, sv.x, fmaf(w.y, sv.y, fmaf(w.z, sv.z, fmaf(w.w, sv.w, acc[m]))));
        }
      }
    }
    const float* Ug = s.Ut + u * s.sV();
#pragma unroll
    for (int m = 0; m < kRPT; ++m) Us[(r4 + m) * kUP + i] = Ug[(r4 + m) * dv + slice * kNS + i] - acc[m];
    // S' = gamma_L S + U^T diag(d) K: column c = tid, the slice's kNS rows
    {
      const int c = tid;
      const float4* Kg = reinterpret_cast<const float4*>(s.K + u * s.sD());
      float a2[kNS];
#pragma unroll
      for (int m = 0; m < kNS; ++m) a2[m] = 0.f;
      constexpr int kKL = kSlabF * kDK / 4 / kThreads;
      float4 kpre[kKL];
      auto load_k = [&](int q0) {
#pragma unroll
        for (int j = 0; j < kKL; ++j) kpre[j] = Kg[q0 * kDK / 4 + tid + j * kThreads];
      };
      load_k(0);
      for (int q0 = 0; q0 < kC; q0 += kSlabF) {
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kKL; ++j) reinterpret_cast<float4*>(Ks)[tid + j * kThreads] = kpre[j];
        __syncthreads();
        if (q0 + kSlabF < kC) load_k(q0 + kSlabF);
#pragma unroll 2
        for (int r = 0; r < kSlabF; ++r) {
          const float kd = dec[q0 + r] * Ks[r * kDK + c];
          const float4* ur = reinterpret_cast<const float4*>(&Us[(q0 + r) * kUP]);
#pragma unroll
          for (int m4 = 0; m4 < kNS / 4; ++m4) {
            const float4 u4 = ur[m4];
            a2[4 * m4] = fmaf(u4.x, kd, a2[4 * m4]);
            a2[4 * m4 + 1] = fmaf(u4.y, kd, a2[4 * m4 + 1]);
            a2[4 * m4 + 2] = fmaf(u4.z, kd, a2[4 * m4 + 2]);
            a2[4 * m4 + 3] = fmaf(u4.w, kd, a2[4 * m4 + 3]);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < kNS; ++m) Ss[m * kSP + c] = fmaf(gL, Ss[m * kSP + c], a2[m]);
    }
  }
}

// ------------------------------------------------------------------ dgamma_L partials
// <dS', S_start> of each (chunk, head) over 16-row slices of the state, as
// the CUDA-core reverse pass leaves them (used with the tensor-core one):
// one CTA per (unit, slice).
// kBf: dS' and the states are bf16 (the tiled layout at dv = 256, both in
// the same element order), else fp32
__device__ __forceinline__ float4 widen_bf16x4(uint2 w) {
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}
template <bool kBf>
__global__ void __launch_bounds__(kThreads) dgl_kernel(Bwd s) {
  __shared__ float red[kThreads / 32];
  const int64_t u = blockIdx.x;
  const int sl = blockIdx.y, tid = threadIdx.x;
  const size_t off = u * s.sS() + (size_t)sl * kNS * kDK;
  auto bf = [&](const float* base) {
    return reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(base) + off);
  };
  float part = 0.f;
  for (int e = tid; e < kNS * kDK / 4; e += kThreads) {
    const float4 x = kBf ? widen_bf16x4(bf(s.dSp)[e])
                         : reinterpret_cast<const float4*>(s.dSp + off)[e];
    const float4 y = kBf ? widen_bf16x4(bf(s.Sst)[e])
                         : reinterpret_cast<const float4*>(s.Sst + off)[e];
    part = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, part))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if ((tid & 31) == 0) red[tid >> 5] = part;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) t += red[w];
    s.dgLp[u * (s.dv / kNS) + sl] = t;
  }
}

// ------------------------------------------------------------------ reverse states
__global__ void __launch_bounds__(kThreads)
rev_states_kernel(const float* __restrict__ dS_final, float* __restrict__ dS0, SeqMap map,
                  int32_t H, Bwd s) {
  extern __shared__ __align__(16) float sm[];
  float* Ds = sm;                   // [kNS][kSP]  this CTA's rows of dS
  float* Kt = Ds + kNS * kSP;       // [C][kKSP]   32 columns of K
  float* Os = Kt + kC * kKSP;       // [C][kUP]    dO columns of the slice
  float* Us = Os + kC * kUP;        // [C][kUP]    dU columns of the slice
  float* Qs = Us + kC * kUP;        // [kSlabR][256]
  float* Ws = Qs + kSlabR * kDK;    // [kSlabR][256]
  float* Pt = Ws + kSlabR * kDK;    // [C][kPP]
  float* dec = Pt + kC * kPP;       // [C]
  float* gq = dec + kC;             // [C]  s * gamma_r
  float* red = gq + kC;             // [8]
  const int n = blockIdx.x, h = blockIdx.y, slice = blockIdx.z;
  const int tid = threadIdx.x, i = tid % kNS, r4 = (tid / kNS) * kRPT;
  const int dv = s.dv;
  const int64_t sbase = ((int64_t)n * H + h) * dv * kDK + (int64_t)slice * kNS * kDK;
  for (int e = tid; e < kNS * kDK; e += kThreads)
    Ds[(e / kDK) * kSP + e % kDK] = dS_final ? dS_final[sbase + e] : 0.f;
  const int64_t cb = map.chunk_begin(n), ce = map.chunk_end(n);
  for (int64_t ci = ce - 1; ci >= cb; --ci) {
    const int64_t u = ci * H + h;
    __syncthreads();
    // dS' of this chunk, and its part of <dS', S_start>
    float* dst = s.dSp + u * s.sS() + (size_t)slice * kNS * kDK;
    const float* Sg = s.Sst + u * s.sS() + (size_t)slice * kNS * kDK;
    float part = 0.f;
    for (int e = tid; e < kNS * kDK; e += kThreads) {
      const float d = Ds[(e / kDK) * kSP + e % kDK];
      dst[e] = d;
      part = fmaf(d, Sg[e], part);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if ((tid & 31) == 0) red[tid >> 5] = part;
    const float* G = s.G + u * kC;
    const float GL = G[kC - 1];
    if (tid < kC) {
      dec[tid] = expf(GL - G[tid]);
      gq[tid] = kScale * expf(G[tid]);
    }
    const float gL = expf(GL);
    const float* Og = s.dO + u * s.sV();
    for (int e = tid; e < kC * kNS; e += kThreads)
      Os[(e / kNS) * kUP + e % kNS] = Og[(e / kNS) * dv + slice * kNS + e % kNS];
    const float* Pg = s.Ph + u * kCC;
    for (int e = tid; e < kCC / 4; e += kThreads)
      *reinterpret_cast<float4*>(&Pt[(e >> 4) * kPP + 4 * (e & 15)]) =
          *reinterpret_cast<const float4*>(Pg + 4 * e);
    // K dS^T for rows r4 .. r4+3, column i
    float acc[kRPT];
#pragma unroll
    for (int m = 0; m < kRPT; ++m) acc[m] = 0.f;
    const float* Kg = s.K + u * s.sD();
    constexpr int kKL = kC * kKS / 4 / kThreads;     // float4 loads a thread a slab
    float4 kpre[kKL];
    auto load_k = [&](int c0) {
#pragma unroll
      for (int j = 0; j < kKL; ++j) {
        const int e = tid + j * kThreads;
        kpre[j] = *reinterpret_cast<const float4*>(Kg + (e / (kKS / 4)) * kDK + c0 + 4 * (e % (kKS / 4)));
      }
    };
    load_k(0);
    for (int c0 = 0; c0 < kDK; c0 += kKS) {
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kKL; ++j) {
        const int e = tid + j * kThreads;
        *reinterpret_cast<float4*>(&Kt[(e / (kKS / 4)) * kKSP + 4 * (e % (kKS / 4))]) = kpre[j];
      }
      __syncthreads();
      if (c0 + kKS < kDK) load_k(c0 + kKS);
#pragma unroll
      for (int cc = 0; cc < kKS; cc += 4) {
        const float4 dsv = *reinterpret_cast<const float4*>(&Ds[i * kSP + c0 + cc]);
#pragma unroll
        for (int m = 0; m < kRPT; ++m) {
          const float4 kk = *reinterpret_cast<const float4*>(&Kt[(r4 + m) * kKSP + cc]);
          acc[m] = fmaf(kk.x, dsv.x, fmaf(kk.y, dsv.y, fmaf(kk.z, dsv.z, fmaf(kk.w, dsv.w, acc[m]))));
        }
      }
    }
    if (tid == 0) {
      float t = 0.f;
      for (int w = 0; w < kThreads / 32; ++w) t += red[w];
      s.dgLp[u * (dv / kNS) + slice] = t;
    }
    // dU = Ph^T dO + diag(d) K dS^T; Ph[j][r] = 0 for j < r
    float* dUg = s.dU + u * s.sV();
    {
      float x[kRPT];
#pragma unroll
      for (int m = 0; m < kRPT; ++m) x[m] = dec[r4 + m] * acc[m];
      for (int j = r4; j < kC; ++j) {
        const float4 p = *reinterpret_cast<const float4*>(&Pt[j * kPP + r4]);
        const float o = Os[j * kUP + i];
        x[0] = fmaf(p.x, o, x[0]);
        x[1] = fmaf(p.y, o, x[1]);
        x[2] = fmaf(p.z, o, x[2]);
        x[3] = fmaf(p.w, o, x[3]);
      }
#pragma unroll
      for (int m = 0; m < kRPT; ++m) {
        Us[(r4 + m) * kUP + i] = x[m];
        dUg[(r4 + m) * dv + slice * kNS + i] = x[m];
      }
    }
    __syncthreads();
    // dS = gamma_L dS' + dO^T Qh - dU^T W, column c = tid; Q and W staged kSlabR rows at a time
    {
      const int c = tid;
      const float4* Qg = reinterpret_cast<const float4*>(s.Q + u * s.sD());
      const float4* Wg = reinterpret_cast<const float4*>(s.W + u * s.sD());
      float a2[kNS];
#pragma unroll
      for (int m = 0; m < kNS; ++m) a2[m] = 0.f;
      constexpr int kQL = kSlabR * kDK / 4 / kThreads;
      float4 qpre[kQL], wpre[kQL];
      auto load_qw = [&](int q0) {
#pragma unroll
        for (int j = 0; j < kQL; ++j) {
          qpre[j] = Qg[q0 * kDK / 4 + tid + j * kThreads];
          wpre[j] = Wg[q0 * kDK / 4 + tid + j * kThreads];
        }
      };
      load_qw(0);
      for (int q0 = 0; q0 < kC; q0 += kSlabR) {
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kQL; ++j) {
          reinterpret_cast<float4*>(Qs)[tid + j * kThreads] = qpre[j];
          reinterpret_cast<float4*>(Ws)[tid + j * kThreads] = wpre[j];
        }
        __syncthreads();
        if (q0 + kSlabR < kC) load_qw(q0 + kSlabR);
#pragma unroll 2
        for (int r = 0; r < kSlabR; ++r) {
          const float qh = gq[q0 + r] * Qs[r * kDK + c], w = Ws[r * kDK + c];
          const float4* orow = reinterpret_cast<const float4*>(&Os[(q0 + r) * kUP]);
          const float4* urow = reinterpret_cast<const float4*>(&Us[(q0 + r) * kUP]);
#pragma unroll
          for (int m4 = 0; m4 < kNS / 4; ++m4) {
            const float4 o4 = orow[m4], u4 = urow[m4];
            a2[4 * m4] = fmaf(o4.x, qh, fmaf(-u4.x, w, a2[4 * m4]));
            a2[4 * m4 + 1] = fmaf(o4.y, qh, fmaf(-u4.y, w, a2[4 * m4 + 1]));
            a2[4 * m4 + 2] = fmaf(o4.z, qh, fmaf(-u4.z, w, a2[4 * m4 + 2]));
            a2[4 * m4 + 3] = fmaf(o4.w, qh, fmaf(-u4.w, w, a2[4 * m4 + 3]));
          }
        }
      }
#pragma unroll
      for (int m = 0; m < kNS; ++m) Ds[m * kSP + c] = fmaf(gL, Ds[m * kSP + c], a2[m]);
    }
  }
  __syncthreads();
  if (dS0)
    for (int e = tid; e < kNS * kDK; e += kThreads) dS0[sbase + e] = Ds[(e / kDK) * kSP + e % kDK];
}

// ------------------------------------------------------------------ C x C terms
// Ms = M + M^T with M = dA o Gam o beta_r;  FG = s dPh o Gam;
// dGc_r = rowsum_r(X) - colsum_r(X) with X = (dA beta_r KK + s dPh QK) o Gam;
// dBc_r = sum_j dA_rj Gam_rj KK_rj.
__global__ void __launch_bounds__(kThreads) cc_kernel(Bwd s) {
  __shared__ float Mt[kC][kC + 1];
  __shared__ float Xt[kC][kC + 1];
  __shared__ float Gs[kC], Bs[kC];
  const int64_t u = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid < kC) { Gs[tid] = s.G[u * kC + tid]; Bs[tid] = s.B[u * kC + tid]; }
  __syncthreads();
  for (int e = tid; e < kCC; e += kThreads) {
    const int r = e >> 6, j = e & 63;
    const float gam = j <= r ? expf(Gs[r] - Gs[j]) : 0.f;
    const float dA = s.dA[u * kCC + e], dP = s.dPh[u * kCC + e];
    const float kk = s.KK[u * kCC + e], qk = s.QK[u * kCC + e];
    Mt[r][j] = dA * gam * Bs[r];
    Xt[r][j] = (dA * Bs[r] * kk + kScale * dP * qk) * gam;
    s.FG[u * kCC + e] = kScale * dP * gam;
  }
  __syncthreads();
  for (int e = tid; e < kCC; e += kThreads) {
    const int r = e >> 6, j = e & 63;
    s.Ms[u * kCC + e] = Mt[r][j] + Mt[j][r];
  }
  if (tid < kC) {
    const int r = tid;
    float rs = 0.f, cs = 0.f, db = 0.f;
    for (int j = 0; j < kC; ++j) {
      rs += Xt[r][j];
      cs += Xt[j][r];
    }
    for (int j = 0; j < r; ++j)   // dA is strictly lower
      db = fmaf(s.dA[u * kCC + r * kC + j] * expf(Gs[r] - Gs[j]), s.KK[u * kCC + r * kC + j], db);
    s.dGc[u * kC + r] = rs - cs;
    s.dBc[u * kC + r] = db;
  }
}

// ------------------------------------------------------------------ assemble
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}
__device__ __forceinline__ void st4_out(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4_out(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&lo);
  w.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = w;
}
template <typename T>
__global__ void __launch_bounds__(kThreads)
assemble_kernel(const float* __restrict__ alpha, const T* __restrict__ q,
                const T* __restrict__ k, const T* __restrict__ v, T* __restrict__ dq,
                T* __restrict__ dk, T* __restrict__ dv_out, float* __restrict__ dalpha,
                float* __restrict__ dbeta, SeqMap map, int32_t H, Bwd s) {
  __shared__ float dG[kC], dB[kC], dsum[kC];
  const int64_t ci = blockIdx.x;
  const int h = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int n, L;
  int64_t t0;
  if (!map.locate(ci, n, t0, L)) return;
  const int64_t u = ci * H + h;
  const int dv = s.dv;
  const float* G = s.G + u * kC;
  const float GL = G[kC - 1];
  for (int rr = 0; rr < kC / 8; ++rr) {
    const int r = warp * (kC / 8) + rr;
    const float gam = expf(G[r]), d = expf(GL - G[r]);
    const float be = s.B[u * kC + r], bg = s.BG[u * kC + r];
    float kTdW = 0.f, qdQh = 0.f, vTdU = 0.f, dd = 0.f;
    // four consecutive columns a lane: 16-byte loads, 4-element stores.  q,
    // k and v come from the caller's arrays (rows past the sequence end are
    // zero, as in the per-chunk copies the GEMMs read)
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 4 * lane; c < kDK; c += 128) {
      const size_t o = u * s.sD() + (size_t)r * kDK + c;
      const size_t g = ((t0 + r) * H + h) * kDK + c;
      const float4 tdw = ld4(s.TdW + o), dqh = ld4(s.dQh + o);
      const float4 kk = r < L ? ld4_in(k + g) : z, qq = r < L ? ld4_in(q + g) : z;
      const float4 dk1 = ld4(s.dK1 + o);
      kTdW += dot4(kk, tdw);
      qdQh += dot4(qq, dqh);
      dd += dot4(kk, dk1);   // u_r . (dS' k_r) = k_r . (U dS')_r
      if (r < L) {
        const float4 dqa = ld4(s.dQa + o), dka = ld4(s.dKa + o);
        const float sg = kScale * gam;
        st4_out(dq + g, make_float4(fmaf(sg, dqh.x, dqa.x), fmaf(sg, dqh.y, dqa.y),
                                    fmaf(sg, dqh.z, dqa.z), fmaf(sg, dqh.w, dqa.w)));
        st4_out(dk + g, make_float4(fmaf(bg, tdw.x, fmaf(d, dk1.x, dka.x)),
                                    fmaf(bg, tdw.y, fmaf(d, dk1.y, dka.y)),
                                    fmaf(bg, tdw.z, fmaf(d, dk1.z, dka.z)),
                                    fmaf(bg, tdw.w, fmaf(d, dk1.w, dka.w))));
      }
    }
    for (int c = 4 * lane; c < dv; c += 128) {
      const size_t o = u * s.sV() + (size_t)r * dv + c;
      const size_t g = ((t0 + r) * H + h) * dv + c;
      const float4 tdu = ld4(s.TdU + o);
      vTdU += dot4(r < L ? ld4_in(v + g) : z, tdu);
      if (r < L)
        st4_out(dv_out + g, make_float4(be * tdu.x, be * tdu.y, be * tdu.z, be * tdu.w));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kTdW += __shfl_xor_sync(0xffffffffu, kTdW, o);
      qdQh += __shfl_xor_sync(0xffffffffu, qdQh, o);
      vTdU += __shfl_xor_sync(0xffffffffu, vTdU, o);
      dd += __shfl_xor_sync(0xffffffffu, dd, o);
    }
    if (lane == 0) {
      const float dgam = be * kTdW + kScale * qdQh;
      dG[r] = gam * dgam + s.dGc[u * kC + r] - d * dd;
      dB[r] = gam * kTdW + vTdU + s.dBc[u * kC + r];
      dsum[r] = d * dd;
    }
  }
  __syncthreads();
  if (tid == 0) {
    float extra = 0.f;
    for (int r = 0; r < kC; ++r) extra += dsum[r];
    float dgl = 0.f;
    for (int sl = 0; sl < dv / kNS; ++sl) dgl += s.dgLp[u * (dv / kNS) + sl];
    dG[kC - 1] += extra + expf(GL) * dgl;
    float acc = 0.f;   // d log alpha_i = sum_{r >= i} dG_r
    for (int r = kC - 1; r >= 0; --r) {
      acc += dG[r];
      dG[r] = acc;
    }
  }
  __syncthreads();
  if (tid < L) {
    const int64_t g = (t0 + tid) * H + h;
    dalpha[g] = dG[tid] / alpha[g];
    dbeta[g] = dB[tid];
  }
}

// ------------------------------------------------------------------ host helpers
struct Mat {
  const float* p; size_t stride; int ld;
};

cudaError_t gemm(cudaStream_t st, bool tA, bool tB, Mat A, Mat B, float* C, size_t sC, int ldc,
                 int N, int K, float alpha, const float* Cin, float beta, int mask,
                 const float* col, size_t sCol, int64_t batch) {
  BG g{A.p, A.stride, A.ld, B.p, B.stride, B.ld, Cin, C, sC, ldc, col, sCol, N, K, alpha,
       beta, mask, batch};
  const unsigned by = (unsigned)(batch < 65535 ? batch : 65535);
  if (N % 128 == 0) {
    const dim3 grid((unsigned)(N / 128), by);
    if (!tA && !tB) bgemm_kernel<false, false, 128><<<grid, kThreads, 0, st>>>(g);
    else if (!tA && tB) bgemm_kernel<false, true, 128><<<grid, kThreads, 0, st>>>(g);
    else if (tA && !tB) bgemm_kernel<true, false, 128><<<grid, kThreads, 0, st>>>(g);
    else bgemm_kernel<true, true, 128><<<grid, kThreads, 0, st>>>(g);
  } else {
    const dim3 grid((unsigned)(N / 64), by);
    if (!tA && !tB) bgemm_kernel<false, false, 64><<<grid, kThreads, 0, st>>>(g);
    else if (!tA && tB) bgemm_kernel<false, true, 64><<<grid, kThreads, 0, st>>>(g);
    else if (tA && !tB) bgemm_kernel<true, false, 64><<<grid, kThreads, 0, st>>>(g);
    else bgemm_kernel<true, true, 64><<<grid, kThreads, 0, st>>>(g);
  }
  count_launches(1);
  return cudaGetLastError();
}

// bf16 I/O: the tensor-core GEMM where its shapes allow (dv = 256), else
// the CUDA-core one.  b_tiled > 0: B is a unit of states in the tiled
// layout, which only the tensor-core GEMM reads.
cudaError_t gemm_io(int io_dtype, unsigned* status, cudaStream_t st, bool tA, bool tB, Mat A,
                    Mat B, float* C, size_t sC, int ldc, int N, int K, float alpha,
                    const float* Cin, float beta, int mask, const float* col, size_t sCol,
                    int64_t batch, int b_tiled = 0, int b_bf16 = 0) {
  if (io_dtype == GDN_BF16 && tgemm_shape_ok(N, K, A.ld, B.ld, ldc, tA, tB, b_tiled))
    return launch_tgemm(A.p, A.stride, A.ld, B.p, B.stride, B.ld, Cin, C, sC, ldc, col, sCol, N,
                        K, alpha, beta, mask, batch, tA, tB, b_tiled, b_bf16, status, st);
  if (b_tiled) return cudaErrorInvalidValue;
  return gemm(st, tA, tB, A, B, C, sC, ldc, N, K, alpha, Cin, beta, mask, col, sCol, batch);
}

constexpr size_t kFwdSmem = sizeof(float) * (kNS * kSP + kC * kWS + kC * kUP + kSlabF * kDK + kC);
constexpr size_t kRevSmem = sizeof(float) * (kNS * kSP + kC * kKSP + 2 * kC * kUP +
                                             2 * kSlabR * kDK + kC * kPP + 2 * kC + 8);
static_assert(kSP % 4 == 0 && kWS % 4 == 0 && kKSP % 4 == 0 && kUP % 4 == 0 && kPP % 4 == 0,
              "16-byte rows");
static_assert((kNS * kSP + kC * kWS + kC * kUP) % 4 == 0, "16-byte aligned slab");
static_assert((kNS * kSP + kC * kKSP + 2 * kC * kUP) % 4 == 0, "16-byte aligned slabs");
static_assert(kRPT == 4 && kNS % 4 == 0, "thread mapping of the state passes");
static_assert(kC * 16 % kThreads == 0 && kSlabF * kDK / 4 % kThreads == 0 &&
              kC * kKS / 4 % kThreads == 0 && kSlabR * kDK / 4 % kThreads == 0,
              "whole float4 loads a thread for every staged slab");
static_assert(3 * (kFwdSmem + 1024) <= 228 * 1024 && 3 * (kRevSmem + 1024) <= 228 * 1024,
              "three state-pass CTAs a SM");

}  // namespace

size_t prefill_backward_scratch_bytes(int64_t max_chunks, int32_t H, int32_t dv, int64_t T_total,
                                      int io_dtype) {
  size_t b = align_up(bwd_scratch_bytes(max_chunks * H, dv), 1024);
  (void)T_total;
  if (io_dtype == GDN_BF16) b += align_up(prefill_tc_scratch_bytes(max_chunks, H, dv), 1024);
  return b;
}

// A stream of the greatest priority per device for the reverse state pass,
// created on first use (nullptr if that fails: the call then stays on the
// caller's stream).  Its 48-odd CTAs each take a whole SM; the priority puts
// them on their SMs before the concurrent chunk-gradient work fills the rest.
cudaStream_t reverse_stream() {
  static cudaStream_t streams[64] = {};
  static bool tried[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!tried[dev]) {
    tried[dev] = true;
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&streams[dev], cudaStreamNonBlocking, greatest) !=
            cudaSuccess) {
      streams[dev] = nullptr;
      (void)cudaGetLastError();
    }
  }
  return streams[dev];
}

cudaError_t launch_prefill_backward(const PrefillLaunch& a, const void* dout,
                                    const float* dS_final, void* dq, void* dk, void* dv_out,
                                    float* dalpha, float* dbeta, float* dS0, int io_dtype,
                                    cudaStream_t st) {
  const int64_t units = a.max_chunks * a.H;
  const int dv = a.dv;
  Bwd s = carve(a.scratch, units, dv);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(fwd_states_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kFwdSmem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(rev_states_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kRevSmem)) != cudaSuccess)
    return e;
  const dim3 gu((unsigned)a.max_chunks, (unsigned)a.H);
  const dim3 gs((unsigned)a.map.N, (unsigned)a.H, (unsigned)(dv / kNS));
  const size_t D = s.sD(), V = s.sV(), S = s.sS(), CC = kCC;
  struct G {
    bool tA, tB; Mat A, B; float* C; size_t sC; int ldc, N, K; float alpha;
    const float* Cin; float beta; int mask; const float* col;
  };
  // bf16 I/O at dv = 256: the forward re-run and the reverse pass leave the
  // chunk states and dS' in the tiled layout
  const bool tiled = io_dtype == GDN_BF16 && tiled_states(dv);
  auto run = [&](const G* list, int n, cudaStream_t q) -> cudaError_t {
    for (int i = 0; i < n; ++i) {
      const G& g = list[i];
      const int bt = tiled && (g.B.p == s.Sst || g.B.p == s.dSp) ? dv : 0;
      const int bbf = bt ? 1 : 0;   // the states and dS' are bf16 there
      const cudaError_t r = gemm_io(io_dtype, a.status, q, g.tA, g.tB, g.A, g.B, g.C, g.sC, g.ldc,
                                    g.N, g.K, g.alpha, g.Cin, g.beta, g.mask, g.col, kC, units, bt,
                                    bbf);
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  };
  // the per-chunk factors: q, k, v, dO tiles, KK^T, QK^T, T, P^, W, U~
  // (bf16 I/O) the forward re-run's per-chunk kernel leaves K K^T, Q K^T,
  // P^, T and its scaled forms in fp32 (PrepSide): the per-chunk factors are
  // then the gather and, once that kernel is done (wait_prep), the W and U~
  // products
  const bool side = io_dtype == GDN_BF16;
  auto local_factors = [&](cudaStream_t q,
                           const std::function<cudaError_t()>& wait_prep) -> cudaError_t {
    if (io_dtype == GDN_BF16)
      gather_kernel<__nv_bfloat16><<<gu, kThreads, 0, q>>>(
          (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v,
          (const __nv_bfloat16*)dout, a.alpha, a.beta, a.map, a.H, s);
    else
      gather_kernel<float><<<gu, kThreads, 0, q>>>((const float*)a.q, (const float*)a.k,
                                                    (const float*)a.v, (const float*)dout,
                                                    a.alpha, a.beta, a.map, a.H, s);
    count_launches(1);
    cudaError_t r = cudaGetLastError();
    if (r != cudaSuccess) return r;
    if (side) {
      if ((r = wait_prep()) != cudaSuccess) return r;
    } else {
      const G f1[] = {
          {false, true, {s.K, D, kDK}, {s.K, D, kDK}, s.KK, CC, kC, kC, kDK, 1.f, nullptr, 0.f, 0, nullptr},
          {false, true, {s.Q, D, kDK}, {s.K, D, kDK}, s.QK, CC, kC, kC, kDK, 1.f, nullptr, 0.f, 0, nullptr},
      };
      if ((r = run(f1, 2, q)) != cudaSuccess) return r;
      tprep_kernel<<<(unsigned)units, kThreads, 0, q>>>(s);
      count_launches(1);
      if ((r = cudaGetLastError()) != cudaSuccess) return r;
    }
    // W = T diag(beta gamma) K, U~ = T diag(beta) V
    const G f2[] = {
        {false, false, {s.TmB, CC, kC}, {s.K, D, kDK}, s.W, D, kDK, kDK, kC, 1.f, nullptr, 0.f, 0, nullptr},
        {false, false, {s.TmU, CC, kC}, {s.V, V, dv}, s.Ut, V, dv, dv, kC, 1.f, nullptr, 0.f, 0, nullptr},
    };
    return run(f2, 2, q);
  };
  // the chunk products that need no reverse-pass output ...
  const G pre[] = {
      // U = U~ - W S^T
      {false, true, {s.W, D, kDK}, {s.Sst, S, kDK}, s.U, V, dv, dv, kDK, -1.f, s.Ut, 1.f, 0, nullptr},
      // dQh = dO S ; dPh = lower(dO U^T)
      {false, false, {s.dO, V, dv}, {s.Sst, S, kDK}, s.dQh, D, kDK, kDK, dv, 1.f, nullptr, 0.f, 0, nullptr},
      {false, true, {s.dO, V, dv}, {s.U, V, dv}, s.dPh, CC, kC, kC, dv, 1.f, nullptr, 0.f, 1, nullptr},
  };
  // ... and those that do
  const G post[] = {
      // dW = -dU S ; dK1 = U dS' (its rows dotted with k_r also give
      // dd_r = u_r . (dS' k_r) in assemble)
      {false, false, {s.dU, V, dv}, {s.Sst, S, kDK}, s.dW, D, kDK, kDK, dv, -1.f, nullptr, 0.f, 0, nullptr},
      {false, false, {s.U, V, dv}, {s.dSp, S, kDK}, s.dK1, D, kDK, kDK, dv, 1.f, nullptr, 0.f, 0, nullptr},
      // dT = (dW K^T) diag(beta gamma) + (dU V^T) diag(beta)
      {false, true, {s.dW, D, kDK}, {s.K, D, kDK}, s.dTm, CC, kC, kC, kDK, 1.f, nullptr, 0.f, 0, s.BG},
      {false, true, {s.dU, V, dv}, {s.V, V, dv}, s.dTm, CC, kC, kC, dv, 1.f, s.dTm, 1.f, 0, s.B},
      // T^T dW, T^T dU, dA = -(T^T dT) T^T strictly lower
      {true, false, {s.Tm, CC, kC}, {s.dW, D, kDK}, s.TdW, D, kDK, kDK, kC, 1.f, nullptr, 0.f, 0, nullptr},
      {true, false, {s.Tm, CC, kC}, {s.dU, V, dv}, s.TdU, V, dv, dv, kC, 1.f, nullptr, 0.f, 0, nullptr},
      {true, false, {s.Tm, CC, kC}, {s.dTm, CC, kC}, s.X, CC, kC, kC, kC, 1.f, nullptr, 0.f, 0, nullptr},
      {false, true, {s.X, CC, kC}, {s.Tm, CC, kC}, s.dA, CC, kC, kC, kC, -1.f, nullptr, 0.f, 2, nullptr},
  };
  constexpr int kPre = sizeof pre / sizeof pre[0], kPost = sizeof post / sizeof post[0];

  if (io_dtype == GDN_BF16) {
    // chunk-start states from the tensor-core forward (bf16 operands, fp32
    // state), without outputs: its state units then load W alone (no Q^ or
    // P^) and skip the output products
    char* extra = (char*)a.scratch + align_up(bwd_scratch_bytes(units, dv), 1024);
    PrefillLaunch f = a;
    f.scratch = extra;
    f.out = nullptr;
    f.S_final = nullptr;
    // the split form: its per-chunk kernel takes every SM briefly, then its
    // state units hold one SM each and the caller's stream gets the rest (the
    // fused cooperative form would hold every SM until its workers finish)
    f.allow_overlap = false;
    f.state_dump = s.Sst;
    f.side = PrepSide{s.KK, s.QK, s.Ph, s.Tm, s.TmB, s.TmU};
    PrefillLaunch f_state = f;   // the re-run's state pass, after its per-chunk kernel
    f_state.state_only = true;
    // the forward re-run and then the reverse pass on the tensor cores (on
    // the re-run's operand images) go to the high-priority stream; on the
    // caller's stream meanwhile, the per-chunk factors take the SMs the
    // re-run's state units leave, then (after the re-run) the products that
    // need no reverse output take those the reverse pass leaves free
    ReverseLaunch r;
    r.k = a.k;
    r.dout = dout;
    r.map = a.map;
    r.H = a.H;
    r.dv = dv;
    r.T_total = a.map.cu_seqlens ? a.map.T : (int64_t)a.map.N * a.map.T;
    r.images = (const uint8_t*)extra;
    r.dS_final = dS_final;
    r.dS0 = dS0;
    r.dSp = s.dSp;
    r.dU = s.dU;
    r.status = a.status;
    cudaStream_t rs = units > 0 ? reverse_stream() : nullptr;
    // inputs ready, re-run's per-chunk kernel done, re-run done, reverse done
    cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
    for (int i = 0; rs && i < 4; ++i) {
      if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
        for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
        rs = nullptr;
        (void)cudaGetLastError();
      }
    }
    if (!rs) {   // one stream, in dependency order
      if ((e = launch_prefill_tc(f, st)) != cudaSuccess) return e;
      if ((e = launch_reverse_tc(r, st)) != cudaSuccess) return e;
      if (units == 0) return cudaSuccess;
      if ((e = local_factors(st, [] { return cudaSuccess; })) != cudaSuccess) return e;
      if ((e = run(pre, kPre, st)) != cudaSuccess) return e;
    } else {
      e = cudaEventRecord(ev[0], st);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(rs, ev[0], 0);
      if (e == cudaSuccess) e = launch_prefill_tc(f, rs, /*prep_only=*/true);
      if (e == cudaSuccess) e = cudaEventRecord(ev[1], rs);
      if (e == cudaSuccess) e = launch_prefill_tc(f_state, rs);
      if (e == cudaSuccess) e = cudaEventRecord(ev[2], rs);
      if (e == cudaSuccess) e = launch_reverse_tc(r, rs);
      if (e == cudaSuccess) e = cudaEventRecord(ev[3], rs);
      if (e == cudaSuccess)
        e = local_factors(st, [&] { return cudaStreamWaitEvent(st, ev[1], 0); });
      if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev[2], 0);
      if (e == cudaSuccess) e = run(pre, kPre, st);
      // join (also on an error above, so that nothing of this call is left
      // running on the internal stream unordered with the caller's)
      const cudaError_t ew = cudaStreamWaitEvent(st, ev[3], 0);
      for (int i = 0; i < 4; ++i) cudaEventDestroy(ev[i]);
      if (e == cudaSuccess) e = ew;
      if (e != cudaSuccess) return e;
    }
    // <dS', S_start> partials
    if (tiled)
      dgl_kernel<true><<<dim3((unsigned)units, (unsigned)(dv / kNS)), kThreads, 0, st>>>(s);
    else
      dgl_kernel<false><<<dim3((unsigned)units, (unsigned)(dv / kNS)), kThreads, 0, st>>>(s);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  } else {
    if (units > 0 && (e = local_factors(st, [] { return cudaSuccess; })) != cudaSuccess) return e;
    fwd_states_kernel<<<gs, kThreads, kFwdSmem, st>>>(a.S0, a.map, a.H, s);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    rev_states_kernel<<<gs, kThreads, kRevSmem, st>>>(dS_final, dS0, a.map, a.H, s);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (units == 0) return cudaSuccess;
    if ((e = run(pre, kPre, st)) != cudaSuccess) return e;
  }
  if ((e = run(post, kPost, st)) != cudaSuccess) return e;
  cc_kernel<<<(unsigned)units, kThreads, 0, st>>>(s);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const G list2[] = {
      // dK: (M + M^T) K + FG^T Q ; dQ: FG K
      {false, false, {s.Ms, CC, kC}, {s.K, D, kDK}, s.dKa, D, kDK, kDK, kC, 1.f, nullptr, 0.f, 0, nullptr},
      {true, false, {s.FG, CC, kC}, {s.Q, D, kDK}, s.dKa, D, kDK, kDK, kC, 1.f, s.dKa, 1.f, 0, nullptr},
      {false, false, {s.FG, CC, kC}, {s.K, D, kDK}, s.dQa, D, kDK, kDK, kC, 1.f, nullptr, 0.f, 0, nullptr},
  };
  if ((e = run(list2, 3, st)) != cudaSuccess) return e;
  if (io_dtype == GDN_BF16)
    assemble_kernel<__nv_bfloat16><<<gu, kThreads, 0, st>>>(
        a.alpha, (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v,
        (__nv_bfloat16*)dq, (__nv_bfloat16*)dk, (__nv_bfloat16*)dv_out, dalpha, dbeta, a.map, a.H,
        s);
  else
    assemble_kernel<float><<<gu, kThreads, 0, st>>>(
        a.alpha, (const float*)a.q, (const float*)a.k, (const float*)a.v, (float*)dq, (float*)dk,
        (float*)dv_out, dalpha, dbeta, a.map, a.H, s);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace gdn
