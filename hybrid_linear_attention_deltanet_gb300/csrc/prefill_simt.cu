// Chunkwise-parallel prefill on the CUDA cores (fp32 FFMA throughout).
//
// This is the fp32-I/O path: tf32/bf16 tensor-core operands cannot hold a
// 1e-4 relative error, so every product here is an fp32 FFMA.
//
// Chunked form of the gated delta rule (Appendix A.3 of "Long-Context Aware
// Upcycling": chunks of C = 64 tokens, delta corrections inside a chunk
// batched through the WY representation, state carried across chunks
// sequentially).  For a chunk with start state S (dv x dk), rows r, j < L,
// G = cumsum(log alpha), gamma = exp(G), Gam_rj = exp(G_r - G_j):
//   A  = strict_lower(beta_r Gam_rj k_r.k_j),     T = (I + A)^{-1}
//   W  = T diag(beta gamma) K                     (C x dk)
//   U~ = T diag(beta) V                           (C x dv)
//   P  = lower(Gam_rj q_r.k_j) / sqrt(dk)         (C x C, diagonal included)
//   U  = U~ - W S^T
//   O  = diag(gamma) Q S^T / sqrt(dk) + P U
//   S' = gamma_L S + U^T diag(gamma_L / gamma) K
// Decay only ever appears as exp of a non-positive log difference, so
// nothing overflows however small the cumulative decay gets.
//
// Kernel 1 (chunk_prep): one CTA per (chunk, head), fully parallel; writes
//   W, U~, P and G for the chunk to scratch.
// Kernel 2 (state_pass): one CTA per (sequence, head, 32-row slice of S);
//   rows of S are independent (every row of U, O and S' depends only on the
//   same row of S), so the d_v axis splits with no communication.  It walks
//   the sequence's chunks in order, carrying its S slice in shared memory.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kPad = kDK + 1;    // row stride of 64 x 256 fp32 tiles (bank-conflict padding)
constexpr int kCP = kC + 1;      // row stride of 64 x 64 tiles
constexpr int kNS = 32;          // rows of S per state-pass CTA

// scratch per (chunk, head): W [C][dk], U~ [C][dv], P [C][C], G [C]
struct SimtScratch {
  float* W; float* Ut; float* P; float* G;
  int32_t dv;
  __host__ __device__ static size_t stride_W() { return (size_t)kC * kDK; }
  __host__ __device__ size_t stride_U() const { return (size_t)kC * dv; }
  __host__ __device__ static size_t stride_P() { return (size_t)kC * kC; }
  __host__ __device__ static size_t stride_G() { return (size_t)kC; }
};

inline SimtScratch carve(void* base, int64_t max_chunks, int32_t H, int32_t dv) {
  const size_t units = (size_t)max_chunks * H;
  char* p = (char*)base;
  SimtScratch s;
  s.dv = dv;
  s.W = (float*)p;  p += align_up(units * SimtScratch::stride_W() * 4, 256);
  s.Ut = (float*)p; p += align_up(units * s.stride_U() * 4, 256);
  s.P = (float*)p;  p += align_up(units * SimtScratch::stride_P() * 4, 256);
  s.G = (float*)p;
  return s;
}

// --------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads)
chunk_prep_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                  const float* __restrict__ alpha, const float* __restrict__ beta,
                  SeqMap map, int32_t H, SimtScratch scr) {
  extern __shared__ float smem[];
  float* Ks = smem;                 // [C][kPad]
  float* QVs = Ks + kC * kPad;      // [C][kPad]  Q for the Gram, then V
  float* As = QVs + kC * kPad;      // [C][kCP]
  float* Ts = As + kC * kCP;        // [C][kCP]
  float* Gs = Ts + kC * kCP;        // [C]
  float* bs = Gs + kC;              // [C]  beta (0 on pad rows)
  float* bgs = bs + kC;             // [C]  beta * gamma

  const int64_t ci = blockIdx.x;
  const int h = blockIdx.y;
  int n, L;
  int64_t t0;
  if (!map.locate(ci, n, t0, L)) return;
  const int tid = threadIdx.x;

  // decay prefix in log space: pad rows get log alpha = 0 and beta = 0, so
  // they neither decay the chunk nor write anything
  if (tid < kC) {
    const bool ok = tid < L;
    Gs[tid] = ok ? logf(alpha[(t0 + tid) * H + h]) : 0.f;
    bs[tid] = ok ? beta[(t0 + tid) * H + h] : 0.f;
  }
  // K, Q rows (pad rows zero)
  for (int e = tid; e < kC * kDK; e += kThreads) {
    const int r = e / kDK, c = e % kDK;
    const int64_t g = ((t0 + r) * H + h) * kDK + c;
    Ks[r * kPad + c] = r < L ? ld_in(k + g) : 0.f;
    QVs[r * kPad + c] = r < L ? ld_in(q + g) : 0.f;
  }
  __syncthreads();
  if (tid == 0) {
    float acc = 0.f;
    for (int r = 0; r < kC; ++r) { acc += Gs[r]; Gs[r] = acc; }
  }
  __syncthreads();
  if (tid < kC) bgs[tid] = bs[tid] * expf(Gs[tid]);

  // Gram products: thread -> row r = tid/4, columns j = tid%4 + 4m
  {
    const int r = tid >> 2, j0 = tid & 3;
    float kk[16], qk[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) { kk[m] = 0.f; qk[m] = 0.f; }
    for (int c = 0; c < kDK; ++c) {
      const float kr = Ks[r * kPad + c], qr = QVs[r * kPad + c];
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float kj = Ks[(j0 + 4 * m) * kPad + c];
        kk[m] = fmaf(kr, kj, kk[m]);
        qk[m] = fmaf(qr, kj, qk[m]);
      }
    }
    const float Gr = Gs[r], br = bs[r];
    float* Pg = scr.P + (size_t)(ci * H + h) * SimtScratch::stride_P();
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const int j = j0 + 4 * m;
      const float gam = j <= r ? expf(Gr - Gs[j]) : 0.f;
      As[r * kCP + j] = j < r ? br * gam * kk[m] : 0.f;
      Pg[r * kC + j] = j <= r ? kScale * gam * qk[m] : 0.f;
    }
  }
  __syncthreads();

  // V block 0 (columns 0 .. 255) replaces Q
  const int dv = scr.dv;
  auto load_v = [&](int vb) {
    for (int e = tid; e < kC * kDK; e += kThreads) {
      const int r = e / kDK, c = e % kDK;
      QVs[r * kPad + c] = r < L ? ld_in(v + ((t0 + r) * H + h) * dv + kDK * vb + c) : 0.f;
    }
  };
  load_v(0);
  // T = (I + A)^{-1} by forward substitution, one column per thread
  if (tid < kC) {
    const int c = tid;
    for (int r = 0; r < kC; ++r) Ts[r * kCP + c] = r == c ? 1.f : 0.f;
    for (int r = 1; r < kC; ++r) {
      float a0 = 0.f, a1 = 0.f;
      int j = 0;
      for (; j + 1 < r; j += 2) {
        a0 = fmaf(As[r * kCP + j], Ts[j * kCP + c], a0);
        a1 = fmaf(As[r * kCP + j + 1], Ts[(j + 1) * kCP + c], a1);
      }
      if (j < r) a0 = fmaf(As[r * kCP + j], Ts[j * kCP + c], a0);
      if (r > c) Ts[r * kCP + c] = -(a0 + a1);
    }
  }
  __syncthreads();

  // W = T diag(beta gamma) K ; U~ = T diag(beta) V ; one output column per
  // thread, V in blocks of 256 columns
  {
    const int c = tid;
    float* Wg = scr.W + (size_t)(ci * H + h) * SimtScratch::stride_W();
    float* Ug = scr.Ut + (size_t)(ci * H + h) * scr.stride_U();
    for (int r = 0; r < kC; ++r) {
      float w = 0.f, u = 0.f;
      for (int j = 0; j <= r; ++j) {
        const float t = Ts[r * kCP + j];
        w = fmaf(t * bgs[j], Ks[j * kPad + c], w);
        u = fmaf(t * bs[j], QVs[j * kPad + c], u);
      }
      Wg[r * kDK + c] = w;
      Ug[r * dv + c] = u;
    }
    for (int vb = 1; vb * kDK < dv; ++vb) {
      __syncthreads();
      load_v(vb);
      __syncthreads();
      for (int r = 0; r < kC; ++r) {
        float u = 0.f;
        for (int j = 0; j <= r; ++j) u = fmaf(Ts[r * kCP + j] * bs[j], QVs[j * kPad + c], u);
        Ug[r * dv + kDK * vb + c] = u;
      }
    }
  }
  if (tid < kC) scr.G[(size_t)(ci * H + h) * SimtScratch::stride_G() + tid] = Gs[tid];
}

// --------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads)
state_pass_kernel(const T* __restrict__ q, const T* __restrict__ k,
                  const float* __restrict__ S0, T* __restrict__ out,
                  float* __restrict__ S_final, SeqMap map, int32_t H, SimtScratch scr,
                  SegRoute route) {
  extern __shared__ float smem[];
  float* Ss = smem;                  // [kNS][kPad]  this CTA's rows of S
  float* Wt = Ss + kNS * kPad;       // [C][33]
  float* Qt = Wt + kC * 33;          // [C][33]
  float* Us = Qt + kC * 33;          // [C][33]
  float* gam = Us + kC * 33;         // [C]  gamma_r * scale
  float* dec = gam + kC;             // [C]  gamma_L / gamma_r (0 on pad rows)

  const int x = blockIdx.x, h = blockIdx.y, slice = blockIdx.z;
  const int n = x >= map.N ? x - map.N : x;
  const int tid = threadIdx.x, i = tid & 31, rg = tid >> 5;
  const int dv = scr.dv;
  const UnitRoute ur = route_unit(route, S0, S_final, x, map.N, (int64_t)H * dv * kDK);
  // an A chain (identity start, no U~) has dk rows
  if (!ur.run || (ur.ident && slice * kNS >= kDK)) return;
  // this CTA's rows of the unit's [H][dv][dk] start and end blocks
  const int64_t state_base = (int64_t)h * dv * kDK + (int64_t)slice * kNS * kDK;

  for (int e = tid; e < kNS * kDK; e += kThreads) {
    const int r = e / kDK, c = e % kDK;
    Ss[r * kPad + c] = ur.S0      ? ur.S0[state_base + e]
                       : ur.ident ? (slice * kNS + r == c ? 1.f : 0.f)
                                  : 0.f;
  }
  __syncthreads();

  const int64_t cb = map.chunk_begin(n), ce = map.chunk_end(n);
  const int64_t s_begin = map.seq_begin(n), s_end = map.seq_end(n);
  for (int64_t ci = cb; ci < ce; ++ci) {
    const int64_t t0 = s_begin + (ci - cb) * kC;
    const int L = (int)min((int64_t)kC, s_end - t0);
    const size_t u = (size_t)(ci * H + h);
    const float* G = scr.G + u * SimtScratch::stride_G();
    __syncthreads();   // the previous chunk's phases 2-3 are done with gam / dec / Us
    if (tid < kC) {
      const float GL = G[L - 1];
      gam[tid] = tid < L ? expf(G[tid]) * kScale : 0.f;
      dec[tid] = tid < L ? expf(GL - G[tid]) : 0.f;
    }
    const float gL = expf(G[L - 1]);

    // phase 1: U = U~ - W S^T and Q S^T for rows r = rg*8 .. rg*8+7, column i
    float accU[8], accQ[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) { accU[m] = 0.f; accQ[m] = 0.f; }
    const float* Wg = scr.W + u * SimtScratch::stride_W();
    for (int c0 = 0; c0 < kDK; c0 += 32) {
      __syncthreads();
      for (int e = tid; e < kC * 32; e += kThreads) {
        const int r = e >> 5, cc = e & 31;
        Wt[r * 33 + cc] = Wg[r * kDK + c0 + cc];
        Qt[r * 33 + cc] = r < L ? ld_in(q + ((t0 + r) * H + h) * kDK + c0 + cc) : 0.f;
      }
      __syncthreads();
#pragma unroll 4
      for (int cc = 0; cc < 32; ++cc) {
        const float sv = Ss[i * kPad + c0 + cc];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          accU[m] = fmaf(Wt[(rg * 8 + m) * 33 + cc], sv, accU[m]);
          accQ[m] = fmaf(Qt[(rg * 8 + m) * 33 + cc], sv, accQ[m]);
        }
      }
    }
    const float* Ug = scr.Ut + u * scr.stride_U();
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int r = rg * 8 + m;
      // an A chain drops U~ (the homogeneous part of the recurrence)
      Us[r * 33 + i] = (ur.ident ? 0.f : Ug[r * dv + slice * kNS + i]) - accU[m];
    }
    __syncthreads();

    // phase 2: O = gamma Q S^T / sqrt(dk) + P U
    const float* Pg = scr.P + u * SimtScratch::stride_P();
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (!ur.write_out) break;
      const int r = rg * 8 + m;
      if (r < L) {
        float o = gam[r] * accQ[m];
        for (int j = 0; j <= r; ++j) o = fmaf(Pg[r * kC + j], Us[j * 33 + i], o);
        st_out(out + ((t0 + r) * H + h) * dv + slice * kNS + i, o);
      }
    }

    // phase 3: S' = gamma_L S + U^T diag(gamma_L / gamma) K, column c = tid
    {
      const int c = tid;
      float acc[kNS];
#pragma unroll
      for (int m = 0; m < kNS; ++m) acc[m] = 0.f;
      for (int r = 0; r < L; ++r) {
        const float kd = dec[r] * ld_in(k + ((t0 + r) * H + h) * kDK + c);
#pragma unroll
        for (int m = 0; m < kNS; ++m) acc[m] = fmaf(Us[r * 33 + m], kd, acc[m]);
      }
#pragma unroll
      for (int m = 0; m < kNS; ++m) Ss[m * kPad + c] = fmaf(gL, Ss[m * kPad + c], acc[m]);
    }
  }
  __syncthreads();
  if (ur.S_final)
    for (int e = tid; e < kNS * kDK; e += kThreads)
      ur.S_final[state_base + e] = Ss[(e / kDK) * kPad + (e % kDK)];
}

constexpr size_t kPrepSmem = sizeof(float) * (2 * kC * kPad + 2 * kC * kCP + 3 * kC);
constexpr size_t kStateSmem = sizeof(float) * (kNS * kPad + 3 * kC * 33 + 2 * kC);

template <typename T>
cudaError_t launch_typed(const PrefillLaunch& a, cudaStream_t stream) {
  SimtScratch scr = carve(a.scratch, a.max_chunks, a.H, a.dv);
  cudaError_t e;
  e = cudaFuncSetAttribute(chunk_prep_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kPrepSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(state_pass_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kStateSmem);
  if (e != cudaSuccess) return e;
  if (a.max_chunks > 0 && !a.state_only) {
    dim3 g1((unsigned)a.max_chunks, (unsigned)a.H);
    chunk_prep_kernel<T><<<g1, kThreads, kPrepSmem, stream>>>(
        (const T*)a.q, (const T*)a.k, (const T*)a.v, a.alpha, a.beta, a.map, a.H, scr);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  dim3 g2((unsigned)a.map.N * (a.route.pass == 1 ? 2u : 1u), (unsigned)a.H,
          (unsigned)(a.dv / kNS));
  state_pass_kernel<T><<<g2, kThreads, kStateSmem, stream>>>(
      (const T*)a.q, (const T*)a.k, a.S0, (T*)a.out, a.S_final, a.map, a.H, scr, a.route);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_simt_scratch_bytes(int64_t max_chunks, int32_t H, int32_t dv) {
  const size_t units = (size_t)max_chunks * H;
  return align_up(units * SimtScratch::stride_W() * 4, 256) +
         align_up(units * (size_t)kC * dv * 4, 256) +
         align_up(units * SimtScratch::stride_P() * 4, 256) +
         align_up(units * SimtScratch::stride_G() * 4, 256);
}

cudaError_t launch_prefill_simt(const PrefillLaunch& a, int io_dtype, cudaStream_t stream) {
  if (io_dtype == GDN_BF16) return launch_typed<__nv_bfloat16>(a, stream);
  return launch_typed<float>(a, stream);
}

}  // namespace gdn
