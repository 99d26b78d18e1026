// One decode step of the whole Gated DeltaNet mixer core in a single launch:
// the pre-recurrence steps (short convolution + SiLU on q, k, v, q/k L2
// normalisation, decay and write strength), the gated delta rule update of
// the cached state, and Eq. 20's gated RMSNorm of the read-out ("Long-Context
// Aware Upcycling", Appendix A.3: the paragraph after Table 8, the text under
// Eq. 16-21, Eq. 16-20).  The projections stay outside.
//
// Two launches and no synchronisation between CTAs.  The first has the plain
// decode step's shape (dv / 64 CTAs of 256 threads per (sequence, head), each
// warp streaming 8 rows of the fp32 state through HBM once, the first rows
// already in flight while the pre-recurrence steps run); its pre-recurrence
// work is spread over all of its threads so the one CTA barrier is short, and
// q and k reach the dot products straight from shared memory.  It writes the
// read-outs to a small fp32 buffer.  The second applies Eq. 20 per (sequence,
// head) and shifts the q / k convolution history in place, which is safe
// because every read of that history belongs to the first.
#include "gdn_internal.cuh"

namespace gdn {

// stream-ordered scratch from the library's per-device pool (api.cu)
cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t stream);
cudaError_t scratch_free(void* p, cudaStream_t stream);

namespace {

constexpr int kRows = 64;                  // state rows per CTA (the plain decode's split)
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = kRows / kWarps;
constexpr int kBatch = 4;                  // rows a warp works on together
constexpr int kTaps = 4;
constexpr float kL2Eps = 1e-6f;

struct LayerArgs {
  const void* qkv;        // [N, C] io dtype, C = H (2 dk + dv)
  const float* conv_w;    // [C, 4]
  const float* a_raw;     // [N, H]
  const float* b_raw;     // [N, H]
  const float* A_log;     // [H]
  const float* dt_bias;   // [H]
  void* conv_state;       // [N, 3, C] io dtype, in place
  float* S;               // [N, H, dv, dk] fp32, in place
  const void* gate;       // [N, H, dv] io dtype (W_G x)
  const float* norm_w;    // [dv]
  float eps;
  void* y;                // [N, H, dv] io dtype
  int32_t H, dv;
  float* o_buf;           // [N, H, dv] scratch: read-outs before the norm
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// the stream's activations use the fast exponential and divide (a few ulp)
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// conv + SiLU of channel c of one token from its 3-token history
template <typename T>
__device__ __forceinline__ float conv1(const T* x, const T* st, int64_t C, int64_t c,
                                       const float* __restrict__ conv_w, float& h1, float& h2,
                                       float& xc) {
  const float4 w = __ldg(reinterpret_cast<const float4*>(conv_w + c * kTaps));
  const float h0 = ld_in(st + c);
  h1 = ld_in(st + C + c);
  h2 = ld_in(st + 2 * C + c);
  xc = ld_in(x + c);
  return silu_fast(fmaf(w.w, xc, fmaf(w.z, h2, fmaf(w.y, h1, w.x * h0))));
}

// Launch 1: pre-recurrence steps and the state update, in the plain decode
// step's shape.  The pre-recurrence work is spread over every thread (q and k
// of the head: 2 channels a thread; this CTA's 64 v channels: 1 for the first
// 64 threads, which also shift that channel's history in place; the gates: one
// thread), so the single CTA barrier that follows is short.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32, 3) decode_layer_kernel(LayerArgs a) {
  const int ranks = a.dv / kRows;
  const int rank = (int)(blockIdx.x % ranks);
  const int64_t unit = blockIdx.x / ranks;          // n * H + h
  const int64_t n = unit / a.H;
  const int h = (int)(unit % a.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t C = (int64_t)a.H * (2 * kDK + a.dv);
  const T* x = static_cast<const T*>(a.qkv) + n * C;
  T* st = static_cast<T*>(a.conv_state) + n * 3 * C;
  const int row0 = rank * kRows + warp * kRowsPerWarp;
  float* Srow0 = a.S + (unit * a.dv + row0) * kDK;
  __shared__ __align__(16) float qk[2 * kDK];      // q then k, before the norm
  __shared__ float vs[kRows];
  __shared__ float part[kWarps];
  __shared__ float ab[2];

  // the first rows of state are in flight while the pre-recurrence steps run
  float4 s[kBatch][2];
#pragma unroll
  for (int r = 0; r < kBatch; ++r) {
    const float4* rowp = reinterpret_cast<const float4*>(Srow0 + r * kDK);
    s[r][0] = __ldcs(rowp + lane);
    s[r][1] = __ldcs(rowp + 32 + lane);
  }
  {
    // threads 0..127: q channels 2t, 2t+1; threads 128..255: k channels
    const int e = 2 * tid;                             // 0 .. 511 over q | k
    const int64_t base = e < kDK ? (int64_t)h * kDK : (int64_t)a.H * kDK + (int64_t)h * kDK - kDK;
    float h1, h2, xc, ss = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float y = conv1<T>(x, st, C, base + e + i, a.conv_w, h1, h2, xc);
      qk[e + i] = y;
      ss = fmaf(y, y, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) part[warp] = ss;                  // warps 0-3: q, 4-7: k
    if (tid < kRows) {
      const int64_t c = 2 * (int64_t)a.H * kDK + (int64_t)h * a.dv + rank * kRows + tid;
      vs[tid] = conv1<T>(x, st, C, c, a.conv_w, h1, h2, xc);
      st_out(st + c, h1);
      st_out(st + C + c, h2);
      st_out(st + 2 * C + c, xc);
    } else if (tid == kRows) {
      const float z = a.a_raw[unit] + a.dt_bias[h];
      ab[0] = expf(-expf(a.A_log[h]) * (z > 20.f ? z : log1pf(expf(z))));
      ab[1] = 1.f / (1.f + expf(-a.b_raw[unit]));
    }
  }
  __syncthreads();
  const float rqn = rsqrtf(part[0] + part[1] + part[2] + part[3] + kL2Eps);
  const float rkn = rsqrtf(part[4] + part[5] + part[6] + part[7] + kL2Eps);
  float kr[8], qr[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    qr[j] = qk[4 * lane + j] * rqn;
    qr[4 + j] = qk[128 + 4 * lane + j] * rqn;
    kr[j] = qk[kDK + 4 * lane + j] * rkn;
    kr[4 + j] = qk[kDK + 128 + 4 * lane + j] * rkn;
  }
  const float al = ab[0], be = ab[1];
  const float vj = lane < kRowsPerWarp ? vs[warp * kRowsPerWarp + lane] : 0.f;

  // ---- the gated delta rule on this warp's rows (Eq. 16-19)
  float kq = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) kq = fmaf(kr[j], qr[j], kq);
  kq = warp_sum(kq);
  float o_mine = 0.f;
#pragma unroll
  for (int rb = 0; rb < kRowsPerWarp; rb += kBatch) {
    if (rb > 0) {
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        const float4* rowp = reinterpret_cast<const float4*>(Srow0 + (rb + r) * kDK);
        s[r][0] = __ldcs(rowp + lane);
        s[r][1] = __ldcs(rowp + 32 + lane);
      }
    }
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
      const float xs[8] = {s[r][0].x, s[r][0].y, s[r][0].z, s[r][0].w,
                           s[r][1].x, s[r][1].y, s[r][1].z, s[r][1].w};
      float rk = 0.f, rq = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        rk = fmaf(xs[j], kr[j], rk);
        rq = fmaf(xs[j], qr[j], rq);
      }
      rk = warp_sum(rk);
      rq = warp_sum(rq);
      const float vi = __shfl_sync(0xffffffffu, vj, rb + r);
      const float delta = be * (vi - al * rk);
      float yv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) yv[j] = fmaf(al, xs[j], delta * kr[j]);
      float4* roww = reinterpret_cast<float4*>(Srow0 + (rb + r) * kDK);
      __stcs(roww + lane, make_float4(yv[0], yv[1], yv[2], yv[3]));
      __stcs(roww + 32 + lane, make_float4(yv[4], yv[5], yv[6], yv[7]));
      const float o = (al * rq + delta * kq) * kScale;
      if (lane == rb + r) o_mine = o;
    }
  }
  if (lane < kRowsPerWarp) a.o_buf[unit * a.dv + row0 + lane] = o_mine;
}

// Launch 2: Eq. 20 for every (sequence, head), one CTA of 256 threads each
// (one or two read-outs a thread, a block reduction for the mean square), and
// the in-place shift of the head's q and k convolution history (two channels
// a thread; the first launch has finished reading it).
template <typename T, bool kSilu>
__global__ void __launch_bounds__(kWarps * 32) finish_kernel(LayerArgs a) {
  const int64_t unit = blockIdx.x;
  const int64_t n = unit / a.H;
  const int h = (int)(unit % a.H);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float part[kWarps];
  const float* o = a.o_buf + unit * a.dv;
  float ov[2] = {0.f, 0.f}, ss = 0.f;
  for (int i = 0; i * kWarps * 32 < a.dv; ++i) {
    ov[i] = o[i * kWarps * 32 + tid];
    ss = fmaf(ov[i], ov[i], ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) part[warp] = ss;
  // the q / k history shift does not depend on the norm: issue it meanwhile
  const int64_t C = (int64_t)a.H * (2 * kDK + a.dv);
  const T* x = static_cast<const T*>(a.qkv) + n * C;
  T* st = static_cast<T*>(a.conv_state) + n * 3 * C;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int e = i * kWarps * 32 + tid;               // 0 .. 511 over q | k
    const int64_t c = (e < kDK ? 0 : (int64_t)a.H * kDK - kDK) + (int64_t)h * kDK + e;
    const float h1 = ld_in(st + C + c), h2 = ld_in(st + 2 * C + c), xc = ld_in(x + c);
    st_out(st + c, h1);
    st_out(st + C + c, h2);
    st_out(st + 2 * C + c, xc);
  }
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) tot += part[w];
  const float rs = rsqrtf(tot / a.dv + a.eps);
  for (int i = 0; i * kWarps * 32 < a.dv; ++i) {
    const int r = i * kWarps * 32 + tid;
    const float g = ld_in(static_cast<const T*>(a.gate) + unit * a.dv + r);
    const float act = kSilu ? silu_fast(g) : __fdividef(1.f, 1.f + __expf(-g));
    st_out(static_cast<T*>(a.y) + unit * a.dv + r, ov[i] * rs * a.norm_w[r] * act);
  }
}

bool aligned(const void* p, uintptr_t al) { return ((uintptr_t)p & (al - 1)) == 0; }
struct Span {
  uintptr_t lo, hi;
};
Span span_of(const void* p, size_t b) { return {(uintptr_t)p, (uintptr_t)p + (p ? b : 0)}; }
bool intersect(Span x, Span y) { return x.lo < x.hi && y.lo < y.hi && x.lo < y.hi && y.lo < x.hi; }

template <typename T, bool kSilu>
cudaError_t launch(const LayerArgs& a, int64_t units, cudaStream_t stream) {
  decode_layer_kernel<T><<<(unsigned)(units * (a.dv / kRows)), kWarps * 32, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  finish_kernel<T, kSilu><<<(unsigned)units, kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" int gdn_decode_layer_step(const void* qkv, const float* conv_w, const float* a_raw,
                                     const float* b_raw, const float* A_log,
                                     const float* dt_bias, void* conv_state, float* S,
                                     const void* gate, const float* norm_w, float eps,
                                     int32_t act, void* y, int32_t batch, int32_t heads,
                                     int32_t dk, int32_t dv, int32_t io_dtype,
                                     gdn_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (batch < 1 || heads < 1 || !(eps >= 0.f)) return GDN_ERR_INVALID_ARG;
  if (dk != kDK || !supported_dv(dv) || (io_dtype != GDN_F32 && io_dtype != GDN_BF16) ||
      (act != GDN_GATE_SILU && act != GDN_GATE_SIGMOID))
    return GDN_ERR_UNSUPPORTED;
  if (!qkv || !conv_w || !a_raw || !b_raw || !A_log || !dt_bias || !conv_state || !S || !gate ||
      !norm_w || !y)
    return GDN_ERR_INVALID_ARG;
  const void* a16[] = {qkv, conv_w, conv_state, S, gate, y};
  for (const void* p : a16)
    if (!aligned(p, 16)) return GDN_ERR_ALIGNMENT;
  const void* a4[] = {a_raw, b_raw, A_log, dt_bias, norm_w};
  for (const void* p : a4)
    if (!aligned(p, 4)) return GDN_ERR_ALIGNMENT;
  const size_t es = io_dtype == GDN_BF16 ? 2 : 4;
  const int64_t C = (int64_t)heads * (2 * dk + dv);
  const size_t nh = (size_t)batch * heads;
  const Span ins[] = {span_of(qkv, (size_t)batch * C * es), span_of(conv_w, (size_t)C * 16),
                      span_of(a_raw, nh * 4), span_of(b_raw, nh * 4),
                      span_of(A_log, heads * 4), span_of(dt_bias, heads * 4),
                      span_of(gate, nh * dv * es), span_of(norm_w, (size_t)dv * 4)};
  const Span outs[] = {span_of(conv_state, (size_t)batch * 3 * C * es),
                       span_of(S, nh * dv * dk * 4), span_of(y, nh * dv * es)};
  for (const Span& o : outs) {
    for (const Span& i : ins)
      if (intersect(i, o)) return GDN_ERR_INVALID_ARG;
    for (const Span& o2 : outs)
      if (&o2 != &o && intersect(o, o2)) return GDN_ERR_INVALID_ARG;
  }
  const int64_t units = (int64_t)batch * heads;
  if (units > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  // scratch: the read-outs between the two launches
  void* scratch = nullptr;
  if (scratch_alloc(&scratch, (size_t)units * dv * 4, stream) != cudaSuccess) return GDN_ERR_CUDA;
  LayerArgs a{qkv, conv_w, a_raw, b_raw, A_log, dt_bias, conv_state, S, gate, norm_w, eps, y,
              heads, dv, (float*)scratch};
  const bool silu = act == GDN_GATE_SILU;
  cudaError_t e;
  if (io_dtype == GDN_BF16)
    e = silu ? launch<__nv_bfloat16, true>(a, units, stream)
             : launch<__nv_bfloat16, false>(a, units, stream);
  else
    e = silu ? launch<float, true>(a, units, stream) : launch<float, false>(a, units, stream);
  count_launches(2);
  const cudaError_t ef = scratch_free(scratch, stream);
  return (e == cudaSuccess && ef == cudaSuccess) ? GDN_OK : GDN_ERR_CUDA;
}
