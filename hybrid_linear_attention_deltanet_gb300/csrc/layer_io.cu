// The steps of a Gated DeltaNet layer on either side of the recurrence
// ("Long-Context Aware Upcycling", Appendix A.3):
//
//  * before it (the paragraph after Table 8 and the text under Eq. 16-21):
//    a short causal depthwise convolution of width 4 + SiLU on q, k and v,
//    L2 normalisation of q and k per head, the decay
//    alpha = exp(-exp(A_log) * softplus(W_alpha x + Delta_bias)) (Eq. 16's
//    e^{g_t}) and the write strength beta = sigmoid(W_beta x);
//  * after it (Eq. 20): the read-out o_t RMS-normalised per head, times a
//    learned weight and an activated gate computed from W_G x_t.
//
// The projections themselves (W_Q, W_K, W_V, W_alpha, W_beta, W_G, W_O) are
// plain GEMMs and stay outside.  Every kernel here is an HBM stream: one warp
// owns 256 channels of one token row (8 per lane, one 16-byte vector at bf16)
// so that each global access is a fully coalesced 512 B (bf16) or 1 KiB
// (fp32) row piece, and the per-head reductions are warp shuffles.
//
// Layouts and argument contracts are those of include/gdn.h.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kTaps = 4;            // short convolution width (Table 8's paragraph)
constexpr int kHist = kTaps - 1;    // inputs carried across calls per channel
constexpr int kSeg = 256;           // channels per warp unit (one q/k head)
constexpr int kTile = 64;           // tokens one warp walks in the prefill form
constexpr int kWarpsPerCta = 8;
// The prefill form streams its input rows through a per-warp ring in shared
// memory filled by cp.async: kRing tokens a warp in flight without holding
// registers (16 warps an SM x 8 tokens x 512 B = 64 KB of loads in flight, about
// what HBM's bandwidth x latency asks of one SM).  16-byte copies a lane per
// token: 1 at bf16, 2 at fp32 (4 tokens deep: the same 32 KB a CTA).
template <typename T> __host__ __device__ constexpr int vecs_of() { return (int)sizeof(T) * 8 / 16; }
template <typename T> __host__ __device__ constexpr int ring_of() { return 8 / vecs_of<T>(); }
template <typename T> __host__ __device__ constexpr size_t ring_bytes() {
  return (size_t)kWarpsPerCta * ring_of<T>() * vecs_of<T>() * 32 * 16;
}
constexpr float kL2Eps = 1e-6f;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// 16-byte global -> shared copy of this thread, completed by cp_async_wait;
// each lane later reads back only what it copied itself
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(smem)),
               "l"((uint64_t)__cvta_generic_to_global(gmem))
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// at most N of this thread's most recent groups still pending
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 8 consecutive elements <-> 8 floats.  bf16 widens exactly (a shift); the
// narrowing rounds to nearest even.
struct Raw8 {
  uint4 a, b;  // bf16 uses a only
};

__device__ __forceinline__ Raw8 load8(const __nv_bfloat16* p) {
  Raw8 r;
  r.a = __ldcs(reinterpret_cast<const uint4*>(p));
  r.b = make_uint4(0, 0, 0, 0);
  return r;
}
__device__ __forceinline__ Raw8 load8(const float* p) {
  Raw8 r;
  r.a = __ldcs(reinterpret_cast<const uint4*>(p));
  r.b = __ldcs(reinterpret_cast<const uint4*>(p) + 1);
  return r;
}
__device__ __forceinline__ Raw8 load8_cached(const __nv_bfloat16* p) {
  Raw8 r;
  r.a = __ldg(reinterpret_cast<const uint4*>(p));
  r.b = make_uint4(0, 0, 0, 0);
  return r;
}
__device__ __forceinline__ Raw8 load8_cached(const float* p) {
  Raw8 r;
  r.a = __ldg(reinterpret_cast<const uint4*>(p));
  r.b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T>
__device__ __forceinline__ void widen8(const Raw8& r, float (&f)[8]);
template <>
__device__ __forceinline__ void widen8<__nv_bfloat16>(const Raw8& r, float (&f)[8]) {
  const uint32_t w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_lo(w[i]);
    f[2 * i + 1] = bf16_hi(w[i]);
  }
}
template <>
__device__ __forceinline__ void widen8<float>(const Raw8& r, float (&f)[8]) {
  const uint32_t w[8] = {r.a.x, r.a.y, r.a.z, r.a.w, r.b.x, r.b.y, r.b.z, r.b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(w[i]);
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float* p, const float (&f)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
// The same 8 elements as four fp32 pairs (element 2i in the low half of
// pair i), for the packed arithmetic of the convolution.
template <typename T>
__device__ __forceinline__ void widen8(const Raw8& r, F2 (&f)[4]);
template <>
__device__ __forceinline__ void widen8<__nv_bfloat16>(const Raw8& r, F2 (&f)[4]) {
  const uint32_t w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = f2(bf16_lo(w[i]), bf16_hi(w[i]));
}
template <>
__device__ __forceinline__ void widen8<float>(const Raw8& r, F2 (&f)[4]) {
  const uint32_t w[8] = {r.a.x, r.a.y, r.a.z, r.a.w, r.b.x, r.b.y, r.b.z, r.b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = f2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const F2 (&f)[4]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo, hi;
    f2_split(f[i], lo, hi);
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float* p, const F2 (&f)[4]) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) f2_split(f[i], v[2 * i], v[2 * i + 1]);
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// Elementwise activations of the streams are approximate to a few ulp (far
// inside the fp32 output tolerance): the convolution's SiLU is silu_pair
// (gdn_internal.cuh), the read-out gate's uses the fast exponential and
// divide intrinsics; at e^-x = inf either gives 0, the correct limit.  The
// per-head gates use expf/log1pf.
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.f + __expf(-x)); }
__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + expf(-x)); }
// log(1 + e^x); above 20 the correction e^-x is below fp32 resolution
__device__ __forceinline__ float softplusf_(float x) { return x > 20.f ? x : log1pf(expf(x)); }

// Conv taps of 8 channels, tap-major in registers as pairs: w[j][i] holds
// tap j of channels c0 + 2i and c0 + 2i + 1.
__device__ __forceinline__ void load_taps(const float* __restrict__ conv_w, int64_t c0,
                                          F2 (&w)[kTaps][4]) {
  const float4* p = reinterpret_cast<const float4*>(conv_w + c0 * kTaps);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 a = __ldg(p + 2 * i), b = __ldg(p + 2 * i + 1);  // taps 0..3 of two channels
    w[0][i] = f2(a.x, b.x); w[1][i] = f2(a.y, b.y); w[2][i] = f2(a.z, b.z); w[3][i] = f2(a.w, b.w);
  }
}

// The same one channel at a time: w[j][i] for channel c0 + i.
__device__ __forceinline__ void load_taps(const float* __restrict__ conv_w, int64_t c0,
                                          float (&w)[kTaps][8]) {
  const float4* p = reinterpret_cast<const float4*>(conv_w + c0 * kTaps);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 t = __ldg(p + i);  // channel c0 + i: taps 0..3
    w[0][i] = t.x; w[1][i] = t.y; w[2][i] = t.z; w[3][i] = t.w;
  }
}

// The three inputs before a sequence's first token: its carried state, or
// zeros.  kNC: the state is read-only for the whole launch (it may then take
// the non-coherent path); the in-place decode form reads it coherently.
template <typename T, bool kNC>
__device__ __forceinline__ void history(const T* state_in, int64_t n, int64_t C, int64_t c0,
                                        F2 (&win)[kHist][4]) {
#pragma unroll
  for (int j = 0; j < kHist; ++j) {
    if (state_in) {
      const T* p = state_in + (n * kHist + j) * C + c0;
      widen8<T>(kNC ? load8_cached(p) : load8(p), win[j]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) win[j][i] = f2(0.f, 0.f);
    }
  }
}

// The decode step's form: the carried state of one sequence, one channel at
// a time.
template <typename T>
__device__ __forceinline__ void history8(const T* state, int64_t n, int64_t C, int64_t c0,
                                         float (&win)[kHist][8]) {
#pragma unroll
  for (int j = 0; j < kHist; ++j) widen8<T>(load8(state + (n * kHist + j) * C + c0), win[j]);
}

// One token of one 256-channel segment, one channel at a time, with the
// window shifting in x: the same roundings as conv_rot below, channel by
// channel (the decode step's single token a warp is bound by the latency of
// this chain, where the pair form's packing costs more than it saves).
__device__ __forceinline__ void conv_token(const float (&w)[kTaps][8], float (&win)[kHist][8],
                                           const float (&x)[8], bool l2, float (&y)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float acc = __fmul_rn(w[0][i], win[0][i]);
    acc = fmaf(w[1][i], win[1][i], acc);
    acc = fmaf(w[2][i], win[2][i], acc);
    acc = fmaf(w[3][i], x[i], acc);
    y[i] = silu_sfu(acc);
    win[0][i] = win[1][i];
    win[1][i] = win[2][i];
    win[2][i] = x[i];
  }
  if (l2) {  // warp-uniform branch: the segment is one q or k head
    const float r = rsqrtf(warp_sum(sumsq8(y)) + kL2Eps);
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(y[i], r);
  }
}

// One token of one 256-channel segment: conv + SiLU (+ L2 norm over the
// segment when it is a q or k head).  The taps run as fp32 pairs (the same
// roundings as one channel at a time).  The window is kept in rotation:
// slot R holds the oldest input, R + 1 (mod 3) the next, R + 2 the newest; x
// replaces the oldest, so the next token takes rotation R + 1, and three
// tokens bring the slots back to their order with no register moves.
template <int R>
__device__ __forceinline__ void conv_rot(const F2 (&w)[kTaps][4], F2 (&win)[kHist][4],
                                         const F2 (&x)[4], bool l2, F2 (&y)[4]) {
  constexpr int a = R % 3, b = (R + 1) % 3, c = (R + 2) % 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    F2 acc = f2_mul(w[0][i], win[a][i]);
    acc = f2_fma(w[1][i], win[b][i], acc);
    acc = f2_fma(w[2][i], win[c][i], acc);
    acc = f2_fma(w[3][i], x[i], acc);
    y[i] = silu_pair(acc);
    win[a][i] = x[i];
  }
  if (l2) {  // warp-uniform branch: the segment is one q or k head
    const float r = rsqrtf(warp_sum(sumsq8(y)) + kL2Eps);
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = f2_mul(y[i], f2(r, r));
  }
}
// The same with the window in order (slot 0 the oldest) before and after.
__device__ __forceinline__ void conv_token(const F2 (&w)[kTaps][4], F2 (&win)[kHist][4],
                                           const F2 (&x)[4], bool l2, F2 (&y)[4]) {
  conv_rot<0>(w, win, x, l2, y);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const F2 t = win[0][i];
    win[0][i] = win[1][i];
    win[1][i] = win[2][i];
    win[2][i] = t;
  }
}
// Two consecutive tokens of one sequence with the window at rotation R:
// their arithmetic has no branch between it, so the two dependent chains
// (taps, SiLU, the L2 reduction) interleave.  o: the first token's output row.
template <typename T, int R>
__device__ __forceinline__ void pair_rot(const F2 (&w)[kTaps][4], F2 (&win)[kHist][4],
                                         const Raw8& r0, const Raw8& r1, bool l2, T* o,
                                         int64_t stride) {
  F2 x0[4], x1[4], y0[4], y1[4];
  widen8<T>(r0, x0);
  widen8<T>(r1, x1);
  conv_rot<R>(w, win, x0, l2, y0);
  conv_rot<(R + 1) % 3>(w, win, x1, l2, y1);
  store8(o, y0);
  store8(o + stride, y1);
}

struct PrepareArgs {
  const void* qkv;          // [T_total, C] io dtype
  const float* conv_w;      // [C, 4]
  const float* a_raw;       // [T_total, H]
  const float* b_raw;       // [T_total, H]
  const float* A_log;       // [H]
  const float* dt_bias;     // [H]
  const void* state_in;     // [N, 3, C] io dtype or null
  void* state_out;          // [N, 3, C] io dtype or null
  void* q; void* k; void* v;
  float* alpha; float* beta;
  const int32_t* cu;        // [N + 1] or null (dense)
  int32_t N;
  int64_t T;                // dense: tokens per sequence; varlen: T_total
  int64_t T_total;
  int32_t H, dk, dv;
  int64_t n_tiles;
  int32_t n_seg;            // C / 256
  unsigned* status;         // device status word (malformed cu_seqlens)
};

struct Seqs {
  const int32_t* cu;
  int64_t T;
  __device__ __forceinline__ int64_t begin(int64_t n) const { return cu ? (int64_t)cu[n] : n * T; }
  __device__ __forceinline__ int64_t end(int64_t n) const {
    return cu ? (int64_t)cu[n + 1] : (n + 1) * T;
  }
  // sequence holding token t (the last n with begin(n) <= t, skipping empties)
  __device__ __forceinline__ int64_t find(int64_t t, int32_t N) const {
    if (!cu) return t / T;
    int lo = 0, hi = N - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
  }
};

__device__ __forceinline__ void gates_one(const PrepareArgs& a, int64_t idx) {
  const int h = (int)(idx % a.H);
  const float decay_rate = expf(__ldg(a.A_log + h));
  const float g = -decay_rate * softplusf_(__ldcs(a.a_raw + idx) + __ldg(a.dt_bias + h));
  a.alpha[idx] = expf(g);
  a.beta[idx] = sigmoidf_(__ldcs(a.b_raw + idx));
}

// Warp units: for each tile of kTile tokens, n_seg channel segments and one
// gate unit; then one unit per sequence that copies the carried state of an
// empty sequence through.
// At most 128 registers a thread and 32 KB of ring a CTA, so that two CTAs
// (16 warps, each with kRing tokens in flight) share an SM.
template <typename T>
__global__ void __launch_bounds__(kWarpsPerCta * 32, 2)
prepare_kernel(PrepareArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t unit = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t C = (int64_t)a.H * (2 * a.dk + a.dv);
  const int64_t per_tile = a.n_seg + 1;
  const Seqs seqs{a.cu, a.T};
  const T* state_in = static_cast<const T*>(a.state_in);
  T* state_out = static_cast<T*>(a.state_out);

  if (unit >= a.n_tiles * per_tile) {  // per-sequence units
    const int64_t n = unit - a.n_tiles * per_tile;
    if (n >= a.N) return;
    if (a.cu && lane == 0 &&
        (a.cu[n + 1] < a.cu[n] || (n == 0 && a.cu[0] != 0) ||
         (n == a.N - 1 && (int64_t)a.cu[a.N] != a.T_total)))
      flag_status(a.status, GDN_ERR_BAD_SEQLENS);
    if (!state_out || seqs.end(n) > seqs.begin(n)) return;   // only empty sequences copy
    for (int64_t e = lane * 8; e < kHist * C; e += 32 * 8) {
      float f[8];
      if (state_in) widen8<T>(load8_cached(state_in + n * kHist * C + e), f);
      else for (int i = 0; i < 8; ++i) f[i] = 0.f;
      store8(state_out + n * kHist * C + e, f);
    }
    return;
  }
  const int64_t tile = unit / per_tile;
  const int seg = (int)(unit % per_tile);
  const int64_t t0 = tile * kTile;
  const int64_t t1 = min(t0 + (int64_t)kTile, a.T_total);

  if (seg == a.n_seg) {  // decay and write strength of the tile's tokens
    for (int64_t idx = t0 * a.H + lane; idx < t1 * a.H; idx += 32) gates_one(a, idx);
    return;
  }

  const int64_t c0 = (int64_t)seg * kSeg + lane * 8;
  const bool l2 = seg < 2 * a.H * a.dk / kSeg;   // q and k heads
  T* dst;
  int64_t dst_stride, dst_c;
  if (c0 < (int64_t)a.H * a.dk) {
    dst = static_cast<T*>(a.q); dst_stride = (int64_t)a.H * a.dk; dst_c = c0;
  } else if (c0 < 2 * (int64_t)a.H * a.dk) {
    dst = static_cast<T*>(a.k); dst_stride = (int64_t)a.H * a.dk; dst_c = c0 - (int64_t)a.H * a.dk;
  } else {
    dst = static_cast<T*>(a.v); dst_stride = (int64_t)a.H * a.dv;
    dst_c = c0 - 2 * (int64_t)a.H * a.dk;
  }
  F2 w[kTaps][4];
  load_taps(a.conv_w, c0, w);
  const T* x = static_cast<const T*>(a.qkv);

  // window before t0: inputs of the same sequence, or the slots of its
  // carried history that precede the sequence start (slot p - sb + 3)
  int64_t n = seqs.find(t0, a.N);
  int64_t sb = seqs.begin(n), se = seqs.end(n);
  F2 win[kHist][4];
#pragma unroll
  for (int j = 0; j < kHist; ++j) {
    const int64_t p = t0 - kHist + j;
    if (p >= sb) {
      widen8<T>(load8_cached(x + p * C + c0), win[j]);
    } else if (state_in) {
      widen8<T>(load8_cached(state_in + (n * kHist + (p - sb + kHist)) * C + c0), win[j]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) win[j][i] = f2(0.f, 0.f);
    }
  }

  // The ring: slot i of this warp holds token t0 + i (mod kRing), one
  // cp.async group per token; groups past the tile's end are empty, so that
  // "all but the kRing - 1 newest groups complete" always means "token t is in".
  // Inside the tile tokens are counted from t0 in 32 bits and the row pointers
  // advance by one row a token (no 64-bit index products on the way).
  constexpr int kRing = ring_of<T>(), kVec = vecs_of<T>();
  extern __shared__ uint4 ring_smem[];
  uint4* ring = ring_smem + (threadIdx.x >> 5) * (kRing * kVec * 32) + lane;
  const int n_tok = (int)(t1 - t0);
  const T* src = x + t0 * C + c0;          // row of the next token to fetch
  int fetched = 0;                          // tokens fetched so far
  auto issue = [&]() {
    if (fetched < n_tok) {
      uint4* slot = ring + (fetched & (kRing - 1)) * (kVec * 32);
      const uint4* g = reinterpret_cast<const uint4*>(src);
#pragma unroll
      for (int u = 0; u < kVec; ++u) cp_async16(slot + u * 32, g + u);
      src += C;
    }
    ++fetched;
    cp_async_commit();
  };
#pragma unroll
  for (int d = 0; d < kRing; ++d) issue();
  auto read = [&](int i) {
    Raw8 r;
    const uint4* slot = ring + (i & (kRing - 1)) * (kVec * 32);
    r.a = slot[0];
    r.b = kVec > 1 ? slot[32] : make_uint4(0, 0, 0, 0);
    return r;
  };
  T* out_row = dst + t0 * dst_stride + dst_c;   // row of token t0 + i: out_row + i rows
  // the current sequence's end relative to t0, clamped so that it fits 32 bits
  // and stays above i + 2 for every i of the tile when the sequence runs on
  auto rel_end = [&]() { return (int)min(se - t0, (int64_t)kTile + 2); };
  int se_rel = rel_end();
  // one token, with the sequence bookkeeping
  auto one = [&](int i, const Raw8& r) {
    const int64_t t = t0 + i;
    if (t >= se && n + 1 < a.N) {  // a new sequence starts here (skipping empty ones)
      do { ++n; } while (n + 1 < a.N && seqs.end(n) <= t);
      sb = seqs.begin(n);
      se = seqs.end(n);
      se_rel = rel_end();
      history<T, true>(state_in, n, C, c0, win);
    }
    F2 xf[4], y[4];
    widen8<T>(r, xf);
    conv_token(w, win, xf, l2, y);
    store8(out_row + i * dst_stride, y);
    if (t == se - 1 && state_out) {
#pragma unroll
      for (int j = 0; j < kHist; ++j) store8(state_out + (n * kHist + j) * C + c0, win[j]);
    }
  };
  // Six tokens an iteration while they all lie inside the current sequence
  // (three pairs, the window in rotation: back in order after six), else a
  // pair, with the sequence bookkeeping where a sequence ends inside it.
  // Each pair waits for its two tokens, then refills their two slots.
  int i = 0;
  while (i < n_tok) {
    if (i + 6 <= n_tok && i + 6 <= se_rel) {
      T* o = out_row + i * dst_stride;
      cp_async_wait<kRing - 2>();
      pair_rot<T, 0>(w, win, read(i), read(i + 1), l2, o, dst_stride);
      issue();
      issue();
      cp_async_wait<kRing - 2>();
      pair_rot<T, 2>(w, win, read(i + 2), read(i + 3), l2, o + 2 * dst_stride, dst_stride);
      issue();
      issue();
      cp_async_wait<kRing - 2>();
      pair_rot<T, 1>(w, win, read(i + 4), read(i + 5), l2, o + 4 * dst_stride, dst_stride);
      issue();
      issue();
      if (i + 6 == se_rel && state_out) {   // token i + 5 ends the sequence
#pragma unroll
        for (int j = 0; j < kHist; ++j) store8(state_out + (n * kHist + j) * C + c0, win[j]);
      }
      i += 6;
      continue;
    }
    cp_async_wait<kRing - 2>();   // tokens i and i + 1 are in
    const Raw8 r0 = read(i);
    const bool pair = i + 1 < n_tok;
    const Raw8 r1 = pair ? read(i + 1) : r0;
    if (pair && i + 1 < se_rel) {
      F2 x0[4], x1[4], y0[4], y1[4];
      widen8<T>(r0, x0);
      widen8<T>(r1, x1);
      conv_token(w, win, x0, l2, y0);
      conv_token(w, win, x1, l2, y1);
      T* o = out_row + i * dst_stride;
      store8(o, y0);
      store8(o + dst_stride, y1);
      if (i + 2 == se_rel && state_out) {   // token i + 1 ends the sequence
#pragma unroll
        for (int j = 0; j < kHist; ++j) store8(state_out + (n * kHist + j) * C + c0, win[j]);
      }
    } else {
      one(i, r0);
      if (pair) one(i + 1, r1);
    }
    // both slots' values are in registers (consumed above): refill them
    issue();
    issue();
    i += 2;
  }
  cp_async_wait<0>();
}

// One token per sequence against the carried convolution state, which is
// updated in place (each lane reads its channels' history before writing it).
template <typename T>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
prepare_decode_kernel(PrepareArgs a, T* __restrict__ state) {
  const int lane = threadIdx.x & 31;
  const int64_t unit = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t per_seq = a.n_seg + 1;
  if (unit >= (int64_t)a.N * per_seq) return;
  const int64_t n = unit / per_seq;
  const int seg = (int)(unit % per_seq);
  const int64_t C = (int64_t)a.H * (2 * a.dk + a.dv);
  if (seg == a.n_seg) {
    for (int64_t idx = n * a.H + lane; idx < (n + 1) * a.H; idx += 32) gates_one(a, idx);
    return;
  }
  const int64_t c0 = (int64_t)seg * kSeg + lane * 8;
  const bool l2 = seg < 2 * a.H * a.dk / kSeg;
  float w[kTaps][8], win[kHist][8], xf[8], y[8];
  load_taps(a.conv_w, c0, w);
  history8<T>(state, n, C, c0, win);
  widen8<T>(load8(static_cast<const T*>(a.qkv) + n * C + c0), xf);
  conv_token(w, win, xf, l2, y);
  if (c0 < (int64_t)a.H * a.dk) {
    store8(static_cast<T*>(a.q) + n * a.H * a.dk + c0, y);
  } else if (c0 < 2 * (int64_t)a.H * a.dk) {
    store8(static_cast<T*>(a.k) + n * a.H * a.dk + (c0 - (int64_t)a.H * a.dk), y);
  } else {
    store8(static_cast<T*>(a.v) + n * a.H * a.dv + (c0 - 2 * (int64_t)a.H * a.dk), y);
  }
#pragma unroll
  for (int j = 0; j < kHist; ++j) store8(state + (n * kHist + j) * C + c0, win[j]);
}

// Eq. 20 read-out: y = o / sqrt(mean(o^2) + eps) * w * act(g) over the dv
// values of one (token, head) row; one warp per row, NV groups of 8 per lane.
template <typename T, int NV, bool kSilu>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
norm_gate_kernel(const T* o, const T* __restrict__ g, const float* __restrict__ w, float eps,
                 T* y, int64_t rows) {   // y may be o itself
  constexpr int dv = NV * kSeg;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * kWarpsPerCta;
  float wr[NV][8];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int i = 0; i < 8; ++i) wr[v][i] = __ldg(w + v * kSeg + lane * 8 + i);
  // two rows per iteration: both rows' loads are in flight before either is used
  for (int64_t r0 = ((int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5)) * 2; r0 < rows;
       r0 += 2 * warps) {
    Raw8 ro[2][NV], rg[2][NV];
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (r0 + u < rows) {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          ro[u][v] = load8(o + (r0 + u) * dv + v * kSeg + lane * 8);
          rg[u][v] = load8(g + (r0 + u) * dv + v * kSeg + lane * 8);
        }
      }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t r = r0 + u;
      if (r >= rows) break;
      float of[NV][8], ss = 0.f;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        widen8<T>(ro[u][v], of[v]);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(of[v][i], of[v][i], ss);
      }
      const float rs = rsqrtf(warp_sum(ss) * (1.f / dv) + eps);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        float gf[8], out[8];
        widen8<T>(rg[u][v], gf);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float act = kSilu ? silu_fast(gf[i]) : sigmoid_fast(gf[i]);
          out[i] = of[v][i] * rs * wr[v][i] * act;
        }
        store8(y + r * dv + v * kSeg + lane * 8, out);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// host side
bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

struct Span {
  uintptr_t lo, hi;
};
Span span_of(const void* p, size_t bytes) { return {(uintptr_t)p, (uintptr_t)p + (p ? bytes : 0)}; }
bool intersect(Span a, Span b) { return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 148;
  return n;
}

bool geometry_ok(int32_t dk, int32_t dv, int32_t io_dtype) {
  return dk == kDK && supported_dv(dv) && (io_dtype == GDN_F32 || io_dtype == GDN_BF16);
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

int gdn_prepare(const void* qkv, const float* conv_w, const float* a_raw, const float* b_raw,
                const float* A_log, const float* dt_bias, const int32_t* cu_seqlens,
                const void* conv_state_in, void* conv_state_out, void* q, void* k, void* v,
                float* alpha, float* beta, int32_t batch, int64_t seqlen, int32_t heads,
                int32_t dk, int32_t dv, int32_t io_dtype, gdn_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (batch < 1 || seqlen < 0 || heads < 1) return GDN_ERR_INVALID_ARG;
  if (!geometry_ok(dk, dv, io_dtype)) return GDN_ERR_UNSUPPORTED;
  const bool varlen = cu_seqlens != nullptr;
  const int64_t T_total = varlen ? seqlen : (int64_t)batch * seqlen;
  if (!conv_w || !A_log || !dt_bias) return GDN_ERR_INVALID_ARG;
  if (T_total > 0 && (!qkv || !a_raw || !b_raw || !q || !k || !v || !alpha || !beta))
    return GDN_ERR_INVALID_ARG;
  if (varlen && T_total > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  const void* v16[] = {qkv, conv_w, conv_state_in, conv_state_out, q, k, v};
  for (const void* p : v16)
    if (!aligned(p, 16)) return GDN_ERR_ALIGNMENT;
  const void* v4[] = {a_raw, b_raw, A_log, dt_bias, cu_seqlens, alpha, beta};
  for (const void* p : v4)
    if (!aligned(p, 4)) return GDN_ERR_ALIGNMENT;
  const size_t es = io_dtype == GDN_BF16 ? 2 : 4;
  const int64_t C = (int64_t)heads * (2 * dk + dv);
  const size_t nt = (size_t)T_total, nh = nt * heads;
  const size_t state_bytes = (size_t)batch * kHist * C * es;
  const Span ins[] = {span_of(qkv, nt * C * es), span_of(conv_w, (size_t)C * kTaps * 4),
                      span_of(a_raw, nh * 4), span_of(b_raw, nh * 4),
                      span_of(A_log, heads * 4), span_of(dt_bias, heads * 4),
                      span_of(cu_seqlens, varlen ? ((size_t)batch + 1) * 4 : 0),
                      span_of(conv_state_in, state_bytes)};
  const Span outs[] = {span_of(q, nh * dk * es), span_of(k, nh * dk * es),
                       span_of(v, nh * dv * es), span_of(alpha, nh * 4), span_of(beta, nh * 4),
                       span_of(conv_state_out, state_bytes)};
  for (const Span& o : outs) {
    for (const Span& i : ins)
      if (intersect(i, o)) return GDN_ERR_INVALID_ARG;   // includes state_in == state_out
    for (const Span& o2 : outs)
      if (&o2 != &o && intersect(o, o2)) return GDN_ERR_INVALID_ARG;
  }

  PrepareArgs a{};
  a.qkv = qkv; a.conv_w = conv_w; a.a_raw = a_raw; a.b_raw = b_raw; a.A_log = A_log;
  a.dt_bias = dt_bias; a.state_in = conv_state_in; a.state_out = conv_state_out;
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta;
  a.cu = cu_seqlens; a.N = batch; a.T = varlen ? T_total : seqlen; a.T_total = T_total;
  a.H = heads; a.dk = dk; a.dv = dv;
  a.n_tiles = (T_total + kTile - 1) / kTile;
  a.n_seg = (int32_t)(C / kSeg);
  a.status = status_ptr();
  if (!a.status) return GDN_ERR_CUDA;
  const int64_t units = a.n_tiles * (a.n_seg + 1) + batch;
  const int64_t blocks = (units + kWarpsPerCta - 1) / kWarpsPerCta;
  if (blocks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  if (blocks == 0) return GDN_OK;
  if (io_dtype == GDN_BF16)
    prepare_kernel<__nv_bfloat16>
        <<<(unsigned)blocks, kWarpsPerCta * 32, ring_bytes<__nv_bfloat16>(), stream>>>(a);
  else
    prepare_kernel<float><<<(unsigned)blocks, kWarpsPerCta * 32, ring_bytes<float>(), stream>>>(a);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_prepare_decode_step(const void* qkv, const float* conv_w, const float* a_raw,
                            const float* b_raw, const float* A_log, const float* dt_bias,
                            void* conv_state, void* q, void* k, void* v, float* alpha,
                            float* beta, int32_t batch, int32_t heads, int32_t dk, int32_t dv,
                            int32_t io_dtype, gdn_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (batch < 1 || heads < 1) return GDN_ERR_INVALID_ARG;
  if (!geometry_ok(dk, dv, io_dtype)) return GDN_ERR_UNSUPPORTED;
  if (!qkv || !conv_w || !a_raw || !b_raw || !A_log || !dt_bias || !conv_state || !q || !k ||
      !v || !alpha || !beta)
    return GDN_ERR_INVALID_ARG;
  const void* v16[] = {qkv, conv_w, conv_state, q, k, v};
  for (const void* p : v16)
    if (!aligned(p, 16)) return GDN_ERR_ALIGNMENT;
  const void* v4[] = {a_raw, b_raw, A_log, dt_bias, alpha, beta};
  for (const void* p : v4)
    if (!aligned(p, 4)) return GDN_ERR_ALIGNMENT;
  const size_t es = io_dtype == GDN_BF16 ? 2 : 4;
  const int64_t C = (int64_t)heads * (2 * dk + dv);
  const size_t nh = (size_t)batch * heads;
  const Span ins[] = {span_of(qkv, (size_t)batch * C * es), span_of(conv_w, (size_t)C * kTaps * 4),
                      span_of(a_raw, nh * 4), span_of(b_raw, nh * 4),
                      span_of(A_log, heads * 4), span_of(dt_bias, heads * 4)};
  const Span outs[] = {span_of(q, nh * dk * es), span_of(k, nh * dk * es),
                       span_of(v, nh * dv * es), span_of(alpha, nh * 4), span_of(beta, nh * 4),
                       span_of(conv_state, (size_t)batch * kHist * C * es)};
  for (const Span& o : outs) {
    for (const Span& i : ins)
      if (intersect(i, o)) return GDN_ERR_INVALID_ARG;
    for (const Span& o2 : outs)
      if (&o2 != &o && intersect(o, o2)) return GDN_ERR_INVALID_ARG;
  }
  PrepareArgs a{};
  a.qkv = qkv; a.conv_w = conv_w; a.a_raw = a_raw; a.b_raw = b_raw; a.A_log = A_log;
  a.dt_bias = dt_bias; a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta;
  a.N = batch; a.H = heads; a.dk = dk; a.dv = dv;
  a.n_seg = (int32_t)(C / kSeg);
  const int64_t units = (int64_t)batch * (a.n_seg + 1);
  const int64_t blocks = (units + kWarpsPerCta - 1) / kWarpsPerCta;
  if (blocks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  if (io_dtype == GDN_BF16)
    prepare_decode_kernel<__nv_bfloat16><<<(unsigned)blocks, kWarpsPerCta * 32, 0, stream>>>(
        a, static_cast<__nv_bfloat16*>(conv_state));
  else
    prepare_decode_kernel<float><<<(unsigned)blocks, kWarpsPerCta * 32, 0, stream>>>(
        a, static_cast<float*>(conv_state));
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_output_norm_gate(const void* o, const void* g, const float* w, float eps, int32_t act,
                         void* y, int64_t tokens, int32_t heads, int32_t dv, int32_t io_dtype,
                         gdn_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (tokens < 0 || heads < 1 || !(eps >= 0.f)) return GDN_ERR_INVALID_ARG;
  if (!supported_dv(dv) || (io_dtype != GDN_F32 && io_dtype != GDN_BF16) ||
      (act != GDN_GATE_SILU && act != GDN_GATE_SIGMOID))
    return GDN_ERR_UNSUPPORTED;
  if (tokens == 0) return GDN_OK;
  if (!o || !g || !w || !y) return GDN_ERR_INVALID_ARG;
  if (!aligned(o, 16) || !aligned(g, 16) || !aligned(y, 16) || !aligned(w, 4))
    return GDN_ERR_ALIGNMENT;
  const size_t es = io_dtype == GDN_BF16 ? 2 : 4;
  const size_t bytes = (size_t)tokens * heads * dv * es;
  const Span so = span_of(o, bytes), sg = span_of(g, bytes), sy = span_of(y, bytes),
             sw = span_of(w, (size_t)dv * 4);
  // y may be o itself (in place) but may not overlap it partially, nor g or w
  if ((y != o && intersect(sy, so)) || intersect(sy, sg) || intersect(sy, sw))
    return GDN_ERR_INVALID_ARG;
  const int64_t rows = tokens * heads;
  const int64_t want = ((rows + 1) / 2 + kWarpsPerCta - 1) / kWarpsPerCta;
  const int64_t cap = (int64_t)sm_count() * 8;   // grid-stride beyond 8 CTAs per SM
  const unsigned blocks = (unsigned)(want < cap ? want : cap);
  const bool silu = act == GDN_GATE_SILU;
#define GDN_NG(T, NV, S)                                                              \
  norm_gate_kernel<T, NV, S><<<blocks, kWarpsPerCta * 32, 0, stream>>>(              \
      (const T*)o, (const T*)g, w, eps, (T*)y, rows)
  if (io_dtype == GDN_BF16) {
    if (dv == 256) { if (silu) GDN_NG(__nv_bfloat16, 1, true); else GDN_NG(__nv_bfloat16, 1, false); }
    else           { if (silu) GDN_NG(__nv_bfloat16, 2, true); else GDN_NG(__nv_bfloat16, 2, false); }
  } else {
    if (dv == 256) { if (silu) GDN_NG(float, 1, true); else GDN_NG(float, 1, false); }
    else           { if (silu) GDN_NG(float, 2, true); else GDN_NG(float, 2, false); }
  }
#undef GDN_NG
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // extern "C"
