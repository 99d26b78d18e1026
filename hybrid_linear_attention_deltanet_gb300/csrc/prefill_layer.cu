// gdn_prefill_layer -- the mixer core of a Gated DeltaNet layer over whole
// sequences ("Long-Context Aware Upcycling", Appendix A.3): the
// pre-recurrence steps (short convolution + SiLU, q / k L2 normalisation, the
// gates; the paragraph after Table 8 and the text under Eq. 16-21), the
// chunked recurrence and Eq. 20's gated RMSNorm in one call.
//
// Up to the long-sequence length the pre-recurrence steps run as their own
// pass into scratch (gdn_prepare), then the tensor-core prefill with the
// read-out inside: in the fused form the per-chunk workers, once their
// chunks' operands are out, apply Eq. 20 to each chunk's output rows behind
// the state chains (o exists only in y's memory in between); in the split
// form the two 128-row units of a head finish their rows as a 2-CTA cluster.
// Measured alternative: the convolution inside the per-chunk prep on its
// input tiles (q, k, v, alpha and beta never in HBM) more than doubled each
// prep item, which the chains then waited for.  For sequences that take the
// segmented form that is still the path taken: there the prep runs over all
// items before the state passes anyway, and the keys the prep processes are
// left in scratch for the state passes' K tiles.
#include <algorithm>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

bool aligned_to(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

struct Span {
  uintptr_t lo, hi;
};
Span span_of(const void* p, size_t bytes) { return {(uintptr_t)p, (uintptr_t)p + (p ? bytes : 0)}; }
bool meet(Span a, Span b) { return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi; }

// The carried convolution state of an empty sequence passes through
// unchanged (zero without a state in): nothing else writes it.  cu = nullptr:
// a dense batch of empty sequences.
__global__ void empty_state_kernel(const int32_t* __restrict__ cu, int32_t N, int64_t C,
                                   const __nv_bfloat16* __restrict__ state_in,
                                   __nv_bfloat16* __restrict__ state_out) {
  const int64_t per = 3 * C / 8;   // 16-byte pieces of one sequence's state
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)N * per;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = i / per;
    if (cu && cu[n + 1] != cu[n]) continue;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (state_in) v = reinterpret_cast<const uint4*>(state_in)[i];
    reinterpret_cast<uint4*>(state_out)[i] = v;
  }
}

size_t k_out_bytes(int64_t T_total, int32_t heads) {
  return align_up((size_t)T_total * heads * kDK * 2, 1024);
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" int gdn_prefill_layer(const void* qkv, const float* conv_w, const float* a_raw,
                                 const float* b_raw, const float* A_log, const float* dt_bias,
                                 const void* conv_state_in, void* conv_state_out, const float* S0,
                                 const int32_t* cu_seqlens, const void* gate,
                                 const float* norm_w, float eps, int32_t act, void* y,
                                 float* S_final, int32_t batch, int64_t seqlen, int32_t heads,
                                 int32_t dk, int32_t dv, int32_t io_dtype, gdn_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (batch < 1 || seqlen < 0 || heads < 1 || !(eps >= 0.f)) return GDN_ERR_INVALID_ARG;
  if (act != GDN_GATE_SILU && act != GDN_GATE_SIGMOID) return GDN_ERR_INVALID_ARG;
  if (io_dtype != GDN_BF16 || dk != kDK || dv != kDK) return GDN_ERR_UNSUPPORTED;
  const bool varlen = cu_seqlens != nullptr;
  const int64_t T_total = varlen ? seqlen : (int64_t)batch * seqlen;
  if (T_total > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  if (T_total > 0 && (!qkv || !conv_w || !a_raw || !b_raw || !A_log || !dt_bias || !gate ||
                      !norm_w || !y))
    return GDN_ERR_INVALID_ARG;
  const void* a16[] = {qkv, conv_w, conv_state_in, conv_state_out, S0, gate, y, S_final};
  for (const void* p : a16)
    if (!aligned_to(p, 16)) return GDN_ERR_ALIGNMENT;
  const void* a4[] = {a_raw, b_raw, A_log, dt_bias, norm_w, cu_seqlens};
  for (const void* p : a4)
    if (!aligned_to(p, 4)) return GDN_ERR_ALIGNMENT;
  const int64_t C = (int64_t)3 * heads * kDK;
  const size_t ntok = (size_t)T_total, nth = ntok * heads;
  const size_t state = (size_t)batch * heads * dv * dk * 4, conv_state = (size_t)batch * 3 * C * 2;
  const Span ins[] = {span_of(qkv, ntok * C * 2),       span_of(conv_w, (size_t)C * 16),
                      span_of(a_raw, nth * 4),          span_of(b_raw, nth * 4),
                      span_of(A_log, heads * 4u),       span_of(dt_bias, heads * 4u),
                      span_of(conv_state_in, conv_state), span_of(S0, state),
                      span_of(cu_seqlens, varlen ? ((size_t)batch + 1) * 4 : 0),
                      span_of(gate, nth * dv * 2),      span_of(norm_w, (size_t)dv * 4)};
  const Span outs[] = {span_of(y, nth * dv * 2), span_of(S_final, S_final ? state : 0),
                       span_of(conv_state_out, conv_state_out ? conv_state : 0)};
  for (const Span& o : outs) {
    for (const Span& i : ins)
      if (meet(o, i)) return GDN_ERR_INVALID_ARG;
  }
  if (meet(outs[0], outs[1]) || meet(outs[0], outs[2]) || meet(outs[1], outs[2]))
    return GDN_ERR_INVALID_ARG;
  if (takes_long_form(seqlen, 0) &&
      plan_long(batch, seqlen, varlen, heads, dv, GDN_BF16, 0).n_slots * 2 > 0x7fffffffLL)
    return GDN_ERR_UNSUPPORTED;

  unsigned* status = status_ptr();
  if (!status) return GDN_ERR_CUDA;

  if (!takes_long_form(seqlen, 0)) {
    // The pre-recurrence steps as their own pass (gdn_prepare, into scratch),
    // then the prefill with the read-out inside: in the fused form its
    // per-chunk workers, once their chunks' operands are out, apply Eq. 20
    // to each chunk's rows behind the state chains; in the split form the
    // two units of a head finish their rows as a cluster.  (Keeping the
    // convolution inside the per-chunk prep instead measured slower: it
    // more than doubles each prep item, which the chains then wait for.)
    const size_t nth = (size_t)T_total * heads;
    const size_t qb = align_up(nth * kDK * 2, 1024), gb = align_up(nth * 4, 1024);
    const size_t pb = align_up(nth * 8, 1024);
    const int64_t max_chunks = max_chunks_bound(batch, T_total, varlen, seqlen);
    const size_t fb = align_up((size_t)batch * heads * (dv / 128) * 4, 1024);
    const size_t need =
        3 * qb + 2 * gb + pb + fb + prefill_scratch_bytes(batch, seqlen, heads, dv, GDN_BF16,
                                                          varlen, 0);
    void* scratch = nullptr;
    if (scratch_alloc(&scratch, need, stream) != cudaSuccess) return GDN_ERR_CUDA;
    char* p = (char*)scratch;
    void* q = p;
    void* k = p + qb;
    void* v = p + 2 * qb;
    float* alpha = (float*)(p + 3 * qb);
    float* beta = (float*)(p + 3 * qb + gb);
    float* part = (float*)(p + 3 * qb + 2 * gb);
    uint32_t* flags = (uint32_t*)(p + 3 * qb + 2 * gb + pb);
    char* pre = p + 3 * qb + 2 * gb + pb + fb;
    int rc = gdn_prepare(qkv, conv_w, a_raw, b_raw, A_log, dt_bias, cu_seqlens, conv_state_in,
                         conv_state_out, q, k, v, alpha, beta, batch, seqlen, heads, kDK, dv,
                         GDN_BF16, stream_);
    cudaError_t e = cudaSuccess;
    if (rc == GDN_OK && fb) e = cudaMemsetAsync(flags, 0, fb, stream);
    if (rc == GDN_OK && e == cudaSuccess) {
      PrefillLaunch a{};
      a.q = q;
      a.k = k;
      a.v = v;
      a.alpha = alpha;
      a.beta = beta;
      a.S0 = S0;
      a.out = y;
      a.S_final = S_final;
      a.H = heads;
      a.dv = dv;
      a.status = status;
      a.map.cu_seqlens = cu_seqlens;
      a.map.N = batch;
      a.map.T = varlen ? T_total : seqlen;
      a.map.chunks_per_seq = varlen ? 0 : (seqlen + kC - 1) / kC;
      a.max_chunks = max_chunks;
      a.allow_overlap = true;
      a.ng.gate = (const __nv_bfloat16*)gate;
      a.ng.w = norm_w;
      a.ng.eps = eps;
      a.ng.act = act;
      a.ng.part = part;
      a.ng.flags = flags;
      e = launch_prefill_any(a, GDN_BF16, seqlen, 0, pre, stream);
    }
    const cudaError_t ef = scratch_free(scratch, stream);
    if (rc != GDN_OK) return rc;
    return (e == cudaSuccess && ef == cudaSuccess) ? GDN_OK : GDN_ERR_CUDA;
  }

  const size_t kb = k_out_bytes(T_total, heads);
  const size_t pb = align_up((size_t)T_total * heads * 8, 1024);   // the norm's partial sums
  const size_t need =
      kb + pb + prefill_scratch_bytes(batch, seqlen, heads, dv, GDN_BF16, varlen, 0);
  void* scratch = nullptr;
  if (scratch_alloc(&scratch, need, stream) != cudaSuccess) return GDN_ERR_CUDA;

  PrefillLaunch a{};
  a.S0 = S0;
  a.out = y;
  a.S_final = S_final;
  a.H = heads;
  a.dv = dv;
  a.status = status;
  a.map.cu_seqlens = cu_seqlens;
  a.map.N = batch;
  a.map.T = varlen ? T_total : seqlen;
  a.map.chunks_per_seq = varlen ? 0 : (seqlen + kC - 1) / kC;
  a.max_chunks = max_chunks_bound(batch, T_total, varlen, seqlen);
  a.allow_overlap = false;
  a.ng.gate = (const __nv_bfloat16*)gate;
  a.ng.w = norm_w;
  a.ng.eps = eps;
  a.ng.act = act;
  a.ng.part = (float*)((char*)scratch + kb);
  a.cv.qkv = (const __nv_bfloat16*)qkv;
  a.cv.conv_w = conv_w;
  a.cv.state_in = (const __nv_bfloat16*)conv_state_in;
  a.cv.state_out = (__nv_bfloat16*)conv_state_out;
  a.cv.a_raw = a_raw;
  a.cv.b_raw = b_raw;
  a.cv.A_log = A_log;
  a.cv.dt_bias = dt_bias;
  a.cv.k_out = (__nv_bfloat16*)scratch;
  cudaError_t e = launch_prefill_any(a, GDN_BF16, seqlen, 0, (char*)scratch + kb + pb, stream);
  if (e == cudaSuccess && conv_state_out && (varlen || seqlen == 0)) {
    empty_state_kernel<<<(unsigned)std::min<int64_t>(((int64_t)batch * 3 * C / 8 + 255) / 256, 4096),
                         256, 0, stream>>>(cu_seqlens, batch, C,
                                           (const __nv_bfloat16*)conv_state_in,
                                           (__nv_bfloat16*)conv_state_out);
    count_launches(1);
    e = cudaGetLastError();
  }
  const cudaError_t ef = scratch_free(scratch, stream);
  return (e == cudaSuccess && ef == cudaSuccess) ? GDN_OK : GDN_ERR_CUDA;
}
