// gdn_prefill_scan -- prefill of long sequences as a scan over segments.
//
// Over the chunks of one sequence the state pass is affine in its start state:
// S_end = S_start A_seg + B_seg, where B_seg is the end state from a zero start
// and A_seg (dk x dk) is the product of the segment's per-token transitions
// alpha_t (I - beta_t k_t k_t^T) (the recurrence of "Long-Context Aware
// Upcycling", Appendix A.3, Eq. 16-18).  A sequence cut into P segments
// therefore runs as P independent chains joined by one sequential scan over the
// segments' (A, B) pairs:
//   1. per-chunk prep over the segmented packing, then the state pass with the
//      caller's S0 as the first segment's start and zero for the others -> B
//      (for the first segment, its true end state);
//   2. the state pass again, on the same per-chunk images, from S0 = [I; 0]
//      (identity in the first dk rows) -> F, and by linearity A = F - B over
//      those rows;
//   3. the scan: start(1) = B(0); start(j) = start(j-1) A(j-1) + B(j-1);
//   4. the state pass from the true starts -> every output and the end state.
// Three state passes over P-times-shorter chains replace one long chain, which
// pays when a batch has few (sequence, head) units and long sequences: the
// sequential chain, not arithmetic, bounds the prefill there.
#include "gdn_internal.cuh"

namespace gdn {

cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t stream);
cudaError_t scratch_free(void* p, cudaStream_t stream);

namespace {

constexpr int kScanRows = 16;     // state rows per scan CTA
constexpr int kScanSlab = 16;     // rows of A staged at a time

// cu_seqlens of the segmented packing of a dense [B, T] batch: segment j of
// sequence b covers tokens [b T + j L, b T + min((j + 1) L, T)).
__global__ void seg_cu_kernel(int32_t* cu, int32_t B, int64_t T, int64_t seg_len, int32_t P) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t n = (int64_t)B * P;
  if (i > n) return;
  const int64_t b = i / P, j = i % P;
  cu[i] = (int32_t)(i == n ? (int64_t)B * T : b * T + min(j * seg_len, T));
}

// starts of pass 1 (the caller's S0 for each first segment, zero otherwise)
// and of pass 2 ([I; 0] everywhere)
__global__ void seg_init_kernel(float* __restrict__ S0seg, float* __restrict__ Iseg,
                                const float* __restrict__ S0, int32_t P, int32_t H, int32_t dv,
                                int64_t total) {
  const int64_t st = (int64_t)dv * kDK;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t s = e / (H * st), rem = e % (H * st);
    const int64_t in_state = rem % st;
    const int64_t row = in_state / kDK, col = in_state % kDK;
    S0seg[e] = (s % P == 0 && S0) ? S0[(s / P) * H * st + rem] : 0.f;
    Iseg[e] = row == col ? 1.f : 0.f;
  }
}

// The scan, one CTA per (16 rows of the state, head, sequence): rows of S are
// independent under right-multiplication by A, so each CTA walks the segments
// on its own.  Thread c owns column c.
__global__ void __launch_bounds__(256) seg_scan_kernel(float* __restrict__ S0seg,
                                                       const float* __restrict__ Bseg,
                                                       const float* __restrict__ Fseg, int32_t H,
                                                       int32_t dv, int32_t P) {
  __shared__ float prev[kScanRows][kDK];
  __shared__ float slab[kScanSlab][kDK];
  const int r0 = blockIdx.x * kScanRows, h = blockIdx.y, b = blockIdx.z, c = threadIdx.x;
  const int64_t st = (int64_t)dv * kDK;
  auto at = [&](const float* base, int j) { return base + ((int64_t)(b * P + j) * H + h) * st; };
  // start(1) = B(0): the first segment started from the caller's S0
#pragma unroll
  for (int r = 0; r < kScanRows; ++r) {
    const float x = at(Bseg, 0)[(r0 + r) * kDK + c];
    prev[r][c] = x;
    S0seg[((int64_t)(b * P + 1) * H + h) * st + (r0 + r) * kDK + c] = x;
  }
  for (int j = 2; j < P; ++j) {
    const float* Bj = at(Bseg, j - 1);
    const float* Fj = at(Fseg, j - 1);
    float acc[kScanRows];
#pragma unroll
    for (int r = 0; r < kScanRows; ++r) acc[r] = Bj[(r0 + r) * kDK + c];
    for (int k0 = 0; k0 < kDK; k0 += kScanSlab) {
      __syncthreads();
      for (int e = c; e < kScanSlab * kDK; e += blockDim.x) {
        const int64_t g = (int64_t)(k0 + e / kDK) * kDK + e % kDK;
        slab[e / kDK][e % kDK] = Fj[g] - Bj[g];        // A = F - B (first dk rows)
      }
      __syncthreads();
#pragma unroll 4
      for (int kk = 0; kk < kScanSlab; ++kk) {
        const float a = slab[kk][c];
#pragma unroll
        for (int r = 0; r < kScanRows; ++r) acc[r] = fmaf(prev[r][k0 + kk], a, acc[r]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kScanRows; ++r) {
      prev[r][c] = acc[r];
      S0seg[((int64_t)(b * P + j) * H + h) * st + (r0 + r) * kDK + c] = acc[r];
    }
  }
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace gdn

using namespace gdn;

namespace gdn {
namespace {

// Segmentation of a dense batch of B sequences of T tokens into P pieces of
// whole chunks (P = 1: nothing to split).
struct ScanPlan {
  int64_t seg_len = 0;   // tokens per segment (a multiple of the chunk)
  int32_t P = 1;
  int64_t max_chunks = 0;
  size_t cu_bytes = 0, tc_bytes = 0, ss = 0;
  size_t bytes() const { return P > 1 ? 2 * cu_bytes + tc_bytes + 5 * ss : 0; }
};

ScanPlan plan_scan(int32_t batch, int64_t seqlen, int32_t heads, int32_t dv, int32_t segments) {
  ScanPlan sp;
  const int64_t chunks = (seqlen + kC - 1) / kC;
  const int64_t seg_chunks = (chunks + segments - 1) / segments;
  sp.seg_len = seg_chunks * kC;
  const int64_t P64 = sp.seg_len > 0 ? (seqlen + sp.seg_len - 1) / sp.seg_len : 1;
  sp.P = P64 > 1 && P64 < 0x7fffffffLL ? (int32_t)P64 : 1;
  if (sp.P <= 1) return sp;
  const int64_t n_seg = (int64_t)batch * sp.P;
  const int64_t T_total = (int64_t)batch * seqlen;
  sp.max_chunks = max_chunks_bound((int32_t)n_seg, T_total, true, 0);
  // segmented cu_seqlens and chunk offsets, the per-chunk images, and five
  // per-(segment, head) states: starts of passes 1 and 2, B, F, ends
  sp.cu_bytes = align_up((size_t)(n_seg + 1) * 4, 1024);
  sp.tc_bytes = align_up(prefill_tc_scratch_bytes(sp.max_chunks, heads, dv), 1024);
  sp.ss = align_up((size_t)n_seg * heads * dv * kDK * 4, 1024);
  return sp;
}

int scan_common(const void* q, const void* k, const void* v, const float* alpha,
                const float* beta, const float* S0, void* out, float* S_final, int32_t batch,
                int64_t seqlen, int32_t heads, int32_t dk, int32_t dv, int32_t segments,
                cudaStream_t stream, bool use_ws, void* ws, size_t ws_bytes) {
  if (batch < 1 || seqlen < 0 || heads < 1 || segments < 1) return GDN_ERR_INVALID_ARG;
  if (dk != kDK || !supported_dv(dv)) return GDN_ERR_UNSUPPORTED;
  const ScanPlan sp = plan_scan(batch, seqlen, heads, dv, segments);
  if (sp.P <= 1)   // nothing to split: the plain prefill
    return use_ws ? gdn_prefill_ws(q, k, v, alpha, beta, S0, nullptr, out, S_final, batch, seqlen,
                                   heads, dk, dv, GDN_BF16, ws, ws_bytes, (gdn_stream_t)stream)
                  : gdn_prefill(q, k, v, alpha, beta, S0, nullptr, out, S_final, batch, seqlen,
                                heads, dk, dv, GDN_BF16, (gdn_stream_t)stream);
  const int32_t P = sp.P;
  const int64_t T_total = (int64_t)batch * seqlen;
  const int64_t n_seg = (int64_t)batch * P;
  if (T_total > 0x7fffffffLL || n_seg * heads > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  if (!q || !k || !v || !alpha || !beta || !out) return GDN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(S0) ||
      !aligned16(S_final) || ((uintptr_t)alpha & 3u) || ((uintptr_t)beta & 3u))
    return GDN_ERR_ALIGNMENT;
  if (batch > 65535) return GDN_ERR_UNSUPPORTED;   // the scan's grid
  // out and S_final may overlap no input and not each other
  const size_t nth = (size_t)T_total * heads;
  const size_t state_bytes = (size_t)batch * heads * dv * dk * 4;
  struct R { uintptr_t lo, hi; };
  auto span = [](const void* p, size_t n) { return R{(uintptr_t)p, (uintptr_t)p + (p ? n : 0)}; };
  auto ov = [](R a, R b) { return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi; };
  const R ins[] = {span(q, nth * dk * 2), span(k, nth * dk * 2), span(v, nth * dv * 2),
                   span(alpha, nth * 4), span(beta, nth * 4), span(S0, state_bytes)};
  const R ro = span(out, nth * dv * 2), rs = span(S_final, state_bytes);
  for (const R& r : ins)
    if (ov(r, ro) || ov(r, rs)) return GDN_ERR_INVALID_ARG;
  if (ov(ro, rs)) return GDN_ERR_INVALID_ARG;
  const size_t need = sp.bytes();
  if (use_ws) {   // the caller's workspace: large enough, 1024-byte aligned, apart from the tensors
    if (!ws || ws_bytes < need) return GDN_ERR_INVALID_ARG;
    if ((uintptr_t)ws & 1023u) return GDN_ERR_ALIGNMENT;
    const R w = span(ws, need);
    for (const R& r : ins)
      if (ov(w, r)) return GDN_ERR_INVALID_ARG;
    if (ov(w, ro) || ov(w, rs)) return GDN_ERR_INVALID_ARG;
  }

  unsigned* status = status_ptr();
  if (!status) return GDN_ERR_CUDA;
  PrefillLaunch a{};
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.H = heads; a.dv = dv;
  a.status = status; a.out = out;
  a.map.N = (int32_t)n_seg;
  a.map.T = T_total;
  a.max_chunks = sp.max_chunks;
  a.allow_overlap = false;   // prep on every SM first: the state passes need most of them

  void* scratch = use_ws ? ws : nullptr;
  if (!use_ws && scratch_alloc(&scratch, need, stream) != cudaSuccess) return GDN_ERR_CUDA;
  char* p = (char*)scratch;
  int32_t* seg_cu = (int32_t*)p; p += sp.cu_bytes;
  int32_t* chunk_off = (int32_t*)p; p += sp.cu_bytes;
  a.scratch = p; p += sp.tc_bytes;
  float* S0seg = (float*)p; p += sp.ss;
  float* Iseg = (float*)p; p += sp.ss;
  float* Bseg = (float*)p; p += sp.ss;
  float* Fseg = (float*)p; p += sp.ss;
  float* Eseg = (float*)p;
  a.map.cu_seqlens = seg_cu;
  a.map.chunk_off = chunk_off;
  cudaError_t e = cudaSuccess;
  seg_cu_kernel<<<(unsigned)((n_seg + 1 + 255) / 256), 256, 0, stream>>>(seg_cu, batch, seqlen,
                                                                          sp.seg_len, P);
  count_launches(1);
  if ((e = cudaGetLastError()) == cudaSuccess)
    e = launch_chunk_offsets(seg_cu, (int32_t)n_seg, T_total, chunk_off, status, stream);
  if (e == cudaSuccess) {
    const int64_t total = (int64_t)n_seg * heads * dv * dk;
    seg_init_kernel<<<1216, 256, 0, stream>>>(S0seg, Iseg, S0, P, heads, dv, total);
    count_launches(1);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {   // 1. prep, then the chains from (S0 | 0) -> B
    a.S0 = S0seg; a.S_final = Bseg; a.state_only = false;
    e = launch_prefill_tc(a, stream);
  }
  if (e == cudaSuccess) {   // 2. the chains from [I; 0] on the same images -> F = A + B
    a.S0 = Iseg; a.S_final = Fseg; a.state_only = true;
    e = launch_prefill_tc(a, stream);
  }
  if (e == cudaSuccess) {   // 3. the scan writes every segment's true start
    seg_scan_kernel<<<dim3((unsigned)(dv / kScanRows), (unsigned)heads, (unsigned)batch), 256, 0,
                      stream>>>(S0seg, Bseg, Fseg, heads, dv, P);
    count_launches(1);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {   // 4. the chains from the true starts -> out and the end states
    a.S0 = S0seg; a.S_final = Eseg; a.state_only = true;
    e = launch_prefill_tc(a, stream);
  }
  if (e == cudaSuccess && S_final) {
    const size_t one = (size_t)heads * dv * dk;
    for (int32_t b = 0; b < batch && e == cudaSuccess; ++b)
      e = cudaMemcpyAsync(S_final + b * one, Eseg + ((size_t)b * P + P - 1) * one, one * 4,
                          cudaMemcpyDeviceToDevice, stream);
  }
  const cudaError_t ef = use_ws ? cudaSuccess : scratch_free(scratch, stream);
  return (e == cudaSuccess && ef == cudaSuccess) ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_prefill_scan(const void* q, const void* k, const void* v, const float* alpha,
                                const float* beta, const float* S0, void* out, float* S_final,
                                int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                                int32_t dv, int32_t segments, gdn_stream_t stream) {
  return scan_common(q, k, v, alpha, beta, S0, out, S_final, batch, seqlen, heads, dk, dv,
                     segments, (cudaStream_t)stream, false, nullptr, 0);
}

extern "C" size_t gdn_prefill_scan_workspace_size(int32_t batch, int64_t seqlen, int32_t heads,
                                                  int32_t dk, int32_t dv, int32_t segments) {
  if (batch < 1 || seqlen < 0 || heads < 1 || segments < 1 || dk != kDK || !supported_dv(dv))
    return SIZE_MAX;
  const ScanPlan sp = plan_scan(batch, seqlen, heads, dv, segments);
  if (sp.P <= 1) return gdn_prefill_workspace_size(batch, seqlen, heads, dk, dv, GDN_BF16, 0);
  return sp.bytes();
}

extern "C" int gdn_prefill_scan_ws(const void* q, const void* k, const void* v,
                                   const float* alpha, const float* beta, const float* S0,
                                   void* out, float* S_final, int32_t batch, int64_t seqlen,
                                   int32_t heads, int32_t dk, int32_t dv, int32_t segments,
                                   void* workspace, size_t workspace_bytes, gdn_stream_t stream) {
  return scan_common(q, k, v, alpha, beta, S0, out, S_final, batch, seqlen, heads, dk, dv,
                     segments, (cudaStream_t)stream, true, workspace, workspace_bytes);
}
